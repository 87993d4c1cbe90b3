// Body of one launcher translation unit.  The including file defines
// GEMM_OUT_KIND; GEMM_LAUNCH_NAME (the general instances) unless GEMM_SPEC_ONLY
// is set; GEMM_LAUNCH_SPEC_NAME for the specialised instances it holds, of set
// GEMM_SPEC_SET (see spec_set; 0 = all sets); and GEMM_F8 (8-bit operands) when
// it is set.
#ifndef GEMM_F8
#define GEMM_F8 false
#endif
#ifndef GEMM_SPEC_SET
#define GEMM_SPEC_SET 0
#endif
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gemm_tc {

namespace {
constexpr int kMaxDevices = 64;

template <int BN, bool PAIR, int SPLIT, int SPEC = 0>
cudaError_t launch_inst(const OperandMaps& m, const KernelArgs& args, int grid,
                        cudaStream_t stream, int dev) {
  constexpr int ST = stages_for(BN, PAIR);
  constexpr int KO = ko_for(BN, PAIR);
  using L = SmemLayout<BN, ST, PAIR, KO>;
  auto kern = gemm_tcgen05_kernel<BN, ST, GEMM_OUT_KIND, PAIR, SPLIT, KO, GEMM_F8, SPEC>;
  static volatile bool attr_set[kMaxDevices] = {};
  static volatile int max_clusters[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = stream;
  if (SPLIT > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = SPLIT;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (grid % SPLIT != 0) return cudaErrorInvalidConfiguration;
  } else if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters[dev] == 0) {
      cfg.gridDim = dim3(2, 1, 1);
      int n = 0;
      cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_clusters[dev] = n;
    }
    if (grid > 2 * max_clusters[dev]) grid = 2 * max_clusters[dev];
    grid &= ~1;
    if (grid < 2) return cudaErrorInvalidConfiguration;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, m.a, m.b, m.a3, m.b3, m.c, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

#ifdef GEMM_LAUNCH_SPEC_NAME
namespace {
// The specialised instances of one layout in this unit's set (see spec_set).
template <int LAYOUT>
cudaError_t launch_spec_layout(int bn, bool pair, int split, bool sk, bool readc, bool epi,
                               bool ragged, const OperandMaps& m, const KernelArgs& args, int grid,
                               cudaStream_t stream, int dev) {
  constexpr int S = spec_bits(LAYOUT, false, false);
#if GEMM_SPEC_SET == 0 || GEMM_SPEC_SET == 3
  if (ragged) {
    constexpr int R = spec_bits(LAYOUT, false, false, false, true);
    if (!pair && split == 1 && bn == 64) return launch_inst<64, false, 1, R>(m, args, grid, stream, dev);
    if (!pair && split == 1 && bn == 128) return launch_inst<128, false, 1, R>(m, args, grid, stream, dev);
    return cudaErrorNotSupported;
  }
#else
  if (ragged) return cudaErrorNotSupported;
#endif
#if GEMM_SPEC_SET == 0 || GEMM_SPEC_SET == 4
  if (epi && !pair) {
    constexpr int E = spec_bits(LAYOUT, false, false, true);
    if (split == 1 && bn == 64) return launch_inst<64, false, 1, E>(m, args, grid, stream, dev);
    if (split == 1 && bn == 128) return launch_inst<128, false, 1, E>(m, args, grid, stream, dev);
    if (split == 2 && bn == 64) return launch_inst<64, false, 2, E>(m, args, grid, stream, dev);
    if (split == 2 && bn == 128) return launch_inst<128, false, 2, E>(m, args, grid, stream, dev);
    return cudaErrorNotSupported;
  }
#else
  if (epi && !pair) return cudaErrorNotSupported;
#endif
#if GEMM_SPEC_SET == 0 || GEMM_SPEC_SET == 1
  if (pair && !epi) {
    if (sk) return launch_inst<256, true, 1, spec_bits(LAYOUT, true, false)>(m, args, grid, stream, dev);
    if (readc) return launch_inst<256, true, 1, spec_bits(LAYOUT, false, true)>(m, args, grid, stream, dev);
    return launch_inst<256, true, 1, S>(m, args, grid, stream, dev);
  }
  if (split == 2 && bn == 128) return launch_inst<128, false, 2, S>(m, args, grid, stream, dev);
  if (split == 2 && bn == 64) return launch_inst<64, false, 2, S>(m, args, grid, stream, dev);
  if (split == 1 && bn == 64) return launch_inst<64, false, 1, S>(m, args, grid, stream, dev);
#endif
#if GEMM_SPEC_SET == 0 || GEMM_SPEC_SET == 2
  if (pair) {
    if (!epi)   // stream-K reading C
      return launch_inst<256, true, 1, spec_bits(LAYOUT, true, true)>(m, args, grid, stream, dev);
    constexpr int E = spec_bits(LAYOUT, false, false, true);
    if (sk) return launch_inst<256, true, 1, spec_bits(LAYOUT, true, false, true)>(m, args, grid, stream, dev);
    return launch_inst<256, true, 1, E>(m, args, grid, stream, dev);
  }
  if (split == 1 && bn == 128) return launch_inst<128, false, 1, S>(m, args, grid, stream, dev);
  if (split == 4 && bn == 128) return launch_inst<128, false, 4, S>(m, args, grid, stream, dev);
  if (split == 4 && bn == 64) return launch_inst<64, false, 4, S>(m, args, grid, stream, dev);
  if (split == 2 && bn == 256) return launch_inst<256, false, 2, S>(m, args, grid, stream, dev);
  if (split == 8 && bn == 128) return launch_inst<128, false, 8, S>(m, args, grid, stream, dev);
#endif
  return cudaErrorNotSupported;
}
}  // namespace

cudaError_t GEMM_LAUNCH_SPEC_NAME(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m,
                                  const KernelArgs& args, int grid, cudaStream_t stream, int dev) {
  if (!spec_supported(bn, pair, split, layout, GEMM_F8, sk, readc, epi, ragged))
    return cudaErrorNotSupported;
  if (GEMM_SPEC_SET != 0 && spec_set(bn, pair, split, sk, readc, epi, ragged) != GEMM_SPEC_SET)
    return cudaErrorNotSupported;
  if constexpr (GEMM_F8) {   // 8-bit operands are K-major only
    return launch_spec_layout<2>(bn, pair, split, sk, readc, epi, ragged, m, args, grid, stream, dev);
  } else {
    switch (layout) {
      case 0: return launch_spec_layout<0>(bn, pair, split, sk, readc, epi, ragged, m, args, grid, stream, dev);
      case 1: return launch_spec_layout<1>(bn, pair, split, sk, readc, epi, ragged, m, args, grid, stream, dev);
      case 2: return launch_spec_layout<2>(bn, pair, split, sk, readc, epi, ragged, m, args, grid, stream, dev);
      case 3: return launch_spec_layout<3>(bn, pair, split, sk, readc, epi, ragged, m, args, grid, stream, dev);
      default: return cudaErrorNotSupported;
    }
  }
}
#endif

#ifndef GEMM_SPEC_ONLY
cudaError_t GEMM_LAUNCH_NAME(int bn, bool pair, int split, const OperandMaps& m,
                             const KernelArgs& args, int grid, cudaStream_t stream, int dev) {
  if (split > 1) {
    if (pair) return cudaErrorInvalidValue;
    if (bn == 256 && split == 2) return launch_inst<256, false, 2>(m, args, grid, stream, dev);
    if (bn == 256 && split == 4) return launch_inst<256, false, 4>(m, args, grid, stream, dev);
    if (bn == 128 && split == 2) return launch_inst<128, false, 2>(m, args, grid, stream, dev);
    if (bn == 128 && split == 4) return launch_inst<128, false, 4>(m, args, grid, stream, dev);
    if (bn == 128 && split == 8) return launch_inst<128, false, 8>(m, args, grid, stream, dev);
    if (bn == 64 && split == 2) return launch_inst<64, false, 2>(m, args, grid, stream, dev);
    if (bn == 64 && split == 4) return launch_inst<64, false, 4>(m, args, grid, stream, dev);
    return cudaErrorInvalidValue;
  }
  if (pair) {
    switch (bn) {
      case 128: return launch_inst<128, true, 1>(m, args, grid, stream, dev);
      case 256: return launch_inst<256, true, 1>(m, args, grid, stream, dev);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 64: return launch_inst<64, false, 1>(m, args, grid, stream, dev);
    case 128: return launch_inst<128, false, 1>(m, args, grid, stream, dev);
    case 256: return launch_inst<256, false, 1>(m, args, grid, stream, dev);
    default: return cudaErrorInvalidValue;
  }
}
#endif

}  // namespace gemm_tc
