// Launchers of the tcgen05 GEMM kernel instances, one translation unit per
// output format (compiled in parallel).  Host-only declarations.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace gemm_tc {

// B columns one CTA holds: the whole tile width, or half of it in pair mode.
constexpr int b_cols_per_cta(int bn, bool pair) { return pair ? bn / 2 : bn; }

// k-blocks per ring stage: two, so that each operand copy reads at least 256
// contiguous bytes of every row it touches (GB300's DRAM delivers ~3.7 TB/s to
// 128-byte row pieces and ~5.3 TB/s to 256-byte ones, measured with a TMA
// streaming probe).
constexpr int ko_for(int /*bn*/, bool /*pair*/) { return 2; }

// Pipeline depth: as many stages as fit in 192 KB of shared memory (the rest
// holds the epilogue staging buffers and barriers).
constexpr int stages_for(int bn, bool pair) {
  return (192 * 1024) / (ko_for(bn, pair) * (BM * BK * 2 + b_cols_per_cta(bn, pair) * BK * 2));
}

// Dynamic shared memory bytes of an instance (layout + alignment slack).
int smem_alloc_bytes(int bn, bool pair);

// Launch the instance (tile width bn; single CTA, CTA pair, or a split-K
// cluster of `split` CTAs).  `grid` is the number of CTAs (a multiple of the
// cluster size).  Pair launches are capped at the number of co-resident 2-CTA
// clusters (the pair kernel is persistent); split-K launches run exactly one
// tile per cluster.  `dev` indexes the per-device attribute cache.
// The operand maps: 2-D (one k-block or one atom per copy, exact bounds) and
// 3-D (several whole 64-element blocks per copy), plus the C map.
struct OperandMaps {
  CUtensorMap a, b, a3, b3, c;
};

cudaError_t launch_gemm_f32(int bn, bool pair, int split, const OperandMaps& m,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_bf16(int bn, bool pair, int split, const OperandMaps& m,
                             const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f16(int bn, bool pair, int split, const OperandMaps& m,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_f32(int bn, bool pair, int split, const OperandMaps& m,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_bf16(int bn, bool pair, int split, const OperandMaps& m,
                             const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_f16(int bn, bool pair, int split, const OperandMaps& m,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);

// Configurations with specialised instances (plain path, fixed layout; see
// specialise_args), by the set of translation units that holds them (0: none):
// set 1, the 256-wide CTA pair (with a stream-K tail, sk, or with a C read,
// readc, or neither), the 2-way split-K clusters of width 128 and 64 and the
// single 64-wide CTA; set 2, the CTA pair with the fused epilogue (epi; with or
// without a stream-K tail) or with both a stream-K tail and a C read, and the
// other single-panel choices (the single
// 128-wide CTA, 4-way clusters of width 64 and 128, 8-way clusters of width 128,
// 2-way clusters of width 256); set 3, the single CTA of width 64 or 128 when N times the output size is
// not a multiple of 16 bytes (the ragged right edge, stored element by element,
// stays a run-time choice): small and odd shapes, where the general kernel's
// larger code costs microseconds of instruction fetches; set 4, the fused
// epilogue (bias and/or activation, their kinds chosen at run time) on the single
// CTA and the 2-way split-K cluster of width 64 or 128.  8-bit operands keep
// every set in their own units.
constexpr int spec_set(int bn, bool pair, int split, bool sk, bool readc, bool epi,
                       bool ragged = false) {
  if (ragged)
    return (!pair && split == 1 && (bn == 64 || bn == 128) && !sk && !readc && !epi) ? 3 : 0;
  if (epi && !pair)
    return (!sk && !readc && (split == 1 || split == 2) && (bn == 64 || bn == 128)) ? 4 : 0;
  if (pair) {
    if (bn != 256 || split != 1) return 0;
    if (epi) return readc ? 0 : 2;
    return (sk && readc) ? 2 : 1;
  }
  if (sk || readc || epi) return 0;
  if ((split == 2 && (bn == 128 || bn == 64)) || (split == 1 && bn == 64)) return 1;
  if ((split == 1 && bn == 128) || (split == 4 && (bn == 128 || bn == 64)) ||
      (split == 2 && bn == 256) || (split == 8 && bn == 128))
    return 2;
  return 0;
}

// Every layout has them (8-bit operands: A row-major with B column-major only).
constexpr bool spec_supported(int bn, bool pair, int split, int layout, bool fp8, bool sk,
                              bool readc, bool epi, bool ragged = false) {
  if (layout < 0 || layout > 3 || (fp8 && layout != 2)) return false;
  return spec_set(bn, pair, split, sk, readc, epi, ragged) != 0;
}

// Launch the specialised instance of (bn, pair, split, layout, sk, readc, epi, ragged), or return
// cudaErrorNotSupported when spec_supported() says there is none.  Only for
// calls on the plain path.
cudaError_t launch_gemm_spec_f32(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                 bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                 int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec_bf16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                  int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec_f16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                 bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                 int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec2_f32(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                  int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec2_bf16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                   bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                   int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec2_f16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                  int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec3_f32(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m,
                                  const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec3_bf16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                   bool epi, bool ragged, const OperandMaps& m,
                                   const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec3_f16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m,
                                  const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec4_f32(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m,
                                  const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec4_bf16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                   bool epi, bool ragged, const OperandMaps& m,
                                   const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_spec4_f16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                  bool epi, bool ragged, const OperandMaps& m,
                                  const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_spec_f32(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                    bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                    int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_spec_bf16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                     bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                     int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f8_spec_f16(int bn, bool pair, int split, int layout, bool sk, bool readc,
                                    bool epi, bool ragged, const OperandMaps& m, const KernelArgs& args,
                                    int grid, cudaStream_t stream, int dev);

// Split-K cluster shapes that have kernel instances: (bn, split).
constexpr bool split_supported(int bn, int split) {
  return (bn == 256 && (split == 2 || split == 4)) ||
         (bn == 128 && (split == 2 || split == 4 || split == 8)) ||
         (bn == 64 && (split == 2 || split == 4));
}

}  // namespace gemm_tc
