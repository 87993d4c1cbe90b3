// Body of one launcher translation unit; GEMM_OUT_KIND and GEMM_LAUNCH_NAME are
// defined by the including file.
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gemm_tc {

namespace {
constexpr int kMaxDevices = 64;

template <int BN>
cudaError_t launch_bn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                      const KernelArgs& args, int grid, cudaStream_t stream, int dev) {
  constexpr int ST = stages_for_bn(BN);
  using L = SmemLayout<BN, ST>;
  auto kern = gemm_tcgen05_kernel<BN, ST, GEMM_OUT_KIND>;
  static volatile bool attr_set[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<grid, NUM_THREADS, L::ALLOC, stream>>>(a, b, c, args);
  return cudaGetLastError();
}
}  // namespace

cudaError_t GEMM_LAUNCH_NAME(int bn, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& c, const KernelArgs& args, int grid,
                             cudaStream_t stream, int dev) {
  switch (bn) {
    case 64: return launch_bn<64>(a, b, c, args, grid, stream, dev);
    case 128: return launch_bn<128>(a, b, c, args, grid, stream, dev);
    case 256: return launch_bn<256>(a, b, c, args, grid, stream, dev);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gemm_tc
