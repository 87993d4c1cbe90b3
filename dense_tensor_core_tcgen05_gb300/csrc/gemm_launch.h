// Launchers of the tcgen05 GEMM kernel instances, one translation unit per
// output format (compiled in parallel).  Host-only declarations.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace gemm_tc {

// Pipeline depth for a tile width: as many ring slots as fit in 192 KB of
// shared memory (the rest holds the epilogue staging buffers and barriers).
constexpr int stages_for_bn(int bn) { return (192 * 1024) / (BM * BK * 2 + bn * BK * 2); }

// Dynamic shared memory bytes of an instance (layout + alignment slack).
int smem_alloc_bytes(int bn);

// Launch the instance for tile width `bn` (64, 128 or 256).  `dev` indexes the
// per-device "attribute already set" cache.  Returns the launch status.
cudaError_t launch_gemm_f32(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_bf16(int bn, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& c, const KernelArgs& args, int grid,
                             cudaStream_t stream, int dev);
cudaError_t launch_gemm_f16(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                            const KernelArgs& args, int grid, cudaStream_t stream, int dev);

}  // namespace gemm_tc
