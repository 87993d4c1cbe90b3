// Launchers of the tcgen05 GEMM kernel instances, one translation unit per
// output format (compiled in parallel).  Host-only declarations.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace gemm_tc {

// B columns one CTA holds: the whole tile width, or half of it in pair mode.
constexpr int b_cols_per_cta(int bn, bool pair) { return pair ? bn / 2 : bn; }

// Pipeline depth: as many ring slots as fit in 192 KB of shared memory (the rest
// holds the epilogue staging buffers and barriers).
constexpr int stages_for(int bn, bool pair) {
  return (192 * 1024) / (BM * BK * 2 + b_cols_per_cta(bn, pair) * BK * 2);
}

// Dynamic shared memory bytes of an instance (layout + alignment slack).
int smem_alloc_bytes(int bn, bool pair);

// Launch the instance (tile width bn; single CTA, CTA pair, or a split-K
// cluster of `split` CTAs).  `grid` is the number of CTAs (a multiple of the
// cluster size).  Pair launches are capped at the number of co-resident 2-CTA
// clusters (the pair kernel is persistent); split-K launches run exactly one
// tile per cluster.  `dev` indexes the per-device attribute cache.
cudaError_t launch_gemm_f32(int bn, bool pair, int split, const CUtensorMap& a,
                            const CUtensorMap& b, const CUtensorMap& c, const KernelArgs& args,
                            int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_bf16(int bn, bool pair, int split, const CUtensorMap& a,
                             const CUtensorMap& b, const CUtensorMap& c, const KernelArgs& args,
                             int grid, cudaStream_t stream, int dev);
cudaError_t launch_gemm_f16(int bn, bool pair, int split, const CUtensorMap& a,
                            const CUtensorMap& b, const CUtensorMap& c, const KernelArgs& args,
                            int grid, cudaStream_t stream, int dev);

// Split-K cluster shapes that have kernel instances: (bn, split).
constexpr bool split_supported(int bn, int split) {
  return (bn == 256 && (split == 2 || split == 4)) || (bn == 128 && split == 2);
}

}  // namespace gemm_tc
