// Specialised tcgen05 GEMM kernel instances (plain path, fixed operand layout)
// with bf16 output: the third set (single CTAs with a ragged right edge).
#define GEMM_OUT_KIND OUT_BF16
#define GEMM_SPEC_ONLY
#define GEMM_SPEC_SET 3
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_spec3_bf16
#include "gemm_launch_impl.cuh"
