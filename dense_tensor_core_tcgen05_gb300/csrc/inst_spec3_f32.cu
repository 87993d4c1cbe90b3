// Specialised tcgen05 GEMM kernel instances (plain path, fixed operand layout)
// with f32 output: the third set (single CTAs with a ragged right edge).
#define GEMM_OUT_KIND OUT_F32
#define GEMM_SPEC_ONLY
#define GEMM_SPEC_SET 3
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_spec3_f32
#include "gemm_launch_impl.cuh"
