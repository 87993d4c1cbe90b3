// Specialised tcgen05 GEMM kernel instances (plain path, fixed operand layout)
// with f32 output: the fourth set (the fused epilogue on single CTAs and 2-way
// split-K clusters).
#define GEMM_OUT_KIND OUT_F32
#define GEMM_SPEC_ONLY
#define GEMM_SPEC_SET 4
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_spec4_f32
#include "gemm_launch_impl.cuh"
