// Specialised tcgen05 GEMM kernel instances (plain path, fixed operand layout)
// with f16 output: the second set (the other single-panel choices).
#define GEMM_OUT_KIND OUT_F16
#define GEMM_SPEC_ONLY
#define GEMM_SPEC_SET 2
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_spec2_f16
#include "gemm_launch_impl.cuh"
