// tcgen05 GEMM kernel instances with 8-bit (E4M3 / E5M2) operands and f32 output.
#define GEMM_OUT_KIND OUT_F32
#define GEMM_F8 true
#define GEMM_LAUNCH_NAME launch_gemm_f8_f32
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_f8_spec_f32
#include "gemm_launch_impl.cuh"
