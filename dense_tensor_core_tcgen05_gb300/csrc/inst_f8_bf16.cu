// tcgen05 GEMM kernel instances with 8-bit (E4M3 / E5M2) operands and bf16 output.
#define GEMM_OUT_KIND OUT_BF16
#define GEMM_F8 true
#define GEMM_LAUNCH_NAME launch_gemm_f8_bf16
#define GEMM_LAUNCH_SPEC_NAME launch_gemm_f8_spec_bf16
#include "gemm_launch_impl.cuh"
