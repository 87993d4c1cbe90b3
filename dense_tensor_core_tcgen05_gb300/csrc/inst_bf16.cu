// tcgen05 GEMM kernel instances with bf16 output.
#define GEMM_OUT_KIND OUT_BF16
#define GEMM_LAUNCH_NAME launch_gemm_bf16
#include "gemm_launch_impl.cuh"
