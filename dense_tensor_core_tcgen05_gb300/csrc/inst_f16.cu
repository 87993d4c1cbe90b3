// tcgen05 GEMM kernel instances with f16 output.
#define GEMM_OUT_KIND OUT_F16
#define GEMM_LAUNCH_NAME launch_gemm_f16
#include "gemm_launch_impl.cuh"
