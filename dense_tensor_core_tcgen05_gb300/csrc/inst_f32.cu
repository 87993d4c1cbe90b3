// tcgen05 GEMM kernel instances with f32 output.
#define GEMM_OUT_KIND OUT_F32
#define GEMM_LAUNCH_NAME launch_gemm_f32
#include "gemm_launch_impl.cuh"
