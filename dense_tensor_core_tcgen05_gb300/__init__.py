"""Dense GEMM for NVIDIA GB300 (sm_103a): C <- alpha*A*B + beta*C.

fp16/bf16 inputs, fp32 accumulation in Tensor Memory (tcgen05), fp32/bf16/fp16
output, behind the C ABI of include/gemm_tcgen05.h.  This package is the thin
Python binding of that library.  The binding is loaded on first use of any of
its names and raises ImportError if the CUDA library has not been built
(``dense_tensor_core_tcgen05_gb300.build.build()``); there is no CPU fallback.
"""
import importlib

_BINDING_NAMES = frozenset((
    "EXPORTS", "GEMM_A_COL", "GEMM_A_ROW", "GEMM_ACT_NONE", "GEMM_ACT_RELU", "GEMM_B_COL",
    "GEMM_B_ROW", "GEMM_BF16", "GEMM_BIAS_COL", "GEMM_BIAS_NONE", "GEMM_BIAS_ROW",
    "GEMM_E4M3", "GEMM_E5M2",
    "GEMM_ERR_ARCH", "GEMM_ERR_CUDA", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_SCRATCH",
    "GEMM_ERR_TIMEOUT", "GEMM_ERR_UNSUPPORTED", "GEMM_F16", "GEMM_F32",
    "GEMM_NOALLOC_SCRATCH_BYTES", "GEMM_OK", "GEMM_ORDER_AUTO", "GEMM_ORDER_GROUPED",
    "GEMM_ORDER_HILBERT", "LIB_PATH", "GemmError",
    "gemm", "gemm_config_t", "gemm_debug_set", "gemm_encode_idesc", "gemm_encode_sdesc",
    "gemm_bias_act", "gemm_ex", "gemm_ex_noalloc", "gemm_host", "gemm_plan", "gemm_plan_t", "gemm_split_tile_item", "gemm_fastdiv",
    "gemm_sync_status",
    "gemm_tile_coord", "gemm_tile_order", "gemm_version", "gemm_work_items", "library", "matmul", "status_string"))


def __getattr__(name):
    if name in _BINDING_NAMES:
        binding = importlib.import_module(".binding", __name__)
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def __dir__():
    return sorted(set(globals()) | _BINDING_NAMES)
