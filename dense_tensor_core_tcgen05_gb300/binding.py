"""ctypes binding of libgemm_tcgen05.so (the C ABI of include/gemm_tcgen05.h).

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  There is no fallback: if the shared library is missing, importing
this module raises.  PyTorch is used (by ``matmul``) only to hand over device
pointers and the current stream.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgemm_tcgen05.so")

GEMM_F16, GEMM_BF16, GEMM_F32, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4
GEMM_A_ROW, GEMM_A_COL, GEMM_B_ROW, GEMM_B_COL = 0, 1, 0, 2
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_ARCH, GEMM_ERR_CUDA, \
    GEMM_ERR_TIMEOUT, GEMM_ERR_SCRATCH = range(7)
GEMM_NOALLOC_SCRATCH_BYTES = 24 * 1024 * 1024
GEMM_BIAS_NONE, GEMM_BIAS_COL, GEMM_BIAS_ROW = 0, 1, 2
GEMM_ACT_NONE, GEMM_ACT_RELU = 0, 1
GEMM_ORDER_AUTO, GEMM_ORDER_GROUPED, GEMM_ORDER_HILBERT = 0, 1, 2

# Symbols declared in include/gemm_tcgen05.h.
EXPORTS = ("gemm", "gemm_bias_act", "gemm_ex", "gemm_ex_noalloc", "gemm_host", "gemm_status_string",
           "gemm_sync_status",
           "gemm_debug_set", "gemm_plan", "gemm_tile_coord", "gemm_tile_order", "gemm_work_items",
           "gemm_split_tile_item", "gemm_fastdiv",
           "gemm_encode_idesc", "gemm_encode_sdesc", "gemm_version")


class gemm_config_t(ctypes.Structure):
    _fields_ = [("bn", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("cta_group", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("stream_k", ctypes.c_int32),
                ("order", ctypes.c_int32), ("general", ctypes.c_int32)]


class gemm_plan_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "bm", "bn", "bk", "stages", "m_tiles", "n_tiles", "k_blocks", "num_tiles",
        "grid", "group_m", "threads", "smem_bytes", "tmem_cols", "a_mn", "b_mn",
        "epi_chunk_cols", "cta_group", "split_k", "groups", "dp_tiles", "order",
        "specialised")] + [
        ("sk_iters", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64),
        ("tile_split", ctypes.c_int32), ("owner_groups", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run dense_tensor_core_tcgen05_gb300.build.build() "
                          "(the GEMM has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    i64, f32, vp, ci, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_int32
    gemm_args = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, ci, ci, ci, vp]
    lib.gemm.argtypes = gemm_args
    lib.gemm.restype = ci
    lib.gemm_ex.argtypes = gemm_args + [ctypes.POINTER(gemm_config_t)]
    lib.gemm_ex.restype = ci
    lib.gemm_bias_act.argtypes = gemm_args[:-1] + [vp, ci, ci, vp, ctypes.POINTER(gemm_config_t)]
    lib.gemm_bias_act.restype = ci
    lib.gemm_ex_noalloc.argtypes = gemm_args + [ctypes.POINTER(gemm_config_t)]
    lib.gemm_ex_noalloc.restype = ci
    lib.gemm_host.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, ci, ci, ci,
                              vp, vp, vp, vp]
    lib.gemm_host.restype = ci
    lib.gemm_status_string.argtypes = [ci]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_sync_status.argtypes = [vp, ctypes.POINTER(ci)]
    lib.gemm_sync_status.restype = ci
    lib.gemm_debug_set.argtypes = [ctypes.c_uint64, i32]
    lib.gemm_debug_set.restype = None
    lib.gemm_plan.argtypes = [i64, i64, i64, ci, ci, ci, i32, ctypes.POINTER(gemm_config_t),
                              ctypes.POINTER(gemm_plan_t)]
    lib.gemm_plan.restype = ci
    lib.gemm_tile_coord.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.gemm_tile_coord.restype = None
    lib.gemm_tile_order.argtypes = [ci, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32), i32]
    lib.gemm_tile_order.restype = i32
    lib.gemm_work_items.argtypes = [i32, i32, i32, i64, i32, ctypes.POINTER(i32), i32]
    lib.gemm_work_items.restype = i32
    lib.gemm_fastdiv.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.gemm_fastdiv.restype = ctypes.c_uint32
    lib.gemm_split_tile_item.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32)]
    lib.gemm_split_tile_item.restype = i32
    lib.gemm_encode_idesc.argtypes = [ci, ci, ci, ci, ci]
    lib.gemm_encode_idesc.restype = ctypes.c_uint32
    lib.gemm_encode_sdesc.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
    lib.gemm_encode_sdesc.restype = ctypes.c_uint64
    lib.gemm_version.argtypes = []
    lib.gemm_version.restype = i32
    return lib


_lib = _load()


def library():
    """The loaded ctypes.CDLL."""
    return _lib


def status_string(status: int) -> str:
    return _lib.gemm_status_string(int(status)).decode()


def _cfg(cfg):
    if cfg is None:
        return None
    if isinstance(cfg, gemm_config_t):
        return ctypes.byref(cfg)
    c = gemm_config_t()
    c.bn, c.group_m, c.grid = int(cfg.get("bn", 0)), int(cfg.get("group_m", 0)), int(cfg.get("grid", 0))
    c.cta_group, c.split_k = int(cfg.get("cta_group", 0)), int(cfg.get("split_k", 0))
    c.stream_k = int(cfg.get("stream_k", 0))
    c.order = int(cfg.get("order", 0))
    c.general = int(cfg.get("general", 0))
    return ctypes.byref(c)


def gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout, stream):
    """Raw C-ABI call; pointers and stream as integers.  Returns the status code."""
    return _lib.gemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                     stream)


def gemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout, stream,
            cfg=None):
    return _lib.gemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                        stream, _cfg(cfg))


def gemm_bias_act(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                  bias, bias_kind, act, stream, cfg=None):
    """Raw C-ABI call of the fused-epilogue GEMM (bias: device pointer or 0)."""
    return _lib.gemm_bias_act(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype,
                              layout, bias, bias_kind, act, stream, _cfg(cfg))


def gemm_ex_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, layout,
                    stream, cfg=None):
    """gemm_ex with stream-K scratch taken from the library's fixed per-device
    buffer instead of cudaMalloc (calls that overlap on the device race)."""
    return _lib.gemm_ex_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype,
                                layout, stream, _cfg(cfg))


def gemm_host(M, N, K, alpha, hA, lda, hB, ldb, beta, hC, ldc, in_dtype, out_dtype, layout,
              dA, dB, dC, stream):
    return _lib.gemm_host(M, N, K, alpha, hA, lda, hB, ldb, beta, hC, ldc, in_dtype, out_dtype,
                          layout, dA, dB, dC, stream)


def gemm_sync_status(stream=0):
    site = ctypes.c_int(0)
    s = _lib.gemm_sync_status(stream, ctypes.byref(site))
    return s, site.value


def gemm_debug_set(wait_timeout_ns=0, inject_skip=0):
    _lib.gemm_debug_set(int(wait_timeout_ns), int(inject_skip))


def gemm_plan(M, N, K, in_dtype, out_dtype, layout, num_sms, cfg=None):
    p = gemm_plan_t()
    s = _lib.gemm_plan(M, N, K, in_dtype, out_dtype, layout, num_sms, _cfg(cfg), ctypes.byref(p))
    return s, p


def gemm_tile_coord(t, m_tiles, n_tiles, group_m):
    m, n = ctypes.c_int32(0), ctypes.c_int32(0)
    _lib.gemm_tile_coord(t, m_tiles, n_tiles, group_m, ctypes.byref(m), ctypes.byref(n))
    return m.value, n.value


def gemm_tile_order(order, m_tiles, n_tiles, group_m=1):
    """The whole tile order as a list of (m_blk, n_blk), or None if unavailable."""
    n = m_tiles * n_tiles
    mb = (ctypes.c_int32 * max(n, 1))()
    nb = (ctypes.c_int32 * max(n, 1))()
    got = _lib.gemm_tile_order(order, m_tiles, n_tiles, group_m, mb, nb, n)
    if got < 0:
        return None
    return [(mb[i], nb[i]) for i in range(got)]


def gemm_work_items(unit, units, dp_tiles, sk_iters, groups, max_items=4096):
    buf = (ctypes.c_int32 * (3 * max_items))()
    n = _lib.gemm_work_items(unit, units, dp_tiles, sk_iters, groups, buf, max_items)
    return [tuple(buf[3 * i:3 * i + 3]) for i in range(min(n, max_items))]


def gemm_split_tile_item(unit, tile_split, owner_groups, groups):
    """(tile, first k-group, end k-group) of a unit under a split-tile plan, or None."""
    buf = (ctypes.c_int32 * 3)()
    n = _lib.gemm_split_tile_item(unit, tile_split, owner_groups, groups, buf)
    return tuple(buf) if n == 1 else None


def gemm_fastdiv(n, d):
    """n // d the kernel's way (multiply and shift); 0xFFFFFFFF out of range."""
    return _lib.gemm_fastdiv(n, d)


def gemm_encode_idesc(in_dtype, a_mn, b_mn, m, n):
    return _lib.gemm_encode_idesc(in_dtype, a_mn, b_mn, m, n)


def gemm_encode_sdesc(addr, lbo, sbo):
    return _lib.gemm_encode_sdesc(addr, lbo, sbo)


def gemm_version():
    return _lib.gemm_version()


# ------------------------------------------------------------ torch helpers

def _torch_dtype_code(dt):
    import torch
    if dt == torch.float16:
        return GEMM_F16
    if dt == torch.bfloat16:
        return GEMM_BF16
    if dt == torch.float32:
        return GEMM_F32
    if dt == getattr(torch, "float8_e4m3fn", None):
        return GEMM_E4M3
    if dt == getattr(torch, "float8_e5m2", None):
        return GEMM_E5M2
    raise TypeError(f"unsupported dtype {dt}")


def _ld(t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("operands must be 2-D with unit stride along the last dimension")
    return t.stride(0) if t.size(0) > 1 else max(t.stride(0), t.size(1))


def matmul(a, b, c, alpha=1.0, beta=0.0, a_col=False, b_col=False, stream=None, cfg=None,
           bias=None, bias_rows=False, relu=False):
    """C <- act(alpha * A * B + beta * C + bias) on CUDA tensors (in place in ``c``).

    ``a`` is the stored A: [M, K] (a_col False) or [K, M] (a_col True, i.e. A
    column-major).  ``b`` is the stored B: [K, N] or [N, K] (b_col True).
    ``c`` is [M, N] with unit column stride; its dtype is the output format.
    ``bias``: optional fp32 CUDA tensor of N values (added per column) or, with
    ``bias_rows``, M values (added per row); ``relu`` clamps negative results to 0
    after the bias.  Either one selects the fused-epilogue entry point.
    Runs on ``stream`` (default: torch's current stream).  Raises GemmError.
    """
    import torch
    if not (a.is_cuda and b.is_cuda and c.is_cuda):
        raise ValueError("a, b and c must be CUDA tensors (there is no CPU path)")
    if a.dtype != b.dtype:
        raise TypeError("A and B must share a dtype")
    M, K = (a.shape[1], a.shape[0]) if a_col else (a.shape[0], a.shape[1])
    N, Kb = (b.shape[0], b.shape[1]) if b_col else (b.shape[1], b.shape[0])
    if Kb != K or tuple(c.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(a.shape)}, B {tuple(b.shape)}, C {tuple(c.shape)}")
    if stream is None:
        stream = torch.cuda.current_stream(c.device).cuda_stream
    layout = (GEMM_A_COL if a_col else 0) | (GEMM_B_COL if b_col else 0)
    if bias is None and not relu:
        s = gemm_ex(M, N, K, float(alpha), a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), float(beta),
                    c.data_ptr(), _ld(c), _torch_dtype_code(a.dtype), _torch_dtype_code(c.dtype),
                    layout, int(stream), cfg)
    else:
        kind = GEMM_BIAS_NONE
        bptr = 0
        if bias is not None:
            if not bias.is_cuda or bias.dtype != torch.float32 or not bias.is_contiguous():
                raise ValueError("bias must be a contiguous fp32 CUDA tensor")
            if bias.numel() != (M if bias_rows else N):
                raise ValueError(f"bias has {bias.numel()} values, expected {M if bias_rows else N}")
            kind = GEMM_BIAS_ROW if bias_rows else GEMM_BIAS_COL
            bptr = bias.data_ptr()
        s = gemm_bias_act(M, N, K, float(alpha), a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                          float(beta), c.data_ptr(), _ld(c), _torch_dtype_code(a.dtype),
                          _torch_dtype_code(c.dtype), layout, bptr, kind,
                          GEMM_ACT_RELU if relu else GEMM_ACT_NONE, int(stream), cfg)
    if s != GEMM_OK:
        raise GemmError(s, "gemm")
    return c
