"""CPU oracle for dense GEMM  C <- alpha*A*B + beta*C  -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The library
(``dense_tensor_core_tcgen05_gb300``) never imports it and shares no code with
it; the only module both sides use is ``seeded_inputs`` (random operands, no
GEMM arithmetic).

The arithmetic lives in ``gemm_oracle.c`` (plain C, binary64 accumulation,
k ascending, round-to-nearest-even output); this file only compiles it with gcc
and marshals numpy arrays.  See that file's header for the definition and the
passages it follows ("GEMM From Naive CUDA to Tensor Cores", leetllm.com:
the worked example, the GEMM definition, the rounded-input reference).

Parity status: pinned.  ``tests/test_oracle_pins.py`` checks it against the
page's worked example, exact rational brute force, identity and permutation
products, the all-ones closed form, and the format facts the page prints.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None

FMT = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4}
_BITS_DT = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32, "e4m3": np.uint8,
            "e5m2": np.uint8}


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into _build/liboracle_gemm.so (gcc, no -march:
    the same source builds on x86-64 and aarch64).  -ffp-contract=off keeps
    every binary64 multiply and add separately rounded on both."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, f64, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [i64, i64, i64, f64, vp, i64, ci, vp, i64, ci, ci,
                                        f64, vp, i64, ci, vp, i64, vp, vp, vp, ci]
            lib.oracle_gemm.restype = ci
            lib.oracle_gemm_epilogue.argtypes = [i64, i64, i64, f64, vp, i64, ci, vp, i64, ci, ci,
                                                 f64, vp, i64, ci, vp, ci, ci, vp, i64, vp, vp,
                                                 vp, ci]
            lib.oracle_gemm_epilogue.restype = ci
            lib.oracle_decode.argtypes = [vp, ci, i64, vp]
            lib.oracle_encode.argtypes = [vp, ci, i64, vp]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Exact binary64 values of fp16 / bf16 / fp32 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=_BITS_DT[fmt])
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(b), FMT[fmt], b.size, _ptr(out))
    return out


def encode(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round binary64 values to fp16 / bf16 / fp32 (nearest, ties to even); bit patterns."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=_BITS_DT[fmt])
    _load().oracle_encode(_ptr(v), FMT[fmt], v.size, _ptr(out))
    return out


BIAS_KIND = {None: 0, "col": 1, "row": 2}


def gemm(A, B, *, M, N, K, in_dtype, out_dtype, a_col=False, b_col=False,
         alpha=1.0, beta=0.0, C=None, rows=None, nthreads=0, bias=None, bias_kind=None,
         relu=False):
    """Oracle GEMM on bit-pattern operands.

    A: [M, K] (a_col False) or [K, M] (a_col True) array of input bit patterns;
    B: [K, N] (b_col False) or [N, K] (b_col True); the leading dimension of each
    is its second extent.  C: [M, N'] (N' >= N) output-format bit patterns, read
    only when beta != 0.  rows: optional list of row indices (default all M).
    bias: float32 values, N of them (bias_kind "col": bias[j] added to column j) or
    M (bias_kind "row": bias[i] added to row i), added after alpha*s + beta*c;
    relu: then negative results become 0 (NaN stays NaN), before the rounding.
    Returns (out_bits [R, N], exact [R, N] binary64 before rounding, scale [R, N]
    = sum_k |a_ik||b_kj|).
    """
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    assert A.ndim == 2 and B.ndim == 2
    assert A.shape == ((K, M) if a_col else (M, K)) or (A.shape[0] == (K if a_col else M)
                                                      and A.shape[1] >= (M if a_col else K))
    assert B.shape[0] == (N if b_col else K) and B.shape[1] >= (K if b_col else N)
    if rows is None:
        r = None
        nr = M
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        nr = r.size
    Cc = None
    ldc = 0
    if beta != 0.0:
        Cc = np.ascontiguousarray(C, dtype=_BITS_DT[out_dtype])
        assert Cc.shape[0] == M and Cc.shape[1] >= N
        ldc = Cc.shape[1]
    bk = BIAS_KIND[bias_kind]
    bv = None
    if bk:
        bv = np.ascontiguousarray(bias, dtype=np.float32)
        assert bv.ndim == 1 and bv.size == (N if bk == 1 else M)
    out_bits = np.empty((nr, N), dtype=_BITS_DT[out_dtype])
    exact = np.empty((nr, N), dtype=np.float64)
    scale = np.empty((nr, N), dtype=np.float64)
    rc = _load().oracle_gemm_epilogue(M, N, K, float(alpha), _ptr(A), A.shape[1], int(a_col),
                                      _ptr(B), B.shape[1], int(b_col), FMT[in_dtype],
                                      float(beta), _ptr(Cc), ldc, FMT[out_dtype],
                                      _ptr(bv), bk, int(bool(relu)),
                                      _ptr(r), nr, _ptr(out_bits), _ptr(exact), _ptr(scale),
                                      int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return out_bits, exact, scale


def flops(M: int, N: int, K: int) -> int:
    """Logical floating-point operations of one GEMM: one multiply and one add per
    inner-loop step, 2*M*N*K (the counting convention of the leetllm page,
    "Compute one output before launching a warp")."""
    return 2 * M * N * K
