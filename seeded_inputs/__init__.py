"""Seeded synthetic operands for the dense GEMM workloads.

This module is the one piece shared by the CUDA path's tests/bench and the
CPU oracle.  It holds no GEMM arithmetic: it only draws numbers and stores
them in the element formats the GEMM reads (IEEE binary16, bfloat16, binary32).

Generator (a counter-based stream, so every element is addressable on its own):

* ``splitmix64`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): element ``i`` of the stream with seed ``s`` is
  ``mix(s + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)`` with the published
  two-multiply finaliser.
* uniform[-1, 1): ``(x >> 40) * 2**-23 - 1`` -- exact in binary32 (24-bit grid).
* normal(0, sigma): Box-Muller on two 53-bit uniforms in (0, 1] drawn from
  stream positions 2i and 2i+1, evaluated in binary64, scaled by sigma, then
  rounded to binary32.
* integers uniform in {-4, ..., 4}: ``x mod 9 - 4``.

The GEMM pages only say "from seed" (no generator, no seed); the choice above is
this library's reading and is recorded with the seeds in every bench receipt.

Rounding to the stored input format is round-to-nearest-even from binary32
(the IEEE default the GEMM pages' format examples use): numpy's float16 cast
for binary16 and an integer RNE on the binary32 bit pattern for bfloat16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

F16, BF16, F32 = "f16", "bf16", "f32"
E4M3, E5M2 = "e4m3", "e5m2"


_CHUNK = 1 << 22


def _chunked(count, fn):
    """Run fn(lo, hi) over [0, count) in chunks on a few threads (numpy drops
    the GIL inside its array loops); chunks write disjoint output slices."""
    spans = [(lo, min(count, lo + _CHUNK)) for lo in range(0, count, _CHUNK)]
    if len(spans) <= 1:
        for lo, hi in spans:
            fn(lo, hi)
        return
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        list(ex.map(lambda sp: fn(*sp), spans))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Elements ``start .. start+count-1`` of the splitmix64 stream ``seed``."""
    out = np.empty(count, dtype=np.uint64)
    s0 = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    s30, s27, s31 = np.uint64(30), np.uint64(27), np.uint64(31)

    def fill(lo, hi):
        with np.errstate(over="ignore"):
            z = out[lo:hi]
            z[:] = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            z *= GAMMA
            z += s0
            z ^= z >> s30
            z *= _M1
            z ^= z >> s27
            z *= _M2
            z ^= z >> s31
    _chunked(count, fill)
    return out


def uniform_pm1(seed: int, count: int) -> np.ndarray:
    """uniform[-1, 1) on a 2**-23 grid, as binary32 (exactly representable)."""
    x = splitmix64(seed, 0, count)
    x >>= np.uint64(40)
    v = x.astype(np.float64)
    v *= 2.0 ** -23
    v -= 1.0
    return v.astype(np.float32)


def normal(seed: int, count: int, sigma: float) -> np.ndarray:
    """normal(0, sigma) by Box-Muller (cosine branch), rounded to binary32."""
    out = np.empty(count, dtype=np.float32)
    x = splitmix64(seed, 0, 2 * count)

    def fill(lo, hi):
        xx = x[2 * lo:2 * hi] >> np.uint64(11)
        u = xx.astype(np.float64)
        u += 1.0
        u *= 2.0 ** -53                       # (0, 1]
        r = np.log(u[0::2])
        r *= -2.0
        np.sqrt(r, out=r)
        c = u[1::2] * (2.0 * np.pi)
        np.cos(c, out=c)
        r *= c
        r *= sigma
        out[lo:hi] = r
    _chunked(count, fill)
    return out


def int_pm4(seed: int, count: int) -> np.ndarray:
    """Integers uniform in {-4..4}, as binary32."""
    x = splitmix64(seed, 0, count)
    return ((x % np.uint64(9)).astype(np.int64) - 4).astype(np.float32)


def f32_to_f16_bits(v: np.ndarray) -> np.ndarray:
    """binary32 -> binary16 (round to nearest even), as uint16 bit patterns."""
    return np.asarray(v, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 (round to nearest even), as uint16 bit patterns.

    Integer RNE on the top 16 bits; NaNs are kept quiet.  Inputs here are finite.
    """
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(v, dtype=np.float32))
    if nan.any():
        r = r.copy()
        r[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16)) | np.uint16(0x40)
    return r


def _fp8_positive_values(exp_bits: int, man_bits: int) -> np.ndarray:
    """Values of the 128 non-negative codes of an OCP FP8 format (NaN where the
    code is not a finite number): E4M3 (4, 3) has no infinities and S.1111.111 as
    NaN; E5M2 (5, 2) has IEEE-style infinities and NaNs."""
    bias = (1 << (exp_bits - 1)) - 1
    vals = np.empty(128, dtype=np.float64)
    for code in range(128):
        e, m = code >> man_bits, code & ((1 << man_bits) - 1)
        if e == 0:
            vals[code] = m / (1 << man_bits) * 2.0 ** (1 - bias)
        elif e == (1 << exp_bits) - 1 and (exp_bits == 5 or m == (1 << man_bits) - 1):
            vals[code] = np.nan
        else:
            vals[code] = (1 + m / (1 << man_bits)) * 2.0 ** (e - bias)
    return vals


def f32_to_fp8_bits(v: np.ndarray, dtype: str) -> np.ndarray:
    """binary32 -> E4M3 / E5M2 (round to nearest, ties to the even code), uint8
    bit patterns.  Inputs must be finite and within the format's range."""
    pos = _fp8_positive_values(4, 3) if dtype == E4M3 else _fp8_positive_values(5, 2)
    finite = np.flatnonzero(np.isfinite(pos))     # codes in increasing value order
    table = pos[finite]
    x = np.asarray(v, dtype=np.float64)
    a = np.abs(x)
    if np.any(~np.isfinite(a)) or np.any(a > table[-1]):
        raise ValueError("value outside the FP8 format's finite range")
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, table.size - 1)
    lo = np.clip(hi - 1, 0, table.size - 1)
    dlo, dhi = a - table[lo], table[hi] - a
    code_lo, code_hi = finite[lo], finite[hi]
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (code_hi % 2 == 0) & (code_lo % 2 == 1))
    code = np.where(pick_hi, code_hi, code_lo).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def to_bits(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round binary32 values to the stored input format; returns the bit patterns."""
    if dtype == F16:
        return f32_to_f16_bits(v)
    if dtype == BF16:
        return f32_to_bf16_bits(v)
    if dtype in (E4M3, E5M2):
        return f32_to_fp8_bits(v, dtype)
    if dtype == F32:
        return np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    raise ValueError(dtype)


def draw(dist: str, seed: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """Dispatch on a distribution name: 'uniform', 'normal', 'int'."""
    if dist == "uniform":
        return uniform_pm1(seed, count)
    if dist == "normal":
        return normal(seed, count, sigma)
    if dist == "int":
        return int_pm4(seed, count)
    raise ValueError(dist)


def matrix(dist: str, seed: int, rows: int, cols: int, dtype: str,
           sigma: float = 1.0, ld: int | None = None) -> np.ndarray:
    """A [rows, cols] row-major array of bit patterns in ``dtype`` with leading
    dimension ``ld`` (>= cols).  Stream element (r, c) is ``r * cols + c`` so the
    logical values do not depend on ``ld``; padding columns are filled with a
    fixed non-zero pattern (a guard band, never read by a correct GEMM)."""
    ld = cols if ld is None else ld
    vals = draw(dist, seed, rows * cols, sigma).reshape(rows, cols)
    bits = to_bits(vals, dtype)
    if ld == cols:
        return np.ascontiguousarray(bits)
    out = np.empty((rows, ld), dtype=bits.dtype)
    guard = {np.dtype(np.uint8): 0x7F, np.dtype(np.uint16): 0x7E00, np.dtype(np.uint32): 0x7FC00000}
    out[:] = bits.dtype.type(guard[bits.dtype])   # a NaN of the format
    out[:, :cols] = bits
    return out


# The five synthetic workloads (shape, formats, storage orders, value
# distributions, alpha/beta).  Seeds: A = 1000+cfg, B = 2000+cfg, C = 3000+cfg.
WORKLOADS = {
    1: dict(name="gemm_512_f16_f32_rowrow", M=512, N=512, K=512, in_dtype=F16,
            out_dtype=F32, a_col=False, b_col=False, dist="uniform", sigma=1.0,
            alpha=1.0, beta=0.0, c_dist=None),
    2: dict(name="gemm_2048_f16_f32_rowrow", M=2048, N=2048, K=2048, in_dtype=F16,
            out_dtype=F32, a_col=False, b_col=False, dist="uniform", sigma=1.0,
            alpha=1.0, beta=0.0, c_dist=None),
    3: dict(name="gemm_4096_bf16_bf16_rowrow", M=4096, N=4096, K=4096, in_dtype=BF16,
            out_dtype=BF16, a_col=False, b_col=False, dist="normal", sigma=1.0,
            alpha=1.0, beta=0.0, c_dist=None),
    4: dict(name="gemm_8192_bf16_f32_rowcol_beta", M=8192, N=8192, K=8192,
            in_dtype=BF16, out_dtype=F32, a_col=False, b_col=True, dist="normal",
            sigma=0.5, alpha=1.0, beta=0.5, c_dist="normal"),
    5: dict(name="gemm_skinny_128x8192x8192_bf16_bf16_rowcol", M=128, N=8192, K=8192,
            in_dtype=BF16, out_dtype=BF16, a_col=False, b_col=True, dist="normal",
            sigma=0.02, alpha=1.0, beta=0.0, c_dist=None),
}


def workload_operands(cfg: int, integer: bool = False, scale: int = 1):
    """Bit-pattern operands for workload ``cfg``.

    ``integer=True`` gives the {-4..4} variant used for bit-exact checks (C_in too).
    ``scale`` divides M, N and K (for reduced-size parity cases of the same recipe).
    Returns dict(A=..., B=..., C=... or None, plus the workload fields).
    A is stored [M, K] (row-major) or [K, M] (column-major); B is stored [K, N]
    (row-major) or [N, K] (column-major); C is [M, N] row-major in out_dtype.
    """
    w = dict(WORKLOADS[cfg])
    M, N, K = w["M"] // scale, w["N"] // scale, w["K"] // scale
    if cfg == 5 and scale != 1:
        M = 128
    w.update(M=M, N=N, K=K)
    dist = "int" if integer else w["dist"]
    sig = w["sigma"]
    a_shape = (K, M) if w["a_col"] else (M, K)
    b_shape = (N, K) if w["b_col"] else (K, N)
    w["A"] = matrix(dist, 1000 + cfg, *a_shape, w["in_dtype"], sig)
    w["B"] = matrix(dist, 2000 + cfg, *b_shape, w["in_dtype"], sig)
    w["C"] = None
    if w["beta"] != 0.0:
        cdist = "int" if integer else w["c_dist"]
        w["C"] = matrix(cdist, 3000 + cfg, M, N, w["out_dtype"], 1.0)
    return w
