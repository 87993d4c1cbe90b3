"""Helpers for the GPU parity tests: move seeded bit-pattern operands to the
device, call the library through its C ABI, and compare with the CPU oracle."""
import numpy as np
import torch

import oracle
import seeded_inputs as si

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
BITS_DT = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32, "e4m3": np.uint8,
           "e5m2": np.uint8}
# Error bound |C_gpu - C_oracle| <= TOL * sum_k |a_ik||b_kj| + 1e-6 per output format.
TOL = {"f32": 1e-3, "bf16": 8e-3, "f16": 8e-3}
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "f32": 0x7FC00000}


def to_device(bits: np.ndarray, fmt: str, device="cuda") -> torch.Tensor:
    """Upload a bit-pattern array as a tensor of the matching dtype (same shape)."""
    b = np.ascontiguousarray(bits)
    if fmt == "f32":
        t = torch.from_numpy(b.view(np.int32).copy()).view(torch.float32)
    elif fmt in ("e4m3", "e5m2"):
        t = torch.from_numpy(b.view(np.uint8).copy()).view(TORCH_DT[fmt])
    else:
        t = torch.from_numpy(b.view(np.int16).copy()).view(TORCH_DT[fmt])
    return t.to(device)


def to_bits(t: torch.Tensor, fmt: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if fmt == "f32":
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def alloc_c(M, N, ldc, fmt, init_bits=None, device="cuda"):
    """[M, ldc] buffer (logical C = first N columns) filled with NaN (poison) or
    with given bits; returns (full buffer, view [M, N])."""
    buf = np.full((M, ldc), NAN_BITS[fmt], dtype=BITS_DT[fmt])
    if init_bits is not None:
        buf[:, :N] = init_bits[:, :N]
    full = to_device(buf, fmt, device)
    return full, full[:, :N]


def run_library(A, B, *, M, N, K, in_dtype, out_dtype, a_col, b_col, alpha=1.0, beta=0.0,
                C=None, ldc=None, cfg=None, bias=None, bias_kind=None, relu=False):
    """Run the GPU GEMM; returns (out bits [M, N], full C buffer bits [M, ldc]).
    bias (float32 numpy, N or M values) with bias_kind "col"/"row", and relu,
    select the fused epilogue."""
    import dense_tensor_core_tcgen05_gb300 as g
    ldc = N if ldc is None else ldc
    dA = to_device(A, in_dtype)[:, :(M if a_col else K)]
    dB = to_device(B, in_dtype)[:, :(K if b_col else N)]
    full, c = alloc_c(M, N, ldc, out_dtype, C)
    dbias = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).cuda()
    g.matmul(dA, dB, c, alpha=alpha, beta=beta, a_col=a_col, b_col=b_col, cfg=cfg, bias=dbias,
             bias_rows=(bias_kind == "row"), relu=relu)
    s, site = g.gemm_sync_status(torch.cuda.current_stream().cuda_stream)
    assert s == g.GEMM_OK, f"kernel status {s} site {site}"
    fb = to_bits(full, out_dtype)
    return fb[:, :N].copy(), fb


def check_against_oracle(gpu_bits, A, B, *, M, N, K, in_dtype, out_dtype, a_col, b_col,
                         alpha=1.0, beta=0.0, C=None, rows=None, exact=False, bias=None,
                         bias_kind=None, relu=False, strict=False):
    """Element-wise comparison on the given rows (default all).  exact=True demands
    identical bit patterns; otherwise the error bound of TOL[out_dtype].  strict=True
    checks the bound exactly as stated (TOL * sum|a||b| + 1e-6), without the extra
    fp32 rounding allowed for beta * C and for the bias."""
    obits, oexact, oscale = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype=in_dtype,
                                        out_dtype=out_dtype, a_col=a_col, b_col=b_col,
                                        alpha=alpha, beta=beta, C=C, rows=rows, bias=bias,
                                        bias_kind=bias_kind, relu=relu)
    g = gpu_bits if rows is None else gpu_bits[np.asarray(rows)]
    if exact:
        bad = np.argwhere(g != obits)
        assert bad.size == 0, (f"{len(bad)} mismatches, first at {tuple(bad[0])}: "
                               f"gpu {g[tuple(bad[0])]:#x} oracle {obits[tuple(bad[0])]:#x}")
        return 0.0
    gv = oracle.decode(g, out_dtype)
    err = np.abs(gv - oexact)
    bound = TOL[out_dtype] * oscale + 1e-6
    if beta != 0.0 and not strict:
        # beta*C is rounded once in fp32 on the GPU: allow its rounding on top
        cin = oracle.decode(np.asarray(C)[:, :N] if rows is None else np.asarray(C)[np.asarray(rows), :N],
                            out_dtype)
        bound = bound + 2.0 ** -23 * np.abs(beta * cin)
    if bias_kind is not None and not strict:
        # the bias is added in fp32 on the GPU: one more rounding of a value at
        # most |alpha| S + |beta c| + |bias| in size (ReLU is 1-Lipschitz)
        bv = np.asarray(bias, np.float64)
        rr = np.arange(M) if rows is None else np.asarray(rows)
        b2 = bv[None, :N] if bias_kind == "col" else bv[rr][:, None]
        bound = bound + 2.0 ** -23 * (np.abs(b2) + abs(alpha) * oscale)
    worst = np.argmax(err - bound)
    assert np.all(np.isfinite(gv)), "non-finite output"
    assert np.all(err <= bound), (f"error bound exceeded at {np.unravel_index(worst, err.shape)}: "
                                  f"err {err.flat[worst]:.3g} bound {bound.flat[worst]:.3g}")
    return float(np.max(err / (oscale + 1e-30)))


def sample_rows(M, count=48, seed=0):
    """Rows to check on large problems: the first and last rows of several
    128-row tiles (tile edges, lane-quarter edges) plus seeded random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, 31, 32, 63, 64, 95, 96, 127, 128, M - 1, M - 2, M - 128, M - 97}
    fixed = {r for r in fixed if 0 <= r < M}
    extra = rng.choice(M, size=min(M, max(0, count - len(fixed))), replace=False)
    return sorted(fixed | set(int(x) for x in extra))


def pad8(n):
    """Leading dimension with a 16-byte row pitch for 16-bit elements."""
    return max(8, (n + 7) // 8 * 8)


def operands(M, N, K, in_dtype, a_col, b_col, dist="uniform", seed=1, sigma=1.0, pad=False):
    """Seeded A and B in the requested storage orders (bit patterns); with pad=True
    the leading dimensions are rounded up to 16-byte pitches (guard columns)."""
    a_shape = (K, M) if a_col else (M, K)
    b_shape = (N, K) if b_col else (K, N)
    A = si.matrix(dist, 1000 + seed, *a_shape, in_dtype, sigma,
                  ld=pad8(a_shape[1]) if pad else None)
    B = si.matrix(dist, 2000 + seed, *b_shape, in_dtype, sigma,
                  ld=pad8(b_shape[1]) if pad else None)
    return A, B
