"""GPU parity of the accumulator preload and the stream-K partial prefetch.

With alpha == 1 and beta != 0 the epilogue warps write beta * C into a tile's
TMEM accumulator before its first MMA, for every work item of a persistent CTA
(or CTA pair) after its first two; the MMAs then accumulate A * B onto it and the
epilogue reads no C.  A stream-K owner whose tile has a single later unit finds
that unit's partial sum prefetched into its draining ring.  Small grids put many
tiles on each unit so both paths run; integer inputs in {-4..4} (and C_in integer,
beta a power of two) keep every partial sum exact, so the result is unique and
must equal the oracle's bits; ragged shapes check the bounds of the C loads.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import check_against_oracle, operands, pad8, run_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# (M, N, K, cfg): every case runs several tiles per unit
PRELOAD_CASES = [
    (768, 512, 320, {"cta_group": 2, "grid": 2}),                  # one pair, 6 tiles
    (768, 512, 320, {"cta_group": 2, "bn": 128, "grid": 4}),       # two pairs of 128-wide tiles
    (700, 500, 200, {"cta_group": 2, "grid": 2}),                  # ragged rows and columns
    (640, 640, 256, {"cta_group": 1, "bn": 256, "grid": 3}),
    (600, 520, 192, {"cta_group": 1, "bn": 128, "grid": 5}),
    (520, 300, 128, {"cta_group": 1, "bn": 64, "grid": 4}),
]


def _case_id(c):
    return f"{c[0]}x{c[1]}x{c[2]}-" + "-".join(f"{k}{v}" for k, v in c[3].items())


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("beta", [0.5, -1.0, 2.0])
@pytest.mark.parametrize("case", PRELOAD_CASES, ids=_case_id)
def test_c_preload_integer_exact(case, beta, out_dtype):
    M, N, K, cfg = case
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=M + N, pad=True)
    ldc = pad8(N)
    C = si.matrix("int", 3100 + M, M, N, out_dtype, ld=ldc)
    out, full = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                            a_col=False, b_col=True, alpha=1.0, beta=beta, C=C, ldc=ldc, cfg=cfg)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=1.0, beta=beta, C=C, exact=True)


@pytest.mark.parametrize("a_col,b_col", [(False, False), (True, False), (True, True)])
def test_c_preload_layouts(a_col, b_col):
    M, N, K = 768, 768, 256
    A, B = operands(M, N, K, "f16", a_col, b_col, dist="int", seed=11)
    C = si.matrix("int", 3111, M, N, "f32")
    cfg = {"cta_group": 2, "grid": 2}
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32", a_col=a_col,
                         b_col=b_col, alpha=1.0, beta=0.5, C=C, cfg=cfg)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32", a_col=a_col,
                         b_col=b_col, alpha=1.0, beta=0.5, C=C, exact=True)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_c_preload_normal_tolerance(out_dtype):
    """Normal draws (the 8192^3 workload's recipe at a smaller size, one pair
    doing all tiles): within the error bound of the output format."""
    M, N, K = 1024, 768, 512
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=12, sigma=0.5)
    C = si.matrix("normal", 3112, M, N, out_dtype, 1.0)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype, a_col=False,
                         b_col=True, alpha=1.0, beta=0.5, C=C, cfg={"cta_group": 2, "grid": 2})
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=1.0, beta=0.5, C=C)


def test_c_preload_general_kernel():
    """The general kernel (every parameter a run-time value) takes the same
    preload path and gives the oracle's bits."""
    M, N, K = 768, 512, 320
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=13)
    C = si.matrix("int", 3113, M, N, "f32")
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, alpha=1.0, beta=0.5, C=C,
                         cfg={"cta_group": 2, "grid": 2, "general": 1})
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, alpha=1.0, beta=0.5, C=C, exact=True)


# Stream-K plans with at least two waves: every owner has at most one later unit,
# whose partial the producer lane prefetches; with beta != 0 the owner's
# accumulator also starts from beta * C when it is the unit's third item or later.
SK_PREFETCH_CASES = [
    (2048, 2048, 2048, {"stream_k": 2, "cta_group": 2, "grid": 48}),
    (2048, 1536, 1024, {"stream_k": 2, "cta_group": 1, "grid": 20}),
    (1900, 1500, 1000, {"stream_k": 2, "cta_group": 1, "bn": 128, "grid": 40}),
    (2048, 2048, 1024, {"stream_k": 2, "cta_group": 2, "grid": 22}),
]


def _plan(M, N, K, cfg, out_dtype="f32"):
    import dense_tensor_core_tcgen05_gb300 as g
    code = {"f32": g.GEMM_F32, "bf16": g.GEMM_BF16}[out_dtype]
    s, p = g.gemm_plan(M, N, K, g.GEMM_BF16, code, g.GEMM_B_COL, _sms(), cfg)
    assert s == 0
    return p


@pytest.mark.parametrize("beta", [0.0, 0.5])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", SK_PREFETCH_CASES, ids=_case_id)
def test_stream_k_prefetch_integer_exact(case, out_dtype, beta):
    M, N, K, cfg = case
    p = _plan(M, N, K, cfg, out_dtype)
    units = p.grid // p.cta_group
    assert p.sk_iters > 0 and p.sk_iters // units >= p.groups, "owners must have one later unit"
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=M + K, pad=True)
    ldc = pad8(N)
    C = si.matrix("int", 3200 + M, M, N, out_dtype, ld=ldc) if beta else None
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype, a_col=False,
                         b_col=True, alpha=1.0, beta=beta, C=C, ldc=ldc, cfg=cfg)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=1.0, beta=beta, C=C, exact=True)


def test_stream_k_prefetch_deterministic():
    M, N, K = 2048, 2048, 2048
    cfg = {"stream_k": 2, "cta_group": 2, "grid": 48}
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=31, sigma=0.5)
    C = si.matrix("normal", 3231, M, N, "f32", 1.0)
    outs = [run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                        b_col=True, alpha=1.0, beta=0.5, C=C, cfg=cfg)[0] for _ in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    check_against_oracle(outs[0], A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, alpha=1.0, beta=0.5, C=C,
                         rows=list(range(0, M, 7)))
