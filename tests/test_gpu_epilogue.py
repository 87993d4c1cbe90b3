"""GPU parity of the fused epilogue C <- act(alpha*A*B + beta*C + bias) against the
oracle, through the C ABI (gemm_bias_act), in every kernel mode: integer inputs
and integer biases are bit-exact, general inputs within the error bound."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import check_against_oracle, operands, pad8, run_library, sample_rows

pytestmark = pytest.mark.gpu

MODES = [{"cta_group": 1, "bn": 256}, {"cta_group": 1, "bn": 64}, {"cta_group": 2},
         {"split_k": 2}, {"split_k": 4}, {"split_k": 4, "bn": 64}, {"split_k": 8, "bn": 128},
         {"cta_group": 1, "stream_k": 2}, {"cta_group": 2, "stream_k": 2},
         {"stream_k": 3}, {"stream_k": 3, "split_k": 4, "bn": 64}]
MODE_IDS = ["cta1", "cta1-bn64", "pair", "splitk2", "splitk4", "splitk4-bn64", "splitk8-bn128",
            "streamk1", "streamk2", "splittile2", "splittile4-bn64"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


def _int_bias(n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(-40, 41, size=n).astype(np.float32)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("kind", ["col", "row"])
@pytest.mark.parametrize("relu", [False, True])
def test_integer_bit_exact(mode, kind, relu):
    """Several tiles with ragged edges in M, N and K; integers keep every step exact,
    so the output must match the oracle bit for bit."""
    M, N, K = (128, 1000, 2048) if "split_k" in mode else (520, 392, 456)
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=M + N, pad=True)
    bias = _int_bias(N if kind == "col" else M, 5)
    for out_dtype in ("f32", "bf16"):
        out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                             a_col=False, b_col=True, cfg=mode, ldc=pad8(N), bias=bias,
                             bias_kind=kind, relu=relu)
        check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                             a_col=False, b_col=True, exact=True, bias=bias, bias_kind=kind,
                             relu=relu)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("a_col,b_col", [(False, False), (True, True)])
def test_uniform_alpha_beta_within_bound(mode, a_col, b_col):
    M, N, K = (128, 768, 3072) if "split_k" in mode else (384, 520, 640)
    A, B = operands(M, N, K, "f16", a_col, b_col, dist="uniform", seed=K, pad=True)
    C = si.matrix("uniform", 3000 + K, M, N, "bf16")
    bias = si.uniform_pm1(91, N).astype(np.float32) * 4
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16", a_col=a_col,
                         b_col=b_col, alpha=0.75, beta=-0.5, C=C, cfg=mode, ldc=pad8(N),
                         bias=bias, bias_kind="col", relu=True)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16", a_col=a_col,
                         b_col=b_col, alpha=0.75, beta=-0.5, C=C, bias=bias, bias_kind="col",
                         relu=True)


def test_ragged_fp32_edge_and_row_bias():
    """N * 4 bytes not a multiple of 16: the right edge takes predicated stores and
    the last bias elements the guarded loads."""
    M, N, K = 200, 203, 136
    A, B = operands(M, N, K, "bf16", False, False, dist="int", seed=3, pad=True)
    for kind in ("col", "row"):
        bias = _int_bias(N if kind == "col" else M, 11)
        out, full = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                                a_col=False, b_col=False, ldc=pad8(N) + 4, bias=bias,
                                bias_kind=kind, relu=True)
        check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                             a_col=False, b_col=False, exact=True, bias=bias, bias_kind=kind,
                             relu=True)
        # the guard columns past N keep their NaN poison
        assert np.all(np.isnan(full[:, N:].view(np.float32)))


def test_k_zero_bias_relu():
    """K == 0: C <- relu(beta * C + bias), exact on dyadic values."""
    import dense_tensor_core_tcgen05_gb300 as g
    M, N = 70, 96
    c0 = (torch.arange(M * N, device="cuda", dtype=torch.float32).reshape(M, N) - 3000) / 8
    bias = (torch.arange(N, device="cuda", dtype=torch.float32) - 40) / 4
    c = c0.clone()
    a = torch.empty(M, 0, device="cuda", dtype=torch.float16)
    b = torch.empty(0, N, device="cuda", dtype=torch.float16)
    g.matmul(a, b, c, beta=0.5, bias=bias, relu=True)
    torch.cuda.synchronize()
    assert torch.equal(c, torch.clamp_min(0.5 * c0 + bias, 0.0))


def test_relu_keeps_nan_and_zero_epilogue_is_plain_gemm():
    import dense_tensor_core_tcgen05_gb300 as g
    M, N, K = 256, 256, 512
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=21)
    C = si.matrix("uniform", 77, M, N, "f32")
    C[5, 9] = 0x7FC00000
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, beta=1.0, C=C, relu=True)
    assert np.isnan(out[5, 9].view(np.float32))
    # a zero bias without activation is the plain GEMM, bit for bit
    plain, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                           b_col=True)
    zero, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                          b_col=True, bias=np.zeros(N, np.float32), bias_kind="col")
    np.testing.assert_array_equal(plain, zero)


def test_workload_size_sampled_rows():
    """The 4096^3 bf16 workload with a per-column bias and ReLU, in the launch
    configuration the planner picks, checked on sampled rows."""
    M = N = K = 4096
    A, B = operands(M, N, K, "bf16", False, False, dist="normal", seed=4)
    bias = si.normal(303, N, 1.0).astype(np.float32)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="bf16", a_col=False,
                         b_col=False, bias=bias, bias_kind="col", relu=True)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="bf16",
                         a_col=False, b_col=False, rows=sample_rows(M, 24), bias=bias,
                         bias_kind="col", relu=True)
