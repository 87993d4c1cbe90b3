"""Small-M ("decode-like") GEMMs beyond the 128-row skinny workload: one to a few
dozen rows against wide, deep B, where the planner splits K over a cluster.  The
split keeps a fixed reduction order, so repeated runs are bitwise identical (the
Ada page's warning: a library that switches to split-K for skinny matrices drifts
run to run)."""
import numpy as np
import pytest
import torch

from gpu_util import check_against_oracle, operands, run_library, sample_rows

pytestmark = pytest.mark.gpu

DECODE = [(1, 4096, 4096), (8, 8192, 4096), (16, 4096, 8192), (32, 2048, 8192), (64, 8192, 2048),
          (96, 3000, 5000)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


@pytest.mark.parametrize("shape", DECODE, ids=lambda s: "x".join(map(str, s)))
def test_decode_integer_exact(shape):
    M, N, K = shape
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=M + N, pad=True)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, ldc=(N + 7) // 8 * 8)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, exact=True)


@pytest.mark.parametrize("shape", DECODE[:3], ids=lambda s: "x".join(map(str, s)))
def test_decode_normal_bf16_deterministic(shape):
    M, N, K = shape
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=K, sigma=0.02)
    outs = [run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="bf16", a_col=False,
                        b_col=True)[0] for _ in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    check_against_oracle(outs[0], A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="bf16",
                         a_col=False, b_col=True, rows=sample_rows(M, 16))


def test_decode_plans_split_k():
    import dense_tensor_core_tcgen05_gb300 as g
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N, K in DECODE:
        s, p = g.gemm_plan(M, N, K, 1, 2, 2, sms)
        assert s == 0 and p.m_tiles == 1
        if K >= 4096:
            assert p.split_k >= 2, (M, N, K)
