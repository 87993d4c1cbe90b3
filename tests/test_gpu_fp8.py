"""GPU parity of FP8 (E4M3, E5M2) operands, multiplied by tcgen05.mma kind::f8f6f4
with fp32 accumulation, against the oracle on the same stored bits: integer
inputs bit-exact, general inputs within the error bound of the output format
(the inputs are exact; only the fp32 sums and the output rounding differ)."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import check_against_oracle, run_library, sample_rows

pytestmark = pytest.mark.gpu

MODES = [{"cta_group": 1, "bn": 256}, {"cta_group": 1, "bn": 64}, {"cta_group": 2},
         {"cta_group": 1, "stream_k": 2}, {"cta_group": 2, "stream_k": 2}]
MODE_IDS = ["cta1", "cta1-bn64", "pair", "streamk1", "streamk2"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


def _ld16(n):
    return (n + 15) // 16 * 16


def _operands(M, N, K, fmt, dist, seed, sigma=1.0):
    """A [M, K] row-major and B stored [N, K] (column-major), leading dimensions
    rounded up to 16 elements (16-byte row pitches)."""
    A = si.matrix(dist, 1000 + seed, M, K, fmt, sigma, ld=_ld16(K))
    B = si.matrix(dist, 2000 + seed, N, K, fmt, sigma, ld=_ld16(K))
    return A, B


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_fp8_integer_exact(fmt, mode):
    """Ragged in every dimension, K not a multiple of the 128-element k-block."""
    M, N, K = 520, 392, 456
    A, B = _operands(M, N, K, fmt, "int", seed=K)
    for out_dtype in ("f32", "bf16"):
        out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype=out_dtype,
                             a_col=False, b_col=True, cfg=mode, ldc=(N + 7) // 8 * 8)
        check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype=out_dtype,
                             a_col=False, b_col=True, exact=True)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("split", [2, 4])
def test_fp8_split_k_integer_exact(fmt, split):
    M, N, K = 128, 1000, 4000
    A, B = _operands(M, N, K, fmt, "int", seed=split)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32", a_col=False,
                         b_col=True, cfg={"split_k": split, "bn": 128}, ldc=1000)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32", a_col=False,
                         b_col=True, exact=True)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_fp8_normal_within_bound(fmt, out_dtype):
    M, N, K = 777, 640, 2048
    A, B = _operands(M, N, K, fmt, "normal", seed=7, sigma=1.0)
    C = si.matrix("uniform", 3007, M, N, out_dtype)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype=out_dtype, a_col=False,
                         b_col=True, alpha=0.5, beta=-1.0, C=C)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=0.5, beta=-1.0, C=C)


def test_fp8_workload_size_sampled_rows():
    M = N = K = 4096
    A, B = _operands(M, N, K, "e4m3", "normal", seed=11)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="e4m3", out_dtype="bf16", a_col=False,
                         b_col=True)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="e4m3", out_dtype="bf16",
                         a_col=False, b_col=True, rows=sample_rows(M, 24))
