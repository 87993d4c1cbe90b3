"""GPU parity under the Hilbert tile order: every kernel mode maps tile indices
through the order's table, so integer problems must still match the oracle bit
for bit, on square and ragged, non-square tile grids."""
import numpy as np
import pytest
import torch

from gpu_util import check_against_oracle, operands, pad8, run_library

pytestmark = pytest.mark.gpu

MODES = [{"cta_group": 1, "bn": 128}, {"cta_group": 2}, {"split_k": 2},
         {"cta_group": 1, "stream_k": 2}, {"cta_group": 2, "stream_k": 2}]
MODE_IDS = ["cta1", "pair", "splitk2", "streamk1", "streamk2"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", [(1792, 1280, 384), (1000, 2600, 264)], ids=["7x5", "ragged"])
def test_hilbert_order_integer_exact(mode, shape):
    M, N, K = shape
    if "split_k" in mode:
        # one 128-row panel; N keeps the 1 x n tile grid inside 16x its Hilbert square
        M, N = 128, min(N, 1800)
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=N, pad=True)
    cfg = dict(mode, order=2)
    import dense_tensor_core_tcgen05_gb300 as g
    s, p = g.gemm_plan(M, N, K, 1, 2, 2, torch.cuda.get_device_properties(0).multi_processor_count, cfg)
    assert s == 0 and p.order == g.GEMM_ORDER_HILBERT
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, cfg=cfg, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, exact=True)


def test_hilbert_and_grouped_orders_agree_bitwise():
    """The order only changes which CTA computes a tile, not how: normal inputs give
    identical bits under both orders."""
    M, N, K = 2304, 1792, 1024
    A, B = operands(M, N, K, "f16", False, False, dist="normal", seed=9)
    outs = [run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16", a_col=False,
                        b_col=False, cfg={"order": o})[0] for o in (1, 2)]
    np.testing.assert_array_equal(outs[0], outs[1])
