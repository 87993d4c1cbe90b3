"""gemm_ex_noalloc: the stream-K launch with its scratch in the library's fixed
per-device buffer (no cudaMalloc) against gemm_ex, which takes the scratch from
its per-stream cache.  Two no-alloc calls in a row must each match gemm_ex
within the parity tolerance of the output format.

The file is named to be collected last, so that it also runs after every other
GPU test has used the library (and the fixed buffer's epochs have advanced).
"""
import pytest
import torch

from gpu_util import TOL

pytestmark = pytest.mark.gpu

# (M, N, K, cfg, in dtype, out dtype, alpha, beta): stream-K on CTA-pair tiles of
# 256 x 256 over every SM (the largest scratch a 152-SM GPU can need), and on
# single-CTA 128-wide tiles with a ragged shape and beta != 0.
CASES = [
    (2048, 2048, 2048, {"stream_k": 2, "cta_group": 2}, torch.float16, torch.float32, 1.0, 0.0),
    (1000, 1096, 1504, {"stream_k": 2, "cta_group": 1, "bn": 128}, torch.bfloat16,
     torch.bfloat16, 0.75, -0.5),
]
CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
TOL_OF = {torch.float32: TOL["f32"], torch.bfloat16: TOL["bf16"], torch.float16: TOL["f16"]}


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as lib
    lib.gemm_debug_set(0, 0)
    return lib


def _call(fn, a, b, c, alpha, beta, cfg):
    M, K = a.shape
    N = b.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return fn(M, N, K, alpha, a.data_ptr(), K, b.data_ptr(), N, beta, c.data_ptr(), N,
              CODE[a.dtype], CODE[c.dtype], 0, stream, cfg)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-cta{c[3]['cta_group']}")
def test_noalloc_matches_gemm_ex_twice(g, case):
    M, N, K, cfg, idt, odt, alpha, beta = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, p = g.gemm_plan(M, N, K, CODE[idt], CODE[odt], 0, sms, cfg)
    assert s == g.GEMM_OK and p.sk_iters > 0, "case does not exercise stream-K"
    assert 0 < p.scratch_bytes <= g.GEMM_NOALLOC_SCRATCH_BYTES

    gen = torch.Generator(device="cuda").manual_seed(M + N + K)
    a = (torch.rand(M, K, device="cuda", generator=gen) * 2 - 1).to(idt)
    b = (torch.rand(K, N, device="cuda", generator=gen) * 2 - 1).to(idt)
    c0 = (torch.rand(M, N, device="cuda", generator=gen) * 2 - 1).to(odt)

    ref = c0.clone()
    assert _call(g.gemm_ex, a, b, ref, alpha, beta, cfg) == g.GEMM_OK
    # error bound of the format: TOL * |alpha| * sum_k |a_ik||b_kj| + 1e-6
    bound = TOL_OF[odt] * abs(alpha) * (a.float().abs() @ b.float().abs()) + 1e-6
    outs = []
    for _ in range(2):
        c = c0.clone()
        assert _call(g.gemm_ex_noalloc, a, b, c, alpha, beta, cfg) == g.GEMM_OK
        outs.append(c)
    s, site = g.gemm_sync_status(torch.cuda.current_stream().cuda_stream)
    assert s == g.GEMM_OK, f"kernel status {s} site {site}"
    for c in outs:
        assert torch.isfinite(c.float()).all()
        err = (c.float() - ref.float()).abs()
        assert bool((err <= bound).all()), f"max excess {(err - bound).max().item()}"
