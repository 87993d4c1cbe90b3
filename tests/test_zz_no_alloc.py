"""gemm_ex_noalloc: the stream-K and split-tile launches with their scratch in
the library's fixed per-device buffer instead of memory from cudaMalloc.

It exists for callers that cannot allocate device memory on the call path: a
framework whose caching allocator already holds the GPU's memory, or a serving
loop that must not synchronise or fail on an allocation.  For those callers the
properties that matter are checked here:

- the results are those of gemm_ex bit for bit (the same plan runs the same
  deterministic kernel, whose stream-K partials are added in a fixed order, so
  only a wrong scratch offset or a stale ready flag could change a bit), on two
  calls in a row, and on integer inputs bit-exact against the CPU oracle;
- the calls allocate nothing: they run on a stream that gemm_ex never used (so
  the library's per-stream scratch cache cannot serve them), and the device's
  free memory and torch's reserved memory are unchanged across them;
- the Hilbert tile order, whose device table gemm_ex allocates, is served
  without allocating (gemm_ex_noalloc walks the grouped order instead) and gives
  the same bits on integer inputs.

The file is named to be collected last, so that it also runs after every other
GPU test has used the library (and the fixed buffer's epochs have advanced).
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import to_bits, to_device

pytestmark = pytest.mark.gpu

CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
FMT = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}
ORDER_HILBERT = 2

# (M, N, K, cfg, in dtype, out dtype, alpha, beta): stream-K on CTA-pair tiles of
# 256 x 256 over every SM (the largest scratch a 152-SM GPU can need), and on
# single-CTA 128-wide tiles with a ragged shape and beta != 0; the split-tile
# plan of a 128-row panel (every tile split over two CTAs through the scratch).
CASES = [
    (2048, 2048, 2048, {"stream_k": 2, "cta_group": 2}, torch.float16, torch.float32, 1.0, 0.0),
    (1000, 1096, 1504, {"stream_k": 2, "cta_group": 1, "bn": 128}, torch.bfloat16,
     torch.bfloat16, 0.75, -0.5),
    (128, 8192, 8192, {"stream_k": 3}, torch.bfloat16, torch.bfloat16, 1.0, 0.0),
]


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as lib
    lib.gemm_debug_set(0, 0)
    return lib


def _call(fn, a, b, c, alpha, beta, cfg, stream):
    M, K = a.shape
    N = b.shape[1]
    return fn(M, N, K, alpha, a.data_ptr(), K, b.data_ptr(), N, beta, c.data_ptr(), N,
              CODE[a.dtype], CODE[c.dtype], 0, stream.cuda_stream, cfg)


def _check_plan(g, M, N, K, idt, odt, cfg):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, p = g.gemm_plan(M, N, K, CODE[idt], CODE[odt], 0, sms, cfg)
    assert s == g.GEMM_OK and (p.sk_iters > 0 or p.tile_split > 0), \
        "case does not use the scratch"
    assert 0 < p.scratch_bytes <= g.GEMM_NOALLOC_SCRATCH_BYTES


def _noalloc_twice(g, a, b, c0, alpha, beta, cfg):
    """Two gemm_ex_noalloc calls in a row on a fresh stream, after a warm-up call
    on another fresh stream (the first call on a device does the one-time set-up,
    and lazily loaded kernel code is allocated when a kernel first runs).
    Returns the two outputs and asserts that nothing was allocated."""
    outs = [c0.clone(), c0.clone()]
    warm = c0.clone()
    ws, st = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    assert _call(g.gemm_ex_noalloc, a, b, warm, alpha, beta, cfg, ws) == g.GEMM_OK
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for c in outs:
        assert _call(g.gemm_ex_noalloc, a, b, c, alpha, beta, cfg, st) == g.GEMM_OK
    torch.cuda.synchronize()
    free1, reserved1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    s, site = g.gemm_sync_status(st.cuda_stream)
    assert s == g.GEMM_OK, f"kernel status {s} site {site}"
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert reserved1 == reserved0
    assert torch.equal(warm, outs[0])
    return outs


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-" +
                         "-".join(f"{k}{v}" for k, v in c[3].items()))
def test_noalloc_matches_gemm_ex_twice(g, case):
    M, N, K, cfg, idt, odt, alpha, beta = case
    _check_plan(g, M, N, K, idt, odt, cfg)
    gen = torch.Generator(device="cuda").manual_seed(M + N + K)
    a = (torch.rand(M, K, device="cuda", generator=gen) * 2 - 1).to(idt)
    b = (torch.rand(K, N, device="cuda", generator=gen) * 2 - 1).to(idt)
    c0 = (torch.rand(M, N, device="cuda", generator=gen) * 2 - 1).to(odt)

    ref = c0.clone()
    cur = torch.cuda.current_stream()
    assert _call(g.gemm_ex, a, b, ref, alpha, beta, cfg, cur) == g.GEMM_OK
    torch.cuda.synchronize()
    for c in _noalloc_twice(g, a, b, c0, alpha, beta, cfg):
        assert torch.isfinite(c.float()).all()
        assert torch.equal(c, ref), "gemm_ex_noalloc differs from gemm_ex"


@pytest.mark.parametrize("order", [0, ORDER_HILBERT], ids=["grouped", "hilbert"])
def test_noalloc_integer_bit_exact_against_oracle(g, order):
    """Integer inputs in {-4..4}: every product and fp32 partial sum is exact, so
    the output is unique and must equal the oracle's bits, whatever the tile
    order or stream-K split."""
    M = N = K = 2048
    cfg = {"stream_k": 2, "cta_group": 2, "order": order}
    _check_plan(g, M, N, K, torch.float16, torch.float32, cfg)
    A = si.matrix("int", 1000 + 71, M, K, "f16")
    B = si.matrix("int", 2000 + 71, K, N, "f16")
    a, b = to_device(A, "f16"), to_device(B, "f16")
    c0 = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)

    ref = c0.clone()
    assert _call(g.gemm_ex, a, b, ref, 1.0, 0.0, cfg, torch.cuda.current_stream()) == g.GEMM_OK
    torch.cuda.synchronize()
    outs = _noalloc_twice(g, a, b, c0, 1.0, 0.0, cfg)
    obits, _, _ = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32")
    assert np.array_equal(to_bits(ref, "f32"), obits)
    for c in outs:
        assert torch.equal(c, ref)
        assert np.array_equal(to_bits(c, "f32"), obits), "gemm_ex_noalloc differs from the oracle"
