"""Specialised kernel instances (the plain path -- beta == 0, no bias or activation,
grouped tiles, data-parallel or with a stream-K tail on the CTA pair, a ragged
right edge only on single CTAs of width 64 or 128 -- with the operand layout fixed
at compile time) against the general kernel and the oracle.  The same call with
gemm_config_t.general = 0 and = 1 must give identical bits, and integer inputs
must match the oracle exactly, in every layout and every configuration that has
specialised instances."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import check_against_oracle, operands, pad8, run_library

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]
# (config, M, N, K): several tiles, ragged M and K (N * 4 and N * 2 bytes stay
# multiples of 16, so the calls stay on the plain path)
CASES = [({"cta_group": 2, "bn": 256}, 520, 776, 456),
         ({"cta_group": 2, "bn": 256, "stream_k": 2}, 1032, 1288, 1000),
         ({"cta_group": 1, "split_k": 2, "bn": 128}, 200, 392, 648),
         ({"cta_group": 1, "split_k": 2, "bn": 64}, 136, 328, 520),
         ({"cta_group": 1, "bn": 64}, 300, 200, 200),
         ({"cta_group": 1, "bn": 128}, 136, 520, 392),
         ({"cta_group": 1, "split_k": 4, "bn": 128}, 120, 392, 1096),
         ({"cta_group": 1, "split_k": 4, "bn": 64}, 72, 200, 1096),
         ({"cta_group": 1, "split_k": 2, "bn": 256}, 130, 776, 648),
         ({"cta_group": 1, "split_k": 8, "bn": 128}, 40, 264, 1096)]
CASE_IDS = ["pair256", "pair256-streamk", "splitk2-bn128", "splitk2-bn64", "cta1-bn64", "cta1-bn128",
            "splitk4-bn128", "splitk4-bn64", "splitk2-bn256", "splitk8-bn128"]
# single CTAs whose right edge is ragged for every output format (N * 2 bytes not
# a multiple of 16): their own specialised instances keep the predicated edge
# stores and fold everything else
RAGGED_CASES = [({"cta_group": 1, "bn": 64}, 73, 61, 67), ({"cta_group": 1, "bn": 64}, 257, 263, 251),
                ({"cta_group": 1, "bn": 128}, 136, 517, 392), ({"cta_group": 1, "bn": 64}, 17, 65, 19)]
RAGGED_IDS = ["bn64-73x61x67", "bn64-257x263x251", "bn128-136x517x392", "bn64-17x65x19"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


def _layout(a_col, b_col):
    return (1 if a_col else 0) | (2 if b_col else 0)


@pytest.mark.parametrize("case", CASES + RAGGED_CASES, ids=CASE_IDS + RAGGED_IDS)
@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("in_dtype,out_dtype", [("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_specialised_matches_general_and_oracle(_lib, case, a_col, b_col, in_dtype, out_dtype):
    g = _lib
    cfg, M, N, K = case
    codes = {"f16": 0, "bf16": 1, "f32": 2}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, p = g.gemm_plan(M, N, K, codes[in_dtype], codes[out_dtype], _layout(a_col, b_col), sms, cfg)
    assert s == 0 and p.specialised == 1, p.as_dict()
    s, p = g.gemm_plan(M, N, K, codes[in_dtype], codes[out_dtype], _layout(a_col, b_col), sms,
                       dict(cfg, general=1))
    assert s == 0 and p.specialised == 0
    A, B = operands(M, N, K, in_dtype, a_col, b_col, dist="int", seed=M + K, pad=True)
    spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                          a_col=a_col, b_col=b_col, cfg=cfg, ldc=pad8(N))
    gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                         a_col=a_col, b_col=b_col, cfg=dict(cfg, general=1), ldc=pad8(N))
    np.testing.assert_array_equal(spec, gen)
    check_against_oracle(spec, A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                         a_col=a_col, b_col=b_col, exact=True)


@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_specialised_normal_inputs_identical_to_general(_lib, case):
    """Non-integer inputs: the two kernels sum in the same order, so the fp32
    results agree bit for bit (and with alpha != 1)."""
    cfg, M, N, K = case
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=N)
    spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                          b_col=True, alpha=0.375, cfg=cfg)
    gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, alpha=0.375, cfg=dict(cfg, general=1))
    np.testing.assert_array_equal(spec, gen)
    check_against_oracle(spec, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, alpha=0.375)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_specialised_fp8(_lib, fmt, case):
    g = _lib
    cfg, M, N, K = case
    ldk = (K + 15) // 16 * 16
    A = si.matrix("int", 1000 + K, M, K, fmt, 1.0, ld=ldk)
    B = si.matrix("int", 2000 + K, N, K, fmt, 1.0, ld=ldk)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    code = {"e4m3": 3, "e5m2": 4}[fmt]
    s, p = g.gemm_plan(M, N, K, code, 2, 2, sms, cfg)
    assert s == 0 and p.specialised == 1
    spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32", a_col=False,
                          b_col=True, cfg=cfg, ldc=pad8(N))
    gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32", a_col=False,
                         b_col=True, cfg=dict(cfg, general=1), ldc=pad8(N))
    np.testing.assert_array_equal(spec, gen)
    check_against_oracle(spec, A, B, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32", a_col=False,
                         b_col=True, exact=True)


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("streamk", [False, True], ids=["dp", "streamk"])
def test_specialised_beta(_lib, a_col, b_col, out_dtype, streamk):
    """The CTA pair's C-reading instances (data-parallel, and with a stream-K
    tail, where only the item finishing a tile takes beta * C): exact on
    integers, and the same bits as the general kernel."""
    M, N, K = (1032, 1288, 1000) if streamk else (520, 776, 456)
    cfg = {"cta_group": 2, "bn": 256, "stream_k": 2} if streamk else {"cta_group": 2, "bn": 256}
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=N + K, pad=True)
    C = si.matrix("int", 77, M, pad8(N), out_dtype)
    for beta in (1.0, -2.0):
        spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                              a_col=a_col, b_col=b_col, beta=beta, C=C, cfg=cfg, ldc=pad8(N))
        gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                             a_col=a_col, b_col=b_col, beta=beta, C=C, cfg=dict(cfg, general=1),
                             ldc=pad8(N))
        np.testing.assert_array_equal(spec, gen)
        check_against_oracle(spec, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                             a_col=a_col, b_col=b_col, beta=beta, C=C, exact=True)


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("mode", [{"cta_group": 2, "bn": 256},
                                  {"cta_group": 2, "bn": 256, "stream_k": 2},
                                  {"cta_group": 1, "bn": 64}, {"cta_group": 1, "bn": 128},
                                  {"cta_group": 1, "split_k": 2, "bn": 128},
                                  {"cta_group": 1, "split_k": 2, "bn": 64}],
                         ids=["dp", "streamk", "cta1-bn64", "cta1-bn128", "splitk2-bn128",
                              "splitk2-bn64"])
def test_specialised_fused_epilogue(_lib, a_col, b_col, mode):
    """The fused-epilogue instances (bias per column or row, with and without
    ReLU) of the CTA pair, the single CTA and the 2-way split-K cluster: exact on
    integers and identical to the general kernel."""
    M, N, K = ((1032, 1288, 1000) if "stream_k" in mode else
               (120, 776, 1096) if "split_k" in mode else (520, 776, 456))
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=M + 3, pad=True)
    rng = np.random.default_rng(N)
    for kind in ("col", "row"):
        bias = rng.integers(-40, 41, size=N if kind == "col" else M).astype(np.float32)
        for relu in (False, True):
            spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                                  a_col=a_col, b_col=b_col, cfg=mode, ldc=pad8(N), bias=bias,
                                  bias_kind=kind, relu=relu)
            gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                                 a_col=a_col, b_col=b_col, cfg=dict(mode, general=1), ldc=pad8(N),
                                 bias=bias, bias_kind=kind, relu=relu)
            np.testing.assert_array_equal(spec, gen)
            check_against_oracle(spec, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                                 a_col=a_col, b_col=b_col, exact=True, bias=bias,
                                 bias_kind=kind, relu=relu)


def test_workload_2048_specialised(_lib):
    """The 2048^3 fp16 -> fp32 workload runs a specialised instance; same bits as
    the general kernel."""
    g = _lib
    M = N = K = 2048
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, p = g.gemm_plan(M, N, K, 0, 2, 0, sms)
    assert s == 0 and p.specialised == 1
    A, B = operands(M, N, K, "f16", False, False, dist="uniform", seed=5)
    spec, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32", a_col=False,
                          b_col=False)
    gen, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32", a_col=False,
                         b_col=False, cfg={"general": 1})
    np.testing.assert_array_equal(spec, gen)
