"""GPU parity: the tcgen05 GEMM (called through the C ABI) against the CPU oracle.

Bar: bit-exact on integer inputs in {-4..4} (every product and fp32 partial sum
is exact, so any summation order gives the same value), and otherwise
|C_gpu - C_oracle| <= tol * sum_k |a_ik||b_kj| + 1e-6 with tol 1e-3 for fp32
output and 8e-3 for bf16/fp16 output.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import (check_against_oracle, operands, pad8, run_library, sample_rows, to_device,
                      to_bits)

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


# ------------------------------------------------------------ single-tile probes
# One CTA tile with operands whose every output is a single exact product:
# identity and permutation matrices move unique values to known places, so a
# wrong shared-memory descriptor, swizzle, TMEM lane/column map or operand major
# shows up as a misplaced value (checked by exact equality).

MODES = [{"cta_group": 1}, {"cta_group": 2}]
# every way the kernel can split the work: single CTA, CTA pair, split-K clusters
ALL_MODES = [{"cta_group": 1}, {"cta_group": 2}, {"split_k": 2}, {"split_k": 4},
             {"cta_group": 1, "stream_k": 2}, {"cta_group": 2, "stream_k": 2}, {"stream_k": 3}]
MODE_IDS = ["cta1", "pair", "splitk2", "splitk4", "streamk1", "streamk2", "splittile2"]


def _mode_fits(mode, K, M=1, N=1):
    """Whether the mode can run this shape: enough k-blocks (split-K) or k-groups
    (split-tile) for its parts, and split-tile units within the SM count."""
    if mode.get("stream_k") == 3:
        parts, bn = mode.get("split_k", 2), mode.get("bn", 128)
        tiles = ((M + 127) // 128) * ((N + bn - 1) // bn)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        return (K + 127) // 128 >= parts and tiles * parts <= sms
    return (K + 63) // 64 >= mode.get("split_k", 1)


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("mode", ALL_MODES, ids=MODE_IDS)
def test_probe_identity_left(a_col, b_col, in_dtype, mode):
    M, N, K = 128 * mode.get("cta_group", 1), 256, 256
    eye = si.to_bits(np.eye(M, K, dtype=np.float32), in_dtype)
    A = np.ascontiguousarray(eye.T) if a_col else eye
    Bv = si.normal(77, K * N, 1.0).reshape(K, N)
    Bl = si.to_bits(Bv, in_dtype)
    B = np.ascontiguousarray(Bl.T) if b_col else Bl
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype="f32",
                         a_col=a_col, b_col=b_col, cfg=dict(mode, bn=256))
    np.testing.assert_array_equal(oracle.decode(out, "f32"), oracle.decode(Bl, in_dtype)[:M])


PROBE_CFGS = [{"bn": 64}, {"bn": 128}, {"bn": 256}, {"bn": 128, "cta_group": 2},
              {"bn": 256, "cta_group": 2}, {"bn": 128, "split_k": 2}, {"bn": 256, "split_k": 2},
              {"bn": 256, "split_k": 4}, {"bn": 128, "split_k": 4}, {"bn": 128, "split_k": 8},
              {"bn": 64, "split_k": 2}, {"bn": 64, "split_k": 4}]


@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("cfg", PROBE_CFGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_probe_permutations(a_col, b_col, cfg):
    """A = P (rows pick unique-valued rows of B): every output is one exact product,
    so a misplaced operand row/column or accumulator lane/column is caught."""
    bn, cta_group = cfg["bn"], cfg.get("cta_group", 1)
    M, N, K = 128 * cta_group, bn, 64 * cfg.get("split_k", 1)
    rng = np.random.default_rng(bn + 7 * a_col + 13 * b_col)
    P = np.zeros((M, K), np.float32)
    rows = rng.integers(0, K, size=M)
    P[np.arange(M), rows] = 1.0
    Bv = (np.arange(K * N, dtype=np.float32).reshape(K, N) % 2039) - 1019.0  # exact in fp16
    Al = si.to_bits(P, "f16")
    Bl = si.to_bits(Bv, "f16")
    A = np.ascontiguousarray(Al.T) if a_col else Al
    B = np.ascontiguousarray(Bl.T) if b_col else Bl
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=a_col, b_col=b_col, cfg=cfg)
    np.testing.assert_array_equal(oracle.decode(out, "f32"), Bv[rows])


# ------------------------------------------------------------ the five workloads

def _workload(cfg, integer, scale=1):
    return si.workload_operands(cfg, integer=integer, scale=scale)


def _run_w(w, ldc=None, cfg=None):
    return run_library(w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"], in_dtype=w["in_dtype"],
                       out_dtype=w["out_dtype"], a_col=w["a_col"], b_col=w["b_col"],
                       alpha=w["alpha"], beta=w["beta"], C=w["C"], ldc=ldc, cfg=cfg)


def _check_w(w, out, rows=None, exact=False, strict=False):
    return check_against_oracle(out, w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"],
                                in_dtype=w["in_dtype"], out_dtype=w["out_dtype"],
                                a_col=w["a_col"], b_col=w["b_col"], alpha=w["alpha"],
                                beta=w["beta"], C=w["C"], rows=rows, exact=exact,
                                strict=strict)


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_workload_integer_bit_exact_full(cfg):
    w = _workload(cfg, integer=True)
    out, _ = _run_w(w)
    _check_w(w, out, exact=True)


@pytest.mark.parametrize("mode", ALL_MODES, ids=MODE_IDS)
def test_workload2_integer_bit_exact_each_mode(mode):
    if not _mode_fits(mode, 2048, 2048, 2048):
        pytest.skip("more split-tile units than SMs")
    w = _workload(2, integer=True)
    out, _ = _run_w(w, cfg=mode)
    _check_w(w, out, exact=True)


@pytest.mark.parametrize("mode", [{"cta_group": 1, "bn": 64}, {"split_k": 2}, {"split_k": 4},
                                  {"split_k": 2, "bn": 128}, {"stream_k": 3},
                                  {"stream_k": 3, "split_k": 4, "bn": 256}],
                         ids=["bn64", "splitk2", "splitk4", "splitk2-bn128", "splittile2",
                              "splittile4-bn256"])
def test_workload5_skinny_integer_each_mode(mode):
    w = _workload(5, integer=True)
    out, _ = _run_w(w, cfg=mode)
    _check_w(w, out, exact=True)


def _check_w_blocks(w, out, exact=False, block=1024, strict=False):
    """Every element, in blocks of rows (bounded host memory for the oracle's
    binary64 results at 8192^3)."""
    for r0 in range(0, w["M"], block):
        _check_w(w, out, rows=list(range(r0, min(w["M"], r0 + block))), exact=exact,
                 strict=strict)


def test_workload4_integer_bit_exact_full():
    """8192^3 bf16 -> fp32 with beta = 0.5 on integer inputs (C_in integer too, so
    beta * c is exact): every element equals the oracle's bits."""
    w = _workload(4, integer=True)
    out, _ = _run_w(w)
    _check_w_blocks(w, out, exact=True)


@pytest.mark.parametrize("cfg", [3, 4])
def test_workload_normal_tolerance_full(cfg):
    """4096^3 bf16 -> bf16 and 8192^3 bf16 -> fp32 (beta 0.5) on their normal
    draws: every element within the error bound of its output format, as stated
    (no extra allowance for the fp32 rounding of beta * C)."""
    w = _workload(cfg, integer=False)
    out, _ = _run_w(w)
    _check_w_blocks(w, out, strict=True)


def test_workload4_integer_bit_exact_sampled():
    w = _workload(4, integer=True)
    out, _ = _run_w(w)
    _check_w(w, out, rows=sample_rows(w["M"], 40), exact=True)


@pytest.mark.parametrize("cfg", [1, 2])
def test_workload_uniform_tolerance_full(cfg):
    w = _workload(cfg, integer=False)
    out, _ = _run_w(w)
    _check_w(w, out, strict=True)


@pytest.mark.parametrize("cfg", [3, 4])
def test_workload_normal_tolerance_sampled(cfg):
    w = _workload(cfg, integer=False)
    out, _ = _run_w(w)
    _check_w(w, out, rows=sample_rows(w["M"], 48, seed=cfg))


def test_workload5_skinny_tolerance_full():
    w = _workload(5, integer=False)
    out, _ = _run_w(w)
    _check_w(w, out, strict=True)


@pytest.mark.parametrize("cfg", [1, 3, 4, 5])
def test_workload_reduced_size_every_element(cfg):
    """The same recipe at a size the oracle checks completely (several tiles)."""
    w = _workload(cfg, integer=False, scale=8 if cfg != 1 else 1)
    out, _ = _run_w(w)
    _check_w(w, out)


# ------------------------------------------------------------ shapes, layouts, formats

ODD_SHAPES = [(257, 263, 251), (31, 29, 37), (17, 65, 19), (73, 61, 67), (1, 1, 1),
              (129, 257, 65), (300, 520, 1000)]


@pytest.mark.parametrize("shape", ODD_SHAPES)
@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
@pytest.mark.parametrize("mode", ALL_MODES, ids=MODE_IDS)
def test_odd_shapes_integer_exact(shape, a_col, b_col, mode):
    M, N, K = shape
    if not _mode_fits(mode, K, M, N):
        pytest.skip("fewer k-blocks than splits")
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=M + N + K, pad=True)
    ldc = pad8(N) + 8
    out, full = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                            a_col=a_col, b_col=b_col, ldc=ldc, cfg=mode)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=a_col, b_col=b_col, exact=True)
    # guard columns of C (beyond N) untouched: still the NaN poison
    assert np.all(full[:, N:] == 0x7FC00000)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cfg", PROBE_CFGS, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_formats_and_tile_widths(out_dtype, in_dtype, cfg):
    M, N, K = 300, 520, 333
    if not _mode_fits(cfg, K):
        K = 64 * cfg["split_k"] + 13   # enough k-blocks for every split, still ragged
    A, B = operands(M, N, K, in_dtype, False, False, dist="uniform", seed=cfg["bn"], pad=True)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                         a_col=False, b_col=False, cfg=cfg, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                         a_col=False, b_col=False)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.5), (-2.0, 1.0), (0.5, -1.0)])
@pytest.mark.parametrize("mode", ALL_MODES, ids=MODE_IDS)
def test_alpha_beta(out_dtype, alpha, beta, mode):
    M, N, K = 512, 384, 320
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=3)
    C = si.matrix("int", 3003, M, N, out_dtype)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=alpha, beta=beta, C=C, cfg=mode)
    # integer inputs and power-of-two alpha/beta keep alpha*acc + beta*c exact in
    # fp32, so both sides round the same exact value once: bit-exact for every format
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=alpha, beta=beta, C=C, exact=True)


@pytest.mark.parametrize("K", [32, 256, 4096])
def test_k_sweep_64x64(K):
    """The leetllm lab's M = N = 64 K-sweep, against the rounded-input reference."""
    A, B = operands(64, 64, K, "f16", False, False, dist="uniform", seed=K)
    out, _ = run_library(A, B, M=64, N=64, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=False, b_col=False)
    check_against_oracle(out, A, B, M=64, N=64, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=False, b_col=False)


@pytest.mark.parametrize("K", [32, 256, 4096])
def test_k_sweep_64x64_against_both_references(K):
    """The lab's K-sweep against its two references ("The two-reference testing
    protocol"): the rounded-input oracle (the gate) and the original fp32 draws.
    The second differs from the first by the fp16 rounding of the inputs, at most
    (2u + u^2) sum_k |a_ik||b_kj| with u = 2^-11, whatever K is."""
    M = N = 64
    A, B = operands(M, N, K, "f16", False, False, dist="uniform", seed=K)
    a0 = si.draw("uniform", 1000 + K, M * K, 1.0).reshape(M, K).astype(np.float64)
    b0 = si.draw("uniform", 2000 + K, K * N, 1.0).reshape(K, N).astype(np.float64)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=False, b_col=False)
    gv = oracle.decode(out, "f32")
    _, exact, scale = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32")
    err_rounded = np.abs(gv - exact)
    assert np.all(err_rounded <= 1e-3 * scale + 1e-6)
    err_original = np.abs(gv - a0 @ b0)
    u = 2.0 ** -11
    assert np.all(err_original <= err_rounded + (2 * u + u * u) * (np.abs(a0) @ np.abs(b0)) + 1e-9)


# ------------------------------------------------------------ stream-K

SK_CASES = [
    (1024, 1024, 2048, {"stream_k": 2, "cta_group": 2}),
    (1024, 1024, 2048, {"stream_k": 2, "cta_group": 1}),
    (1000, 1100, 1500, {"stream_k": 2, "cta_group": 2}),
    (1000, 1100, 1500, {"stream_k": 2, "cta_group": 1, "bn": 128}),
    (2048, 1536, 1024, {"stream_k": 2, "cta_group": 1, "grid": 20}),   # 2 data-parallel waves + stream-K
    (2048, 1536, 1024, {"stream_k": 2, "cta_group": 2, "grid": 22}),   # 11 pairs
    (640, 2304, 4096, {"stream_k": 2, "cta_group": 1, "bn": 64}),
]


def _assert_stream_k(M, N, K, cfg, layout=0):
    import dense_tensor_core_tcgen05_gb300 as g
    s, p = g.gemm_plan(M, N, K, g.GEMM_BF16, g.GEMM_F32, layout, torch.cuda.get_device_properties(0).multi_processor_count, cfg)
    assert s == 0 and p.sk_iters > 0, "case does not exercise stream-K"


@pytest.mark.parametrize("case", SK_CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-" + "-".join(f"{k}{v}" for k, v in c[3].items()))
@pytest.mark.parametrize("a_col,b_col", [(False, False), (False, True), (True, True)])
def test_stream_k_integer_exact(case, a_col, b_col):
    M, N, K, cfg = case
    _assert_stream_k(M, N, K, cfg, (1 if a_col else 0) | (2 if b_col else 0))
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=M + K, pad=True)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=a_col,
                         b_col=b_col, cfg=cfg, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=a_col, b_col=b_col, exact=True)


@pytest.mark.parametrize("case", SK_CASES[:4], ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-cta{c[3]['cta_group']}")
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_stream_k_uniform_beta(case, out_dtype):
    M, N, K, cfg = case
    _assert_stream_k(M, N, K, cfg)
    A, B = operands(M, N, K, "f16", False, True, dist="uniform", seed=K, pad=True)
    C = si.matrix("uniform", 3000 + K, M, N, out_dtype)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype=out_dtype, a_col=False,
                         b_col=True, alpha=0.75, beta=-0.5, C=C, cfg=cfg, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=0.75, beta=-0.5, C=C)


def test_stream_k_deterministic_and_repeated():
    """Stream-K partials are added in a fixed order: repeated launches (epochs
    advancing on the same scratch) give bitwise-identical results."""
    M, N, K, cfg = SK_CASES[0]
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=11)
    outs = [run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                        b_col=True, cfg=cfg)[0] for _ in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    check_against_oracle(outs[0], A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, rows=sample_rows(M, 40))


# ------------------------------------------------------------ edge cases

def test_k_zero_scales_c(_lib):
    g = _lib
    M, N = 70, 96
    for out_dtype, tdt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        c = torch.arange(M * N, device="cuda", dtype=torch.float32).reshape(M, N).to(tdt)
        ref = (c.float() * 0.5).to(tdt)
        a = torch.empty(M, 0, device="cuda", dtype=torch.float16)
        b = torch.empty(0, N, device="cuda", dtype=torch.float16)
        g.matmul(a, b, c, alpha=1.0, beta=0.5)
        torch.cuda.synchronize()
        assert torch.equal(c, ref)
        c2 = torch.full((M, N), float("nan"), device="cuda", dtype=tdt)
        g.matmul(a, b, c2, alpha=1.0, beta=0.0)
        torch.cuda.synchronize()
        assert torch.equal(c2, torch.zeros_like(c2))


def test_empty_m_or_n_is_noop(_lib):
    g = _lib
    a = torch.ones(0, 64, device="cuda", dtype=torch.bfloat16)
    b = torch.ones(64, 32, device="cuda", dtype=torch.bfloat16)
    c = torch.empty(0, 32, device="cuda", dtype=torch.float32)
    g.matmul(a, b, c)
    a2 = torch.ones(16, 64, device="cuda", dtype=torch.bfloat16)
    b2 = torch.ones(64, 0, device="cuda", dtype=torch.bfloat16)
    c2 = torch.empty(16, 0, device="cuda", dtype=torch.float32)
    g.matmul(a2, b2, c2)
    torch.cuda.synchronize()


def test_beta_zero_ignores_nan_in_c():
    # run_library poisons C with NaN; beta = 0 output must be finite and correct
    M, N, K = 200, 300, 100
    A, B = operands(M, N, K, "f16", False, False, dist="int", seed=9, pad=True)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=False, b_col=False, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                         a_col=False, b_col=False, exact=True)


def test_deterministic_bitwise():
    w = _workload(3, integer=False, scale=2)
    o1, _ = _run_w(w)
    o2, _ = _run_w(w)
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("grid,group_m,cta_group", [(1, 1, 1), (7, 3, 1), (152, 16, 1),
                                                    (300, 2, 1), (2, 1, 2), (6, 3, 2),
                                                    (152, 8, 2)])
def test_persistent_grid_and_group_override(grid, group_m, cta_group):
    """Every CTA count (one CTA or one pair doing every tile, fewer CTAs than
    tiles) and tile order gives the same exact result."""
    M, N, K = 640, 768, 320
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=grid)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, cfg={"bn": 128, "grid": grid, "group_m": group_m,
                                          "cta_group": cta_group})
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, exact=True)


def test_host_entry_point_e2e(_lib):
    """gemm_host: host operands in, host result out, through the C ABI."""
    g = _lib
    M, N, K = 384, 512, 256
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=21)
    hA = torch.from_numpy(A.view(np.int16).copy()).pin_memory()
    hB = torch.from_numpy(B.view(np.int16).copy()).pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    dA = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    dC = torch.empty(M, N, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    s = g.gemm_host(M, N, K, 1.0, hA.data_ptr(), K, hB.data_ptr(), K, 0.0, hC.data_ptr(), N,
                    g.GEMM_BF16, g.GEMM_F32, g.GEMM_B_COL, dA.data_ptr(), dB.data_ptr(),
                    dC.data_ptr(), st)
    assert s == g.GEMM_OK
    assert g.gemm_sync_status(st)[0] == g.GEMM_OK
    out = hC.numpy().view(np.uint32)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True, exact=True)


@pytest.mark.parametrize("a_col,b_col,beta", [(False, True, 0.5), (True, False, 0.0)])
def test_host_entry_point_pipelined(_lib, a_col, b_col, beta):
    """gemm_host on a problem large enough for its row-panel pipeline (5 panels,
    the last one ragged; copies on internal streams overlapping the panels'
    GEMMs): every element exact against the oracle, C read when beta != 0."""
    g = _lib
    M, N, K = 2148, 4096, 4096
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=23, pad=True)
    C = si.matrix("int", 91, M, N, "f32")
    hA = torch.from_numpy(A.view(np.int16).copy()).pin_memory()
    hB = torch.from_numpy(B.view(np.int16).copy()).pin_memory()
    init = C.view(np.float32) if beta != 0.0 else np.full((M, N), np.nan, np.float32)
    hC = torch.from_numpy(np.ascontiguousarray(init)).pin_memory()
    dA = torch.empty(A.shape, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(B.shape, dtype=torch.bfloat16, device="cuda")
    dC = torch.empty(M, N, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    layout = (g.GEMM_A_COL if a_col else 0) | (g.GEMM_B_COL if b_col else 0)
    s = g.gemm_host(M, N, K, 1.0, hA.data_ptr(), A.shape[1], hB.data_ptr(), B.shape[1], beta,
                    hC.data_ptr(), N, g.GEMM_BF16, g.GEMM_F32, layout, dA.data_ptr(),
                    dB.data_ptr(), dC.data_ptr(), st)
    assert s == g.GEMM_OK
    assert g.gemm_sync_status(st)[0] == g.GEMM_OK
    out = hC.numpy().view(np.uint32)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=a_col, b_col=b_col, beta=beta, C=C if beta != 0.0 else None,
                         exact=True)


def test_device_checks_on_gpu(_lib):
    g = _lib
    a = torch.ones(64, 64, device="cuda", dtype=torch.float16)
    c = torch.ones(64, 64, device="cuda", dtype=torch.float32)
    st = torch.cuda.current_stream().cuda_stream
    # misaligned pointer -> unsupported, nothing launched
    s = g.gemm(64, 64, 64, 1.0, a.data_ptr() + 2, 64, a.data_ptr(), 64, 0.0, c.data_ptr(), 64,
               g.GEMM_F16, g.GEMM_F32, 0, st)
    assert s == g.GEMM_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        g.matmul(a.cpu(), a.cpu(), c.cpu())


# ------------------------------------------------------------ bounded waits

# plus the two-CTA split-K clusters whose slices are exchanged early (each warp
# sends its rows as soon as they are staged, and after an abort all the same)
TIMEOUT_MODES = ALL_MODES + [{"split_k": 2, "bn": 128}, {"split_k": 2, "bn": 64}]
TIMEOUT_IDS = MODE_IDS + ["splitk2-bn128-early", "splitk2-bn64-early"]


@pytest.mark.parametrize("mode", TIMEOUT_MODES, ids=TIMEOUT_IDS)
def test_wait_timeout_is_reported_and_context_survives(_lib, mode):
    """The producer leaves one ring slot unarmed (host-set debug flag): the MMA
    issuer's wait must run out, the kernel must record the timeout and return,
    and the device must stay usable."""
    g = _lib
    M, N, K = 512, 256, 2048   # every mode gets >= 3 ring stages per CTA
    A, B = operands(M, N, K, "bf16", False, False, dist="int", seed=5)
    try:
        g.gemm_debug_set(50_000_000, 3)   # 50 ms limit; skip ring iteration 2
        dA = to_device(A, "bf16")
        dB = to_device(B, "bf16")
        c = torch.zeros(M, N, device="cuda", dtype=torch.float32)
        g.matmul(dA, dB, c, cfg=mode)
        s, site = g.gemm_sync_status(torch.cuda.current_stream().cuda_stream)
        assert s == g.GEMM_ERR_TIMEOUT
        # with partial sums in play an owner's wait for a contributor's flag
        # (site 7) may run out before its MMA issuer's wait does
        assert site in ((2, 3, 4, 1, 7) if mode.get("stream_k") else (2, 3, 4, 1))
    finally:
        g.gemm_debug_set(0, 0)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=False, cfg=mode)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=False, exact=True)
