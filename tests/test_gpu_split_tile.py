"""GPU parity of the split-tile schedule (gemm_config_t.stream_k = 3): every
tile's k-groups split over several one-CTA units without a cluster, the first
unit (the larger share) finishing the tile from the others' partial sums, which
it loads into its spare TMEM accumulator while its own MMAs run.

Bar as everywhere: bit-exact against the oracle on integer inputs, the error
bound otherwise, and identical bits from run to run (the partials are added in
a fixed order).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import check_against_oracle, operands, pad8, run_library

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (False, True), (True, False), (True, True)]

# (M, N, K, cfg): single 128-row panels of the decode and skinny kind, a ragged
# panel (M < 128: only ceil8(M) rows of A copied), several panels, and every
# tile width and part count the plan accepts
CASES = [
    (128, 2048, 4096, {"stream_k": 3}),
    (77, 1000, 3000, {"stream_k": 3}),
    (16, 4096, 8192, {"stream_k": 3, "bn": 128}),
    (1, 2048, 4096, {"stream_k": 3, "split_k": 8}),
    (128, 4096, 2048, {"stream_k": 3, "split_k": 4, "bn": 256}),
    (300, 700, 2000, {"stream_k": 3, "split_k": 3, "bn": 64}),
    (200, 520, 260, {"stream_k": 3, "split_k": 2, "bn": 64}),
]


def _ids(c):
    return f"{c[0]}x{c[1]}x{c[2]}-" + "-".join(f"{k}{v}" for k, v in c[3].items())


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    g.gemm_debug_set(0, 0)
    yield g


def _assert_split_tile(g, M, N, K, cfg, layout=0, in_dtype=1, out_dtype=2):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, p = g.gemm_plan(M, N, K, in_dtype, out_dtype, layout, sms, cfg)
    assert s == 0 and p.tile_split == cfg.get("split_k", 2), p.as_dict()
    assert p.grid == p.num_tiles * p.tile_split
    return p


@pytest.mark.parametrize("case", CASES, ids=_ids)
@pytest.mark.parametrize("a_col,b_col", LAYOUTS)
def test_split_tile_integer_exact(_lib, case, a_col, b_col):
    M, N, K, cfg = case
    _assert_split_tile(_lib, M, N, K, cfg, (1 if a_col else 0) | (2 if b_col else 0))
    A, B = operands(M, N, K, "bf16", a_col, b_col, dist="int", seed=M + N + K, pad=True)
    ldc = pad8(N) + 8
    out, full = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=a_col,
                            b_col=b_col, cfg=cfg, ldc=ldc)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=a_col, b_col=b_col, exact=True)
    assert np.all(full[:, N:] == 0x7FC00000)   # guard columns untouched


@pytest.mark.parametrize("case", CASES[:4] + CASES[5:6], ids=_ids)
@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_split_tile_uniform_alpha_beta(_lib, case, out_dtype):
    M, N, K, cfg = case
    A, B = operands(M, N, K, "f16", False, True, dist="uniform", seed=K, pad=True)
    C = si.matrix("uniform", 3000 + K, M, N, out_dtype)
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype=out_dtype, a_col=False,
                         b_col=True, alpha=0.75, beta=-0.5, C=C, cfg=cfg, ldc=pad8(N))
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype=out_dtype,
                         a_col=False, b_col=True, alpha=0.75, beta=-0.5, C=C)


@pytest.mark.parametrize("bias_kind", ["col", "row"])
def test_split_tile_fused_bias_relu_exact(_lib, bias_kind):
    M, N, K, cfg = CASES[1]
    A, B = operands(M, N, K, "bf16", False, True, dist="int", seed=9, pad=True)
    bias = np.random.default_rng(4100).integers(-40, 41, size=N if bias_kind == "col" else M)
    bias = bias.astype(np.float32)
    C = si.matrix("int", 3100, M, N, "f32")
    out, _ = run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, alpha=2.0, beta=0.5, C=C, cfg=cfg, ldc=pad8(N), bias=bias,
                         bias_kind=bias_kind, relu=True)
    check_against_oracle(out, A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                         b_col=True, alpha=2.0, beta=0.5, C=C, exact=True, bias=bias,
                         bias_kind=bias_kind, relu=True)


def test_split_tile_deterministic_and_repeated(_lib):
    """Repeated launches on the same scratch (the epoch advancing) give identical
    bits, and the same bits as the split-K cluster plan within the bound."""
    M, N, K, cfg = CASES[0]
    A, B = operands(M, N, K, "bf16", False, True, dist="normal", seed=21)
    outs = [run_library(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32", a_col=False,
                        b_col=True, cfg=cfg)[0] for _ in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    check_against_oracle(outs[0], A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                         a_col=False, b_col=True)


def test_split_tile_skinny_workload_full(_lib):
    """The 128 x 8192 x 8192 bf16 -> bf16 workload under the split-tile plan,
    every element against the oracle."""
    w = si.workload_operands(5)
    cfg = {"stream_k": 3}
    _assert_split_tile(_lib, w["M"], w["N"], w["K"], cfg, 2, 1, 1)
    out, _ = run_library(w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"], in_dtype=w["in_dtype"],
                         out_dtype=w["out_dtype"], a_col=w["a_col"], b_col=w["b_col"],
                         alpha=w["alpha"], beta=w["beta"], C=w["C"], cfg=cfg)
    check_against_oracle(out, w["A"], w["B"], M=w["M"], N=w["N"], K=w["K"],
                         in_dtype=w["in_dtype"], out_dtype=w["out_dtype"], a_col=w["a_col"],
                         b_col=w["b_col"], alpha=w["alpha"], beta=w["beta"], C=w["C"])
