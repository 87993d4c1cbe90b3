"""Host-side checks of the C-ABI library that need no GPU: the shared library
loads and exports every symbol the header declares, argument validation returns
the documented codes before touching CUDA, a valid call without a device fails
loudly (no CPU fallback), and the planner / tile order / descriptor encoders."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    from dense_tensor_core_tcgen05_gb300 import build as b
    b.build()
    import dense_tensor_core_tcgen05_gb300 as g
    return g


def _header_functions():
    text = open(os.path.join(ROOT, "include", "gemm_tcgen05.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", text)) -
                  {"if", "sizeof", "defined"})


def test_header_declares_what_binding_exports(g):
    assert _header_functions() == sorted(g.EXPORTS)


def test_library_exports_every_declared_symbol(g):
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _header_functions():
        assert name in syms, name
    lib = ctypes.CDLL(g.LIB_PATH)
    for name in _header_functions():
        assert getattr(lib, name) is not None


def test_header_compiles_as_c():
    src = '#include "gemm_tcgen05.h"\nint main(void){gemm_plan_t p; (void)p; return 0;}\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-", "-fsyntax-only"], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(g):
    for s in range(7):
        assert g.status_string(s) != "unknown status"
    assert g.status_string(99) == "unknown status"
    assert g.gemm_version() >= 100


ALIGNED = 1 << 20   # a fake 16-byte-aligned "pointer": validation never dereferences


@pytest.mark.parametrize("args,expected", [
    # M, N, K, lda, ldb, ldc, in, out, layout, A, B, C
    ((-1, 8, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),
    ((8, -1, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),
    ((8, 8, -1, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),
    ((8, 8, 8, 8, 8, 8, 2, 2, 0, ALIGNED, ALIGNED, ALIGNED), 2),      # fp32 inputs
    ((8, 8, 8, 8, 8, 8, 7, 2, 0, ALIGNED, ALIGNED, ALIGNED), 2),      # bad in dtype
    ((8, 8, 8, 8, 8, 8, 0, 5, 0, ALIGNED, ALIGNED, ALIGNED), 2),      # bad out dtype
    ((8, 8, 8, 8, 8, 8, 0, 2, 4, ALIGNED, ALIGNED, ALIGNED), 1),      # bad layout bits
    ((8, 16, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),     # ldc < N
    ((8, 8, 16, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),     # lda < K (A row)
    ((16, 8, 8, 8, 8, 8, 0, 2, 1, ALIGNED, ALIGNED, ALIGNED), 1),     # lda < M (A col)
    ((8, 16, 8, 8, 8, 16, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 1),    # ldb < N (B row)
    ((8, 8, 16, 16, 8, 8, 0, 2, 2, ALIGNED, ALIGNED, ALIGNED), 1),    # ldb < K (B col)
    ((8, 8, 8, 8, 8, 8, 0, 2, 0, 0, ALIGNED, ALIGNED), 1),            # NULL A
    ((8, 8, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, 0), 1),            # NULL C
    ((8, 8, 8, 8, 8, 8, 0, 2, 0, ALIGNED + 2, ALIGNED, ALIGNED), 2),  # misaligned A
    ((8, 8, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED + 8), 2),  # misaligned C
    ((8, 8, 12, 12, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 2),    # lda*2 not /16
    ((8, 6, 8, 8, 6, 6, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 2),      # ldc*4 not /16
    ((1 << 31, 8, 8, 8, 8, 8, 0, 2, 0, ALIGNED, ALIGNED, ALIGNED), 2),  # M >= 2^31
    ((0, 8, 8, 8, 8, 8, 0, 2, 0, 0, 0, 0), 0),                         # M == 0: no-op
    ((8, 0, 8, 8, 8, 8, 0, 2, 0, 0, 0, 0), 0),                         # N == 0: no-op
])
def test_argument_validation_codes(g, args, expected):
    M, N, K, lda, ldb, ldc, din, dout, layout, A, B, C = args
    assert g.gemm(M, N, K, 1.0, A, lda, B, ldb, 0.0, C, ldc, din, dout, layout, 0) == expected


def test_k_zero_does_not_need_a_or_b(g):
    # valid K == 0 call: passes validation with NULL A/B and then needs a device
    s = g.gemm(8, 8, 0, 1.0, 0, 0, 0, 0, 0.5, ALIGNED, 8, 0, 2, 0, 0)
    assert s in (g.GEMM_ERR_CUDA, g.GEMM_ERR_ARCH, g.GEMM_OK)


def test_no_cpu_fallback_without_device(g):
    """A well-formed call on a machine without a usable GB300 must fail with a CUDA
    or architecture error: the library has no CPU path."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    s = g.gemm(128, 128, 128, 1.0, ALIGNED, 128, ALIGNED, 128, 0.0, ALIGNED, 128, 0, 2, 0, 0)
    assert s == g.GEMM_ERR_CUDA
    # the host entry point too, on its single-panel path and on its row-panel
    # pipeline (>= 64 MiB over the link, M >= 2048): its first copy or stream
    # call fails before any buffer is touched, and the error comes back
    for M, N, K in ((128, 128, 128), (4096, 4096, 4096)):
        s = g.gemm_host(M, N, K, 1.0, ALIGNED, K, ALIGNED, N, 0.5, ALIGNED, N, 0, 2, 0,
                        ALIGNED, ALIGNED, ALIGNED, 0)
        assert s == g.GEMM_ERR_CUDA, (M, s)
    with pytest.raises(ValueError):
        g.matmul(torch.ones(4, 4, dtype=torch.float16), torch.ones(4, 4, dtype=torch.float16),
                 torch.ones(4, 4))


@pytest.mark.parametrize("shape,layout,expect", [
    # big squares: CTA-pair tiles of 256 x 256 (one cta_group::2 MMA over two SMs)
    # one wave of 64 pair tiles on 76 pairs: data-parallel, one tile per pair
    ((2048, 2048, 2048, 0, 2), 0, dict(cta_group=2, bm=256, bn=256, num_tiles=64, grid=128,
                                       k_blocks=32, b_mn=1, stages=3, bk=128, groups=16,
                                       dp_tiles=64, sk_iters=0, scratch_bytes=0)),
    # 3.37 waves, the last one 37% full: two data-parallel waves, the remaining
    # 104 tiles stream-K
    ((4096, 4096, 4096, 1, 1), 0, dict(cta_group=2, bn=256, num_tiles=256, grid=152,
                                       dp_tiles=152, sk_iters=104 * 32)),
    # 1.89 waves (under 2): data-parallel
    ((3072, 3072, 4096, 1, 1), 0, dict(cta_group=2, bn=256, num_tiles=144, grid=152,
                                       dp_tiles=144, sk_iters=0)),
    # 13.47 waves, the last one 47% full: 12 data-parallel waves, the remaining
    # 112 tiles stream-K
    ((8192, 8192, 8192, 1, 2), 2, dict(cta_group=2, bn=256, num_tiles=1024, grid=152, b_mn=0,
                                       dp_tiles=912, sk_iters=112 * 64)),
    # 7.58 waves, the last one 58% full: stream-K; 6.96 waves (the last one 96%
    # full, less than a quarter idle): data-parallel
    ((6144, 6144, 4096, 1, 1), 2, dict(cta_group=2, num_tiles=576, dp_tiles=6 * 76,
                                       sk_iters=(576 - 6 * 76) * 32)),
    ((5888, 5888, 4096, 1, 1), 2, dict(cta_group=2, num_tiles=529, dp_tiles=529, sk_iters=0)),
    # a single 128-row panel with long K: 128-wide tiles, K split over 2-CTA clusters
    ((128, 8192, 8192, 1, 1), 2, dict(cta_group=1, bm=128, bn=128, num_tiles=64, grid=128,
                                      k_blocks=128, stages=3, split_k=2)),
    # N too wide for 128-wide tiles in one wave: 256-wide, split 4
    ((128, 16384, 8192, 1, 1), 2, dict(cta_group=1, bn=256, num_tiles=64, split_k=2)),
    # a single panel with short K: no split (too few k-blocks per CTA)
    ((128, 8192, 256, 1, 1), 2, dict(cta_group=1, split_k=1)),
    ((257, 263, 251, 1, 2), 3, dict(cta_group=1, m_tiles=3, k_blocks=4, a_mn=1, b_mn=0)),
    ((512, 512, 512, 0, 2), 0, dict(cta_group=1, bn=64, num_tiles=32, grid=32)),
])
def test_plan(g, shape, layout, expect):
    M, N, K, din, dout = shape
    s, p = g.gemm_plan(M, N, K, din, dout, layout, 152)
    assert s == 0
    d = p.as_dict()
    for k, v in expect.items():
        assert d[k] == v, (k, d)
    assert d["smem_bytes"] <= 232448
    assert d["tmem_cols"] in (128, 256, 512)
    b_cols = d["bn"] // d["cta_group"]
    assert d["stages"] >= 2
    assert d["stages"] * (d["bk"] // 64) * (128 * 64 * 2 + b_cols * 64 * 2) <= 192 * 1024
    assert d["grid"] % d["cta_group"] == 0


@pytest.mark.parametrize("M,N,expect_sk", [
    (2816, 4864, True),    # 209 pair tiles: 2 waves + 57 (a quarter of 76 units idle)
    (3584, 3840, False),   # 210: 2 waves + 58 (fewer than a quarter idle)
    (2048, 4864, False),   # 152: exactly 2 waves, nothing to balance
    (2816, 3584, True),    # 154: 2 waves + 2
    (2048, 2048, False),   # 64: under 2 waves (every tile would be split)
])
def test_stream_k_rule_boundaries(g, M, N, expect_sk):
    """The planner's automatic stream-K tail: at least 2 waves of tiles and a last
    wave that leaves at least a quarter of the units idle; then all but the last
    whole wave stay data-parallel."""
    s, p = g.gemm_plan(M, N, 4096, 1, 1, 2, 152, {"cta_group": 2, "bn": 256})
    assert s == 0
    d = p.as_dict()
    units = d["grid"] // 2
    if expect_sk:
        waves = d["num_tiles"] // units
        assert d["sk_iters"] > 0 and d["dp_tiles"] == (waves - 1) * units, d
        assert d["sk_iters"] == (d["num_tiles"] - d["dp_tiles"]) * d["groups"]
    else:
        assert d["sk_iters"] == 0 and d["dp_tiles"] == d["num_tiles"], d


def test_plan_prefers_pairs_only_with_more_than_one_panel(g):
    for M in (1, 64, 128):
        s, p = g.gemm_plan(M, 4096, 4096, 1, 1, 0, 152)
        assert s == 0 and p.cta_group == 1
    s, p = g.gemm_plan(4096, 4096, 4096, 1, 1, 0, 152, {"cta_group": 1})
    assert s == 0 and p.cta_group == 1 and p.bm == 128 and p.num_tiles == 512
    s, p = g.gemm_plan(512, 512, 512, 0, 2, 0, 152, {"cta_group": 2, "bn": 128})
    assert s == 0 and (p.cta_group, p.bm, p.bn, p.num_tiles, p.grid) == (2, 256, 128, 8, 16)


def test_plan_split_k_overrides(g):
    s, p = g.gemm_plan(128, 4096, 4096, 1, 1, 2, 152, {"split_k": 2})
    assert s == 0 and (p.split_k, p.bn, p.grid, p.num_tiles) == (2, 256, 32, 16)
    s, p = g.gemm_plan(128, 4096, 4096, 1, 1, 2, 152, {"split_k": 2, "bn": 128})
    assert s == 0 and (p.split_k, p.bn, p.grid) == (2, 128, 64)
    for bad in ({"split_k": 3}, {"split_k": 8, "bn": 256}, {"split_k": 2, "cta_group": 2},
                {"split_k": 8, "bn": 64}, {"split_k": 16, "bn": 128}):
        assert g.gemm_plan(256, 4096, 4096, 1, 1, 2, 152, bad)[0] == g.GEMM_ERR_INVALID_ARG, bad
    # narrower slices: 128-wide split 4 / 8, 64-wide split 2 / 4
    for good, grid in (({"split_k": 4, "bn": 128}, 128), ({"split_k": 8, "bn": 128}, 256),
                       ({"split_k": 2, "bn": 64}, 128), ({"split_k": 4, "bn": 64}, 256)):
        s, p = g.gemm_plan(128, 4096, 4096, 1, 1, 2, 152, good)
        assert s == 0 and (p.split_k, p.bn, p.grid) == (good["split_k"], good["bn"], grid), good
    # small-N decode shapes: as many CTAs as fit one wave (128 for N = 2048)
    s, p = g.gemm_plan(16, 2048, 8192, 1, 1, 2, 152)
    assert s == 0 and (p.bn, p.split_k, p.grid) == (64, 4, 128)
    # a manual tile setting turns the automatic split off
    s, p = g.gemm_plan(128, 8192, 8192, 1, 1, 2, 152, {"cta_group": 1, "bn": 64})
    assert s == 0 and (p.split_k, p.bn, p.num_tiles) == (1, 64, 128)
    # an explicit split overrides an automatic pair choice
    s, p = g.gemm_plan(4096, 4096, 4096, 1, 1, 2, 152, {"split_k": 2})
    assert s == 0 and (p.cta_group, p.split_k, p.bm) == (1, 2, 128)
    # fewer k-blocks than splits
    assert g.gemm_plan(128, 4096, 128, 1, 1, 2, 152, {"split_k": 4})[0] == g.GEMM_ERR_INVALID_ARG
    # general is 0 or 1
    import ctypes
    cfg = g.gemm_config_t()
    cfg.general = 7
    p = g.gemm_plan_t()
    lib = g.library()
    assert lib.gemm_plan(256, 256, 256, 1, 1, 0, 152, ctypes.byref(cfg), ctypes.byref(p)) == 1
    assert g.gemm_plan(256, 256, 256, 1, 1, 0, 152, {"order": 3})[0] == g.GEMM_ERR_INVALID_ARG


def test_stream_k_override(g):
    s, p = g.gemm_plan(4096, 4096, 4096, 1, 1, 0, 152, {"stream_k": 1})
    assert s == 0 and p.sk_iters == 0 and p.dp_tiles == p.num_tiles == 256 and p.scratch_bytes == 0
    s, p = g.gemm_plan(1024, 1024, 1024, 1, 1, 0, 152, {"stream_k": 2, "cta_group": 1, "bn": 128})
    assert s == 0 and p.sk_iters == 64 * 8 and p.dp_tiles == 0 and p.grid == 152
    assert p.scratch_bytes == 4096 + 152 * 128 * 128 * 4
    assert g.gemm_plan(1024, 1024, 1024, 1, 1, 0, 152, {"stream_k": 4})[0] == g.GEMM_ERR_INVALID_ARG
    # split-K plans never stream-K
    s, p = g.gemm_plan(128, 8192, 8192, 1, 1, 2, 152, {"stream_k": 2})
    assert s == 0 and p.split_k == 2 and p.sk_iters == 0


@pytest.mark.parametrize("units,num_tiles,groups,waves_dp", [(76, 64, 16, 0), (76, 256, 32, 2),
                                                             (152, 60, 5, 0), (7, 23, 9, 2),
                                                             (76, 1024, 64, 12), (5, 3, 4, 0)])
def test_stream_k_split_covers_every_k_group_once(g, units, num_tiles, groups, waves_dp):
    dp = waves_dp * units
    sk = (num_tiles - dp) * groups
    seen = {}
    for u in range(units):
        items = g.gemm_work_items(u, units, dp, sk, groups)
        for t, g0, g1 in items:
            assert 0 <= t < num_tiles and 0 <= g0 < g1 <= groups
            if t < dp:
                assert (g0, g1) == (0, groups) and t % units == u
            for k in range(g0, g1):
                assert (t, k) not in seen
                seen[(t, k)] = u
    assert len(seen) == num_tiles * groups
    # the units touching a split tile are consecutive, in k order; the highest
    # one (holding the last k-group) owns the tile and its share is that unit's
    # last stream-K item, while every other unit's share is its first item; so a
    # unit whose share spans tiles starts at k-group 0 of its first tile
    for t in range(dp, num_tiles):
        owners = [seen[(t, k)] for k in range(groups)]
        assert owners == sorted(owners)
        assert set(owners) == set(range(owners[0], owners[-1] + 1))
        for u in set(owners):
            items = [it for it in g.gemm_work_items(u, units, dp, sk, groups) if it[0] >= dp]
            share = [it for it in items if it[0] == t]
            assert len(share) == 1
            if u == owners[-1] and len(set(owners)) > 1:
                assert share[0] == items[-1] and share[0][2] == groups
            elif u != owners[-1]:
                assert share[0] == items[0]
            if u == owners[0]:
                assert share[0][1] == 0
    for u in range(units):
        items = [it for it in g.gemm_work_items(u, units, dp, sk, groups) if it[0] >= dp]
        if len(items) > 1:
            assert items[0][1] == 0
            assert [it[0] for it in items] == sorted((it[0] for it in items), reverse=True)


def test_plan_overrides_and_errors(g):
    s, p = g.gemm_plan(1024, 1024, 1024, 0, 2, 0, 152, {"bn": 128, "group_m": 3, "grid": 10,
                                                         "cta_group": 1})
    assert s == 0 and (p.bn, p.group_m, p.grid, p.cta_group) == (128, 3, 10, 1)
    s, _ = g.gemm_plan(1024, 1024, 1024, 0, 2, 0, 152, {"bn": 96})
    assert s == g.GEMM_ERR_INVALID_ARG
    s, _ = g.gemm_plan(1024, 1024, 1024, 0, 2, 0, 152, {"bn": 64, "cta_group": 2})
    assert s == g.GEMM_ERR_INVALID_ARG
    s, _ = g.gemm_plan(1024, 1024, 1024, 0, 2, 0, 152, {"cta_group": 3})
    assert s == g.GEMM_ERR_INVALID_ARG
    s, _ = g.gemm_plan(1024, 1024, 1024, 0, 2, 0, 0)
    assert s == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("mt,nt,gm", [(1, 1, 1), (32, 16, 8), (32, 16, 16), (5, 7, 3),
                                      (13, 4, 16), (64, 32, 16), (1, 128, 1), (3, 1, 2)])
def test_tile_order_covers_every_tile_once(g, mt, nt, gm):
    seen = np.zeros((mt, nt), np.int32)
    for t in range(mt * nt):
        m, n = g.gemm_tile_coord(t, mt, nt, gm)
        assert 0 <= m < mt and 0 <= n < nt
        seen[m, n] += 1
    assert np.all(seen == 1)


def _avg_panels(order, window):
    counts = []
    for i in range(0, len(order) - window + 1, window):
        w = order[i:i + window]
        counts.append(len({m for m, _ in w}) + len({n for _, n in w}))
    return sum(counts) / len(counts)


def test_grouped_order_panel_counts_from_lecture(g):
    """"Scheduling is geometry" (linearly.space lecture 26.5): eight tiles in flight
    in one row of the tile grid need 1 + 8 = 9 operand panels; the same eight tiles
    as a 4 x 2 block need 4 + 2 = 6.  The grouped order with group_m = 4 visits
    exactly such 4 x 2 blocks."""
    mt, nt = 32, 16
    row_major = [(t // nt, t % nt) for t in range(mt * nt)]
    grouped = [g.gemm_tile_coord(t, mt, nt, 4) for t in range(mt * nt)]
    assert _avg_panels(row_major, 8) == 9
    assert _avg_panels(grouped, 8) == 6
    # a 64-tile wave: row-major spans 4 rows x 16 columns (20 panels), group_m = 8
    # gives 8 x 8 blocks (16 panels)
    grouped8 = [g.gemm_tile_coord(t, mt, nt, 8) for t in range(mt * nt)]
    assert _avg_panels(row_major, 64) == 20
    assert _avg_panels(grouped8, 64) == 16


def test_instruction_descriptor_fields(g):
    d = g.gemm_encode_idesc(1, 0, 1, 128, 256)
    assert (d >> 4) & 3 == 1          # D = f32
    assert (d >> 7) & 7 == 1          # A = bf16
    assert (d >> 10) & 7 == 1         # B = bf16
    assert (d >> 15) & 1 == 0         # A K-major
    assert (d >> 16) & 1 == 1         # B MN-major
    assert (d >> 17) & 0x3F == 256 >> 3
    assert (d >> 24) & 0x1F == 128 >> 4
    assert d & 0b1111 == 0 and (d >> 13) & 3 == 0 and (d >> 23) & 1 == 0 and d >> 29 == 0
    d16 = g.gemm_encode_idesc(0, 1, 0, 128, 64)
    assert (d16 >> 7) & 0x3F == 0 and (d16 >> 15) & 3 == 1 and (d16 >> 17) & 0x3F == 8


def test_smem_descriptor_fields(g):
    d = g.gemm_encode_sdesc(0x10400, 16, 1024)
    assert d & 0x3FFF == 0x10400 >> 4
    assert (d >> 16) & 0x3FFF == 1
    assert (d >> 32) & 0x3FFF == 64
    assert (d >> 46) & 3 == 1
    assert (d >> 49) & 7 == 0
    assert (d >> 61) & 7 == 2
    d2 = g.gemm_encode_sdesc(0x3FFF0, 8192, 1024)
    assert d2 & 0x3FFF == 0x3FFF and (d2 >> 16) & 0x3FFF == 512


@pytest.mark.parametrize("bias,kind,act,M,expect", [
    (0, 1, 0, 64, 1),               # column bias without a pointer
    (0, 2, 1, 64, 1),               # row bias without a pointer
    (ALIGNED, 3, 0, 64, 1),         # unknown bias kind
    (ALIGNED, 1, 2, 64, 1),         # unknown activation
    (ALIGNED, -1, 0, 64, 1),
    (ALIGNED + 4, 1, 0, 64, 2),     # bias not 16-byte aligned
    (0, 1, 1, 0, 0),                # M == 0: quick return, the bias is never read
])
def test_bias_act_argument_checks(g, bias, kind, act, M, expect):
    s = g.gemm_bias_act(M, 64, 64, 1.0, ALIGNED, 64, ALIGNED, 64, 0.0, ALIGNED, 64, 0, 2, 0,
                        bias, kind, act, 0)
    assert s == expect


# ------------------------------------------------------------ tile orders

def _panel_counts(golden):
    out = {}
    for line in open(os.path.join(ROOT, "tests", "golden", golden)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v) if "." in v else int(v)
    return out


def _avg_panels_sliding(order, window):
    """Mean over every run of `window` consecutive tiles of the A panels plus B
    panels it touches (distinct tile rows + distinct tile columns)."""
    tot = 0
    for s0 in range(len(order) - window + 1):
        w = order[s0:s0 + window]
        tot += len({m for m, _ in w}) + len({n for _, n in w})
    return tot / (len(order) - window + 1)


def test_tile_orders_match_the_lectures_panel_counts(g):
    """The lecture's "Scheduling is geometry" counts panels of 8 tiles in flight:
    9.86 row by row, 7.02 grouped, 6.67 along a Hilbert curve (8 x 8 tile grid,
    groups of 4 tile-rows, as in its 4 x 2 block example)."""
    pc = _panel_counts("panel_counts.txt")
    mt = nt = pc["grid"]
    w = pc["window"]
    row = g.gemm_tile_order(g.GEMM_ORDER_GROUPED, mt, nt, 1)
    grp = g.gemm_tile_order(g.GEMM_ORDER_GROUPED, mt, nt, pc["group_rows"])
    hil = g.gemm_tile_order(g.GEMM_ORDER_HILBERT, mt, nt)
    assert round(_avg_panels_sliding(row, w), 2) == pc["row_major"]
    assert round(_avg_panels_sliding(grp, w), 2) == pc["grouped"]
    assert round(_avg_panels_sliding(hil, w), 2) == pc["hilbert"]


@pytest.mark.parametrize("mt,nt", [(1, 1), (8, 8), (32, 32), (24, 24), (28, 20), (3, 17), (17, 3),
                                   (64, 5), (5, 64), (1, 16), (33, 40)])
def test_hilbert_order_covers_each_tile_once(g, mt, nt):
    hil = g.gemm_tile_order(g.GEMM_ORDER_HILBERT, mt, nt)
    if hil is None:   # too elongated for the enclosing square: the planner keeps grouped
        side = 1 << max(0, (max(mt, nt) - 1).bit_length())
        assert side * side > 16 * mt * nt
        s, p = g.gemm_plan(mt * 128, nt * 256, 512, 1, 1, 0, 152,
                           {"order": 2, "cta_group": 1, "bn": 256})
        assert s == 0 and p.order == g.GEMM_ORDER_GROUPED
        return
    assert sorted(hil) == [(m, n) for m in range(mt) for n in range(nt)]


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_hilbert_steps_are_adjacent_on_power_of_two_squares(g, k):
    n = 1 << k
    hil = g.gemm_tile_order(g.GEMM_ORDER_HILBERT, n, n)
    assert hil[0] == (0, 0)
    for (a, b), (c, d) in zip(hil, hil[1:]):
        assert abs(a - c) + abs(b - d) == 1


def test_plan_reports_the_order(g):
    s, p = g.gemm_plan(8192, 8192, 8192, 1, 2, 2, 152, {"order": 2})
    assert s == 0 and p.order == g.GEMM_ORDER_HILBERT
    s, p = g.gemm_plan(8192, 8192, 8192, 1, 2, 2, 152)
    assert s == 0 and p.order == g.GEMM_ORDER_GROUPED


@pytest.mark.parametrize("layout,lda,ldb,expect", [
    (2, 64, 64, 0), (0, 64, 64, 2), (1, 64, 64, 2), (3, 64, 64, 2),   # K-major (A row, B col) only
    (2, 56, 64, 2), (2, 64, 72, 2),                                   # 16-byte pitch: 16 elements
])
def test_fp8_layout_and_pitch_rules(g, layout, lda, ldb, expect):
    for fmt in (g.GEMM_E4M3, g.GEMM_E5M2):
        s = g.gemm(64, 64, 48, 1.0, ALIGNED, lda, ALIGNED, ldb, 0.0, ALIGNED, 64, fmt, 2, layout, 0)
        if expect == 0:
            assert s in (g.GEMM_ERR_CUDA, g.GEMM_ERR_ARCH, g.GEMM_OK)
        else:
            assert s == expect


def test_fp8_plan_uses_128_element_k_blocks(g):
    s, p = g.gemm_plan(4096, 4096, 4096, g.GEMM_E4M3, 1, 2, 152)
    assert s == 0 and p.k_blocks == 32 and p.bk == 256 and p.groups == 16


def test_plan_specialised_flag():
    """gemm_plan_t.specialised: 1 exactly when the plan's configuration has a
    specialised instance for the layout and the plan keeps the plain path."""
    import dense_tensor_core_tcgen05_gb300 as g
    plan = lambda *a, **k: g.gemm_plan(*a, **k)[1].specialised
    # 2048^3 fp16 -> fp32 row/row: the 256-wide CTA pair, every layout
    for layout in range(4):
        assert plan(2048, 2048, 2048, 0, 2, layout, 152) == 1
        assert plan(2048, 2048, 2048, 0, 2, layout, 152, {"general": 1}) == 0
    # 4096^3 plans a stream-K tail: the pair has stream-K instances, the single
    # CTA does not
    s, p = g.gemm_plan(4096, 4096, 4096, 1, 1, 0, 152)
    assert s == 0 and p.sk_iters > 0 and p.specialised == 1
    s, p = g.gemm_plan(4096, 4096, 4096, 1, 1, 0, 152, {"cta_group": 1, "bn": 64, "stream_k": 2})
    assert s == 0 and p.sk_iters > 0 and p.specialised == 0
    # skinny and decode shapes: 2-way split-K clusters
    assert plan(128, 8192, 8192, 1, 1, 2, 152) == 1
    # N * sizeof(out) not a multiple of 16 bytes: ragged right edge
    assert plan(256, 203, 256, 1, 2, 0, 152, {"cta_group": 2}) == 0
    # the Hilbert order reads a tile table
    assert plan(2048, 2048, 2048, 1, 1, 0, 152, {"order": 2}) == 0
    # configurations without specialised instances
    assert plan(2048, 2048, 2048, 1, 1, 0, 152, {"cta_group": 1, "bn": 256}) == 0
    assert plan(128, 8192, 8192, 1, 1, 2, 152, {"split_k": 4, "bn": 256}) == 0
    # the second set: the other single-panel choices
    assert plan(128, 8192, 8192, 1, 1, 2, 152, {"split_k": 4, "bn": 128}) == 1
    assert plan(32, 2048, 8192, 1, 1, 2, 152) == 1   # 8-way clusters of width 128
    assert plan(128, 8192, 8192, 1, 1, 2, 152, {"split_k": 8, "bn": 128}) == 1
    # the third set: single CTAs of width 64 or 128 with a ragged right edge
    assert plan(73, 61, 67, 0, 2, 0, 152) == 1
    assert plan(257, 263, 251, 0, 2, 0, 152) == 1
    assert plan(257, 263, 251, 0, 2, 0, 152, {"bn": 256}) == 0
    assert plan(8, 14336, 4096, 1, 1, 2, 152) == 1   # the single 128-wide CTA
    assert plan(512, 512, 512, 0, 2, 0, 152) == 1   # the single 64-wide CTA
    # 8-bit operands: A row-major with B column-major only
    assert plan(2048, 2048, 2048, 3, 2, 2, 152) == 1


def test_split_tile_plans(g):
    # 128 x 8192 x 8192 bf16, B column-major: 64 tiles of 128 columns, 2 parts each
    s, p = g.gemm_plan(128, 8192, 8192, 1, 1, 2, 152, {"stream_k": 3})
    assert s == 0 and p.tile_split == 2 and p.split_k == 1 and p.cta_group == 1 and p.bn == 128
    assert p.grid == 128 and p.dp_tiles == 0 and p.sk_iters == 0 and p.groups == 64
    assert p.owner_groups == 35   # 32 + a tenth of the tile's k-groups over the 2 parts
    assert p.scratch_bytes == 4096 + 128 * 128 * 128 * 4
    s, p = g.gemm_plan(128, 8192, 8192, 1, 1, 2, 152, {"stream_k": 3, "split_k": 4, "bn": 256})
    assert s == 0 and p.tile_split == 4 and p.grid == 128 and p.owner_groups == 20
    # more units than SMs, a part without a k-group, a CTA pair: refused
    assert g.gemm_plan(1024, 1024, 1024, 1, 1, 0, 152, {"stream_k": 3, "split_k": 4, "bn": 64})[0] == \
        g.GEMM_ERR_UNSUPPORTED
    assert g.gemm_plan(128, 1024, 128, 1, 1, 0, 152, {"stream_k": 3})[0] == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan(256, 1024, 4096, 1, 1, 0, 152, {"stream_k": 3, "cta_group": 2})[0] == \
        g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan(128, 1024, 4096, 1, 1, 0, 152, {"stream_k": 3, "split_k": 17})[0] == \
        g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("units,num_tiles,groups,waves_dp", [
    (76, 256, 16, 2), (76, 1024, 64, 12), (76, 64, 16, 0), (152, 60, 5, 0), (7, 23, 9, 2),
    (5, 3, 4, 0), (76, 576, 32, 6), (3, 2, 40, 0), (64, 200, 3, 1)])
def test_stream_k_schedule_has_no_wait_cycle(g, units, num_tiles, groups, waves_dp):
    """Each unit runs its items in order (the MMA issuer and the epilogue walk the
    same list, with two accumulator buffers); an item that finishes a split tile
    waits until every other unit's segment of that tile is published.  Simulated
    on the host from the kernel's own walk: every unit must get through its list,
    i.e. no owner waits (directly or through its unit's earlier items) on a
    segment that itself waits on that owner."""
    dp = waves_dp * units
    sk = (num_tiles - dp) * groups
    items = {u: [tuple(it) for it in g.gemm_work_items(u, units, dp, sk, groups)]
             for u in range(units)}
    holders = {}
    for u, its in items.items():
        for t, g0, g1 in its:
            if t >= dp:
                holders.setdefault(t, []).append((u, g0, g1))
    done = {u: 0 for u in range(units)}   # items finished per unit
    published = set()                                # (unit, tile) segments published
    progress = True
    while progress:
        progress = False
        for u in range(units):
            while done[u] < len(items[u]):
                t, g0, g1 = items[u][done[u]]
                whole = g0 == 0 and g1 == groups
                if t >= dp and not whole and g1 == groups:
                    # the owner: every other holder's segment must be out
                    if any((v, t) not in published for v, _, _ in holders[t] if v != u):
                        break
                if t >= dp and g1 < groups:
                    published.add((u, t))
                done[u] += 1
                progress = True
    stuck = [u for u in range(units) if done[u] < len(items[u])]
    assert not stuck, f"units {stuck[:8]} wait forever"
    # and the kernel's contributor list is exactly the other holders, in unit order
    for t, hs in holders.items():
        us = sorted(v for v, _, _ in hs)
        assert us == list(range(us[0], us[-1] + 1))


@pytest.mark.parametrize("parts,groups", [(2, 64), (2, 2), (3, 7), (4, 64), (8, 33), (16, 16)])
def test_split_tile_items_cover_each_tile_once(g, parts, groups):
    """Every k-group of a tile is held by exactly one of its parts; the first part
    (the owner) starts at k-group 0 and holds the largest share."""
    extra = max(1, groups // 10)
    owner = min((groups + (parts - 1) * extra) // parts, groups - (parts - 1))
    for tile in range(3):
        items = [g.gemm_split_tile_item(tile * parts + q, parts, owner, groups) for q in range(parts)]
        assert all(it is not None and it[0] == tile for it in items)
        covered = []
        for (_, g0, g1) in items:
            assert g0 < g1
            covered.extend(range(g0, g1))
        assert sorted(covered) == list(range(groups))
        assert items[0][1] == 0 and items[0][2] == owner
        shares = [g1 - g0 for (_, g0, g1) in items]
        assert shares[0] == max(shares)
    assert g.gemm_split_tile_item(0, 1, 1, groups) is None


def test_fastdiv_matches_integer_division(g):
    """The kernel divides by run-time constants with a multiply and a shift
    (Granlund-Montgomery); it must equal integer division for every divisor and
    numerator below 2^31: small and power-of-two divisors, divisors next to powers
    of two, and numerators at the top of the range and at multiples of d."""
    rng = np.random.default_rng(5)
    ds = [1, 2, 3, 5, 6, 7, 9, 76, 152, 255, 256, 257, 1000, 65535, 65536, 65537,
          (1 << 30) - 1, 1 << 30, (1 << 30) + 1, (1 << 31) - 1]
    ds += [int(x) for x in rng.integers(1, 1 << 31, size=60)]
    for d in ds:
        ns = [0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, (1 << 31) - 1, (1 << 31) - 2]
        ns += [int(x) for x in rng.integers(0, 1 << 31, size=40)]
        ns += [(k * d) % (1 << 31) for k in range(1, 6)] + [((k * d) - 1) % (1 << 31) for k in range(1, 6)]
        for n in ns:
            if 0 <= n < (1 << 31):
                assert g.gemm_fastdiv(n, d) == n // d, (n, d)
    assert g.gemm_fastdiv(5, 0) == 0xFFFFFFFF
    assert g.gemm_fastdiv(1 << 31, 3) == 0xFFFFFFFF


@pytest.mark.parametrize("seed", range(6))
def test_grouped_order_kernel_walk_matches_definition(g, seed):
    """gemm_tile_order walks the grouped order the kernel's way (fastdiv);
    gemm_tile_coord computes the definition with plain division."""
    rng = np.random.default_rng(100 + seed)
    for _ in range(8):
        mt, nt = int(rng.integers(1, 70)), int(rng.integers(1, 70))
        gm = int(rng.integers(1, 20))
        order = g.gemm_tile_order(1, mt, nt, gm)
        assert order is not None and len(order) == mt * nt
        for t in range(mt * nt):
            assert order[t] == g.gemm_tile_coord(t, mt, nt, gm), (mt, nt, gm, t)
