"""Host-side checks of bench.py: roofline arithmetic against the pages' numbers,
and the multi-rank aggregation (max over ranks, whole-job value) with two gloo
ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flop_counts.txt")


def test_panel_intensity_and_knees_from_pages():
    for line in open(GOLDEN):
        p = line.split()
        if not p or p[0].startswith("#"):
            continue
        if p[0] == "panel":
            bm, bn, s, want = int(p[1]), int(p[2]), int(p[3]), float(p[4])
            assert round(bench.panel_intensity(bm, bn, s), 1) == want
        elif p[0] == "knee":
            assert round(float(p[1]) / float(p[2]), 2 if float(p[3]) < 100 else 1) == float(p[3])


def test_algorithmic_bytes_and_bound():
    w = dict(M=128, N=8192, K=8192, out_dtype="bf16", beta=0.0)
    assert bench.algorithmic_bytes(w) == 2 * (128 * 8192 + 8192 * 8192) + 2 * 128 * 8192
    assert bench.roofline_bound(w, 1882.2, 6794.1) == "hbm"
    w4 = dict(M=8192, N=8192, K=8192, out_dtype="f32", beta=0.5)
    assert bench.algorithmic_bytes(w4) == 2 * 2 * 8192 * 8192 + 2 * 4 * 8192 * 8192
    assert bench.roofline_bound(w4, 1882.2, 6794.1) == "tensor"
    assert bench.gemm_flops(2, 2, 3) == 24


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.0, 3.0][rank]          # rank 1 is the slow replica
    step_ms, value = bench.aggregate_ranks(local_ms, 1e9, world)
    q.put((rank, step_ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step_ms, value in res:
        assert step_ms == 3.0                       # max over ranks
        assert value == pytest.approx(2 * 1e9 / 3e-3 / 1e12)   # both ranks' FLOPs / slowest time


def test_aggregate_single_rank():
    assert bench.aggregate_ranks(4.0, 2e12, 1) == (4.0, 2e12 / 4e-3 / 1e12)
