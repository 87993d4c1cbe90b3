"""Hardware probes behind the GEMM's design (measurement tooling, not the GEMM path).

    python -m dense_tensor_core_tcgen05_gb300.probes [MODE]

With no MODE: (1) the tcgen05.mma rate per tile width (cycles per instruction and
dense FLOP/clk/SM, one issuing thread per CTA or CTA pair, all SMs busy), (2) TMA
copies from L2 and with cluster multicast, (3) the bandwidth at which TMA tile copies
stream an 8192 x 8192 K-major bf16 matrix from DRAM, per copy shape.  Modes:

    store   the routes by which 128 CTAs can write a 16 MiB fp32 output (the
            epilogue of a one-wave 2048^3 GEMM)
    intake  TMA intake from L2 by footprint, sharing and cold L2; beside cp.async
    values  the same intake with constant and random data
    depth   the intake kernel against the streaming kernel on one access pattern,
            the latter with its indices by division or kept incrementally
    smem    TMA intake while other warps read shared memory
    cross   each TMA probe kernel launched with the other's tensor map

The probes are built from probes.cu into _build/libprobes.so (sm_103a only).
"""
from __future__ import annotations

import ctypes
import os
import statistics
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_PKG = os.path.dirname(_HERE)
_SRC = os.path.join(_HERE, "probes.cu")
_LIB = os.path.join(_PKG, "_build", "libprobes.so")


def build(force=False):
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
                               f"-I{os.path.join(_PKG, 'csrc')}", _SRC, "-o", _LIB])
    lib = ctypes.CDLL(_LIB)
    lib.probe_mma_rate.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p]
    lib.probe_tma_stream.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 11 + [ctypes.c_void_p]
    lib.probe_tma_mcast.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 9 + [ctypes.c_void_p]
    lib.probe_store_rate.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    lib.probe_intake.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_longlong] + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    return lib


def mma_rate(lib, n, pair, grid=152, iters=2000):
    """Median over issuing CTAs: (cycles per MMA, dense FLOP/clk/SM)."""
    import torch
    out = torch.zeros(grid, dtype=torch.int64, device="cuda")
    rc = lib.probe_mma_rate(n, int(pair), grid, iters, out.data_ptr())
    if rc != 0:
        raise RuntimeError(f"probe_mma_rate rc {rc}")
    v = [int(x) for i, x in enumerate(out.cpu().tolist()) if not pair or i % 2 == 0]
    if any(x < 0 for x in v):
        raise RuntimeError("an issuing CTA gave up its wait")
    cyc = statistics.median(v) / (iters * 4)
    flop_per_sm = 2 * (256 if pair else 128) * n * 16 / (2 if pair else 1)
    return cyc, flop_per_sm / cyc


def tma_stream(lib, B, grid, R, KO, S, grouped=False, promo=3, reps=1, variant=0, threads=64):
    """(median in-kernel ns per CTA, TB/s) for streaming B [N, K] bf16 `reps` times."""
    import torch
    N, K = B.shape
    out = torch.zeros(grid, dtype=torch.int64, device="cuda")
    rc = lib.probe_tma_stream(B.data_ptr(), N, K, grid, R, KO, S, int(grouped), promo, reps,
                              variant, threads, out.data_ptr())
    if rc != 0:
        raise RuntimeError(f"probe_tma_stream rc {rc}")
    ns = statistics.median(out.cpu().tolist())
    return ns, reps * N * K * 2 / ns / 1e3


def main(argv=None):
    import sys
    import torch
    argv = sys.argv[1:] if argv is None else argv
    lib = build()
    if argv == ["store"]:
        store_rates(lib)
        return
    if argv == ["intake"]:
        intake_rates(lib)
        return
    if argv == ["values"]:
        intake_by_values(lib)
        return
    if argv == ["depth"]:
        intake_by_depth(lib)
        return
    if argv == ["smem"]:
        intake_with_smem_reads(lib)
        return
    if argv == ["cross"]:
        cross_check(lib)
        return
    print("tcgen05.mma kind::f16 (bf16), K = 16 per instruction, all SMs busy")
    for n, pair in ((64, 0), (128, 0), (256, 0), (128, 1), (256, 1)):
        cyc, fpc = mma_rate(lib, n, pair)
        print(f"  M={256 if pair else 128:3d} N={n:3d} {'pair' if pair else 'cta '}: "
              f"{cyc:6.1f} cycles/MMA, {fpc:6.0f} FLOP/clk/SM")
    l2_rate(lib)
    mcast_rate(lib)
    B = torch.randn(8192, 8192, device="cuda").to(torch.bfloat16)
    flush = torch.empty(512 << 18, dtype=torch.float32, device="cuda")
    print("TMA streaming of an 8192 x 8192 K-major bf16 matrix, 128 CTAs (in-kernel time)")
    promos = ("none", "64B", "128B", "256B")
    for (R, KO, S, grouped, promo) in ((64, 1, 16, 0, 3), (64, 2, 8, 0, 3), (64, 2, 8, 0, 0),
                                       (64, 2, 8, 1, 3), (64, 2, 8, 1, 0), (64, 4, 4, 0, 3),
                                       (64, 4, 4, 1, 3), (32, 4, 8, 0, 3), (64, 8, 3, 0, 3),
                                       (64, 8, 3, 1, 3)):
        res = []
        for _ in range(5):
            flush.zero_()
            res.append(tma_stream(lib, B, 128, R, KO, S, grouped, promo))
        ns, tbs = sorted(res)[len(res) // 2]
        print(f"  copy = {R:3d} rows x {KO} blocks ({KO * 128:4d} B per row), {S:2d} in flight, "
              f"{'8-row groups' if grouped else 'whole box   '}, L2 promotion {promos[promo]:4s}: "
              f"{ns / 1e3:6.1f} us, {tbs:4.2f} TB/s")


def l2_rate(lib):
    """TMA rate from L2 into shared memory: every CTA re-streams its 128 x 512
    slice of a 16 MB matrix (L2-resident after the first pass) 64 times, with the
    GEMM's stage shape (128 rows x 2 blocks)."""
    import torch
    A = torch.randn(16384, 512, device="cuda").to(torch.bfloat16)
    print("TMA from L2 (16 MB matrix re-streamed 64x per CTA, 128 rows x 2 blocks per copy)")
    for grid, S in ((128, 6), (128, 3), (64, 6), (32, 6), (16, 6)):
        ns, tbs = tma_stream(lib, A, grid, 128, 2, S, reps=64)
        print(f"  {grid:3d} CTAs, {S} copies in flight: {tbs:5.2f} TB/s total, "
              f"{tbs * 1e3 / grid:6.1f} GB/s per SM")


def mcast_rate(lib):
    """Bytes each SM receives per second from L2 when clusters of C CTAs share
    every copy by multicast (each CTA issues 1/C of it)."""
    import torch
    A = torch.randn(16384, 512, device="cuda").to(torch.bfloat16)
    N, K = A.shape
    print("TMA multicast from L2 (copies of 128 rows x 2 blocks shared by C CTAs, 128 CTAs)")
    for batched, C in ((0, 1), (0, 2), (0, 4), (1, 1), (1, 2), (1, 4)):
        grid, reps = 128, 48
        out = torch.zeros(grid, dtype=torch.int64, device="cuda")
        rc = lib.probe_tma_mcast(A.data_ptr(), N, K, grid, 128, 2, 6, C, reps, batched,
                                 out.data_ptr())
        if rc != 0:
            raise RuntimeError(f"probe_tma_mcast rc {rc}")
        v = out.cpu().tolist()
        if any(x < 0 for x in v):
            raise RuntimeError("a CTA gave up its wait")
        ns = statistics.median(v)
        per_cta = reps * (N // (grid // C)) * K * 2
        print(f"  {'batches of 6' if batched else 'per-slot release'}, C = {C}: "
              f"{per_cta / ns:6.1f} GB/s received per SM "
              f"({per_cta / C / ns:6.1f} GB/s issued per SM)")


STORE_ROUTES = ("tensor stores, 2 buffers per warp", "tensor stores, a buffer per chunk",
                "16-byte global stores by row", "coalesced 16-byte global stores",
                "one 3-D tensor store per warp")


def store_rates(lib, M=2048, N=2048, grid_m=16, grid_n=8, runs=7):
    """Time for 128 CTAs to write a 2048 x 2048 fp32 C as 128 x 256 blocks (the
    output of a one-wave 2048^3 GEMM on 256 x 256 pair tiles), per route, with L2
    flushed (written, then read back) before every run: median over runs of the
    span first start -> last completion, and of the mean per-CTA duration."""
    import torch
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    flush = torch.empty(512 << 18, dtype=torch.float32, device="cuda")
    rows = flush.view(-1, 1 << 16)
    sink = torch.empty(1 << 16, dtype=torch.float32, device="cuda")
    r = torch.arange(grid_m * 128, device="cuda", dtype=torch.float32)[:, None]
    c = torch.arange(grid_n * 256, device="cuda", dtype=torch.float32)[None, :]
    want = 0.5 * r + c
    out = torch.zeros(grid_m * grid_n * 5, dtype=torch.int64, device="cuda")
    print(f"fp32 output of {grid_m * grid_n} CTAs x 128 x 256 ({M * N * 4 / 2**20:.0f} MiB), L2 flushed")
    for mode, name in enumerate(STORE_ROUTES):
        spans, per = [], []
        for _ in range(runs):
            C.fill_(float("nan"))
            flush.zero_()
            torch.sum(rows, dim=0, out=sink)
            torch.cuda.synchronize()
            rc = lib.probe_store_rate(C.data_ptr(), M, N, N, grid_m, grid_n, mode, out.data_ptr())
            if rc != 0:
                raise RuntimeError(f"probe_store_rate rc {rc}")
            t = out.view(-1, 5).cpu()
            t0, t1 = t[:, 0], t[:, 1:].max(dim=1).values
            spans.append(int(t1.max() - t0.min()))
            per.append(float((t1 - t0).double().mean()))
        ok = torch.equal(C[:grid_m * 128, :grid_n * 256], want)
        sp, pc = statistics.median(spans), statistics.median(per)
        print(f"  {name:36s}: span {sp / 1e3:5.2f} us, per CTA {pc / 1e3:5.2f} us "
              f"({grid_m * grid_n * 128 * 256 * 4 / sp / 1e3:5.2f} TB/s){'' if ok else '  WRONG OUTPUT'}")


def intake(lib, A, P, out, grid, W, copies, cp_iters, share=1, warm=True, bars_after_ring=0):
    """Median per-CTA GB/s of the TMA stream (None when off) and of each cp.async warp."""
    rows, cols = A.shape
    for _ in range(2 if warm else 1):
        rc = lib.probe_intake(A.data_ptr(), rows, cols, share, P.data_ptr(), P.numel(), grid, W,
                              copies, cp_iters, bars_after_ring, out.data_ptr())
        if rc != 0:
            raise RuntimeError(f"probe_intake rc {rc}")
    t = out.view(-1, 8)[:grid].cpu().double()
    if (t < 0).any():
        raise RuntimeError("a CTA gave up its wait")
    tma = copies * 32768 / float(t[:, 0].median()) if copies else None
    cps = [abs(cp_iters) * 4096 / float(t[:, w].median()) for w in range(1, W + 1)]
    return tma, cps


def intake_rates(lib, grid=128):
    """GB/s an SM takes in from L2 by TMA copies of 128 rows x 2 blocks (32 KB,
    3 in flight): by the footprint each CTA cycles through, by how many CTAs
    share it, from a cold L2, and alongside cp.async warps."""
    import torch
    P = torch.zeros(grid * 4 * 6 * 4096, dtype=torch.uint8, device="cuda")
    out = torch.zeros(grid * 8, dtype=torch.int64, device="cuda")
    copies = 192   # 6 MB per CTA
    print(f"TMA from L2, {grid} CTAs, {copies} copies of 32 KB each (GB/s per SM)")
    for cols in (128, 256, 512, 1024, 2048, 4096):
        A = torch.ones(128 * grid, cols, device="cuda", dtype=torch.bfloat16)
        tma, _ = intake(lib, A, P, out, grid, 0, copies, 0)
        print(f"  own rows, {cols * 256 // 1024:5d} KB per CTA ({A.numel() * 2 >> 20:3d} MB in all): {tma:6.1f}")
        del A
    A = torch.ones(128 * grid, 2048, device="cuda", dtype=torch.bfloat16)
    for share in (2, 8, 32, 128):
        tma, _ = intake(lib, A, P, out, grid, 0, copies, 0, share=share)
        print(f"  512 KB per CTA shared by {share:3d} CTAs ({64 // share:2d} MB in all): {tma:6.1f}")
    flush = torch.empty(512 << 18, dtype=torch.float32, device="cuda")
    for share in (1, 8):
        flush.zero_()
        torch.cuda.synchronize()
        tma, _ = intake(lib, A, P, out, grid, 0, 16, 0, share=share, warm=False)
        print(f"  cold L2, one pass over 512 KB per CTA shared by {share} CTAs: {tma:6.1f}")
    A = torch.ones(128 * grid, 256, device="cuda", dtype=torch.bfloat16)
    cp_iters = 1536
    print(f"TMA (64 KB per CTA) with cp.async warps (24 KB each), {grid} CTAs (GB/s per SM)")
    for W, use in ((1, 0), (2, 0), (4, 0), (1, 1), (2, 1), (4, 1)):
        tma, cps = intake(lib, A, P, out, grid, W, copies if use else 0, cp_iters)
        tot = (tma or 0.0) + sum(cps)
        print(f"  W={W} tma={use}: " + (f"TMA {tma:6.1f}, " if tma else "") +
              ", ".join(f"{c:5.1f}" for c in cps) + f"; sum {tot:6.1f}")


def intake_by_values(lib, grid=128):
    """The same TMA and cp.async intake from L2 with constant and with random
    operand values: whether the rate depends on the data moved."""
    import torch
    out = torch.zeros(grid * 8, dtype=torch.int64, device="cuda")
    print(f"TMA from L2 by operand values, {grid} CTAs, 256 KB per CTA (GB/s per SM)")
    for name, make in (("ones", lambda: torch.ones(128 * grid, 1024, device="cuda", dtype=torch.bfloat16)),
                       ("zeros", lambda: torch.zeros(128 * grid, 1024, device="cuda", dtype=torch.bfloat16)),
                       ("normal(0,1)", lambda: torch.randn(128 * grid, 1024, device="cuda").to(torch.bfloat16)),
                       ("random bits", lambda: torch.randint(-2**15, 2**15, (128 * grid, 1024), device="cuda",
                                                             dtype=torch.int16).view(torch.bfloat16)),
                       ("ones, each 8th row random", None)):
        if make is None:
            A = torch.ones(128 * grid, 1024, device="cuda", dtype=torch.bfloat16)
            A[::8] = torch.randn(A[::8].shape, device="cuda").to(torch.bfloat16)
        else:
            A = make()
        P = torch.zeros(grid * 4 * 6 * 4096, dtype=torch.uint8, device="cuda")
        if name != "ones" and name != "zeros":
            P = torch.randint(0, 256, P.shape, device="cuda", dtype=torch.uint8)
        tma, _ = intake(lib, A, P, out, grid, 0, 192, 0)
        _, cps = intake(lib, A, P, out, grid, 2, 0, 1536)
        tma2, cps2 = intake(lib, A, P, out, grid, 2, 192, 1536)
        print(f"  {name:26s}: TMA {tma:6.1f}; cp.async x2 {sum(cps):6.1f}; both {tma2 + sum(cps2):6.1f}")
        B = A.view(-1, 512)[: 32768]
        ns, tbs = tma_stream(lib, B, grid, 128, 2, 4, reps=2)
        ns, tbs = tma_stream(lib, B, grid, 128, 2, 4, reps=32)
        print(f"  {'':26s}  streaming probe (256 rows x 512 per CTA): {tbs * 1e3 / grid:6.1f}")
        del A, P



def intake_by_depth(lib, grid=128):
    """Both TMA probes on one access pattern (CTA b cycles through rows
    [128 b, 128 b + 128) x 512 columns of a bf16 matrix, copies of 128 rows x 2
    blocks), by copies in flight and CTA count."""
    import torch
    out = torch.zeros(152 * 8, dtype=torch.int64, device="cuda")
    P = torch.zeros(152 * 4 * 6 * 4096, dtype=torch.uint8, device="cuda")
    for g in (grid,):
        A = torch.randn(128 * g, 512, device="cuda").to(torch.bfloat16)
        tma, _ = intake(lib, A, P, out, g, 0, 192, 0)
        res = [f"intake probe (S=3): {tma:6.1f}"]
        for S, variant, threads in ((3, 1, 64), (3, 2, 64), (4, 2, 64), (6, 2, 64)):
            tma_stream(lib, A, g, 128, 2, S, reps=2, variant=variant, threads=threads)
            ns, tbs = tma_stream(lib, A, g, 128, 2, S, reps=48, variant=variant, threads=threads)
            how = "incremental indices" if variant & 2 else "indices by division"
            res.append(f"streaming probe, S={S}, {how}: {tbs * 1e3 / g:6.1f}")
        print(f"  {g:3d} CTAs: " + ", ".join(res))



def intake_with_smem_reads(lib, grid=128):
    """TMA intake from L2 while other warps of the CTA read shared memory as
    fast as they can: whether TMA's writes and shared-memory reads share one
    shared-memory bandwidth (GB/s per SM)."""
    import torch
    out = torch.zeros(grid * 8, dtype=torch.int64, device="cuda")
    P = torch.zeros(grid * 4 * 6 * 4096, dtype=torch.uint8, device="cuda")
    A = torch.randn(128 * grid, 512, device="cuda").to(torch.bfloat16)
    n = 12288
    for W, use in ((0, 1), (1, 0), (2, 0), (4, 0), (1, 1), (2, 1), (4, 1)):
        tma, rd = intake(lib, A, P, out, grid, W, 192 if use else 0, -n)
        print(f"  W={W} tma={use}: " + (f"TMA {tma:6.1f}; " if tma else "") +
              "shared reads " + ", ".join(f"{c:6.1f}" for c in rd) +
              f"; reads {sum(rd):6.1f}, all {(tma or 0) + sum(rd):6.1f}")



def cross_check(lib, grid=128):
    """Each TMA probe kernel launched with the other probe's host-built tensor
    map (same matrix and copy pattern): GB/s per SM."""
    import torch
    out = torch.zeros(grid * 8, dtype=torch.int64, device="cuda")
    P = torch.zeros(grid * 4 * 6 * 4096, dtype=torch.uint8, device="cuda")
    A = torch.randn(128 * grid, 512, device="cuda").to(torch.bfloat16)
    for rep in range(2):
        a, _ = intake(lib, A, P, out, grid, 0, 192, 0)
        # the intake host code launching the streaming kernel (out[b], one per CTA)
        for _ in range(2):
            rc = lib.probe_intake(A.data_ptr(), A.shape[0], A.shape[1], 1, P.data_ptr(), P.numel(), grid, 0,
                                  192, 0, 2, out.data_ptr())
            if rc != 0:
                raise RuntimeError(f"probe_intake rc {rc}")
        b = 192 * 32768 / float(out[:grid].double().median())
        _, c = tma_stream(lib, A, grid, 128, 2, 3, reps=48, variant=1)
        # the streaming host code launching the intake kernel (out[8 b])
        o2 = torch.zeros(grid * 8, dtype=torch.int64, device="cuda")
        N, K = A.shape
        for _ in range(2):
            rc = lib.probe_tma_stream(A.data_ptr(), N, K, grid, 128, 2, 3, 0, 3, 48, 4, 64, o2.data_ptr())
            if rc != 0:
                raise RuntimeError(f"probe_tma_stream rc {rc}")
        d = 192 * 32768 / float(o2.view(-1, 8)[:, 0].double().median())
        print(f"  intake kernel + intake map {a:6.1f}, streaming kernel + intake map {b:6.1f}, "
              f"streaming kernel + streaming map {c * 1e3 / grid:6.1f}, intake kernel + streaming map {d:6.1f}")


if __name__ == "__main__":
    main()
