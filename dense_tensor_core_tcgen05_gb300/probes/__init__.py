"""Hardware probes behind the GEMM's design (measurement tooling, not the GEMM path).

    python -m dense_tensor_core_tcgen05_gb300.probes

prints (1) the tcgen05.mma rate per tile width (cycles per instruction and dense
FLOP/clk/SM, one issuing thread per CTA or CTA pair, all SMs busy) and (2) the
bandwidth at which TMA tile copies stream an 8192 x 8192 K-major bf16 matrix, per
copy shape (rows x consecutive 64-element blocks per row).  The probes are built
from probes.cu into _build/libprobes.so (sm_103a only).
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
    lib.probe_tma_stream.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 9 + [ctypes.c_void_p]
    lib.probe_tma_mcast.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 9 + [ctypes.c_void_p]
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


def tma_stream(lib, B, grid, R, KO, S, grouped=False, promo=3, reps=1):
    """(median in-kernel ns per CTA, TB/s) for streaming B [N, K] bf16 `reps` times."""
    import torch
    N, K = B.shape
    out = torch.zeros(grid, dtype=torch.int64, device="cuda")
    rc = lib.probe_tma_stream(B.data_ptr(), N, K, grid, R, KO, S, int(grouped), promo, reps,
                              out.data_ptr())
    if rc != 0:
        raise RuntimeError(f"probe_tma_stream rc {rc}")
    ns = statistics.median(out.cpu().tolist())
    return ns, reps * N * K * 2 / ns / 1e3


def main():
    import torch
    lib = build()
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


if __name__ == "__main__":
    main()
