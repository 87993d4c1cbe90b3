"""Host-side checks of the hardware probes that need no GPU: the probe library
builds and exports its entry points, and each entry point rejects arguments that
would take a copy, a store or a launch outside its buffers (status -10, or -11 for
an unknown MMA shape) before making any CUDA call.  Only rejected argument sets
are passed, with null buffers, and only where no GPU is visible."""
import ctypes

import pytest

ENTRY_POINTS = ("probe_mma_rate", "probe_tma_stream", "probe_tma_mcast", "probe_store_rate",
                "probe_intake")


@pytest.fixture(scope="module")
def lib():
    import torch
    if torch.cuda.is_available():
        pytest.skip("argument checks are exercised only where no GPU can be reached")
    from dense_tensor_core_tcgen05_gb300 import probes
    return probes.build()


def test_probe_library_exports(lib):
    for name in ENTRY_POINTS:
        assert hasattr(lib, name), name


@pytest.mark.parametrize("args", [
    # C, M, N, ldc, grid_m, grid_n, mode
    (0, 2048, 2048, 2048, 16, 8, 5),        # no such route
    (0, 2048, 2048, 2048, 16, 8, -1),
    (0, 2048, 2048, 2048, 17, 8, 0),        # 17 x 128 rows > M
    (0, 2048, 2048, 2048, 16, 9, 0),        # 9 x 256 columns > N
    (0, 2048, 2048, 2047, 16, 8, 0),        # ldc < N
    (0, 2048, 2048, 2050, 16, 8, 0),        # row pitch not a multiple of 16 bytes
    (8, 2048, 2048, 2048, 16, 8, 0),        # base not 16-byte aligned
    (0, 2048, 2048, 2048, 0, 8, 0),         # empty grid
])
def test_store_rate_rejects(lib, args):
    assert lib.probe_store_rate(*args, None) == -10


@pytest.mark.parametrize("args", [
    # A, rows, cols, share, P, p_bytes, grid, W, tma_copies, cp_iters, bars_after_ring
    (0, 16384, 100, 1, 0, 128 * 4 * 6 * 4096, 128, 0, 192, 0, 0),    # cols < 128
    (0, 16384, 192, 1, 0, 128 * 4 * 6 * 4096, 128, 0, 192, 0, 0),    # cols not whole copies
    (0, 16383, 512, 1, 0, 128 * 4 * 6 * 4096, 128, 0, 192, 0, 0),    # rows < 128 per CTA
    (0, 16384, 512, 0, 0, 128 * 4 * 6 * 4096, 128, 0, 192, 0, 0),    # share < 1
    (0, 16384, 512, 1, 0, 128 * 4 * 6 * 4096, 128, 5, 192, 0, 0),    # more than 4 cp.async warps
    (0, 16384, 512, 1, 0, 128 * 4 * 6 * 4096 - 1, 128, 1, 192, 8, 0),  # P too small
    (0, 16384, 512, 1, 8, 128 * 4 * 6 * 4096, 128, 1, 192, 8, 0),    # P not 16-byte aligned
    (0, 16384, 512, 1, 0, 128 * 4 * 6 * 4096, 128, 1, 192, 8, 1),    # barriers over cp.async area
    (0, 16384, 512, 1, 0, 128 * 4 * 6 * 4096, 0, 0, 192, 0, 0),      # empty grid
])
def test_intake_rejects(lib, args):
    lib.probe_intake.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_longlong] + [ctypes.c_int] * 5 + \
                                [ctypes.c_void_p]
    assert lib.probe_intake(*args, None) == -10


@pytest.mark.parametrize("args", [
    # B, N, K, grid, R, KO, S, grouped, promo, reps, variant, threads
    (0, 16384, 512, 128, 128, 2, 3, 0, 3, 4, 0, 96),    # block size not 64 or 160
    (0, 16384, 512, 100, 128, 2, 3, 0, 3, 4, 0, 64),    # rows do not split over the grid
    (0, 16384, 512, 32, 512, 2, 3, 0, 3, 4, 0, 64),     # box taller than 256 rows
    (0, 16384, 480, 128, 128, 2, 3, 0, 3, 4, 0, 64),    # K not whole copies
    (0, 16384, 512, 128, 128, 2, 3, 0, 4, 4, 0, 64),    # no such L2 promotion
    (0, 16384, 512, 128, 128, 2, 0, 0, 3, 4, 0, 64),    # no slots
    (0, 16384, 512, 128, 128, 2, 3, 0, 3, 0, 0, 64),    # no passes
])
def test_tma_stream_rejects(lib, args):
    assert lib.probe_tma_stream(*args, None) == -10


def test_mma_rate_rejects(lib):
    assert lib.probe_mma_rate(256, 1, 151, 10, None) == -10    # a pair needs an even grid
    assert lib.probe_mma_rate(256, 0, 152, 0, None) == -10     # no iterations
    assert lib.probe_mma_rate(96, 0, 152, 10, None) == -11     # no such tile width
