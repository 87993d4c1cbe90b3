"""Pins for the oracle's FP8 inputs (the OCP E4M3 and E5M2 formats of the FP8 GEMM
variant the Ada page lists as written but untested): every bit pattern decodes
like torch's float8 types, the input generator rounds like torch's casts, and a
GEMM on FP8 inputs equals exact rational arithmetic.  No GPU."""
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_decode_all_fp8_patterns(fmt):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.decode(codes, fmt)
    ref = torch.from_numpy(codes).view(TORCH_FP8[fmt]).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(dec[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(dec[ok]), np.signbit(ref[ok]))


@pytest.mark.parametrize("fmt,limit", [("e4m3", 448.0), ("e5m2", 57344.0)])
def test_format_facts(fmt, limit):
    dec = oracle.decode(np.arange(256, dtype=np.uint8), fmt)
    assert np.nanmax(dec[np.isfinite(dec)]) == limit
    if fmt == "e4m3":
        assert not np.any(np.isinf(dec)) and np.sum(np.isnan(dec)) == 2   # S.1111.111
    else:
        assert np.sum(np.isinf(dec)) == 2 and np.sum(np.isnan(dec)) == 6


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_generator_rounds_like_torch(fmt):
    x = (np.random.default_rng(1).standard_normal(200000) * 30).astype(np.float32)
    lim = 448.0 if fmt == "e4m3" else 57344.0
    x = np.clip(x, -lim, lim)
    mine = si.to_bits(x, fmt)
    ref = torch.from_numpy(x).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, ref)


@pytest.mark.parametrize("seed", range(10))
def test_fp8_gemm_brute_force_exact(seed):
    """FP8 values are dyadic with few bits, so the oracle must equal exact rational
    arithmetic of alpha*AB + beta*C."""
    rnd = random.Random(77 + seed)
    fmt = rnd.choice(["e4m3", "e5m2"])
    M, N, K = rnd.randint(1, 6), rnd.randint(1, 6), rnd.randint(1, 12)
    a_col, b_col = rnd.random() < 0.5, rnd.random() < 0.5
    alpha, beta = rnd.choice([1.0, 0.5, -2.0]), rnd.choice([0.0, 1.0, -0.25])
    Av = np.array([[rnd.randint(-48, 48) / 8 for _ in range(K)] for _ in range(M)], np.float32)
    Bv = np.array([[rnd.randint(-48, 48) / 8 for _ in range(N)] for _ in range(K)], np.float32)
    A, B = si.to_bits(Av, fmt), si.to_bits(Bv, fmt)
    a, b = oracle.decode(A, fmt), oracle.decode(B, fmt)   # the stored values
    C = si.to_bits(np.array([[rnd.randint(-64, 64) / 16 for _ in range(N)] for _ in range(M)],
                            np.float32), "f32")
    c = oracle.decode(C, "f32")
    As = np.ascontiguousarray(A.T) if a_col else A
    Bs = np.ascontiguousarray(B.T) if b_col else B
    bits, exact, _ = oracle.gemm(As, Bs, M=M, N=N, K=K, in_dtype=fmt, out_dtype="f32",
                                 a_col=a_col, b_col=b_col, alpha=alpha, beta=beta, C=C)
    for i in range(M):
        for j in range(N):
            r = Fraction(alpha) * sum((Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(K)),
                                      Fraction(0))
            if beta != 0:
                r += Fraction(beta) * Fraction(c[i, j])
            assert Fraction(exact[i, j]) == r
