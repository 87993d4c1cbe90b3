"""Pins for the CPU oracle: each test ties it to something other than itself --
values the GEMM pages print, exact rational arithmetic, closed forms, and
special cases that reduce to a known answer.  No GPU needed."""
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _parse_worked_example():
    rows = _read_golden("worked_example.txt")
    out, i = {}, 0
    while i < len(rows):
        tag = rows[i][0]
        if tag in ("A", "B", "C"):
            r, c = int(rows[i][1]), int(rows[i][2])
            out[tag] = np.array([[float(x) for x in rows[i + 1 + k]] for k in range(r)])
            assert out[tag].shape == (r, c)
            i += 1 + r
        else:
            out[tag] = float(rows[i][1])
            i += 1
    return out


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


# ------------------------------------------------------------ worked example

@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_worked_example(in_dtype, out_dtype):
    g = _parse_worked_example()
    A = si.to_bits(g["A"].astype(np.float32), in_dtype)
    B = si.to_bits(g["B"].astype(np.float32), in_dtype)
    bits, exact, scale = oracle.gemm(A, B, M=2, N=2, K=3, in_dtype=in_dtype,
                                     out_dtype=out_dtype)
    np.testing.assert_array_equal(exact, g["C"])
    np.testing.assert_array_equal(oracle.decode(bits, out_dtype), g["C"])
    assert oracle.flops(2, 2, 3) == g["flops"]
    # the page's two traffic models for FP32 elements
    M, N, K = 2, 2, 3
    assert round(oracle.flops(M, N, K) / (4 * M * N * (2 * K + 1)), 3) == g["scalar_load_model"]
    assert round(oracle.flops(M, N, K) / (4 * (M * K + K * N + M * N)), 3) == g["perfect_reuse_bound"]


def test_worked_example_storage_orders():
    """Same logical product from every storage order (non-symmetric fixture)."""
    g = _parse_worked_example()
    A = si.to_bits(g["A"].astype(np.float32), "f16")
    B = si.to_bits(g["B"].astype(np.float32), "f16")
    for a_col in (False, True):
        for b_col in (False, True):
            As = np.ascontiguousarray(A.T) if a_col else A
            Bs = np.ascontiguousarray(B.T) if b_col else B
            _, exact, _ = oracle.gemm(As, Bs, M=2, N=2, K=3, in_dtype="f16", out_dtype="f32",
                                      a_col=a_col, b_col=b_col)
            np.testing.assert_array_equal(exact, g["C"])


def test_flop_count_facts():
    for row in _read_golden("flop_counts.txt"):
        if row[0] == "flops":
            M, N, K, v = map(int, row[1:])
            assert oracle.flops(M, N, K) == v


# ------------------------------------------------------------ format facts

def test_format_facts_from_page():
    rows = _read_golden("format_facts.txt")
    for row in rows:
        if row[0] == "two_reference":
            continue
        x, fmt, want = float(row[0]), row[1], float(row[2])
        assert oracle.decode(oracle.encode(np.array([x]), fmt), fmt)[0] == want
    # two-reference example: A=[1.0001, 1], B=[1, -1]^T
    want = {r[1]: float(r[2]) for r in rows if r[0] == "two_reference"}
    a = np.array([[1.0001, 1.0]], dtype=np.float32)
    b = np.array([[1.0], [-1.0]], dtype=np.float32)
    bits, exact, _ = oracle.gemm(si.to_bits(a, "f16"), si.to_bits(b, "f16"), M=1, N=1, K=2,
                                 in_dtype="f16", out_dtype="f32")
    assert exact[0, 0] == want["rounded"] == 0.0
    original = float(np.float64(a[0, 0]) - 1.0)
    assert round(original, 8) == want["original"]


def test_decode_all_f16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_decode_all_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_decode_f32_patterns():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    bits[:6] = [0, 1, 0x7F7FFFFF, 0x80000001, 0x7F800000, 0x00800000]
    got = oracle.decode(bits, "f32")
    ref = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def _random_doubles(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(-1, 1, n)
    expo = rng.integers(-30, 20, n)
    x = np.ldexp(mant, expo)
    x[:8] = [0.0, -0.0, 65504.0, 65520.0, 65519.99, 2.0 ** -25, 2.0 ** -24 * 1.5, -1e300]
    return x


def test_encode_f16_matches_ieee_cast():
    x = _random_doubles(300000, 1)
    got = oracle.encode(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)      # numpy: binary64 -> binary16, RNE
    np.testing.assert_array_equal(got, ref)


def test_encode_f32_matches_ieee_cast():
    x = _random_doubles(300000, 2) * 1e10
    got = oracle.encode(x, "f32")
    ref = x.astype(np.float32).view(np.uint32)
    np.testing.assert_array_equal(got, ref)


def test_encode_bf16_matches_torch_on_binary32_values():
    # on values that are exact binary32 numbers, binary32 -> bf16 (torch, RNE)
    # is the same single rounding as binary64 -> bf16
    x = _random_doubles(300000, 3).astype(np.float32)
    got = oracle.encode(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_encode_bf16_ties_and_double_rounding():
    one = 1.0
    ulp = 2.0 ** -7
    cases = [
        (one + ulp / 2, 0x3F80),                    # tie, even below
        (one + 3 * ulp / 2, 0x3F82),                # tie, even above
        (one + ulp / 2 + 2.0 ** -40, 0x3F81),       # just above a tie: rounds up
        (-(one + ulp / 2), 0xBF80),
        (3.3895313892515355e38, 0x7F7F),            # largest finite bf16
        (3.40e38, 0x7F80),                          # rounds past the largest: inf
    ]
    for x, want in cases:
        assert oracle.encode(np.array([x]), "bf16")[0] == want, x


# ------------------------------------------------------------ closed forms

def test_identity_and_permutation():
    rng = np.random.default_rng(7)
    K, N = 24, 40
    Bv = si.normal(11, K * N, 1.0).reshape(K, N)
    B = si.to_bits(Bv, "bf16")
    Bexact = oracle.decode(B, "bf16")
    eye = si.to_bits(np.eye(K, dtype=np.float32), "bf16")
    bits, exact, _ = oracle.gemm(eye, B, M=K, N=N, K=K, in_dtype="bf16", out_dtype="f32")
    np.testing.assert_array_equal(exact, Bexact)
    np.testing.assert_array_equal(_f32(bits), Bexact.astype(np.float32))
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), perm] = 1.0
    bits, exact, _ = oracle.gemm(si.to_bits(P, "bf16"), B, M=K, N=N, K=K, in_dtype="bf16",
                                 out_dtype="f32")
    np.testing.assert_array_equal(exact, Bexact[perm])
    # B = identity on the right gives A back, column-major B storage
    A = si.to_bits(si.uniform_pm1(12, N * K).reshape(N, K), "f16")
    eyeK = si.to_bits(np.eye(K, dtype=np.float32), "f16")
    _, exact, _ = oracle.gemm(A, eyeK, M=N, N=K, K=K, in_dtype="f16", out_dtype="f32", b_col=True)
    np.testing.assert_array_equal(exact, oracle.decode(A, "f16"))


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.0, 0.5), (-0.5, -1.0)])
def test_all_ones_closed_form(alpha, beta):
    M, N, K = 5, 7, 33
    ones_a = si.to_bits(np.ones((M, K), np.float32), "f16")
    ones_b = si.to_bits(np.ones((K, N), np.float32), "f16")
    c = si.to_bits(np.full((M, N), 3.0, np.float32), "f32")
    _, exact, scale = oracle.gemm(ones_a, ones_b, M=M, N=N, K=K, in_dtype="f16",
                                  out_dtype="f32", alpha=alpha, beta=beta, C=c)
    np.testing.assert_array_equal(exact, np.full((M, N), alpha * K + beta * 3.0))
    np.testing.assert_array_equal(scale, np.full((M, N), float(K)))


def test_k_zero_and_beta_zero_skips_c():
    M, N = 3, 4
    a = np.zeros((M, 0), np.uint16)
    b = np.zeros((0, N), np.uint16)
    c = si.to_bits(np.arange(M * N, dtype=np.float32).reshape(M, N), "f32")
    _, exact, _ = oracle.gemm(a, b, M=M, N=N, K=0, in_dtype="f16", out_dtype="f32",
                              beta=2.0, C=c)
    np.testing.assert_array_equal(exact, 2.0 * np.arange(M * N).reshape(M, N))
    # beta == 0: C is not read, so NaN in C does not reach the output
    A = si.to_bits(np.ones((M, 2), np.float32), "f16")
    B = si.to_bits(np.ones((2, N), np.float32), "f16")
    cnan = np.full((M, N), 0x7FC00000, np.uint32)
    bits, exact, _ = oracle.gemm(A, B, M=M, N=N, K=2, in_dtype="f16", out_dtype="f32",
                                 beta=0.0, C=cnan)
    np.testing.assert_array_equal(exact, np.full((M, N), 2.0))


# ------------------------------------------------------------ brute force, exact rationals

def _exact_gemm(Av, Bv, alpha, beta, Cv):
    """Exact rational C = alpha*A*B + beta*C and S = sum |a||b|, as Fractions."""
    M, K = len(Av), len(Av[0])
    N = len(Bv[0])
    out, scl = [], []
    for i in range(M):
        ro, rs = [], []
        for j in range(N):
            s = Fraction(0)
            t = Fraction(0)
            for k in range(K):
                s += Fraction(Av[i][k]) * Fraction(Bv[k][j])
                t += abs(Fraction(Av[i][k])) * abs(Fraction(Bv[k][j]))
            r = Fraction(alpha) * s
            if beta != 0:
                r += Fraction(beta) * Fraction(Cv[i][j])
            ro.append(r)
            rs.append(t)
        out.append(ro)
        scl.append(rs)
    return out, scl


def _round_ref(x: float, fmt: str) -> int:
    """Reference rounding of an exact binary32 value (independent library casts)."""
    if fmt == "f32":
        return int(np.array([x], np.float32).view(np.uint32)[0])
    if fmt == "f16":
        return int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
    t = torch.tensor([x], dtype=torch.float32).to(torch.bfloat16)
    return int(t.view(torch.int16).item()) & 0xFFFF


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_dyadic_exact(seed):
    """Dyadic inputs (multiples of 1/16 in [-4, 4]) make every product and sum exact
    in binary64 and binary32, so the oracle must equal exact rational arithmetic,
    and its rounded output must equal an independent library rounding."""
    rnd = random.Random(seed)
    M, N, K = rnd.randint(1, 6), rnd.randint(1, 6), rnd.randint(1, 9)
    in_dtype = rnd.choice(["f16", "bf16"])
    out_dtype = rnd.choice(["f32", "bf16", "f16"])
    a_col, b_col = rnd.random() < 0.5, rnd.random() < 0.5
    alpha = rnd.choice([1.0, 2.0, -0.5, 1.25])
    beta = rnd.choice([0.0, 0.5, -1.0])
    Av = [[rnd.randint(-64, 64) / 16 for _ in range(K)] for _ in range(M)]
    Bv = [[rnd.randint(-64, 64) / 16 for _ in range(N)] for _ in range(K)]
    Cv = [[rnd.randint(-64, 64) / 16 for _ in range(N)] for _ in range(M)]
    A = si.to_bits(np.array(Av, np.float32).reshape(M, K), in_dtype)
    B = si.to_bits(np.array(Bv, np.float32).reshape(K, N), in_dtype)
    C = si.to_bits(np.array(Cv, np.float32).reshape(M, N), out_dtype)
    Cv = oracle.decode(C, out_dtype).tolist()  # values as stored in the output format
    As = np.ascontiguousarray(A.T) if a_col else A
    Bs = np.ascontiguousarray(B.T) if b_col else B
    bits, exact, scale = oracle.gemm(As, Bs, M=M, N=N, K=K, in_dtype=in_dtype,
                                     out_dtype=out_dtype, a_col=a_col, b_col=b_col,
                                     alpha=alpha, beta=beta, C=C)
    ref, refs = _exact_gemm(Av, Bv, alpha, beta, Cv)
    for i in range(M):
        for j in range(N):
            assert Fraction(exact[i, j]) == ref[i][j]
            assert Fraction(scale[i, j]) == refs[i][j]
            assert int(bits[i, j]) == _round_ref(float(ref[i][j]), out_dtype)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_general_within_fp64_bound(seed):
    """Seeded workload-style inputs (uniform / normal, rounded to fp16 / bf16): the
    oracle's binary64 sum stays within the binary64 accumulation bound
    K * 2^-53 * S of the exact rational value."""
    rnd = random.Random(100 + seed)
    M, N, K = rnd.randint(1, 5), rnd.randint(1, 5), rnd.randint(1, 40)
    in_dtype = rnd.choice(["f16", "bf16"])
    A = si.to_bits(si.normal(seed, M * K, 1.0).reshape(M, K), in_dtype)
    B = si.to_bits(si.uniform_pm1(seed + 50, K * N).reshape(K, N), in_dtype)
    _, exact, scale = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype="f32")
    Av = oracle.decode(A, in_dtype).tolist()
    Bv = oracle.decode(B, in_dtype).tolist()
    ref, refs = _exact_gemm(Av, Bv, 1.0, 0.0, None)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(exact[i, j]) - ref[i][j])
            assert err <= Fraction(K) * Fraction(2) ** -53 * refs[i][j]
            assert abs(Fraction(scale[i, j]) - refs[i][j]) <= Fraction(K) * Fraction(2) ** -53 * refs[i][j]


def test_row_subset_matches_full():
    w = si.workload_operands(1)
    M = N = K = 512
    bits, exact, scale = oracle.gemm(w["A"][:, :], w["B"], M=M, N=N, K=K, in_dtype="f16",
                                     out_dtype="f32")
    rows = [0, 17, 255, 511, 3]
    b2, e2, s2 = oracle.gemm(w["A"], w["B"], M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                             rows=rows)
    np.testing.assert_array_equal(b2, bits[rows])
    np.testing.assert_array_equal(e2, exact[rows])
    np.testing.assert_array_equal(s2, scale[rows])


def test_thread_count_does_not_change_result():
    w = si.workload_operands(1)
    r1 = oracle.gemm(w["A"], w["B"], M=512, N=512, K=512, in_dtype="f16", out_dtype="f32",
                     rows=list(range(40)), nthreads=1)
    r4 = oracle.gemm(w["A"], w["B"], M=512, N=512, K=512, in_dtype="f16", out_dtype="f32",
                     rows=list(range(40)), nthreads=4)
    for x, y in zip(r1, r4):
        np.testing.assert_array_equal(x, y)
