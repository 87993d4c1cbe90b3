"""Pins for the oracle's fused epilogue (bias + ReLU after alpha*AB + beta*C, one
rounding): a hand-worked extension of the GEMM page's printed example, exact
rational arithmetic on dyadic inputs, a closed form and the special cases.  No GPU."""
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "bias_relu_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    out, i = {}, 0
    while i < len(rows):
        tag = rows[i][0]
        if len(rows[i]) == 3:
            r, c = int(rows[i][1]), int(rows[i][2])
            out[tag] = np.array([[float(x) for x in rows[i + 1 + k]] for k in range(r)])
            i += 1 + r
        else:
            out[tag] = np.array([float(x) for x in rows[i + 1]], np.float32)
            assert out[tag].size == int(rows[i][1])
            i += 2
    return out


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", ["col", "row"])
@pytest.mark.parametrize("relu", [False, True])
def test_worked_example_bias_relu(out_dtype, kind, relu):
    g = _golden()
    A = si.to_bits(g["A"].astype(np.float32), "bf16")
    B = si.to_bits(g["B"].astype(np.float32), "bf16")
    bits, exact, _ = oracle.gemm(A, B, M=2, N=2, K=3, in_dtype="bf16", out_dtype=out_dtype,
                                 bias=g["bias_" + kind], bias_kind=kind, relu=relu)
    want = g[kind + ("_relu" if relu else "")]
    np.testing.assert_array_equal(exact, want)
    np.testing.assert_array_equal(oracle.decode(bits, out_dtype), want)


def _exact(Av, Bv, alpha, beta, Cv, bias, kind, relu):
    M, K, N = len(Av), len(Av[0]), len(Bv[0])
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((Fraction(Av[i][k]) * Fraction(Bv[k][j]) for k in range(K)), Fraction(0))
            r = Fraction(alpha) * s
            if beta != 0:
                r += Fraction(beta) * Fraction(Cv[i][j])
            if kind == "col":
                r += Fraction(float(bias[j]))
            elif kind == "row":
                r += Fraction(float(bias[i]))
            if relu and r < 0:
                r = Fraction(0)
            row.append(r)
        out.append(row)
    return out


def _round_ref(x, fmt):
    if fmt == "f32":
        return int(np.array([x], np.float32).view(np.uint32)[0])
    if fmt == "f16":
        return int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
    return int(torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


@pytest.mark.parametrize("seed", range(16))
def test_brute_force_dyadic_exact_bias_relu(seed):
    """Dyadic inputs keep every step exact, so the oracle must equal exact rational
    arithmetic of relu(alpha*AB + beta*C + bias) and round like an independent
    library cast.  Shapes are non-square, so a row/column mix-up of the bias, a
    ReLU before the bias or a bias scaled by alpha all fail."""
    rnd = random.Random(1000 + seed)
    M, N, K = rnd.randint(1, 6), rnd.randint(1, 6), rnd.randint(1, 9)
    while M == N:
        N = rnd.randint(1, 7)
    in_dtype = rnd.choice(["f16", "bf16"])
    out_dtype = rnd.choice(["f32", "bf16", "f16"])
    a_col, b_col = rnd.random() < 0.5, rnd.random() < 0.5
    alpha = rnd.choice([1.0, 2.0, -0.5, 1.25])
    beta = rnd.choice([0.0, 0.5, -1.0])
    kind = rnd.choice(["col", "row"])
    relu = rnd.random() < 0.6
    Av = [[rnd.randint(-64, 64) / 16 for _ in range(K)] for _ in range(M)]
    Bv = [[rnd.randint(-64, 64) / 16 for _ in range(N)] for _ in range(K)]
    Cv = [[rnd.randint(-64, 64) / 16 for _ in range(N)] for _ in range(M)]
    bias = np.array([rnd.randint(-256, 256) / 16 for _ in range(N if kind == "col" else M)],
                    np.float32)
    A = si.to_bits(np.array(Av, np.float32).reshape(M, K), in_dtype)
    B = si.to_bits(np.array(Bv, np.float32).reshape(K, N), in_dtype)
    C = si.to_bits(np.array(Cv, np.float32).reshape(M, N), out_dtype)
    Cv = oracle.decode(C, out_dtype).tolist()
    As = np.ascontiguousarray(A.T) if a_col else A
    Bs = np.ascontiguousarray(B.T) if b_col else B
    bits, exact, _ = oracle.gemm(As, Bs, M=M, N=N, K=K, in_dtype=in_dtype, out_dtype=out_dtype,
                                 a_col=a_col, b_col=b_col, alpha=alpha, beta=beta, C=C,
                                 bias=bias, bias_kind=kind, relu=relu)
    ref = _exact(Av, Bv, alpha, beta, Cv, bias, kind, relu)
    for i in range(M):
        for j in range(N):
            assert Fraction(exact[i, j]) == ref[i][j]
            assert int(bits[i, j]) == _round_ref(float(ref[i][j]), out_dtype)


@pytest.mark.parametrize("kind", ["col", "row"])
def test_all_ones_closed_form_with_bias(kind):
    """A = B = 1 (M x K, K x N): relu(alpha*K + beta*c + bias)."""
    M, N, K, alpha, beta = 5, 7, 11, 0.5, -1.0
    A = si.to_bits(np.ones((M, K), np.float32), "bf16")
    B = si.to_bits(np.ones((K, N), np.float32), "bf16")
    c = np.arange(M * N, dtype=np.float32).reshape(M, N) / 4
    C = si.to_bits(c, "f32")
    bias = (np.arange(N if kind == "col" else M, dtype=np.float32) - 8.0)
    bits, exact, _ = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="bf16", out_dtype="f32",
                                 alpha=alpha, beta=beta, C=C, bias=bias, bias_kind=kind,
                                 relu=True)
    b2 = bias[None, :] if kind == "col" else bias[:, None]
    want = np.maximum(alpha * K + beta * c.astype(np.float64) + b2, 0.0)
    np.testing.assert_array_equal(exact, want)


def test_relu_keeps_nan_and_zero_bias_is_identity():
    M, N, K = 3, 4, 5
    rnd = np.random.default_rng(7)
    A = si.to_bits(rnd.uniform(-1, 1, (M, K)).astype(np.float32), "f16")
    B = si.to_bits(rnd.uniform(-1, 1, (K, N)).astype(np.float32), "f16")
    C = si.to_bits(np.zeros((M, N), np.float32), "f32")
    C[1, 2] = 0x7FC00000                     # NaN in C, read because beta != 0
    bits, exact, _ = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="f32",
                                 beta=1.0, C=C, bias=np.zeros(N, np.float32), bias_kind="col",
                                 relu=True)
    assert np.isnan(exact[1, 2]) and np.isnan(_f32(bits)[1, 2])
    # with a zero bias and no ReLU the epilogue is the plain GEMM, bit for bit
    b0, e0, s0 = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16")
    b1, e1, s1 = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16",
                             bias=np.zeros(M, np.float32), bias_kind="row")
    np.testing.assert_array_equal(b0, b1)
    np.testing.assert_array_equal(e0, e1)
    # ReLU alone clamps exactly the negative results
    b2, e2, _ = oracle.gemm(A, B, M=M, N=N, K=K, in_dtype="f16", out_dtype="bf16", relu=True)
    np.testing.assert_array_equal(e2, np.where(e0 < 0, 0.0, e0))


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_bias_length_is_checked():
    A = si.to_bits(np.ones((2, 3), np.float32), "bf16")
    B = si.to_bits(np.ones((3, 4), np.float32), "bf16")
    with pytest.raises(AssertionError):
        oracle.gemm(A, B, M=2, N=4, K=3, in_dtype="bf16", out_dtype="f32",
                    bias=np.zeros(2, np.float32), bias_kind="col")
