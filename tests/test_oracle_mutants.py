"""The oracle's pins catch plausible mistakes.  Each case plants one mistake in a
temporary copy of the oracle's C source (a dropped term, a wrong sign, index or
precision, a transposed operand, a misplaced epilogue step), builds that copy on
the CPU, and runs the existing pin tests against it with the copy standing in
for the oracle: at least one pin must fail for every mistake.  The oracle
itself is not modified.  No GPU needed."""
import importlib.util
import os
import shutil

import pytest

import test_oracle_epilogue_pins as EP
import test_oracle_fp8_pins as F8
import test_oracle_pins as P

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

# (name, text in gemm_oracle.c, replacement): one planted mistake each
MUTANTS = [
    ("sign of the products", "acc[j] += a * b;", "acc[j] -= a * b;"),
    ("first k term dropped", "acc[j] += a * b;", "if (k > 0) acc[j] += a * b;"),
    ("last k term dropped", "for (int64_t k = 0; k < K; ++k) {\n            /* A is",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n            /* A is"),
    ("A storage orders swapped", "J->a_col ? k * J->lda + i : i * J->lda + k",
     "J->a_col ? i * J->lda + k : k * J->lda + i"),
    ("B storage orders swapped", "b_col ? j * ldb + k : k * ldb + j",
     "b_col ? k * ldb + j : j * ldb + k"),
    ("alpha dropped", "double r = J->alpha * acc[j];", "double r = acc[j];"),
    ("beta term dropped", "r += J->beta * decode(J->C_in, J->out_fmt, i * J->ldc + j);",
     "r += 0.0 * decode(J->C_in, J->out_fmt, i * J->ldc + j);"),
    ("C read transposed", "r += J->beta * decode(J->C_in, J->out_fmt, i * J->ldc + j);",
     "r += J->beta * decode(J->C_in, J->out_fmt, j * J->ldc + i);"),
    ("bias by row and column swapped",
     "if (J->bias_kind == OR_BIAS_COL) r += (double)J->bias[j];",
     "if (J->bias_kind == OR_BIAS_COL) r += (double)J->bias[i];"),
    ("ReLU before the bias",
     "if (J->bias_kind == OR_BIAS_COL) r += (double)J->bias[j];",
     "if (J->act == OR_ACT_RELU && r < 0.0) r = 0.0;\n"
     "            if (J->bias_kind == OR_BIAS_COL) r += (double)J->bias[j];"),
    ("ReLU keeps the negatives", "if (J->act == OR_ACT_RELU && r < 0.0) r = 0.0;",
     "if (J->act == OR_ACT_RELU && r > 0.0) r = 0.0;"),
    ("bf16 output with one extra bit", "double y = round_fmt(x, 8, -126, 127);",
     "double y = round_fmt(x, 9, -126, 127);"),
    ("fp16 subnormal scale", "return s | (uint16_t)ldexp(ay, 24);",
     "return s | (uint16_t)ldexp(ay, 23);"),
    ("scale term without |a|", "scl[j] += aa * fabs(b);", "scl[j] += fabs(b);"),
    ("ties rounded away from zero", "r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;",
     "r = fl + 1.0;"),
    ("rounding by truncation", "if (d > 0.5)\n        r = fl + 1.0;",
     "if (d > 2.0)\n        r = fl + 1.0;"),
    ("no overflow to infinity", "if (y > maxf) return copysign(INFINITY, x);",
     "if (y > maxf) return copysign(maxf, x);"),
    ("subnormal quantum not fixed", "if (E < emin) E = emin;        /* subnormal range: fixed quantum */",
     "/* subnormal range not special-cased */"),
    ("E4M3 exponent bias off by one", "v = ldexp((double)(8 + m), e - 10);",
     "v = ldexp((double)(8 + m), e - 11);"),
    ("E4M3 subnormals scaled as normals", "v = ldexp((double)m, -9);",
     "v = ldexp((double)(8 + m), -10);"),
    ("E4M3 with an infinity", "else if (e == 15 && m == 7)\n        v = NAN;",
     "else if (e == 15 && m == 7)\n        v = INFINITY;"),
    ("E5M2 infinity read as NaN",
     "/* m/4 * 2^(1-15) */\n    else if (e == 31)\n        v = m ? NAN : INFINITY;",
     "/* m/4 * 2^(1-15) */\n    else if (e == 31)\n        v = NAN;"),
    ("E5M2 mantissa with three bits", "int s = (b >> 7) & 1, e = (b >> 2) & 0x1F, m = b & 0x3;",
     "int s = (b >> 7) & 1, e = (b >> 2) & 0x1F, m = b & 0x7;"),
]

# the pins, as (test module, function, keyword arguments)
PINS = [
    (P, "test_worked_example", dict(in_dtype="bf16", out_dtype="f32")),
    (P, "test_worked_example", dict(in_dtype="f16", out_dtype="f16")),
    (P, "test_worked_example", dict(in_dtype="f16", out_dtype="bf16")),
    (P, "test_worked_example_storage_orders", {}),
    (P, "test_encode_f16_matches_ieee_cast", {}),
    (P, "test_encode_bf16_matches_torch_on_binary32_values", {}),
    (P, "test_encode_bf16_ties_and_double_rounding", {}),
    (P, "test_identity_and_permutation", {}),
    (P, "test_all_ones_closed_form", dict(alpha=2.0, beta=0.5)),
    (P, "test_k_zero_and_beta_zero_skips_c", {}),
    (P, "test_brute_force_dyadic_exact", dict(seed=0)),
    (P, "test_brute_force_dyadic_exact", dict(seed=1)),
    (P, "test_brute_force_general_within_fp64_bound", dict(seed=0)),
    (EP, "test_worked_example_bias_relu", dict(out_dtype="f32", kind="col", relu=True)),
    (EP, "test_worked_example_bias_relu", dict(out_dtype="f32", kind="row", relu=False)),
    (EP, "test_brute_force_dyadic_exact_bias_relu", dict(seed=0)),
    (EP, "test_brute_force_dyadic_exact_bias_relu", dict(seed=1)),
    (EP, "test_brute_force_dyadic_exact_bias_relu", dict(seed=2)),
    (EP, "test_brute_force_dyadic_exact_bias_relu", dict(seed=3)),
    (F8, "test_decode_all_fp8_patterns", dict(fmt="e4m3")),
    (F8, "test_decode_all_fp8_patterns", dict(fmt="e5m2")),
    (F8, "test_fp8_gemm_brute_force_exact", dict(seed=0)),
]


def _mutant_oracle(tmp_path, idx, old, new):
    d = tmp_path / f"oracle_mut{idx}"
    shutil.copytree(ORACLE_DIR, d, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    src = d / "gemm_oracle.c"
    text = src.read_text()
    assert text.count(old) == 1, f"the mistake's anchor must be unique: {old!r}"
    src.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mut{idx}", d / "__init__.py",
                                                  submodule_search_locations=[str(d)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def _failing_pins(monkeypatch, mod):
    failed = []
    for module, name, kwargs in PINS:
        with monkeypatch.context() as m:
            m.setattr(module, "oracle", mod)
            try:
                getattr(module, name)(**kwargs)
            except Exception:   # an assertion, or the pin's own check failing otherwise
                failed.append(name)
    return failed


def test_pins_pass_on_the_oracle(monkeypatch):
    """The battery itself is green on the unmodified oracle."""
    import oracle
    assert _failing_pins(monkeypatch, oracle) == []


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, idx):
    name, old, new = MUTANTS[idx]
    mod = _mutant_oracle(tmp_path, idx, old, new)
    failed = _failing_pins(monkeypatch, mod)
    assert failed, f"no pin caught the planted mistake: {name}"
