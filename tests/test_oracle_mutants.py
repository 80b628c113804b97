"""Plants plausible mistakes in a copy of the oracle's C source and checks that
the pins catch every one of them.  CPU only; the mutants are compiled into a
temporary directory and never touch the real oracle library.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

from oracle import ref
from tests.conftest import parse_matrix, read_golden
from tiled_matrix_multiplication_gb300 import inputs

SRC = os.path.join(os.path.dirname(ref.__file__), "gemm_ref.c")

MUTANTS = {
    "drop_last_k_term": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k < K - 1; ++k) {"),
    "reversed_k_on_B": ("const double *b = B + k * ldb;", "const double *b = B + (K - 1 - k) * ldb;"),
    "reversed_k_on_A": ("const double a = A[i * lda + k];", "const double a = A[i * lda + (K - 1 - k)];"),
    "wrong_sign": ("c[j] += p;", "c[j] -= p;"),
    "acc_reset_each_k": ("c[j] += p;", "c[j] = p;"),
    "abs_sum_signed": ("s[j] += fabs(p);", "s[j] += p;"),
    "row_subset_ignored": ("const int64_t i = rows ? rows[r] : r;", "const int64_t i = r;"),
    "decode_exponent_off_by_one": ("(int)e - bias - frac_bits);", "(int)e - bias - frac_bits + 1);"),
    "decode_subnormal_scale": ("ldexp((double)f, 1 - bias - frac_bits);", "ldexp((double)f, -bias - frac_bits);"),
    "encode_truncates": ("rint(ax / quantum)", "floor(ax / quantum)"),
    "encode_bias": ("(uint32_t)(e + bias) << frac_bits", "(uint32_t)(e + bias - 1) << frac_bits"),
    "encode_no_overflow": ("if (v >= ldexp(1.0, emax + 1))", "if (0)"),
    "encode_late_overflow": ("if (v >= ldexp(1.0, emax + 1))", "if (v > ldexp(1.0, emax + 2))"),
    "e4m3_ieee_top_binade": ("if (e == 0xFu && f == 7u)", "if (e == 0xFu)"),
    "e4m3_bias": ("ldexp((double)(f | 8u), (int)e - 7 - 3)", "ldexp((double)(f | 8u), (int)e - 8 - 3)"),
    "e4m3_subnormal_scale": ("ldexp((double)f, 1 - 7 - 3)", "ldexp((double)f, -7 - 3)"),
    "e4m3_encode_overflow_early": ("if (v >= 480.0)", "if (v >= 448.0)"),
    "e4m3_encode_truncates": ("const double v = rint(ax / quantum) * quantum;\n    if (v >= 480.0)",
                              "const double v = floor(ax / quantum) * quantum;\n    if (v >= 480.0)"),
    "e5m2_as_e4m3": ("case ORC_E5M2: return decode_bits(bits & 0xFFu, 5, 2);",
                     "case ORC_E5M2: return decode_bits(bits & 0xFFu, 4, 3);"),
}


def _fsum_ref(A, B):
    M, K = A.shape
    N = B.shape[1]
    return np.array([[math.fsum(float(A[i, k]) * float(B[k, j]) for k in range(K))
                      for j in range(N)] for i in range(M)])


def battery(lib) -> list[str]:
    """Run the oracle pins against ``lib``; returns the names of failed pins."""
    failed = []
    g = read_golden("worked_example.txt")
    A = np.array(parse_matrix(g["A"]))
    B = np.array(parse_matrix(g["B"]))
    C = np.array(parse_matrix(g["C"]))
    for fmt in ("f16", "bf16", "f32"):
        a_bits = ref.encode(A, fmt, lib=lib)
        b_bits = ref.encode(B, fmt, lib=lib)
        got, S = ref.gemm_ref_bits(a_bits, b_bits, K=3, N=2, fmt=fmt, lib=lib)
        if not (np.array_equal(got, C) and np.array_equal(S, C)):
            failed.append(f"worked_example_{fmt}")
    for trial in range(6):
        M, N, K = 3 + trial, 5 + trial, 4 + 2 * trial
        a = inputs.matrix_bits(M, K, "f16", "uniform", 500 + trial)
        b = inputs.matrix_bits(K, N, "f16", "uniform", 600 + trial)
        Ad, Bd = ref.decode(a, "f16", lib=lib), ref.decode(b, "f16", lib=lib)
        Cm, Sm = ref.gemm_ref(Ad, Bd, lib=lib)
        Ax = a.view(np.float16).astype(np.float64)
        Bx = b.view(np.float16).astype(np.float64)
        Sx = np.abs(Ax) @ np.abs(Bx)
        if not np.all(np.abs(Cm - _fsum_ref(Ax, Bx)) <= K * 2.0 ** -52 * Sx):
            failed.append("brute_force")
            break
        if not np.allclose(Sm, Sx, rtol=1e-12, atol=0):
            failed.append("abs_sum")
            break
        rows = [M - 1, 0]
        Cr, _ = ref.gemm_ref(Ad, Bd, rows=rows, lib=lib)
        if not np.array_equal(Cr, Cm[rows]):
            failed.append("row_subset")
            break
    allp = np.arange(65536, dtype=np.uint16)
    vals = allp.view(np.float16).astype(np.float64)
    got = ref.decode(allp, "f16", lib=lib)[0]
    if not ((got == vals) | (np.isnan(got) & np.isnan(vals))).all():
        failed.append("decode_f16")
    x = np.random.default_rng(3).standard_normal(20000) * 100.0
    x = np.concatenate([x, [65520.0, 70000.0, 1e6, 1 + 3 * 2.0 ** -11]])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    if not np.array_equal(ref.encode(x, "f16", lib=lib), want):
        failed.append("encode_f16")
    failed += fp8_pins(lib)
    return failed


def fp8_pins(lib) -> list[str]:
    """FP8 decode of all 256 patterns and encode of random values against
    torch's float8 types; the worked example exact in E4M3."""
    import torch
    failed = []
    allp = np.arange(256, dtype=np.uint8)
    for fmt, tdt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        want = torch.from_numpy(allp).view(tdt).to(torch.float64).numpy()
        got = ref.decode(allp, fmt, lib=lib)[0]
        if not ((got == want) | (np.isnan(got) & np.isnan(want))).all():
            failed.append(f"decode_{fmt}")
        top = 500.0 if fmt == "e4m3" else 60000.0
        x = np.random.default_rng(5).uniform(-top, top, 20000)
        x = np.concatenate([x, np.ldexp(np.random.default_rng(6).uniform(-1, 1, 5000), -8),
                            [464.0, 470.0, 1 + 2.0 ** -4, 1 + 3 * 2.0 ** -4, 2.0 ** -10]])
        if fmt == "e5m2":
            x = x[np.abs(x) < 57344.0]
        tw = torch.from_numpy(x).to(tdt).view(torch.uint8).numpy()
        if not np.array_equal(ref.encode(x, fmt, lib=lib), tw):
            failed.append(f"encode_{fmt}")
    g = read_golden("worked_example.txt")
    A = np.array(parse_matrix(g["A"]))
    B = np.array(parse_matrix(g["B"]))
    C = np.array(parse_matrix(g["C"]))
    got, _ = ref.gemm_ref_bits(ref.encode(A, "e4m3", lib=lib), ref.encode(B, "e4m3", lib=lib),
                               K=3, N=2, fmt="e4m3", lib=lib)
    if not np.array_equal(got, C):
        failed.append("worked_example_e4m3")
    return failed


def _build_variant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new))
    out = str(tmp_path / f"lib{name}.so")
    ref._compile(str(src), out, openmp=False)
    return ref.load(out)


def test_unmutated_copy_passes(tmp_path):
    lib = _build_variant(tmp_path, "control", "int orc_num_threads", "int orc_num_threads")
    assert battery(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert battery(lib), f"mutant {name} passed every pin"
