"""Pins for the CPU oracle: each ties it to the pages or to mathematics, never
to itself.  CPU only.

* worked example and its BK = 2 partial sums (golden fixtures, cited there);
* brute force on tiny random shapes against exactly rounded sums (math.fsum of
  exact products) and against numpy's float64 matmul;
* special cases: identity, permutation, all-ones, zero K;
* the number-format decoders against hand-worked bit patterns and against
  numpy's own float16 / float32 conversions (all 65536 half patterns);
* the round-to-nearest-even encoders against numpy (f16, f32) and torch (bf16
  from exactly representable float32 inputs), with ties and overflow;
* the ulp used by the tolerance against numpy.spacing.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from oracle import tiled_model as tm
from tests.conftest import parse_matrix, parse_numbers, read_golden
from tiled_matrix_multiplication_gb300 import inputs

FMTS = ("f16", "bf16", "f32")


def _bits_of(x: np.ndarray, fmt: str) -> np.ndarray:
    """Exactly representable float64 values -> bit patterns via numpy/torch
    (independent of the oracle's encoder)."""
    if fmt == "f16":
        return x.astype(np.float16).view(np.uint16)
    if fmt == "f32":
        return x.astype(np.float32).view(np.uint32)
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _exact_ref(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """Correctly rounded sum of exact products, element by element."""
    M, K = A.shape
    N = B.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            out[i, j] = math.fsum(float(A[i, k]) * float(B[k, j]) for k in range(K))
    return out


# ------------------------------------------------------------ worked example

@pytest.mark.parametrize("fmt", FMTS)
def test_worked_example(oracle_lib, fmt):
    g = read_golden("worked_example.txt")
    A = np.array(parse_matrix(g["A"]))
    B = np.array(parse_matrix(g["B"]))
    C = np.array(parse_matrix(g["C"]))
    a_bits, b_bits = _bits_of(A, fmt), _bits_of(B, fmt)
    got, S = oracle.gemm_ref_bits(a_bits, b_bits, K=3, N=2, fmt=fmt)
    assert np.array_equal(got, C)
    assert np.array_equal(S, C)  # all products positive


def test_worked_example_bk2_partials():
    g = read_golden("worked_example.txt")
    p = read_golden("bk2_partials.txt")
    A = np.array(parse_matrix(g["A"]))
    B = np.array(parse_matrix(g["B"]))
    run = tm.tiled_gemm(A, B, bm=2, bn=2, bk=int(p["BK"]), trace=(0, 0))
    assert run.trace == parse_numbers(p["C00_partials"])
    assert run.C[0, 0] == float(p["C00"])
    assert np.array_equal(run.C, np.array(parse_matrix(g["C"])))
    # the mistake the lesson warns about -- resetting the accumulator in every
    # K chunk -- would leave only the last partial
    assert run.trace[-1] == float(p["C00_if_acc_reset_per_chunk"])
    assert run.trace[-1] != run.C[0, 0]


# --------------------------------------------------------------- brute force

@pytest.mark.parametrize("fmt", FMTS)
def test_brute_force_tiny_shapes(oracle_lib, fmt):
    rng = np.random.default_rng(1234)
    for trial in range(40):
        M, N, K = (int(x) for x in rng.integers(1, 18, size=3))
        a = inputs.matrix_bits(M, K, fmt, "uniform", 100 + trial)
        b = inputs.matrix_bits(K, N, fmt, "uniform", 200 + trial)
        A = oracle.decode(a, fmt)
        B = oracle.decode(b, fmt)
        C, S = oracle.gemm_ref(A, B)
        exact = _exact_ref(A, B)
        Sx = np.abs(A) @ np.abs(B)
        # sequential double summation: |err| <= (K-1) * 2^-53 * S  (tiny K)
        assert np.all(np.abs(C - exact) <= K * 2.0 ** -52 * Sx + 1e-300), (M, N, K)
        assert np.allclose(S, Sx, rtol=K * 2.0 ** -51, atol=0)
        np.testing.assert_allclose(C, A @ B, rtol=0, atol=float(K * 2.0 ** -50 * Sx.max()))


def test_integer_inputs_exact(oracle_lib):
    for M, N, K in [(5, 7, 5), (17, 3, 33), (1, 1, 1), (8, 9, 64)]:
        a = inputs.matrix_bits(M, K, "f16", "int", 7)
        b = inputs.matrix_bits(K, N, "f16", "int", 8)
        A, B = oracle.decode(a, "f16"), oracle.decode(b, "f16")
        C, _ = oracle.gemm_ref(A, B)
        Ai, Bi = A.astype(np.int64), B.astype(np.int64)
        assert np.array_equal(C, (Ai @ Bi).astype(np.float64))


def test_rows_subset_matches_full(oracle_lib):
    a = inputs.matrix_bits(20, 11, "bf16", "normal", 3)
    b = inputs.matrix_bits(11, 9, "bf16", "normal", 4)
    A, B = oracle.decode(a, "bf16"), oracle.decode(b, "bf16")
    C, S = oracle.gemm_ref(A, B)
    rows = [19, 0, 7, 7]
    Cr, Sr = oracle.gemm_ref(A, B, rows=rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])


def test_strided_operands_ignore_padding(oracle_lib):
    a = inputs.matrix_bits(6, 5, "f16", "uniform", 1, ld=13)   # NaN padding
    b = inputs.matrix_bits(5, 4, "f16", "uniform", 2, ld=9)
    C, _ = oracle.gemm_ref_bits(a, b, K=5, N=4, fmt="f16")
    assert np.isfinite(C).all()
    C2, _ = oracle.gemm_ref_bits(np.ascontiguousarray(a[:, :5]), np.ascontiguousarray(b[:, :4]),
                                 K=5, N=4, fmt="f16")
    assert np.array_equal(C, C2)


# ------------------------------------------------------------- special cases

@pytest.mark.parametrize("fmt", FMTS)
def test_identity_and_permutation(oracle_lib, fmt):
    M, K = 9, 12
    a = inputs.matrix_bits(M, K, fmt, "uniform", 11)
    A = oracle.decode(a, fmt)
    C, _ = oracle.gemm_ref(A, np.eye(K))
    assert np.array_equal(C, A)
    perm = np.random.default_rng(5).permutation(K)
    P = np.zeros((K, K))
    P[perm, np.arange(K)] = 1.0       # column j of P selects row perm[j]
    C, _ = oracle.gemm_ref(A, P)
    assert np.array_equal(C, A[:, perm])
    C, _ = oracle.gemm_ref(P.T, A.T)  # row permutation from the left
    assert np.array_equal(C, A.T[perm])


def test_ones_gives_column_sums(oracle_lib):
    b = inputs.matrix_bits(10, 6, "f32", "uniform", 21)
    B = oracle.decode(b, "f32")
    C, _ = oracle.gemm_ref(np.ones((3, 10)), B)
    for j in range(6):
        assert np.all(C[:, j] == math.fsum(B[:, j])) or np.allclose(C[:, j], math.fsum(B[:, j]),
                                                                   rtol=1e-15, atol=0)


def test_zero_k_is_empty_sum(oracle_lib):
    C, S = oracle.gemm_ref(np.zeros((3, 0)), np.zeros((0, 4)))
    assert C.shape == (3, 4) and not C.any() and not S.any()


def test_rejects_bad_arguments(oracle_lib):
    with pytest.raises(ValueError):
        oracle.gemm_ref(np.zeros((2, 3)), np.zeros((4, 2)))
    with pytest.raises(ValueError):
        oracle.gemm_ref(np.zeros((2, 3)), np.zeros((3, 2)), rows=[2])


# ------------------------------------------------------------------- formats

def test_decode_hand_worked_patterns(oracle_lib):
    cases = {
        "f16": [(0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0400, 2.0 ** -14),
                (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x3555, 0.333251953125),
                (0x8000, -0.0)],
        "bf16": [(0x3F80, 1.0), (0x4049, 3.140625), (0xBF00, -0.5), (0x0080, 2.0 ** -126),
                 (0x0001, 2.0 ** -133), (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127)],
        "f32": [(0x3F800000, 1.0), (0x00000001, 2.0 ** -149), (0x00800000, 2.0 ** -126),
                (0x7F7FFFFF, (2 - 2.0 ** -23) * 2.0 ** 127), (0xC0490FDB, -3.1415927410125732)],
    }
    for fmt, pairs in cases.items():
        for bits, val in pairs:
            got = oracle.decode(np.array([bits], dtype=np.uint32 if fmt == "f32" else np.uint16), fmt)[0, 0]
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (fmt, hex(bits))
    for fmt, inf_bits, nan_bits in [("f16", 0x7C00, 0x7E00), ("bf16", 0x7F80, 0x7FC0),
                                    ("f32", 0x7F800000, 0x7FC00000)]:
        dt = np.uint32 if fmt == "f32" else np.uint16
        assert oracle.decode(np.array([inf_bits], dtype=dt), fmt)[0, 0] == math.inf
        assert math.isnan(oracle.decode(np.array([nan_bits], dtype=dt), fmt)[0, 0])


def test_decode_all_half_and_bfloat_patterns(oracle_lib):
    allp = np.arange(65536, dtype=np.uint16)
    got = oracle.decode(allp, "f16")[0]
    ref = allp.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    got = oracle.decode(allp, "bf16")[0]
    with np.errstate(invalid="ignore"):
        ref = (allp.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_decode_f32_patterns(oracle_lib):
    pats = np.random.default_rng(9).integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    got = oracle.decode(pats, "f32")[0]
    with np.errstate(invalid="ignore"):
        ref = pats.view(np.float32).astype(np.float64)
    assert ((got == ref) | (np.isnan(got) & np.isnan(ref))).all()


def test_encode_half_against_numpy(oracle_lib):
    rng = np.random.default_rng(17)
    x = np.concatenate([
        rng.standard_normal(100_000) * 10.0 ** rng.integers(-9, 6, size=100_000),
        np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65504.0, 65519.99, 65520.0, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -26, -0.0, 0.0, 1e9, -1e9]),
    ])
    got = oracle.encode(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    # every finite half value round-trips
    allp = np.arange(65536, dtype=np.uint16)
    vals = allp.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    assert np.array_equal(oracle.encode(vals[fin], "f16"), allp[fin])


def test_encode_ties_and_overflow(oracle_lib):
    enc = lambda v, f: int(oracle.encode(np.array([v]), f)[0])  # noqa: E731
    assert enc(1 + 2.0 ** -11, "f16") == 0x3C00          # tie -> even (down)
    assert enc(1 + 3 * 2.0 ** -11, "f16") == 0x3C02      # tie -> even (up)
    assert enc(65520.0, "f16") == 0x7C00                 # halfway past max -> Inf
    assert enc(65519.0, "f16") == 0x7BFF
    assert enc(2.0 ** -25, "f16") == 0x0000              # half of min subnormal: tie -> 0
    assert enc(3 * 2.0 ** -25, "f16") == 0x0002          # 1.5 ulp -> 2 (even)
    assert enc(1 + 2.0 ** -8, "bf16") == 0x3F80          # tie -> even
    assert enc(1 + 3 * 2.0 ** -8, "bf16") == 0x3F82
    assert enc(-1.0, "bf16") == 0xBF80


def test_encode_bf16_against_torch(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    x32 = (rng.standard_normal(200_000) * 10.0 ** rng.integers(-30, 30, size=200_000)).astype(np.float32)
    x = x32.astype(np.float64)                       # exactly representable in f32
    got = oracle.encode(x, "bf16")
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_encode_f32_against_numpy(oracle_lib):
    rng = np.random.default_rng(29)
    x = rng.standard_normal(200_000) * 10.0 ** rng.integers(-40, 38, size=200_000)
    assert np.array_equal(oracle.encode(x, "f32"), x.astype(np.float32).view(np.uint32))


def test_ulp_against_numpy_spacing():
    for fmt, npt in [("f16", np.float16), ("f32", np.float32)]:
        x = np.array([1.0, 1.5, 3.0, 1000.0, 2.0 ** -20, 1e-3, 0.1, 60000.0 if fmt == "f16" else 1e30])
        ref = np.spacing(x.astype(npt)).astype(np.float64)
        assert np.array_equal(oracle.ulp(x, fmt), ref), fmt
    assert oracle.ulp(np.array([0.0]), "f16")[0] == 2.0 ** -24
    assert oracle.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert oracle.ulp(np.array([2.0 ** -130]), "bf16")[0] == 2.0 ** -133


def test_check_close_flags_nan_and_outliers():
    C_ref = np.array([[1.0, 2.0]])
    S = np.array([[1.0, 2.0]])
    ok, _ = oracle.check_close(np.array([[1.0, 2.0]]), C_ref, S, "f16", "f16")
    assert ok
    ok, _ = oracle.check_close(np.array([[1.0, np.nan]]), C_ref, S, "f16", "f16")
    assert not ok
    ok, _ = oracle.check_close(np.array([[1.0 + 0.9 * (2e-3 + 2.0 ** -10), 2.0]]), C_ref, S, "f16", "f16")
    assert ok
    ok, _ = oracle.check_close(np.array([[1.0 + 1.1 * (2e-3 + 2.0 ** -10), 2.0]]), C_ref, S, "f16", "f16")
    assert not ok
