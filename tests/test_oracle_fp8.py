"""Pins for the oracle's 8-bit formats (OCP FP8 E4M3 and E5M2): hand-worked
bit patterns, every pattern against torch's float8 types (an independent
library routine), round-to-nearest-even ties and overflow, the pages' worked
example (exact in E4M3), and brute force on small integer operands.  CPU only.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from tests.conftest import parse_matrix, read_golden
from tests.test_oracle_mutants import fp8_pins
from tiled_matrix_multiplication_gb300 import inputs


def test_library_and_worked_example_pins():
    assert fp8_pins(oracle.ref.load()) == []


@pytest.mark.parametrize("fmt,bits,value", [
    ("e4m3", 0x38, 1.0), ("e4m3", 0x7E, 448.0), ("e4m3", 0xFE, -448.0),
    ("e4m3", 0x08, 2.0 ** -6), ("e4m3", 0x07, 7 * 2.0 ** -9), ("e4m3", 0x01, 2.0 ** -9),
    ("e4m3", 0x78, 256.0), ("e4m3", 0x3C, 1.5), ("e4m3", 0x80, -0.0),
    ("e5m2", 0x3C, 1.0), ("e5m2", 0x7B, 57344.0), ("e5m2", 0x7C, math.inf),
    ("e5m2", 0xFC, -math.inf), ("e5m2", 0x04, 2.0 ** -14), ("e5m2", 0x01, 2.0 ** -16),
    ("e5m2", 0x3E, 1.5),
])
def test_hand_worked_patterns(fmt, bits, value):
    got = oracle.decode(np.array([bits], dtype=np.uint8), fmt)[0, 0]
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)
    assert int(oracle.encode(np.array([value]), fmt)[0]) == bits


@pytest.mark.parametrize("fmt,nans", [("e4m3", {0x7F, 0xFF}),
                                      ("e5m2", {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF})])
def test_nan_patterns(fmt, nans):
    v = oracle.decode(np.arange(256, dtype=np.uint8), fmt)[0]
    assert set(np.flatnonzero(np.isnan(v)).tolist()) == nans


def test_ties_and_overflow():
    enc = lambda x, f: int(oracle.encode(np.array([x]), f)[0])   # noqa: E731
    # 1 + 1/16 lies halfway between 1 (fraction 000) and 1.125 (001): even wins
    assert enc(1 + 2 ** -4, "e4m3") == 0x38
    assert enc(1 + 3 * 2 ** -4, "e4m3") == 0x3A                 # 1.1875 -> 1.25
    # E4M3 has no infinity: 464 ties to 448, anything rounding past it is NaN
    assert enc(464.0, "e4m3") == 0x7E and enc(470.0, "e4m3") == 0x7F
    assert enc(-1e9, "e4m3") == 0xFF
    # E5M2 is IEEE-like: 61440 ties away from the odd 57344 to 2^16 = Inf
    assert enc(61440.0, "e5m2") == 0x7C and enc(60000.0, "e5m2") == 0x7B
    assert enc(2.0 ** -10, "e4m3") == 0x00 and enc(3 * 2.0 ** -11, "e4m3") == 0x01


def test_round_trip_every_finite_pattern():
    for fmt in ("e4m3", "e5m2"):
        p = np.arange(256, dtype=np.uint8)
        v = oracle.decode(p, fmt)[0]
        fin = np.isfinite(v)
        assert np.array_equal(oracle.encode(v[fin], fmt), p[fin])


def test_generator_agrees_with_oracle_encoder():
    for fmt in ("e4m3", "e5m2"):
        x = inputs.draw_f64("uniform", 11, 0, 50000)
        assert np.array_equal(inputs.f64_to_bits(x, fmt), oracle.encode(x, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_brute_force_small_integers(fmt):
    M, N, K = 7, 9, 11
    a = inputs.matrix_bits(M, K, fmt, "int", 21)
    b = inputs.matrix_bits(K, N, fmt, "int", 22)
    A = oracle.decode(a, fmt)
    B = oracle.decode(b, fmt)
    assert set(np.unique(A)) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    C, S = oracle.gemm_ref_bits(a, b, K=K, N=N, fmt=fmt)
    want = [[math.fsum(A[i, k] * B[k, j] for k in range(K)) for j in range(N)] for i in range(M)]
    assert np.array_equal(C, want)
    assert np.array_equal(S, np.abs(A) @ np.abs(B))
