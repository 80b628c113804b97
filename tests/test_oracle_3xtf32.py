"""Pins for the 3xTF32 tolerance (oracle/compare.py, rel_tol_3xtf32): a CPU
emulation of the method -- operands split into TF32 parts by round-to-nearest
(ties away) on the FP32 bit pattern, the three kept products summed in FP32 --
must land inside the bound on random and on constant operands, while on
constant operands (whose TF32 rounding error does not average out) one-pass
TF32 and a split that drops the lo * hi cross term must not.  CPU only.
"""
from __future__ import annotations

import numpy as np

import oracle
from tiled_matrix_multiplication_gb300 import inputs


def tf32_rna(x: np.ndarray) -> np.ndarray:
    """Round float32 values to 10 fraction bits, ties away from zero."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x1000) & 0xFFFFE000
    return u.astype(np.uint32).view(np.float32)


def split(x):
    hi = tf32_rna(x)
    lo = tf32_rna((x - hi).astype(np.float32))
    return hi, lo


def fp32_gemm(A, B):
    """Sequential FP32 accumulation in increasing k (numpy float32 ops)."""
    acc = np.zeros((A.shape[0], B.shape[1]), dtype=np.float32)
    for k in range(A.shape[1]):
        acc = (acc + np.outer(A[:, k], B[k, :]).astype(np.float32)).astype(np.float32)
    return acc


def case(M=24, N=40, K=300, seed=3):
    a = inputs.matrix_bits(M, K, "f32", "uniform", seed)
    b = inputs.matrix_bits(K, N, "f32", "uniform", seed + 1)
    A, B = a.view(np.float32), b.view(np.float32)
    C_ref, S = oracle.gemm_ref_bits(a, b, K=K, N=N, fmt="f32")
    return A, B, C_ref, S


def test_split_parts_are_tf32_and_exact_enough():
    x = inputs.matrix_bits(1, 100000, "f32", "uniform", 9).view(np.float32)[0]
    hi, lo = split(x)
    assert np.all(hi.view(np.uint32) & 0x1FFF == 0) and np.all(lo.view(np.uint32) & 0x1FFF == 0)
    r = x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64)
    assert np.max(np.abs(r) / np.abs(x.astype(np.float64))) <= 2.0 ** -21


def test_emulated_3xtf32_is_inside_the_bound():
    A, B, C_ref, S = case()
    ah, al = split(A)
    bh, bl = split(B)
    Ap = np.concatenate([ah, al, ah], axis=1)
    Bp = np.concatenate([bh, bh, bl], axis=0)
    C = fp32_gemm(Ap, Bp).astype(np.float64)
    ok, rep = oracle.check_close(C, C_ref, S, "f32", "f32", rel=oracle.rel_tol_3xtf32(300))
    assert ok, rep


def constant_case(K=300, M=4, N=5):
    """Every operand element 1 + 3 * 2^-12: TF32 rounds it up by 2^-12, the
    same way every time, so a method that keeps that error off its products
    is wrong by about 2.4e-4 * S, well outside the bound at K = 300."""
    x = np.float32(1 + 3 * 2.0 ** -12)
    A = np.full((M, K), x, dtype=np.float32)
    B = np.full((K, N), x, dtype=np.float32)
    C_ref, S = oracle.gemm_ref_bits(A.view(np.uint32), B.view(np.uint32), K=K, N=N, fmt="f32")
    return A, B, C_ref, S


def test_one_pass_tf32_and_a_dropped_cross_term_are_outside():
    A, B, C_ref, S = constant_case()
    rel = oracle.rel_tol_3xtf32(300)
    one = fp32_gemm(tf32_rna(A), tf32_rna(B)).astype(np.float64)
    assert not oracle.check_close(one, C_ref, S, "f32", "f32", rel=rel)[0]
    ah, al = split(A)
    bh, bl = split(B)
    two = fp32_gemm(np.concatenate([ah, ah], axis=1),
                    np.concatenate([bh, bl], axis=0)).astype(np.float64)
    assert not oracle.check_close(two, C_ref, S, "f32", "f32", rel=rel)[0]
    three = fp32_gemm(np.concatenate([ah, al, ah], axis=1),
                      np.concatenate([bh, bh, bl], axis=0)).astype(np.float64)
    assert oracle.check_close(three, C_ref, S, "f32", "f32", rel=rel)[0]


def test_bound_is_tighter_than_tf32():
    for K in (64, 777, 2048):
        assert oracle.rel_tol_3xtf32(K) < oracle.rel_tol_for("f32") / 10
