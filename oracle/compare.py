"""Tolerance rule for comparing a computed C with the FP64 reference.

TEST INFRASTRUCTURE (see the package docstring).

Rule, per element (C_ref and S from ``gemm_ref``):
  * f16 / bf16 / FP8 (e4m3, e5m2) operands:  |C - C_ref| <= 2e-3 * S + ulp_out(C_ref)
  * f32 operands contracted at TF32:  |C - C_ref| <= 1e-2 * S + ulp_out(C_ref)
where S = sum_k |A[m,k] * B[k,n]| and ulp_out(x) is the spacing of the output
format at |x| (the subnormal spacing below the smallest normal).

Why these hold with margin: the products of f16/bf16 (and FP8) operands are exact in the
FP32 accumulator, so the accumulated error is at most about K * 2^-24 * S
(2.4e-4 * S at K = 4096, 9.8e-4 * S at K = 16384), plus half an ulp for the final
rounding to the output format.  TF32 rounds each f32 operand to 10 fraction
bits (relative error 2^-11 each, so about 2^-10 per product), which 1e-2
covers with a factor of ten; the accumulation term is the same as above.
"""
from __future__ import annotations

import numpy as np

# (exponent of the smallest normal, fraction bits) per output format
_FORMAT = {"f16": (-14, 10), "bf16": (-126, 7), "f32": (-126, 23)}

REL_TOL = {"f16": 2e-3, "bf16": 2e-3, "f32": 1e-2, "e4m3": 2e-3, "e5m2": 2e-3}


def rel_tol_for(dtype_in: str) -> float:
    return REL_TOL[dtype_in]


def ulp(x: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of format ``fmt`` at |x| (x in float64)."""
    emin, frac = _FORMAT[fmt]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(ax > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - frac).astype(np.int64))


def tolerance(C_ref: np.ndarray, S: np.ndarray, dtype_in: str, dtype_out: str) -> np.ndarray:
    return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_out)


def rel_tol_3xtf32(K: int) -> float:
    """Relative bound (times S) for FP32 operands contracted as three TF32
    products ("Matrix Multiplication", teenygrad docs, section "T::dot": TF32x3,
    three TF32 products recovering most of FP32's precision).

    Each operand x = hi + lo + r with hi, lo TF32 values and |r| <= 2^-22 |x|;
    the three kept products hi*hi + lo*hi + hi*lo (each exact in FP32) miss
    lo*lo and the r terms, at most about 3 * 2^-22 |a b| per product: 2^-20.
    Their 3K terms are summed in FP32: at most 3K * 2^-24 * S for sequential
    round-to-nearest addition, doubled (3K * 2^-23) for an accumulator that may
    truncate.
    """
    return 2.0 ** -20 + 3.0 * K * 2.0 ** -23


def check_close(C: np.ndarray, C_ref: np.ndarray, S: np.ndarray, dtype_in: str,
                dtype_out: str, rel: float | None = None):
    """Returns ``(ok, report)``; ``report`` describes the worst element.
    ``rel`` overrides the relative term of the rule (e.g. ``rel_tol_3xtf32``)."""
    C = np.asarray(C, dtype=np.float64)
    tol = (tolerance(C_ref, S, dtype_in, dtype_out) if rel is None
           else rel * np.asarray(S, dtype=np.float64) + ulp(C_ref, dtype_out))
    err = np.abs(C - C_ref)
    bad = ~(err <= tol)  # NaN in C counts as a failure
    ok = not bool(bad.any())
    if C.size == 0:
        return True, "empty"
    ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    idx = np.unravel_index(int(np.argmax(ratio)), C.shape)
    report = (f"{int(bad.sum())} of {C.size} outside tolerance; worst at {tuple(int(i) for i in idx)}: "
              f"got {C[idx]!r} ref {C_ref[idx]!r} tol {tol[idx]!r} (err/tol {ratio[idx]:.3g})")
    return ok, report
