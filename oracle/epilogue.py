"""Reference for the GEMM with a fused epilogue, in FP64.

TEST INFRASTRUCTURE (see the package docstring).

The pages end the tiled-matmul chapter by pointing at the work that can be
done while the output tile is still in registers ("Matrix Multiplication",
teenygrad docs, closing line before the "Fusing an Epilogue" chapter), and
the tree they describe fuses a convolution-as-GEMM with a batch-norm (a
per-channel scale and shift) and a SiLU.  They print no formula for it; the
plainest reading, used here, applies in this order to each accumulated
element C[m,n] = sum_k A[m,k] B[k,n]:

    pre[m,n] = alpha * scale[n] * C[m,n] + bias[n]
    D[m,n]   = act(pre[m,n]) + beta * R[m,n]

with an optional per-column scale and bias (absent: 1 and 0), an activation

    none        x
    relu        x if x > 0 else 0
    silu        x / (1 + exp(-x))                         (x * sigmoid(x))
    gelu_tanh   x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))

and an optional residual R read in the output format.  D is rounded once to
the output format.  ``gelu_tanh`` is the tanh form of the Gaussian error
linear unit (Hendrycks and Gimpel, "Gaussian Error Linear Units", 2016).
"""
from __future__ import annotations

import math

import numpy as np

from .compare import REL_TOL, ulp

ACTIVATIONS = ("none", "relu", "silu", "gelu_tanh")
ACT_CODES = {name: i for i, name in enumerate(ACTIVATIONS)}

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)

# Upper bounds of |act'(x)| over the reals (the tests check them on a grid):
# silu' peaks at about 1.0998, the tanh-form GELU' at about 1.1289.
LIPSCHITZ = {"none": 1.0, "relu": 1.0, "silu": 1.1, "gelu_tanh": 1.13}


def activation(x: np.ndarray, act: str) -> np.ndarray:
    """The activation ``act`` applied elementwise in FP64."""
    x = np.asarray(x, dtype=np.float64)
    if act == "none":
        return x.copy()
    if act == "relu":
        return np.where(x > 0, x, 0.0)
    if act == "silu":
        with np.errstate(over="ignore"):
            return x / (1.0 + np.exp(-x))
    if act == "gelu_tanh":
        return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)))
    raise ValueError(f"unknown activation {act!r}")


def epilogue_ref(C_ref: np.ndarray, alpha: float = 1.0, scale=None, bias=None,
                 act: str = "none", beta: float = 0.0, R=None):
    """Returns ``(D, pre)`` in FP64 for the exact accumulated product ``C_ref``
    ([rows, N]); ``scale`` and ``bias`` are length-N vectors or None, ``R`` a
    [rows, N] array of decoded residual values or None."""
    C_ref = np.asarray(C_ref, dtype=np.float64)
    pre = float(alpha) * C_ref
    if scale is not None:
        pre = pre * np.asarray(scale, dtype=np.float64)[None, :]
    if bias is not None:
        pre = pre + np.asarray(bias, dtype=np.float64)[None, :]
    D = activation(pre, act)
    if R is not None:
        D = D + float(beta) * np.asarray(R, dtype=np.float64)
    return D, pre


def epilogue_tolerance(C_ref, S, dtype_in: str, dtype_out: str, alpha: float = 1.0, scale=None,
                       bias=None, act: str = "none", beta: float = 0.0, R=None) -> np.ndarray:
    """Per-element bound on |D - D_ref| for a GPU result computed from an FP32
    accumulator.

    The accumulator is within REL_TOL * S of C_ref (the GEMM rule without its
    output rounding); the affine step multiplies that by |alpha * scale[n]|;
    the activation by at most its Lipschitz constant.  The FP32 evaluation of
    each step (a few roundings and the library exp / tanh, each within a few
    units of 2^-24) is covered by 2^-20 times the magnitudes involved, and the
    final rounding by one ulp of the output format at |D_ref|.
    """
    C_ref = np.asarray(C_ref, dtype=np.float64)
    D, pre = epilogue_ref(C_ref, alpha, scale, bias, act, beta, R)
    gain = abs(float(alpha)) * (np.abs(np.asarray(scale, dtype=np.float64))[None, :]
                                if scale is not None else 1.0)
    mags = np.abs(gain * C_ref) + np.abs(pre) + np.abs(D)
    if bias is not None:
        mags = mags + np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    if R is not None:
        mags = mags + abs(float(beta)) * np.abs(np.asarray(R, dtype=np.float64))
    return (LIPSCHITZ[act] * gain * REL_TOL[dtype_in] * np.asarray(S, dtype=np.float64)
            + 2.0 ** -20 * mags + ulp(D, dtype_out))


def check_epilogue(D, C_ref, S, dtype_in: str, dtype_out: str, **ep):
    """Returns ``(ok, report)`` for a computed D (decoded to FP64)."""
    D = np.asarray(D, dtype=np.float64)
    D_ref, _ = epilogue_ref(C_ref, **ep)
    tol = epilogue_tolerance(C_ref, S, dtype_in, dtype_out, **ep)
    err = np.abs(D - D_ref)
    bad = ~(err <= tol)
    if D.size == 0:
        return True, "empty"
    ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1.0), np.inf)
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    idx = np.unravel_index(int(np.argmax(ratio)), D.shape)
    report = (f"{int(bad.sum())} of {D.size} outside tolerance; worst at "
              f"{tuple(int(i) for i in idx)}: got {D[idx]!r} ref {D_ref[idx]!r} "
              f"tol {tol[idx]!r} (err/tol {ratio[idx]:.3g})")
    return not bool(bad.any()), report
