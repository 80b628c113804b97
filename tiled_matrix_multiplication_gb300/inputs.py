"""Seeded synthetic operands for C = A·B.

This module only draws numbers: it holds none of the matrix-multiply
arithmetic.  The CUDA path (through the tests and the benchmark) and the CPU
oracle both consume the bit patterns it returns, so the two sides always see
the same bytes.

Generator: splitmix64 evaluated as a counter (element i of a stream with seed s
is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)``), following Steele, Lea and Flood,
"Fast splittable pseudorandom number generators" (OOPSLA 2014).  Because it is
a pure function of (seed, index), any row of a huge operand can be regenerated
on its own.

Distributions (the workloads' value recipes):
  * ``uniform``  -- U[-1, 1): ``(x >> 11) * 2**-53 * 2 - 1``
  * ``normal``   -- N(0, sigma): Box-Muller on the draws 2i and 2i+1
  * ``int``      -- integers drawn uniformly from {-2, ..., 2}
The float64 draw is then rounded to nearest-even into the operand dtype
(``f16`` and ``f32`` by numpy's conversion; ``bf16`` by rounding the float32
value's upper half; the 8-bit ``e4m3`` / ``e5m2`` by scaling to an integer
multiple of the value's quantum, see ``_to_fp8``).
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

DTYPES = ("f16", "bf16", "f32", "e4m3", "e5m2")
ELEM_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}
BITS_NP = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32, "e4m3": np.uint8,
           "e5m2": np.uint8}

# (exponent bias, fraction bits, largest finite magnitude) of the 8-bit formats
# of the OCP 8-bit Floating Point Specification: E4M3 has no infinities (its
# only NaN is S.1111.111), E5M2 follows IEEE 754.
_FP8 = {"e4m3": (7, 3, 448.0), "e5m2": (15, 2, 57344.0)}

# Seeds used for the named workloads (A and B streams).
SEED_A = 0x5EED0001
SEED_B = 0x5EED0002


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Elements ``start .. start+count-1`` of the splitmix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _uniform01(x: np.ndarray) -> np.ndarray:
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def draw_f64(dist: str, seed: int, start: int, count: int, sigma: float = 0.02) -> np.ndarray:
    """``count`` float64 draws of distribution ``dist`` starting at element ``start``."""
    if dist == "uniform":
        return _uniform01(splitmix64(seed, start, count)) * 2.0 - 1.0
    if dist == "normal":
        z = splitmix64(seed, 2 * start, 2 * count)
        u1 = (_uniform01(z[0::2]) + 2.0 ** -54)  # in (0, 1]
        u2 = _uniform01(z[1::2])
        return sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    if dist == "int":
        z = splitmix64(seed, start, count)
        return ((z >> np.uint64(32)) % np.uint64(5)).astype(np.float64) - 2.0
    raise ValueError(f"unknown distribution {dist!r}")


def _to_fp8(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round to nearest-even into E4M3 / E5M2 bit patterns.  Draws here are
    small (|x| <= 2 for the uniform and integer recipes), far from the
    formats' overflow; larger magnitudes saturate to the largest finite value
    (not used by any workload)."""
    bias, frac, vmax = _FP8[dtype]
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    ax = np.minimum(np.abs(x), vmax)
    emin = 1 - bias
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, emin)
    q = np.rint(np.ldexp(ax, (frac - e).astype(np.int64)))       # ties to even
    # q in [0, 2^(frac+1)]: q == 2^(frac+1) is the next binade's leading value
    up = q >= 2 ** (frac + 1)
    e = np.where(up, e + 1, e)
    q = np.where(up, q / 2, q)
    normal = q >= 2 ** frac
    code = np.where(normal, (e + bias) * 2 ** frac + (q - 2 ** frac), q)
    return sign | code.astype(np.uint8)


def f64_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to the operand dtype; returns the raw bit patterns."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "f32":
        return x.astype(np.float32).view(np.uint32)
    if dtype in _FP8:
        return _to_fp8(x, dtype)
    if dtype == "bf16":
        w = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        w = w + np.uint64(0x7FFF) + ((w >> np.uint64(16)) & np.uint64(1))
        return (w >> np.uint64(16)).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def matrix_bits(rows: int, cols: int, dtype: str, dist: str, seed: int,
                ld: int | None = None, pad_bits: int | None = None,
                row_start: int = 0, chunk: int = 1 << 22) -> np.ndarray:
    """A ``[rows, ld]`` array of bit patterns; element (r, c) of the logical
    ``[*, cols]`` matrix is stream element ``(row_start + r) * cols + c``.

    Columns ``cols .. ld-1`` hold ``pad_bits`` (default: a quiet NaN) so that a
    kernel that reads past the logical width is caught by a NaN in its output.
    """
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    out = np.empty((rows, ld), dtype=BITS_NP[dtype])
    if ld > cols:
        out[:, cols:] = nan_bits(dtype) if pad_bits is None else pad_bits
    rows_per_chunk = max(1, chunk // max(cols, 1))
    for r0 in range(0, rows, rows_per_chunk):
        r1 = min(rows, r0 + rows_per_chunk)
        x = draw_f64(dist, seed, (row_start + r0) * cols, (r1 - r0) * cols)
        out[r0:r1, :cols] = f64_to_bits(x, dtype).reshape(r1 - r0, cols)
    return out


def nan_bits(dtype: str) -> int:
    return {"f16": 0x7E00, "bf16": 0x7FC0, "f32": 0x7FC00000, "e4m3": 0x7F, "e5m2": 0x7E}[dtype]


def problem(M: int, N: int, K: int, dtype: str, dist: str = "uniform",
            lda: int | None = None, ldb: int | None = None, seed_a: int = SEED_A,
            seed_b: int = SEED_B):
    """Operands of one GEMM problem as bit-pattern arrays ``(A[M, lda], B[K, ldb])``."""
    a = matrix_bits(M, K, dtype, dist, seed_a, ld=lda)
    b = matrix_bits(K, N, dtype, dist, seed_b, ld=ldb)
    return a, b
