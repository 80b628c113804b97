"""ctypes front-end to ``gemm_ref.c`` (test infrastructure; see the package docstring).

``build()`` compiles ``gemm_ref.c`` with the host C compiler into
``oracle/_build/liboracle.so`` (OpenMP when available).  It is rebuilt when the
source is newer than the library.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
FORMATS = {"f16": F16, "bf16": BF16, "f32": F32, "e4m3": E4M3, "e5m2": E5M2}
_BITS = {F16: np.uint16, BF16: np.uint16, F32: np.uint32, E4M3: np.uint8, E5M2: np.uint8}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def _compile(src: str, out: str, openmp: bool = True) -> None:
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found")
    flags = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]
    if openmp:
        flags.append("-fopenmp")
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([cc, *flags, src, "-o", tmp, "-lm"], check=True,
                   stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    os.replace(tmp, out)


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle if needed; returns the library path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        try:
            _compile(src, out, openmp=True)
        except subprocess.CalledProcessError:
            _compile(src, out, openmp=False)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and type the oracle library."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        p = path or build()
        lib = ctypes.CDLL(p)
        i64, dp, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_decode_one.argtypes = [ctypes.c_int, ctypes.c_uint32]
        lib.orc_decode_one.restype = ctypes.c_double
        lib.orc_encode_one.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.orc_encode_one.restype = ctypes.c_uint32
        lib.orc_decode.argtypes = [ctypes.c_int, vp, i64, i64, i64, dp]
        lib.orc_decode.restype = ctypes.c_int
        lib.orc_encode.argtypes = [ctypes.c_int, dp, i64, vp]
        lib.orc_encode.restype = ctypes.c_int
        lib.orc_gemm.argtypes = [i64, i64, i64, dp, i64, dp, i64,
                                 ctypes.POINTER(ctypes.c_int64), i64, dp, dp, i64]
        lib.orc_gemm.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def num_threads() -> int:
    return int(load().orc_num_threads())


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def decode(bits: np.ndarray, fmt, cols: int | None = None, lib=None) -> np.ndarray:
    """Bit patterns ``[rows, ld]`` -> float64 ``[rows, cols]`` (cols defaults to ld)."""
    lib = lib or load()
    f = _fmt(fmt)
    bits = np.ascontiguousarray(bits, dtype=_BITS[f])
    if bits.ndim == 1:
        bits = bits.reshape(1, -1)
    rows, ld = bits.shape
    cols = ld if cols is None else cols
    out = np.empty((rows, cols), dtype=np.float64)
    rc = lib.orc_decode(f, bits.ctypes.data, rows, cols, ld, _dp(out))
    if rc != 0:
        raise ValueError("orc_decode failed")
    return out


def encode(x: np.ndarray, fmt, lib=None) -> np.ndarray:
    """float64 -> bit patterns of ``fmt`` (round to nearest, ties to even)."""
    lib = lib or load()
    f = _fmt(fmt)
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=_BITS[f])
    rc = lib.orc_encode(f, _dp(x), x.size, out.ctypes.data)
    if rc != 0:
        raise ValueError("orc_encode failed")
    return out


def gemm_ref(A: np.ndarray, B: np.ndarray, rows=None, with_abs: bool = True, lib=None):
    """FP64 reference on decoded operands.

    ``A`` is float64 ``[M, K]``, ``B`` float64 ``[K, N]``.  Returns ``(C, S)``
    for the selected rows (all rows if ``rows`` is None); ``S`` is the
    sum of |products| (None when ``with_abs`` is False).
    """
    lib = lib or load()
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if rows is None:
        nr, rp = M, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nr, rp = rows.size, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    C = np.empty((nr, N), dtype=np.float64)
    S = np.empty((nr, N), dtype=np.float64) if with_abs else None
    rc = lib.orc_gemm(M, N, K, _dp(A), K, _dp(B), N, rp, nr, _dp(C),
                      _dp(S) if S is not None else None, N)
    if rc != 0:
        raise ValueError("orc_gemm rejected its arguments")
    return C, S


def gemm_ref_bits(a_bits: np.ndarray, b_bits: np.ndarray, K: int, N: int, fmt,
                  rows=None, with_abs: bool = True, lib=None):
    """Reference from raw operand bit patterns ``A[M, lda]``, ``B[K, ldb]``.

    Only the logical ``[M, K]`` / ``[K, N]`` parts are read; padding columns
    are ignored.  When ``rows`` is given only those rows of A are decoded.
    """
    lib = lib or load()
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = decode(a_bits[rows], fmt, cols=K, lib=lib)
        B = decode(b_bits[:K], fmt, cols=N, lib=lib)
        return gemm_ref(A, B, rows=None, with_abs=with_abs, lib=lib)
    A = decode(a_bits, fmt, cols=K, lib=lib)
    B = decode(b_bits[:K], fmt, cols=N, lib=lib)
    return gemm_ref(A, B, with_abs=with_abs, lib=lib)
