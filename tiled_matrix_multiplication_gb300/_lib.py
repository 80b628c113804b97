"""ctypes binding of ``libtg_gemm.so`` -- argument marshalling only.

The names mirror the C ABI in ``include/tg_gemm.h``.  Every GEMM runs in the
library's CUDA kernels; there is no fallback of any kind: if the library has
not been built, or the device is not an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# TG_CHECKED=1 selects the checked build (device-side bounds and alignment
# checks compiled in; built with ``python -m tiled_matrix_multiplication_gb300.build --checked``)
CHECKED = os.environ.get("TG_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_PKG, "libtg_gemm_checked.so" if CHECKED else "libtg_gemm.so")

TG_F16, TG_BF16, TG_F32, TG_E4M3, TG_E5M2 = 0, 1, 2, 3, 4
DTYPE_CODES = {"f16": TG_F16, "bf16": TG_BF16, "f32": TG_F32, "e4m3": TG_E4M3, "e5m2": TG_E5M2}

TG_OK = 0
TG_ERR_INVALID_VALUE = 1
TG_ERR_UNSUPPORTED = 2
TG_ERR_OUT_OF_MEMORY = 3
TG_ERR_CUDA = 4
TG_ERR_ARCH = 5
TG_ERR_TIMEOUT = 6
TG_ERR_NOT_IMPLEMENTED = 7
TG_ERR_BOUNDS = 8

TG_PATH_AUTO, TG_PATH_TC, TG_PATH_TC_PAIR, TG_PATH_SKINNY = 0, 1, 2, 3

# Every extern "C" symbol the header declares.
EXPORTS = ("tg_gemm", "tg_gemm_ex", "tg_plan_gemm", "tg_status_string",
           "tg_last_device_error", "tg_abi_version", "tg_gemm_splitk_noalloc",
           "tg_gemm_strided_batched", "tg_plan_gemm_strided_batched", "tg_gemm_fused",
           "tg_gemm_host", "tg_selftest_timeout", "tg_gemm_strided_batched_fused",
           "tg_checked_build", "tg_selftest_bounds")

TG_ACT_NONE, TG_ACT_RELU, TG_ACT_SILU, TG_ACT_GELU_TANH = 0, 1, 2, 3
ACT_CODES = {"none": TG_ACT_NONE, "relu": TG_ACT_RELU, "silu": TG_ACT_SILU,
             "gelu_tanh": TG_ACT_GELU_TANH}

# Bytes of the library-owned partial-tile array of tg_gemm_splitk_noalloc.
NOALLOC_SCRATCH_BYTES = 16 << 20


class tg_options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("block_n", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("max_ctas", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("multicast", ctypes.c_int32), ("f32_mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class tg_epilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("ldr", ctypes.c_int64),
                ("activation", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class tg_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("pack_a", ctypes.c_int32), ("pack_b", ctypes.c_int32),
                ("c_vector", ctypes.c_int32), ("kernels", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("multicast", ctypes.c_int32), ("per_batch", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class TgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{status_name(status)}{': ' + what if what else ''}")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the library (raises if it is missing -- build it with ``build()``)."""
    global _lib
    if _lib is not None and path is None:   # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -m tiled_matrix_multiplication_gb300.build)")
        lib = ctypes.CDLL(p)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32
        gemm_args = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int, ctypes.c_int, vp]
        lib.tg_gemm.argtypes = gemm_args
        lib.tg_gemm.restype = ctypes.c_int
        lib.tg_gemm_ex.argtypes = gemm_args + [ctypes.POINTER(tg_options)]
        lib.tg_gemm_ex.restype = ctypes.c_int
        lib.tg_plan_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                     ctypes.c_int, i32, ctypes.POINTER(tg_options),
                                     ctypes.POINTER(tg_plan)]
        lib.tg_plan_gemm.restype = ctypes.c_int
        lib.tg_status_string.argtypes = [ctypes.c_int]
        lib.tg_status_string.restype = ctypes.c_char_p
        lib.tg_last_device_error.argtypes = [vp]
        lib.tg_last_device_error.restype = ctypes.c_int
        lib.tg_abi_version.argtypes = []
        lib.tg_abi_version.restype = i32
        lib.tg_gemm_splitk_noalloc.argtypes = gemm_args[:-1] + [i32, vp]
        lib.tg_gemm_splitk_noalloc.restype = ctypes.c_int
        batched = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, ctypes.c_int,
                   ctypes.c_int]
        lib.tg_gemm_strided_batched.argtypes = batched + [vp, ctypes.POINTER(tg_options)]
        lib.tg_gemm_strided_batched.restype = ctypes.c_int
        lib.tg_plan_gemm_strided_batched.argtypes = batched + [i32, ctypes.POINTER(tg_options),
                                                               ctypes.POINTER(tg_plan)]
        lib.tg_plan_gemm_strided_batched.restype = ctypes.c_int
        lib.tg_gemm_fused.argtypes = gemm_args[:-1] + [ctypes.POINTER(tg_epilogue), vp,
                                                        ctypes.POINTER(tg_options)]
        lib.tg_gemm_fused.restype = ctypes.c_int
        lib.tg_gemm_strided_batched_fused.argtypes = batched + [ctypes.POINTER(tg_epilogue), i64,
                                                                vp, ctypes.POINTER(tg_options)]
        lib.tg_gemm_strided_batched_fused.restype = ctypes.c_int
        lib.tg_gemm_host.argtypes = gemm_args + [ctypes.POINTER(tg_options)]
        lib.tg_gemm_host.restype = ctypes.c_int
        lib.tg_selftest_timeout.argtypes = [i32, vp]
        lib.tg_selftest_timeout.restype = ctypes.c_int
        lib.tg_checked_build.argtypes = []
        lib.tg_checked_build.restype = i32
        lib.tg_selftest_bounds.argtypes = [i32, vp]
        lib.tg_selftest_bounds.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _code(dtype) -> int:
    return DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)


TG_F32_TF32, TG_F32_3XTF32 = 0, 1


def make_options(path=0, splits=0, block_n=0, group_m=0, max_ctas=0, timeout_ms=0,
                 multicast=0, f32_mode=0):
    o = tg_options()
    o.path, o.splits, o.block_n, o.group_m = path, splits, block_n, group_m
    o.max_ctas, o.timeout_ms = max_ctas, timeout_ms
    o.multicast, o.f32_mode, o.reserved = multicast, f32_mode, 0
    return o


def status_name(status: int) -> str:
    try:
        return load().tg_status_string(int(status)).decode()
    except RuntimeError:
        return f"tg_status({int(status)})"


def tg_status_string(status: int) -> str:
    return load().tg_status_string(int(status)).decode()


def tg_abi_version() -> int:
    return int(load().tg_abi_version())


def tg_gemm(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream) -> int:
    """Raw C call; pointers and stream are integers.  Returns the tg_status."""
    return int(load().tg_gemm(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                              _code(dtype_out), stream))


def tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream, options=None) -> int:
    opt = ctypes.byref(options) if options is not None else None
    return int(load().tg_gemm_ex(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                                 _code(dtype_out), stream, opt))


def tg_plan_gemm(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, num_sms, options=None):
    """Returns ``(status, plan_dict)``; host only, needs no GPU."""
    plan = tg_plan()
    opt = ctypes.byref(options) if options is not None else None
    st = int(load().tg_plan_gemm(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                                 _code(dtype_out), num_sms, opt, ctypes.byref(plan)))
    return st, plan.as_dict()


def tg_last_device_error(stream) -> int:
    return int(load().tg_last_device_error(stream))


def tg_gemm_splitk_noalloc(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, splits,
                           stream) -> int:
    """Split-K GEMM whose partial tiles live in the library's fixed device array
    (NOALLOC_SCRATCH_BYTES): for callers that must not have the library
    allocate device memory.  Returns the tg_status (TG_ERR_UNSUPPORTED when
    splits * M * N * 4 exceeds the array, for misaligned operands or TF32)."""
    return int(load().tg_gemm_splitk_noalloc(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                                             _code(dtype_out), splits, stream))


def tg_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc, stride_c,
                            dtype_in, dtype_out, stream, options=None) -> int:
    """``batch`` products C_z = A_z B_z whose operands start ``stride_*`` elements
    apart (0 = one operand shared by all).  Returns the tg_status."""
    opt = ctypes.byref(options) if options is not None else None
    return int(load().tg_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b,
                                              c, ldc, stride_c, _code(dtype_in),
                                              _code(dtype_out), stream, opt))


def tg_plan_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                 stride_c, dtype_in, dtype_out, num_sms, options=None):
    """Returns ``(status, plan_dict)``; host only, needs no GPU."""
    plan = tg_plan()
    opt = ctypes.byref(options) if options is not None else None
    st = int(load().tg_plan_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb,
                                                 stride_b, c, ldc, stride_c, _code(dtype_in),
                                                 _code(dtype_out), num_sms, opt,
                                                 ctypes.byref(plan)))
    return st, plan.as_dict()


def make_epilogue(alpha=1.0, beta=0.0, scale=0, bias=0, residual=0, ldr=0, activation="none"):
    """tg_epilogue from plain values; pointers are integers (0 = NULL)."""
    e = tg_epilogue()
    e.alpha, e.beta = alpha, beta
    e.scale, e.bias, e.residual = scale or None, bias or None, residual or None
    e.ldr = ldr
    e.activation = ACT_CODES[activation] if isinstance(activation, str) else int(activation)
    e.reserved = 0
    return e


def tg_gemm_fused(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, epilogue, stream,
                  options=None) -> int:
    """C = act(alpha * scale * (A B) + bias) + beta * R; ``epilogue`` is a
    tg_epilogue or None.  Returns the tg_status."""
    ep = ctypes.byref(epilogue) if epilogue is not None else None
    opt = ctypes.byref(options) if options is not None else None
    return int(load().tg_gemm_fused(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                                    _code(dtype_out), ep, stream, opt))


def tg_gemm_strided_batched_fused(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, c, ldc,
                                  stride_c, dtype_in, dtype_out, epilogue, stride_r, stream,
                                  options=None) -> int:
    """The batched product with the fused epilogue on every product; residual
    blocks ``stride_r`` elements apart (0 = one shared).  Returns the tg_status."""
    ep = ctypes.byref(epilogue) if epilogue is not None else None
    opt = ctypes.byref(options) if options is not None else None
    return int(load().tg_gemm_strided_batched_fused(batch, M, N, K, a, lda, stride_a, b, ldb,
                                                    stride_b, c, ldc, stride_c, _code(dtype_in),
                                                    _code(dtype_out), ep, stride_r, stream, opt))


def tg_gemm_host(M, N, K, a, lda, b, ldb, c, ldc, dtype_in, dtype_out, stream,
                 options=None) -> int:
    """C = A B with HOST pointers a, b, c (page-locked for overlap); the copies
    and the multiply are pipelined on the device.  Returns the tg_status."""
    opt = ctypes.byref(options) if options is not None else None
    return int(load().tg_gemm_host(M, N, K, a, lda, b, ldb, c, ldc, _code(dtype_in),
                                   _code(dtype_out), stream, opt))


def tg_selftest_timeout(timeout_ms, stream) -> int:
    """Enqueue the failure-detection check (a bounded wait that always runs
    out); tg_last_device_error then reports TG_ERR_TIMEOUT."""
    return int(load().tg_selftest_timeout(timeout_ms, stream))


def tg_checked_build() -> int:
    """1 if the loaded library has the device-side checks compiled in."""
    return int(load().tg_checked_build())


def tg_selftest_bounds(index, stream) -> int:
    """Enqueue the checked-build check: one checked store to element `index`
    of a 32-element array (outside 0..31: skipped, TG_ERR_BOUNDS recorded)."""
    return int(load().tg_selftest_bounds(index, stream))
