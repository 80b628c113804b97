"""GB300-native tiled dense matrix multiply: C = A @ B on sm_103a tensor cores.

The product is the C-ABI library ``libtg_gemm.so`` (header ``include/tg_gemm.h``);
this package is its thin binding.  PyTorch is used only for device memory and
streams: every step of the multiply runs in the library's CUDA kernels.

    import torch, tiled_matrix_multiplication_gb300 as tg
    c = tg.gemm(a, b)                   # a [M,K], b [K,N] on cuda, f16/bf16/f32
    c = tg.gemm(a, b, out_dtype=torch.float32)

The raw C entry points are re-exported under their C names (``tg_gemm``,
``tg_gemm_ex``, ``tg_plan_gemm``, ``tg_status_string``, ``tg_last_device_error``,
``tg_abi_version``) with pointers and streams passed as integers.
"""
from __future__ import annotations

from ._lib import (DTYPE_CODES, EXPORTS, LIB_PATH, TG_BF16, TG_ERR_ARCH, TG_ERR_CUDA,
                   TG_ERR_INVALID_VALUE, TG_ERR_NOT_IMPLEMENTED, TG_ERR_OUT_OF_MEMORY,
                   TG_ERR_TIMEOUT, TG_ERR_UNSUPPORTED, TG_F16, TG_F32, TG_OK, TG_PATH_AUTO,
                   TG_PATH_SKINNY, TG_PATH_TC, TG_PATH_TC_PAIR, NOALLOC_SCRATCH_BYTES, TgError,
                   load, make_options, status_name, tg_abi_version, tg_gemm, tg_gemm_ex,
                   tg_gemm_splitk_noalloc, tg_last_device_error, tg_options, tg_plan,
                   tg_plan_gemm, tg_status_string)

__all__ = [
    "gemm", "plan", "check_device_error", "dtype_code", "TgError", "load", "make_options",
    "tg_gemm", "tg_gemm_ex", "tg_plan_gemm", "tg_status_string", "tg_last_device_error",
    "tg_abi_version", "tg_gemm_splitk_noalloc", "NOALLOC_SCRATCH_BYTES", "tg_options", "tg_plan",
    "EXPORTS", "LIB_PATH",
    "TG_F16", "TG_BF16", "TG_F32", "TG_OK", "TG_ERR_INVALID_VALUE", "TG_ERR_UNSUPPORTED",
    "TG_ERR_OUT_OF_MEMORY", "TG_ERR_CUDA", "TG_ERR_ARCH", "TG_ERR_TIMEOUT",
    "TG_ERR_NOT_IMPLEMENTED", "TG_PATH_AUTO", "TG_PATH_TC", "TG_PATH_TC_PAIR", "TG_PATH_SKINNY",
]


def dtype_code(dtype) -> int:
    """torch dtype (or 'f16'/'bf16'/'f32') -> tg_dtype code."""
    if isinstance(dtype, str):
        return DTYPE_CODES[dtype]
    import torch
    table = {torch.float16: TG_F16, torch.bfloat16: TG_BF16, torch.float32: TG_F32}
    if dtype not in table:
        raise TgError(TG_ERR_UNSUPPORTED, f"dtype {dtype}")
    return table[dtype]


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def gemm(a, b, out_dtype=None, out=None, stream=None, **options):
    """C = A @ B through ``tg_gemm_ex`` on ``stream`` (default: torch's current stream).

    ``a`` is [M, K] and ``b`` is [K, N] CUDA tensors of the same dtype with unit
    column stride (any row stride).  ``out_dtype`` defaults to the input dtype;
    ``out`` may be a preallocated [M, N] tensor with unit column stride.
    ``options`` are tg_options fields (path, splits, block_n, group_m, max_ctas,
    timeout_ms).  Raises ``ValueError`` on a shape mismatch and ``TgError`` on
    any status other than TG_OK.
    """
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("gemm expects [M, K] @ [K, N]")
    if a.dtype != b.dtype:
        raise ValueError("A and B must have the same dtype")
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = a.shape
    N = b.shape[1]
    if (a.stride(1) != 1 and K > 1) or (b.stride(1) != 1 and N > 1):
        raise ValueError("A and B need unit column stride")
    out_dtype = a.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    elif out.shape != (M, N) or out.dtype != out_dtype or (out.stride(1) != 1 and N > 1):
        raise ValueError("out must be [M, N] of out_dtype with unit column stride")
    lda = a.stride(0) if M > 1 else max(K, 1)
    ldb = b.stride(0) if K > 1 else max(N, 1)
    ldc = out.stride(0) if M > 1 else max(N, 1)
    opt = make_options(**options) if options else None
    with torch.cuda.device(a.device):
        st = tg_gemm_ex(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc,
                        dtype_code(a.dtype), dtype_code(out_dtype), _stream_handle(stream), opt)
    if st != TG_OK:
        raise TgError(st, f"tg_gemm_ex(M={M}, N={N}, K={K})")
    return out


def plan(M, N, K, dtype_in="f16", dtype_out=None, num_sms=148, lda=None, ldb=None, ldc=None,
         a=0x1000, b=0x100000000, c=0x200000000, **options) -> dict:
    """What ``tg_gemm_ex`` would launch for these sizes (host only, no GPU).

    The default pointer values are aligned, disjoint placeholders; they are
    only inspected for alignment and overlap.
    """
    dtype_out = dtype_in if dtype_out is None else dtype_out
    opt = make_options(**options) if options else None
    st, p = tg_plan_gemm(M, N, K, a, K if lda is None else lda, b, N if ldb is None else ldb,
                         c, N if ldc is None else ldc, dtype_in, dtype_out, num_sms, opt)
    if st != TG_OK:
        raise TgError(st, "tg_plan_gemm")
    return p


def check_device_error(stream=None) -> None:
    """Synchronise ``stream`` and raise if a kernel recorded a failure."""
    st = tg_last_device_error(_stream_handle(stream))
    if st != TG_OK:
        raise TgError(st, "device-side failure")
