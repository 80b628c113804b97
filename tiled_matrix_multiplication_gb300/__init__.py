"""GB300-native tiled dense matrix multiply: C = A @ B on sm_103a tensor cores.

The product is the C-ABI library ``libtg_gemm.so`` (header ``include/tg_gemm.h``);
this package is its thin binding.  PyTorch is used only for device memory and
streams: every step of the multiply runs in the library's CUDA kernels.

    import torch, tiled_matrix_multiplication_gb300 as tg
    c = tg.gemm(a, b)                   # a [M,K], b [K,N] on cuda, f16/bf16/f32
    c = tg.gemm(a, b, out_dtype=torch.float32)

The raw C entry points are re-exported under their C names (``tg_gemm``,
``tg_gemm_ex``, ``tg_plan_gemm``, ``tg_gemm_strided_batched``, ...) with pointers
and streams passed as integers.  ``bmm`` runs a batch of products
([B, M, K] @ [B, K, N], either side may be a shared 2-D matrix).
"""
from __future__ import annotations

from ._lib import (DTYPE_CODES, EXPORTS, LIB_PATH, TG_BF16, TG_E4M3, TG_E5M2, TG_ERR_ARCH,
                   TG_F32_3XTF32, TG_F32_TF32,
                   TG_ERR_CUDA,
                   TG_ERR_INVALID_VALUE, TG_ERR_NOT_IMPLEMENTED, TG_ERR_OUT_OF_MEMORY,
                   TG_ERR_BOUNDS, CHECKED, tg_checked_build, tg_selftest_bounds,
                   TG_ERR_TIMEOUT, TG_ERR_UNSUPPORTED, TG_F16, TG_F32, TG_OK, TG_PATH_AUTO,
                   TG_PATH_SKINNY, TG_PATH_TC, TG_PATH_TC_PAIR, NOALLOC_SCRATCH_BYTES, TgError,
                   load, make_options, status_name, tg_abi_version, tg_gemm, tg_gemm_ex,
                   ACT_CODES, TG_ACT_GELU_TANH, TG_ACT_NONE, TG_ACT_RELU, TG_ACT_SILU,
                   make_epilogue, tg_epilogue, tg_gemm_fused, tg_gemm_host,
                   tg_selftest_timeout, tg_gemm_strided_batched_fused,
                   tg_gemm_splitk_noalloc, tg_gemm_strided_batched, tg_last_device_error,
                   tg_options, tg_plan, tg_plan_gemm, tg_plan_gemm_strided_batched,
                   tg_status_string)

__all__ = [
    "gemm", "gemm_fused", "bmm", "bmm_fused", "plan", "plan_batched", "check_device_error",
    "tg_gemm_fused", "tg_gemm_strided_batched_fused", "tg_gemm_host", "tg_selftest_timeout", "tg_epilogue", "make_epilogue", "ACT_CODES", "TG_ACT_NONE", "TG_ACT_RELU",
    "TG_ACT_SILU", "TG_ACT_GELU_TANH", "dtype_code", "TgError", "load", "make_options",
    "tg_gemm", "tg_gemm_ex", "tg_plan_gemm", "tg_status_string", "tg_last_device_error",
    "tg_abi_version", "tg_gemm_splitk_noalloc", "tg_gemm_strided_batched",
    "tg_plan_gemm_strided_batched", "NOALLOC_SCRATCH_BYTES", "tg_options", "tg_plan",
    "EXPORTS", "LIB_PATH",
    "TG_F16", "TG_BF16", "TG_F32", "TG_E4M3", "TG_E5M2", "TG_F32_TF32", "TG_F32_3XTF32", "TG_OK", "TG_ERR_INVALID_VALUE", "TG_ERR_UNSUPPORTED",
    "TG_ERR_OUT_OF_MEMORY", "TG_ERR_CUDA", "TG_ERR_ARCH", "TG_ERR_TIMEOUT",
    "TG_ERR_NOT_IMPLEMENTED", "TG_PATH_AUTO", "TG_PATH_TC", "TG_PATH_TC_PAIR", "TG_PATH_SKINNY",
    "TG_ERR_BOUNDS", "CHECKED", "tg_checked_build", "tg_selftest_bounds",
]


_TORCH_CODES = None


def dtype_code(dtype) -> int:
    """torch dtype (or 'f16'/'bf16'/'f32') -> tg_dtype code."""
    global _TORCH_CODES
    if isinstance(dtype, str):
        return DTYPE_CODES[dtype]
    if _TORCH_CODES is None:
        import torch
        _TORCH_CODES = {torch.float16: TG_F16, torch.bfloat16: TG_BF16, torch.float32: TG_F32,
                        torch.float8_e4m3fn: TG_E4M3, torch.float8_e5m2: TG_E5M2}
    code = _TORCH_CODES.get(dtype)
    if code is None:
        raise TgError(TG_ERR_UNSUPPORTED, f"dtype {dtype}")
    return code


class _OnDevice:
    """Makes `device` current for the call, touching the current device only
    when it differs (entering torch's device context on every call costs more
    than a small GEMM on the GPU)."""
    __slots__ = ("index", "prev")

    def __init__(self, device):
        self.index = device.index

    def __enter__(self):
        import torch
        cur = torch.cuda.current_device()
        self.prev = cur if cur != self.index else None
        if self.prev is not None:
            torch.cuda.set_device(self.index)

    def __exit__(self, *exc):
        if self.prev is not None:
            import torch
            torch.cuda.set_device(self.prev)
        return False


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
    timeout_ms, multicast, f32_mode).  Raises ``ValueError`` on a
    shape mismatch and ``TgError`` on any status other than TG_OK.
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
    with _OnDevice(a.device):
        st = tg_gemm_ex(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc,
                        dtype_code(a.dtype), dtype_code(out_dtype), _stream_handle(stream), opt)
    if st != TG_OK:
        raise TgError(st, f"tg_gemm_ex(M={M}, N={N}, K={K})")
    return out


def gemm_fused(a, b, out_dtype=None, out=None, stream=None, alpha=1.0, scale=None, bias=None,
               activation="none", beta=0.0, residual=None, **options):
    """C = act(alpha * scale * (A @ B) + bias) + beta * residual, through
    ``tg_gemm_fused``; the epilogue runs on the FP32 accumulator before the
    one rounding to ``out_dtype``.

    ``scale`` and ``bias`` are optional float32 CUDA vectors of length N;
    ``residual`` an optional [M, N] CUDA tensor of ``out_dtype`` with unit
    column stride (it may be ``out`` itself).  ``activation``: "none", "relu",
    "silu" or "gelu_tanh".  Other arguments as for ``gemm``.
    """
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("gemm_fused expects [M, K] @ [K, N]")
    if a.dtype != b.dtype or not (a.is_cuda and b.is_cuda):
        raise ValueError("A and B must be CUDA tensors of the same dtype")
    M, K = a.shape
    N = b.shape[1]
    if (a.stride(1) != 1 and K > 1) or (b.stride(1) != 1 and N > 1):
        raise ValueError("A and B need unit column stride")
    out_dtype = a.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    elif out.shape != (M, N) or out.dtype != out_dtype or (out.stride(1) != 1 and N > 1):
        raise ValueError("out must be [M, N] of out_dtype with unit column stride")
    for name, v in (("scale", scale), ("bias", bias)):
        if v is not None and (v.dtype != torch.float32 or v.shape != (N,) or not v.is_cuda
                              or (v.stride(0) != 1 and N > 1)):
            raise ValueError(f"{name} must be a contiguous float32 CUDA vector of length N")
    ldr = 0
    if residual is not None:
        if (residual.shape != (M, N) or residual.dtype != out_dtype or not residual.is_cuda
                or (residual.stride(1) != 1 and N > 1)):
            raise ValueError("residual must be [M, N] of out_dtype with unit column stride")
        ldr = residual.stride(0) if M > 1 else max(N, 1)
    lda = a.stride(0) if M > 1 else max(K, 1)
    ldb = b.stride(0) if K > 1 else max(N, 1)
    ldc = out.stride(0) if M > 1 else max(N, 1)
    ep = make_epilogue(alpha=alpha, beta=beta,
                       scale=scale.data_ptr() if scale is not None else 0,
                       bias=bias.data_ptr() if bias is not None else 0,
                       residual=residual.data_ptr() if residual is not None else 0, ldr=ldr,
                       activation=activation)
    opt = make_options(**options) if options else None
    with _OnDevice(a.device):
        st = tg_gemm_fused(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc,
                           dtype_code(a.dtype), dtype_code(out_dtype), ep,
                           _stream_handle(stream), opt)
    if st != TG_OK:
        raise TgError(st, f"tg_gemm_fused(M={M}, N={N}, K={K})")
    return out


def _batch_stride(t, dims: int) -> int:
    """Element stride between the products of a [B, rows, cols] tensor (0 for 2-D)."""
    return 0 if t.dim() == dims - 1 else (t.stride(0) if t.shape[0] > 1 else 0)


def _bmm_args(a, b, out_dtype, out):
    """Shapes, pitches and batch strides of C[z] = A[z] @ B[z] (see ``bmm``)."""
    import torch
    if a.dim() not in (2, 3) or b.dim() not in (2, 3) or (a.dim() == 2 and b.dim() == 2):
        raise ValueError("bmm expects [B, M, K] or [M, K] times [B, K, N] or [K, N]")
    if a.dtype != b.dtype:
        raise ValueError("A and B must have the same dtype")
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    batch = a.shape[0] if a.dim() == 3 else b.shape[0]
    if (a.dim() == 3 and a.shape[0] != batch) or (b.dim() == 3 and b.shape[0] != batch):
        raise ValueError("batch sizes differ")
    M, K = a.shape[-2], a.shape[-1]
    N = b.shape[-1]
    if b.shape[-2] != K:
        raise ValueError("inner dimensions differ")
    if (a.stride(-1) != 1 and K > 1) or (b.stride(-1) != 1 and N > 1):
        raise ValueError("A and B need unit column stride")
    out_dtype = a.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((batch, M, N), dtype=out_dtype, device=a.device)
    elif (out.shape != (batch, M, N) or out.dtype != out_dtype or
          (out.stride(-1) != 1 and N > 1)):
        raise ValueError("out must be [B, M, N] of out_dtype with unit column stride")
    lda = a.stride(-2) if M > 1 else max(K, 1)
    ldb = b.stride(-2) if K > 1 else max(N, 1)
    ldc = out.stride(-2) if M > 1 else max(N, 1)
    sc = out.stride(0) if batch > 1 else (M - 1) * ldc + N
    return (batch, M, N, K, lda, _batch_stride(a, 3), ldb, _batch_stride(b, 3), ldc, sc,
            out_dtype, out)


def bmm(a, b, out_dtype=None, out=None, stream=None, **options):
    """C[z] = A[z] @ B[z] through ``tg_gemm_strided_batched``.

    ``a`` is [B, M, K] or a shared [M, K]; ``b`` is [B, K, N] or a shared
    [K, N] (at least one of them 3-D), same dtype, unit column stride.  The
    result is a new [B, M, N] tensor of ``out_dtype`` (default: the input
    dtype), or ``out`` with unit column stride.  Raises ``ValueError`` on a
    shape mismatch and ``TgError`` on any status other than TG_OK.
    """
    import torch
    batch, M, N, K, lda, sa, ldb, sb, ldc, sc, out_dtype, out = _bmm_args(a, b, out_dtype, out)
    opt = make_options(**options) if options else None
    with _OnDevice(a.device):
        st = tg_gemm_strided_batched(batch, M, N, K, a.data_ptr(), lda, sa, b.data_ptr(), ldb, sb,
                                     out.data_ptr(), ldc, sc, dtype_code(a.dtype),
                                     dtype_code(out_dtype), _stream_handle(stream), opt)
    if st != TG_OK:
        raise TgError(st, f"tg_gemm_strided_batched(batch={batch}, M={M}, N={N}, K={K})")
    return out


def bmm_fused(a, b, out_dtype=None, out=None, stream=None, alpha=1.0, scale=None, bias=None,
              activation="none", beta=0.0, residual=None, **options):
    """C[z] = act(alpha * scale * (A[z] @ B[z]) + bias) + beta * residual[z],
    through ``tg_gemm_strided_batched_fused``.

    Operands as for ``bmm``; ``scale`` / ``bias`` as for ``gemm_fused`` (shared
    by every product); ``residual`` a [B, M, N] tensor (one block per product,
    possibly ``out`` itself) or a shared [M, N] one, of ``out_dtype`` with unit
    column stride.
    """
    import torch
    batch, M, N, K, lda, sa, ldb, sb, ldc, sc, out_dtype, out = _bmm_args(a, b, out_dtype, out)
    for name, v in (("scale", scale), ("bias", bias)):
        if v is not None and (v.dtype != torch.float32 or v.shape != (N,) or not v.is_cuda
                              or (v.stride(0) != 1 and N > 1)):
            raise ValueError(f"{name} must be a contiguous float32 CUDA vector of length N")
    ldr, sr = 0, 0
    if residual is not None:
        if (residual.shape not in ((batch, M, N), (M, N)) or residual.dtype != out_dtype
                or not residual.is_cuda or (residual.stride(-1) != 1 and N > 1)):
            raise ValueError("residual must be [B, M, N] or [M, N] of out_dtype with unit "
                             "column stride")
        ldr = residual.stride(-2) if M > 1 else max(N, 1)
        sr = _batch_stride(residual, 3)
    ep = make_epilogue(alpha=alpha, beta=beta,
                       scale=scale.data_ptr() if scale is not None else 0,
                       bias=bias.data_ptr() if bias is not None else 0,
                       residual=residual.data_ptr() if residual is not None else 0, ldr=ldr,
                       activation=activation)
    opt = make_options(**options) if options else None
    with _OnDevice(a.device):
        st = tg_gemm_strided_batched_fused(batch, M, N, K, a.data_ptr(), lda, sa, b.data_ptr(),
                                           ldb, sb, out.data_ptr(), ldc, sc, dtype_code(a.dtype),
                                           dtype_code(out_dtype), ep, sr,
                                           _stream_handle(stream), opt)
    if st != TG_OK:
        raise TgError(st, f"tg_gemm_strided_batched_fused(batch={batch}, M={M}, N={N}, K={K})")
    return out


def plan_batched(batch, M, N, K, dtype_in="f16", dtype_out=None, num_sms=148, stride_a=None,
                 stride_b=None, stride_c=None, lda=None, ldb=None, ldc=None, a=0x1000,
                 b=0x10000000000, c=0x20000000000, **options) -> dict:
    """What ``tg_gemm_strided_batched`` would launch (host only, no GPU); the
    default strides are those of contiguous [B, rows, cols] operands."""
    dtype_out = dtype_in if dtype_out is None else dtype_out
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sa = M * lda if stride_a is None else stride_a
    sb = K * ldb if stride_b is None else stride_b
    sc = M * ldc if stride_c is None else stride_c
    opt = make_options(**options) if options else None
    st, p = tg_plan_gemm_strided_batched(batch, M, N, K, a, lda, sa, b, ldb, sb, c, ldc, sc,
                                         dtype_in, dtype_out, num_sms, opt)
    if st != TG_OK:
        raise TgError(st, "tg_plan_gemm_strided_batched")
    return p


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
