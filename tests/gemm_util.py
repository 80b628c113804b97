"""Helpers shared by the GPU parity tests: upload seeded bit patterns, run the
library through its binding, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import inputs

_INT_VIEW = {"f16": np.int16, "bf16": np.int16, "f32": np.int32, "e4m3": np.uint8,
             "e5m2": np.uint8}


def torch_dtype(name):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[name]


def to_device(bits: np.ndarray, dtype: str):
    """Bit patterns -> CUDA tensor of ``dtype`` holding exactly those bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(_INT_VIEW[dtype]))
    return t.view(torch_dtype(dtype)).cuda()


def to_bits(t, dtype: str) -> np.ndarray:
    import torch
    ints = {"f16": torch.int16, "bf16": torch.int16, "f32": torch.int32, "e4m3": torch.uint8,
            "e5m2": torch.uint8}[dtype]
    host = t.detach().contiguous().view(ints).cpu().numpy()
    return host.view(inputs.BITS_NP[dtype])


def run_gemm(M, N, K, din, dout, dist="uniform", lda=None, ldb=None, ldc=None,
             seed_a=inputs.SEED_A, seed_b=inputs.SEED_B, poison=None, a_bits=None, b_bits=None,
             **opts):
    """Runs C = A*B on the GPU; returns ``(a_bits, b_bits, c_bits)`` where
    ``c_bits`` is the whole ``[M, ldc]`` output buffer (padding included)."""
    import torch
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    if a_bits is None:
        a_bits = inputs.matrix_bits(M, K, din, dist, seed_a, ld=lda)
    if b_bits is None:
        b_bits = inputs.matrix_bits(K, N, din, dist, seed_b, ld=ldb)
    a_buf = to_device(a_bits, din) if M * lda else torch.empty((M, lda), dtype=torch_dtype(din), device="cuda")
    b_buf = to_device(b_bits, din) if K * ldb else torch.empty((K, ldb), dtype=torch_dtype(din), device="cuda")
    poison = inputs.nan_bits(dout) if poison is None else poison
    c_init = np.full((M, ldc), poison, dtype=inputs.BITS_NP[dout])
    c_buf = to_device(c_init, dout) if M * ldc else torch.empty((M, ldc), dtype=torch_dtype(dout), device="cuda")
    a = a_buf[:, :K]
    b = b_buf[:, :N]
    c = c_buf[:, :N]
    tg.gemm(a, b, out_dtype=torch_dtype(dout), out=c, **opts)
    torch.cuda.synchronize()
    tg.check_device_error()
    return a_bits, b_bits, to_bits(c_buf, dout)


def compare(a_bits, b_bits, c_bits, M, N, K, din, dout, exact=False, rows=None, cols=None):
    """Element-by-element comparison with the oracle on the selected rows
    (all rows by default) and columns (all by default).  ``exact``: integer
    inputs, the bits must match the oracle's correctly rounded result."""
    if rows is None:
        rows = np.arange(M)
    rows = np.asarray(rows, dtype=np.int64)
    if cols is None:
        b_sel = b_bits[:K, :N]
        got_bits = c_bits[rows][:, :N]
    else:
        cols = np.asarray(cols, dtype=np.int64)
        b_sel = b_bits[:K][:, cols]
        got_bits = c_bits[rows][:, cols]
    ncols = b_sel.shape[1]
    C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_bits[rows]), np.ascontiguousarray(b_sel),
                                    K=K, N=ncols, fmt=din)
    if exact:
        want = oracle.encode(C_ref, dout)
        bad = np.argwhere(want != got_bits)
        assert bad.size == 0, (f"{len(bad)} mismatches; first at {tuple(bad[0])}: got "
                               f"{hex(int(got_bits[tuple(bad[0])]))} want {hex(int(want[tuple(bad[0])]))}")
        return
    got = oracle.decode(got_bits, dout)
    ok, report = oracle.check_close(got, C_ref, S, din, dout)
    assert ok, report


def padding_untouched(c_bits, N, dout, poison=None):
    poison = inputs.nan_bits(dout) if poison is None else poison
    return bool(np.all(c_bits[:, N:] == poison))
