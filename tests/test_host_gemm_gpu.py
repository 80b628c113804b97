"""GPU parity of tg_gemm_host (operands and result in page-locked host
memory, copies pipelined with the multiply): every element against the
oracle, one and several row panels, ragged sizes, padded host pitches (the
padding of C untouched), K = 0, FP32 and FP8 operands, and repeated calls on
one stream."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare
from tiled_matrix_multiplication_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


def pinned(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits)).pin_memory()
    return t


def run_host(M, N, K, din, dout, dist="uniform", lda=None, ldb=None, ldc=None, **opts):
    import torch
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    a_bits = inputs.matrix_bits(M, K, din, dist, inputs.SEED_A, ld=lda)
    b_bits = inputs.matrix_bits(K, N, din, dist, inputs.SEED_B, ld=ldb)
    poison = inputs.nan_bits(dout)
    a, b = pinned(a_bits), pinned(b_bits)
    c = pinned(np.full((M, ldc), poison, dtype=inputs.BITS_NP[dout]))
    opt = tg.make_options(**opts) if opts else None
    s = torch.cuda.current_stream()
    st = tg.tg_gemm_host(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, c.data_ptr(), ldc, din,
                         dout, s.cuda_stream, opt)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    s.synchronize()
    tg.check_device_error()
    out = c.numpy().copy()
    if ldc > N:
        assert np.all(out[:, N:] == poison), "padding of C was written"
    return a_bits, b_bits, out


@pytest.mark.parametrize("M,N,K", [(127, 255, 65), (300, 520, 200), (2049, 700, 300),
                                   (4096, 256, 128), (1, 8192, 64)])
def test_panels_every_element(M, N, K):
    a, b, c = run_host(M, N, K, "f16", "f16")
    compare(a, b, c, M, N, K, "f16", "f16")


def test_padded_host_pitches():
    a, b, c = run_host(1500, 300, 130, "bf16", "f32", lda=133, ldb=301, ldc=307)
    compare(a, b, c, 1500, 300, 130, "bf16", "f32")


def test_integer_exact_fp8_and_tf32():
    a, b, c = run_host(1100, 400, 256, "e4m3", "f16", dist="int")
    compare(a, b, c, 1100, 400, 256, "e4m3", "f16", exact=True)
    a, b, c = run_host(1000, 333, 77, "f32", "f32")
    compare(a, b, c, 1000, 333, 77, "f32", "f32")


def test_k_zero():
    a, b, c = run_host(600, 50, 0, "f16", "f32", ldc=53)
    assert np.all(c[:, :50] == 0)


def test_repeated_calls_on_one_stream():
    import torch
    M, N, K = 2048, 512, 256
    outs = []
    bufs = []
    s = torch.cuda.current_stream()
    for i in range(3):
        a_bits = inputs.matrix_bits(M, K, "f16", "int", 50 + i)
        b_bits = inputs.matrix_bits(K, N, "f16", "int", 60 + i)
        a, b = pinned(a_bits), pinned(b_bits)
        c = pinned(np.zeros((M, N), dtype=np.uint16))
        assert tg.tg_gemm_host(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                               "f16", "f16", s.cuda_stream, None) == tg.TG_OK
        bufs.append((a_bits, b_bits, a, b, c))
    s.synchronize()
    for a_bits, b_bits, _, _, c in bufs:
        compare(a_bits, b_bits, c.numpy(), M, N, K, "f16", "f16", exact=True)


def test_argument_errors_before_any_copy():
    assert tg.tg_gemm_host(4, 4, 4, 0, 4, 0, 4, 0, 4, "f16", "f16", 0, None) \
        == tg.TG_ERR_INVALID_VALUE


def test_alternating_streams():
    # consecutive calls on two streams overlap their copies; each result is
    # still complete once its own stream is synchronised
    import torch
    M, N, K = 2048, 1024, 512
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    calls = []
    for i in range(4):
        a_bits = inputs.matrix_bits(M, K, "bf16", "int", 70 + i)
        b_bits = inputs.matrix_bits(K, N, "bf16", "int", 80 + i)
        a, b = pinned(a_bits), pinned(b_bits)
        c = pinned(np.zeros((M, N), dtype=np.uint16))
        s = streams[i % 2]
        assert tg.tg_gemm_host(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                               "bf16", "bf16", s.cuda_stream, None) == tg.TG_OK
        calls.append((a_bits, b_bits, a, b, c, s))
    for a_bits, b_bits, _, _, c, s in calls:
        s.synchronize()
        compare(a_bits, b_bits, c.numpy(), M, N, K, "bf16", "bf16", exact=True)


def test_result_feeds_the_next_call_on_one_stream():
    # the second call reads, as its A, the host buffer the first call writes:
    # stream order makes the first call's copy-back land before the read
    import torch
    n = 1024
    s = torch.cuda.current_stream()
    a_bits = inputs.matrix_bits(n, n, "f32", "int", 90)
    b_bits = inputs.matrix_bits(n, n, "f32", "int", 91)
    a, b = pinned(a_bits), pinned(b_bits)
    c1 = pinned(np.zeros((n, n), dtype=np.uint32))
    c2 = pinned(np.zeros((n, n), dtype=np.uint32))
    assert tg.tg_gemm_host(n, n, n, a.data_ptr(), n, b.data_ptr(), n, c1.data_ptr(), n, "f32",
                           "f32", s.cuda_stream, None) == tg.TG_OK
    assert tg.tg_gemm_host(n, n, n, c1.data_ptr(), n, b.data_ptr(), n, c2.data_ptr(), n, "f32",
                           "f32", s.cuda_stream, None) == tg.TG_OK
    s.synchronize()
    compare(a_bits, b_bits, c1.numpy(), n, n, n, "f32", "f32", exact=True)
    # C1 holds integers up to 4096 in magnitude: exact in TF32 only below 2^11,
    # so the second product is checked within the TF32 tolerance
    compare(c1.numpy(), b_bits, c2.numpy(), n, n, n, "f32", "f32")
