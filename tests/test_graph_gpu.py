"""The library's calls inside a CUDA graph: calls captured on a stream and
replayed must give the results of direct calls (checked element by element
against the oracle) on every launch route -- tile kernel, small-M kernel,
split-K with its workspace and reduce kernel, packed (misaligned) operands,
the fused epilogue, a strided batch -- and a replay after the inputs change
must see the new inputs (the graph holds pointers, not copies)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare, to_bits, to_device
from tiled_matrix_multiplication_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

CASES = [
    # (M, N, K, din, dout, lda_pad, options)
    (300, 520, 200, "f16", "f16", 0, {}),                                   # tile kernel (pairs)
    (64, 1000, 700, "bf16", "bf16", 0, {}),                                # small-M kernel
    (256, 512, 4096, "f16", "f32", 0, dict(path=tg.TG_PATH_TC, splits=4)),  # split-K + reduce
    (127, 255, 65, "f16", "f32", 0, {}),                                   # packed operands
    (200, 264, 130, "f32", "f32", 3, {}),                                  # TF32: pack + transpose
]


def _operands(M, N, K, din, lda, seed):
    a_bits = inputs.matrix_bits(M, K, din, "int", inputs.SEED_A + seed, ld=lda)
    b_bits = inputs.matrix_bits(K, N, din, "int", inputs.SEED_B + seed)
    return a_bits, b_bits


def test_captured_calls_replay_exactly():
    import torch
    stream = torch.cuda.Stream()
    bufs = []
    for i, (M, N, K, din, dout, pad, opts) in enumerate(CASES):
        lda = K + pad
        a_bits, b_bits = _operands(M, N, K, din, lda, i)
        a = to_device(a_bits, din)
        b = to_device(b_bits, din)
        c = to_device(np.full((M, N), inputs.nan_bits(dout), dtype=inputs.BITS_NP[dout]), dout)
        bufs.append((a, b, c, a_bits, b_bits))

    def enqueue():
        for (M, N, K, din, dout, pad, opts), (a, b, c, _, _) in zip(CASES, bufs):
            o = tg.make_options(**opts) if opts else None
            st = tg.tg_gemm_ex(M, N, K, a.data_ptr(), K + pad, b.data_ptr(), N, c.data_ptr(), N,
                               din, dout, stream.cuda_stream, o)
            assert st == tg.TG_OK, tg.tg_status_string(st)

    # warm up outside the capture (first-call device state, pools, kernels)
    with torch.cuda.stream(stream):
        enqueue()
    stream.synchronize()
    tg.check_device_error()
    for _, _, c, _, _ in bufs:
        c.fill_(float("nan"))
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        enqueue()
    graph.replay()
    torch.cuda.synchronize()
    tg.check_device_error()
    for (M, N, K, din, dout, pad, _), (a, b, c, a_bits, b_bits) in zip(CASES, bufs):
        compare(np.ascontiguousarray(a_bits[:, :K]), b_bits, to_bits(c, dout), M, N, K, din, dout,
                exact=True)

    # new inputs in the same buffers, replay again
    for i, ((M, N, K, din, dout, pad, _), (a, b, c, _, _)) in enumerate(zip(CASES, bufs)):
        a_bits, b_bits = _operands(M, N, K, din, K + pad, 100 + i)
        a.copy_(to_device(a_bits, din))
        b.copy_(to_device(b_bits, din))
        bufs[i] = (a, b, c, a_bits, b_bits)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    tg.check_device_error()
    for (M, N, K, din, dout, pad, _), (a, b, c, a_bits, b_bits) in zip(CASES, bufs):
        compare(np.ascontiguousarray(a_bits[:, :K]), b_bits, to_bits(c, dout), M, N, K, din, dout,
                exact=True)


def test_captured_fused_and_batched():
    import torch
    stream = torch.cuda.Stream()
    g = torch.Generator(device="cpu").manual_seed(11)
    a = torch.randint(-2, 3, (3, 150, 96), generator=g).to(torch.bfloat16).cuda()
    b = torch.randint(-2, 3, (3, 96, 200), generator=g).to(torch.bfloat16).cuda()
    r = torch.randint(-2, 3, (3, 150, 200), generator=g).to(torch.bfloat16).cuda()
    bias = torch.randint(-2, 3, (200,), generator=g).float().cuda()
    out = torch.empty(3, 150, 200, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        tg.bmm_fused(a, b, out=out, bias=bias, activation="relu", beta=1.0, residual=r,
                     stream=stream)
    stream.synchronize()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        tg.bmm_fused(a, b, out=out, bias=bias, activation="relu", beta=1.0, residual=r,
                     stream=stream)
    graph.replay()
    torch.cuda.synchronize()
    tg.check_device_error()
    a_bits, b_bits, r_bits = (to_bits(t, "bf16") for t in (a, b, r))
    o_bits = to_bits(out, "bf16")
    for z in range(3):
        C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_bits[z]),
                                        np.ascontiguousarray(b_bits[z]), K=96, N=200, fmt="bf16")
        ok, report = oracle.epilogue.check_epilogue(
            oracle.decode(np.ascontiguousarray(o_bits[z]), "bf16"), C_ref, S, "bf16", "bf16",
            bias=bias.cpu().numpy(), act="relu", beta=1.0,
            R=oracle.decode(np.ascontiguousarray(r_bits[z]), "bf16"))
        assert ok, f"product {z}: {report}"
