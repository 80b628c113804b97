"""GPU parity of the strided-batched product with the fused epilogue
C_z = act(alpha * scale * (A_z B_z) + bias) + beta * R_z: every product is
checked element by element against the oracle's epilogue reference, with its
own seeded operands and residual block (a product reading another one's
residual, or the residual of z = 0 for every z, fails), and every element of
C that no product owns keeps its poison value.

Covers the one-launch kernels (single CTA, CTA pair with and without A
multicast, the small-M kernel with its on-chip K split and two CTAs per SM),
one residual shared by every product (stride 0), residuals in place (R_z =
C_z), C and R interleaved along rows, batch strides that force the scalar
residual loads, the one-call-per-product route (TF32, misaligned operands),
K = 0 and the torch-level ``bmm_fused`` helper.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import to_bits, to_device, torch_dtype
from tests.test_batched_gpu import flat_operand
from tests.test_epilogue_gpu import f32_vector
from tiled_matrix_multiplication_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

SEED_R = 73


def run_batched_fused(batch, M, N, K, din, dout, act="silu", alpha=1.0, beta=0.5,
                      use_scale=True, use_bias=True, residual=True, sr=None, in_place=False,
                      lda=None, ldb=None, ldc=None, ldr=None, sa=None, sb=None, sc=None,
                      a_off=0, **opts):
    import torch
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sa = M * lda if sa is None else sa
    sb = K * ldb if sb is None else sb
    sc = M * ldc if sc is None else sc
    if in_place:
        ldr, sr = ldc, sc
    ldr = N if ldr is None else ldr
    sr = M * ldr if sr is None else sr
    a_flat, a_mats = flat_operand(batch, M, K, lda, sa, din, "uniform", inputs.SEED_A)
    b_flat, b_mats = flat_operand(batch, K, N, ldb, sb, din, "uniform", inputs.SEED_B + 1000)
    a_flat = np.concatenate([np.zeros(a_off, a_flat.dtype), a_flat])
    c_len = max(sc * (batch - 1) + M * ldc, 1)
    poison = inputs.nan_bits(dout)
    c_init = np.full(c_len, poison, dtype=inputs.BITS_NP[dout])
    r_mats = None
    if residual:
        # block z at z*sr + m*ldr + n (sr == 0: one block for every product)
        r_mats = [inputs.matrix_bits(M, N, dout, "uniform", SEED_R + (z if sr else 0))
                  for z in range(batch if sr else 1)]
        r_mats = [r_mats[z if sr else 0] for z in range(batch)]
        r_len = max((batch - 1) * sr + (M - 1) * ldr + N, 1)
        r_flat = c_init if in_place else np.zeros(r_len, dtype=inputs.BITS_NP[dout])
        for z in range(batch):
            idx = z * sr + np.arange(M)[:, None] * ldr + np.arange(N)[None, :]
            r_flat[idx] = r_mats[z]
    scale = f32_vector(N, 71, 0.5, 1.5) if use_scale else None
    bias = f32_vector(N, 72, -1.0, 1.0) if use_bias else None
    a_dev = to_device(a_flat, din)
    b_dev = to_device(b_flat, din)
    c_dev = to_device(c_init, dout)
    r_dev = c_dev if in_place else (to_device(r_flat, dout) if residual else None)
    sc_d = torch.from_numpy(scale).cuda() if use_scale else None
    bi_d = torch.from_numpy(bias).cuda() if use_bias else None
    ep = tg.make_epilogue(alpha=alpha, beta=beta,
                          scale=sc_d.data_ptr() if use_scale else 0,
                          bias=bi_d.data_ptr() if use_bias else 0,
                          residual=r_dev.data_ptr() if residual else 0,
                          ldr=ldr if residual else 0, activation=act)
    opt = tg.make_options(**opts) if opts else None
    es = inputs.BITS_NP[din]().itemsize
    st = tg.tg_gemm_strided_batched_fused(
        batch, M, N, K, a_dev.data_ptr() + a_off * es, lda, sa, b_dev.data_ptr(), ldb, sb,
        c_dev.data_ptr(), ldc, sc, din, dout, ep, sr if residual else 0,
        torch.cuda.current_stream().cuda_stream, opt)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    torch.cuda.synchronize()
    tg.check_device_error()
    c_flat = to_bits(c_dev, dout)
    owned = np.zeros(c_len, dtype=bool)
    for z in range(batch):
        idx = z * sc + np.arange(M)[:, None] * ldc + np.arange(N)[None, :]
        owned[idx] = True
        C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_mats[z][:, :K]),
                                        np.ascontiguousarray(b_mats[z][:, :N]), K=K, N=N,
                                        fmt=din)
        R = oracle.decode(r_mats[z], dout) if residual else None
        got = oracle.decode(np.ascontiguousarray(c_flat[idx]), dout)
        ok, report = oracle.epilogue.check_epilogue(
            got, C_ref, S, din, dout, alpha=alpha, scale=scale, bias=bias, act=act, beta=beta,
            R=R)
        assert ok, f"product {z}: {report}"
    assert np.all(c_flat[~owned] == c_init[~owned]), \
        "an element outside every product's C was written"


def test_single_cta_bf16():
    run_batched_fused(3, 300, 520, 200, "bf16", "bf16", path=tg.TG_PATH_TC)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_pair_multicast(act):
    run_batched_fused(3, 520, 1100, 256, "f16", "f16", act=act, path=tg.TG_PATH_TC_PAIR,
                      multicast=2, block_n=256)


def test_pair_shared_residual_to_f32():
    run_batched_fused(3, 520, 600, 256, "f16", "f32", act="none", beta=1.0, sr=0,
                      path=tg.TG_PATH_TC_PAIR, multicast=1)


def test_in_place():
    run_batched_fused(4, 260, 384, 192, "bf16", "bf16", act="relu", beta=1.0, in_place=True)


def test_interleaved_c_and_residual():
    # C and R stored [M][batch][N]: products sit side by side along a row
    batch, M, N = 3, 200, 136
    run_batched_fused(batch, M, N, 160, "f16", "f16", ldc=batch * N, sc=N, ldr=batch * N, sr=N)


def test_residual_stride_scalar_loads():
    # a residual batch stride of an odd number of elements: no 16-byte loads
    run_batched_fused(3, 300, 520, 200, "f16", "f16", sr=300 * 520 + 1)


def test_small_m_on_chip_split():
    run_batched_fused(3, 64, 512, 2048, "bf16", "bf16", act="gelu_tanh",
                      path=tg.TG_PATH_SKINNY, splits=4)


def test_small_m_two_per_sm():
    p = tg.plan_batched(40, 16, 1024, 512, num_sms=152)
    assert p["path"] == tg.TG_PATH_SKINNY and p["ctas"] > 152
    run_batched_fused(40, 16, 1024, 512, "f16", "f32", act="silu")


def test_per_product_route_tf32():
    run_batched_fused(3, 130, 200, 96, "f32", "f32", act="silu")


def test_per_product_route_misaligned_a():
    # A starts one element past a 16-byte boundary: no rank-3 map, one call per product
    run_batched_fused(3, 200, 264, 128, "f16", "f16", a_off=1)


def test_k_zero():
    run_batched_fused(3, 100, 136, 0, "f16", "f16", act="gelu_tanh")


def test_bmm_fused_helper():
    import torch
    g = torch.Generator(device="cpu").manual_seed(5)
    a = torch.randn(4, 150, 96, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(4, 96, 200, generator=g).to(torch.bfloat16).cuda()
    r = torch.randn(4, 150, 200, generator=g).to(torch.bfloat16).cuda()
    bias = torch.randn(200, generator=g).float().cuda()
    out = tg.bmm_fused(a, b, bias=bias, activation="relu", beta=1.0, residual=r)
    torch.cuda.synchronize()
    tg.check_device_error()
    a_bits, b_bits, r_bits = (to_bits(t, "bf16") for t in (a, b, r))
    o_bits = to_bits(out, "bf16")
    for z in range(4):
        C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_bits[z]),
                                        np.ascontiguousarray(b_bits[z]), K=96, N=200, fmt="bf16")
        ok, report = oracle.epilogue.check_epilogue(
            oracle.decode(np.ascontiguousarray(o_bits[z]), "bf16"), C_ref, S, "bf16", "bf16",
            bias=bias.cpu().numpy(), act="relu", beta=1.0,
            R=oracle.decode(np.ascontiguousarray(r_bits[z]), "bf16"))
        assert ok, f"product {z}: {report}"
    # a shared [M, N] residual
    out2 = tg.bmm_fused(a, b, residual=r[1], beta=1.0)
    torch.cuda.synchronize()
    o2 = to_bits(out2, "bf16")
    for z in range(4):
        C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_bits[z]),
                                        np.ascontiguousarray(b_bits[z]), K=96, N=200, fmt="bf16")
        ok, report = oracle.epilogue.check_epilogue(
            oracle.decode(np.ascontiguousarray(o2[z]), "bf16"), C_ref, S, "bf16", "bf16",
            beta=1.0, R=oracle.decode(np.ascontiguousarray(r_bits[1]), "bf16"))
        assert ok, f"shared residual, product {z}: {report}"
