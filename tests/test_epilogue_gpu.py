"""GPU parity of the fused epilogue C = act(alpha * scale * (A B) + bias) +
beta * R on every kernel path (single CTA, CTA pair, 512-wide pair tiles,
pairs sharing A by multicast, the small-M kernel, K split summed by the
reduce kernel, TF32; C through TMA stores or the warps' own stores), each
activation, with and without residual,
in place (R = C), K = 0, scalar and vector loads of the epilogue operands.
The oracle's epilogue reference and tolerance (oracle/epilogue.py) decide.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import to_bits, to_device
from tiled_matrix_multiplication_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

ACTS = ("none", "relu", "silu", "gelu_tanh")


def f32_vector(n, seed, lo, hi, pad=0):
    """n float32 values in [lo, hi) from the seeded generator (after `pad`
    leading zeros, to misalign the vector's start)."""
    u = inputs.matrix_bits(1, n, "f32", "uniform", seed).view(np.float32).astype(np.float64)
    v = (lo + (hi - lo) * (u[0] + 1.0) / 2.0).astype(np.float32)
    return np.concatenate([np.zeros(pad, np.float32), v])


def run_fused(M, N, K, din, dout, act="none", alpha=1.0, beta=0.0, use_scale=True,
              use_bias=True, residual=True, in_place=False, ldc=None, ldr=None, sb_pad=0,
              dist="uniform", rows=None, **opts):
    import torch
    ldc = N if ldc is None else ldc
    ldr = (ldc if in_place else N) if ldr is None else ldr
    a_bits = inputs.matrix_bits(M, K, din, dist, inputs.SEED_A)
    b_bits = inputs.matrix_bits(K, N, din, dist, inputs.SEED_B)
    a = to_device(a_bits, din) if M * K else torch.empty((M, K), device="cuda",
                                                         dtype={"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[din])
    b = to_device(b_bits, din) if K * N else torch.empty((K, N), device="cuda", dtype=a.dtype)
    scale = f32_vector(N, 71, 0.5, 1.5, sb_pad) if use_scale else None
    bias = f32_vector(N, 72, -1.0, 1.0, sb_pad) if use_bias else None
    sc_d = torch.from_numpy(scale).cuda() if use_scale else None
    bi_d = torch.from_numpy(bias).cuda() if use_bias else None
    poison = inputs.nan_bits(dout)
    r_bits = inputs.matrix_bits(M, N, dout, "uniform", 73, ld=ldr) if residual else None
    if in_place:
        assert ldr == ldc
        c_init = r_bits.copy()
    else:
        c_init = np.full((M, ldc), poison, dtype=inputs.BITS_NP[dout])
    c = to_device(c_init, dout)
    r = c if in_place else (to_device(r_bits, dout) if residual else None)
    ep = tg.make_epilogue(alpha=alpha, beta=beta,
                          scale=(sc_d.data_ptr() + 4 * sb_pad) if use_scale else 0,
                          bias=(bi_d.data_ptr() + 4 * sb_pad) if use_bias else 0,
                          residual=r.data_ptr() if residual else 0, ldr=ldr if residual else 0,
                          activation=act)
    opt = tg.make_options(**opts) if opts else None
    st = tg.tg_gemm_fused(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), ldc, din, dout,
                          ep, torch.cuda.current_stream().cuda_stream, opt)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    torch.cuda.synchronize()
    tg.check_device_error()
    c_bits = to_bits(c, dout)
    sel = np.arange(M) if rows is None else np.asarray(rows)
    C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a_bits[sel]), b_bits, K=K, N=N, fmt=din)
    R = oracle.decode(np.ascontiguousarray(r_bits[sel][:, :N]), dout) if residual else None
    got = oracle.decode(np.ascontiguousarray(c_bits[sel][:, :N]), dout)
    kw = dict(alpha=alpha, scale=scale[sb_pad:] if use_scale else None,
              bias=bias[sb_pad:] if use_bias else None, act=act, beta=beta, R=R)
    ok, report = oracle.epilogue.check_epilogue(got, C_ref, S, din, dout, **kw)
    assert ok, report
    if not in_place and ldc > N:
        assert np.all(c_bits[:, N:] == poison), "padding columns of C were written"
    return c_bits


PATHS = {
    "auto": dict(),
    "single_cta": dict(path=tg.TG_PATH_TC, block_n=128),
    "pair": dict(path=tg.TG_PATH_TC_PAIR, multicast=1, block_n=256),
    "pair_multicast": dict(path=tg.TG_PATH_TC_PAIR, multicast=2, block_n=256),
    "split_k": dict(path=tg.TG_PATH_TC_PAIR, splits=3, multicast=1),
    "pair_wide": dict(path=tg.TG_PATH_TC_PAIR, block_n=512),
    "pair_wide_small_grid": dict(path=tg.TG_PATH_TC_PAIR, block_n=512, max_ctas=2),
}


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("path", sorted(PATHS))
def test_paths_and_activations(path, act):
    M, N, K = (1000, 1100, 600) if path == "pair_wide_small_grid" else (300, 520, 200)
    run_fused(M, N, K, "f16", "f16", act=act, alpha=0.75, beta=-0.5, **PATHS[path])


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M", [1, 40, 128])
def test_small_m_kernel(M, act):
    p = tg.plan(M, 1000, 700, "bf16", num_sms=152, path=tg.TG_PATH_SKINNY)
    assert p["path"] == tg.TG_PATH_SKINNY
    run_fused(M, 1000, 700, "bf16", "bf16", act=act, alpha=1.25, beta=1.0,
              path=tg.TG_PATH_SKINNY)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_tf32(act):
    run_fused(200, 300, 130, "f32", "f32", act=act, alpha=0.5, beta=2.0)


@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_wide_output_and_padding(dout):
    run_fused(257, 300, 96, "bf16", dout, act="silu", ldc=320, ldr=304, beta=0.25)


def test_in_place_residual():
    run_fused(300, 520, 200, "f16", "f16", act="relu", beta=1.0, in_place=True, ldc=528)


def test_in_place_residual_split_and_small_m():
    run_fused(300, 520, 200, "f16", "f16", act="silu", beta=1.0, in_place=True,
              path=tg.TG_PATH_TC_PAIR, splits=2, multicast=1)
    run_fused(64, 640, 512, "f16", "f16", act="silu", beta=1.0, in_place=True)


def test_scalar_loads():
    # scale / bias starting 4 bytes off a 16-byte boundary and an odd residual pitch
    run_fused(300, 520, 200, "f16", "f16", act="gelu_tanh", sb_pad=1, ldr=523, beta=0.5)


def test_alpha_only_and_bias_only():
    run_fused(300, 520, 200, "f16", "f32", alpha=-2.0, use_scale=False, use_bias=False,
              residual=False)
    run_fused(300, 520, 200, "f16", "f32", use_scale=False, residual=False, act="relu")


def test_k_zero_is_epilogue_of_zero():
    run_fused(50, 70, 0, "f16", "f32", act="silu", beta=3.0)


def test_bench_shape_sampled():
    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(4096, 40, replace=False),
                                     [0, 4095]]))
    run_fused(4096, 4096, 4096, "f16", "f16", act="silu", beta=1.0, rows=rows)


def test_torch_helper():
    import torch
    M, N, K = 130, 260, 96
    a_bits = inputs.matrix_bits(M, K, "bf16", "uniform", 1)
    b_bits = inputs.matrix_bits(K, N, "bf16", "uniform", 2)
    a, b = to_device(a_bits, "bf16"), to_device(b_bits, "bf16")
    bias = torch.from_numpy(f32_vector(N, 9, -1, 1)).cuda()
    out = tg.gemm_fused(a, b, out_dtype=torch.float32, bias=bias, activation="relu")
    torch.cuda.synchronize()
    C_ref, S = oracle.gemm_ref_bits(a_bits, b_bits, K=K, N=N, fmt="bf16")
    ok, rep = oracle.epilogue.check_epilogue(out.cpu().numpy().astype(np.float64), C_ref, S,
                                             "bf16", "f32", bias=bias.cpu().numpy(), act="relu")
    assert ok, rep


def test_epilogue_with_unaligned_c_pitch():
    # C's pitch is not a 16-byte multiple: the warps store C themselves
    run_fused(300, 1100, 512, "f16", "f16", act="gelu_tanh", alpha=0.5, beta=1.0,
              path=tg.TG_PATH_TC_PAIR, block_n=512, ldc=1103, ldr=1104)
    run_fused(257, 520, 512, "bf16", "f32", act="silu", beta=0.5,
              path=tg.TG_PATH_TC, block_n=128, ldc=521)
