"""GPU parity of the strided-batched GEMM: every product of the batch is
compared element by element with the oracle (each product has its own seeded
operands, so a product reading another one's data fails), and every element
of the C buffer that no product owns must keep its poison value.

Covers the one-launch kernels (single CTA, CTA pair, pairs sharing A by
multicast, the small-M kernel with and without its on-chip K split and with
two CTAs per SM), shared operands (batch stride 0), C interleaved along rows,
the one-call-per-product route (TF32, misaligned batch strides), K = 0 and the
torch-level ``bmm`` helper.
"""
from __future__ import annotations

import numpy as np
import pytest

import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare, to_bits, to_device, torch_dtype
from tiled_matrix_multiplication_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


def flat_operand(batch, rows, cols, ld, stride, din, dist, seed):
    """Flat element buffer holding `batch` matrices `stride` apart (one if
    stride == 0) and the bits of each product's matrix."""
    mats = [inputs.matrix_bits(rows, cols, din, dist, seed + (z if stride else 0), ld=ld)
            for z in range(batch if stride else 1)]
    length = (len(mats) - 1) * stride + rows * ld
    buf = np.zeros(max(length, 1), dtype=inputs.BITS_NP[din])
    for z, m in enumerate(mats):
        buf[z * stride: z * stride + rows * ld] = m.reshape(-1)
    return buf, [mats[z if stride else 0] for z in range(batch)]


def run_batched(batch, M, N, K, din, dout, dist="uniform", lda=None, ldb=None, ldc=None, sa=None,
                sb=None, sc=None, **opts):
    import torch
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sa = M * lda if sa is None else sa
    sb = K * ldb if sb is None else sb
    sc = M * ldc if sc is None else sc
    a_flat, a_mats = flat_operand(batch, M, K, lda, sa, din, dist, inputs.SEED_A)
    b_flat, b_mats = flat_operand(batch, K, N, ldb, sb, din, dist, inputs.SEED_B + 1000)
    c_len = max(sc * (batch - 1) + M * ldc, 1)
    poison = inputs.nan_bits(dout)
    a_dev = to_device(a_flat, din)
    b_dev = to_device(b_flat, din)
    c_dev = to_device(np.full(c_len, poison, dtype=inputs.BITS_NP[dout]), dout)
    opt = tg.make_options(**opts) if opts else None
    st = tg.tg_gemm_strided_batched(batch, M, N, K, a_dev.data_ptr(), lda, sa, b_dev.data_ptr(),
                                    ldb, sb, c_dev.data_ptr(), ldc, sc, din, dout,
                                    torch.cuda.current_stream().cuda_stream, opt)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    torch.cuda.synchronize()
    tg.check_device_error()
    c_flat = to_bits(c_dev, dout)
    owned = np.zeros(c_len, dtype=bool)
    outs = []
    for z in range(batch):
        idx = z * sc + np.arange(M)[:, None] * ldc + np.arange(N)[None, :]
        owned[idx] = True
        outs.append(c_flat[idx])
    assert np.all(c_flat[~owned] == poison), "an element outside every product's C was written"
    return a_mats, b_mats, outs


def check_all(batch, M, N, K, din, dout, exact=False, **kw):
    a_mats, b_mats, outs = run_batched(batch, M, N, K, din, dout, **kw)
    for z in range(batch):
        compare(a_mats[z], b_mats[z], outs[z], M, N, K, din, dout, exact=exact)


def test_auto_ragged_f16():
    check_all(3, 300, 520, 200, "f16", "f16")


def test_single_cta_bf16_to_f32():
    check_all(2, 200, 300, 130, "bf16", "f32", path=tg.TG_PATH_TC)


@pytest.mark.parametrize("block_n", [128, 256])
def test_pair_no_multicast(block_n):
    check_all(3, 520, 600, 256, "f16", "f16", path=tg.TG_PATH_TC_PAIR, multicast=1,
              block_n=block_n)


def test_pair_multicast_odd_tile_columns():
    # 1100 columns = 5 tiles of 256: the last multicast unit has one empty half
    check_all(3, 520, 1100, 256, "f16", "f16", path=tg.TG_PATH_TC_PAIR, multicast=2,
              block_n=256)


def test_small_m_auto():
    check_all(5, 37, 1000, 700, "f16", "f16")


def test_small_m_on_chip_split():
    check_all(3, 64, 512, 2048, "bf16", "bf16", path=tg.TG_PATH_SKINNY, splits=4)


def test_small_m_two_per_sm():
    p = tg.plan_batched(40, 16, 1024, 512, num_sms=152)
    assert p["path"] == tg.TG_PATH_SKINNY and p["ctas"] > 152
    check_all(40, 16, 1024, 512, "f16", "f32")


@pytest.mark.parametrize("which", ["a", "b"])
@pytest.mark.parametrize("M", [48, 400])
def test_shared_operand(which, M):
    kw = {"sa": 0} if which == "a" else {"sb": 0}
    check_all(4, M, 384, 320, "f16", "f16", **kw)


@pytest.mark.parametrize("M", [40, 300])
def test_interleaved_c(M):
    # C stored [M][batch][N] (ldc = batch * N, stride_c = N)
    check_all(3, M, 136, 200, "f16", "f16", ldc=3 * 136, sc=136)


def test_padded_leading_dims_and_strides():
    check_all(3, 130, 200, 96, "f16", "f16", lda=104, ldb=264, ldc=208, sa=130 * 104 + 64,
              sb=96 * 264 + 8, sc=130 * 208 + 24)


def test_tf32_one_call_per_product():
    p = tg.plan_batched(3, 130, 70, 50, "f32", num_sms=152)
    assert p["per_batch"] == 1
    check_all(3, 130, 70, 50, "f32", "f32")


def test_misaligned_batch_stride():
    # A batch stride of an odd number of elements: each product on its own
    check_all(3, 100, 128, 64, "f16", "f16", sa=100 * 64 + 1)


def test_integer_exact():
    check_all(4, 256, 256, 512, "f16", "f16", exact=True, dist="int")


def test_k_zero_zeroes_every_product():
    a_mats, b_mats, outs = run_batched(3, 20, 30, 0, "f16", "f32")
    for o in outs:
        assert np.all(o == 0)


def test_bmm_helper():
    import torch
    batch, M, N, K = 4, 96, 160, 72
    a_bits = [inputs.matrix_bits(M, K, "bf16", "uniform", inputs.SEED_A + z) for z in range(batch)]
    b_bits = inputs.matrix_bits(K, N, "bf16", "uniform", inputs.SEED_B)
    a = torch.stack([to_device(x, "bf16") for x in a_bits])
    b = to_device(b_bits, "bf16")
    c = tg.bmm(a, b, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert c.shape == (batch, M, N) and c.dtype == torch.float32
    for z in range(batch):
        compare(a_bits[z], b_bits, to_bits(c[z], "f32"), M, N, K, "bf16", "f32")


def test_larger_batch_sampled():
    # 8 products of 2048^3: the whole-GPU one-launch path, sampled rows per product
    batch, n = 8, 2048
    a_mats, b_mats, outs = run_batched(batch, n, n, n, "f16", "f16")
    rng = np.random.default_rng(7)
    for z in range(batch):
        rows = np.unique(np.concatenate([rng.choice(n, 12, replace=False), [0, n - 1]]))
        compare(a_mats[z], b_mats[z], outs[z], n, n, n, "f16", "f16", rows=rows)


def _sampled_batch_check(batch, M, N, K, din, dout, dist, rows_per, seed):
    """The bench's contiguous [batch, rows, cols] layout at full size: every
    product's C is checked on a seeded sample of rows (all columns)."""
    a_mats, b_mats, outs = run_batched(batch, M, N, K, din, dout, dist=dist)
    rng = np.random.default_rng(seed)
    for z in range(batch):
        rows = np.unique(np.concatenate([rng.choice(M, min(rows_per, M), replace=False),
                                         [0, M - 1]]))
        compare(a_mats[z], b_mats[z], outs[z], M, N, K, din, dout, rows=rows)


def test_bench_batch_16x2048_f16():
    _sampled_batch_check(16, 2048, 2048, 2048, "f16", "f16", "uniform", 6, 11)


def test_bench_batch_64x1024_bf16():
    _sampled_batch_check(64, 1024, 1024, 1024, "bf16", "bf16", "normal", 4, 12)


def test_bench_batch_32_small_m():
    # 32 products of 64 x 8192 x 8192 (the small-M kernel, two CTAs per SM):
    # every row of every product
    _sampled_batch_check(32, 64, 8192, 8192, "f16", "f16", "uniform", 64, 13)


def test_wide_tiles_batched():
    # 512-wide pair tiles over a batch: rank-3 tensor maps for A, B and C
    check_all(3, 520, 1100, 256, "f16", "f16", path=tg.TG_PATH_TC_PAIR, block_n=512)
    check_all(4, 300, 600, 300, "bf16", "f32", path=tg.TG_PATH_TC_PAIR, block_n=512, sb=0)
