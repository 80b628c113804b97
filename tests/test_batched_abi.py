"""Host-only rules of the strided-batched entry points (validation and
planning through tg_plan_gemm_strided_batched); no compute call, no GPU."""
from __future__ import annotations

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

A, B, C = 0x10000, 0x10000000000, 0x20000000000   # aligned, disjoint placeholders


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    return tg.load()


def bplan(batch, M, N, K, din="f16", dout=None, lda=None, ldb=None, ldc=None, sa=None, sb=None,
          sc=None, a=A, b=B, c=C, sms=152, **opts):
    dout = din if dout is None else dout
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sa = M * lda if sa is None else sa
    sb = K * ldb if sb is None else sb
    sc = M * ldc if sc is None else sc
    o = tg.make_options(**opts) if opts else None
    return tg.tg_plan_gemm_strided_batched(batch, M, N, K, a, lda, sa, b, ldb, sb, c, ldc, sc,
                                           din, dout, sms, o)


def single(M, N, K, din="f16", **opts):
    o = tg.make_options(**opts) if opts else None
    return tg.tg_plan_gemm(M, N, K, A, K, B, N, C, N, din, din, 152, o)


@pytest.mark.parametrize("kw,status", [
    (dict(batch=-1), tg.TG_ERR_INVALID_VALUE),
    (dict(sa=-1), tg.TG_ERR_INVALID_VALUE),
    (dict(sb=-8), tg.TG_ERR_INVALID_VALUE),
    (dict(sc=-64), tg.TG_ERR_INVALID_VALUE),
    (dict(sc=0), tg.TG_ERR_INVALID_VALUE),            # every product writes the same C
    (dict(sc=64 * 128 - 1), tg.TG_ERR_INVALID_VALUE),  # last row of C_z meets C_{z+1}
    (dict(batch=2 ** 31), tg.TG_ERR_UNSUPPORTED),
    (dict(splits=2), tg.TG_ERR_UNSUPPORTED),           # K split across kernels
    (dict(splits=2, path=tg.TG_PATH_TC_PAIR), tg.TG_ERR_UNSUPPORTED),
    (dict(din="f16", dout="bf16"), tg.TG_ERR_UNSUPPORTED),
    (dict(lda=10), tg.TG_ERR_INVALID_VALUE),           # lda < K, as for one product
])
def test_rejected(kw, status):
    args = dict(batch=4, M=64, N=128, K=96)
    args.update(kw)
    st, _ = bplan(**args)
    assert st == status


def test_rejected_leaves_plan_alone_and_null_plan():
    o = None
    st = tg.load().tg_plan_gemm_strided_batched(2, 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 16, 0, 0,
                                                 152, o, None)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_c_overlapping_a_across_the_batch():
    # A spans 8 products of 64 x 96; C of the last products would land inside it
    M, N, K = 64, 128, 96
    st, _ = bplan(8, M, N, K, a=A, c=A + 2 * (M * K) * 2 * 3)
    assert st == tg.TG_ERR_INVALID_VALUE
    # the same C right after the whole of A is fine
    st, _ = bplan(8, M, N, K, a=A, c=A + 8 * M * K * 2)
    assert st == tg.TG_OK


def test_interleaved_c_rows_are_disjoint():
    # C stored [M][batch][N]: ldc = batch * N, stride_c = N
    st, p = bplan(4, 64, 128, 96, ldc=4 * 128, sc=128)
    assert st == tg.TG_OK and p["per_batch"] == 0
    # stride_c below N overlaps neighbouring products
    st, _ = bplan(4, 64, 128, 96, ldc=4 * 128, sc=127)
    assert st == tg.TG_ERR_INVALID_VALUE
    # interleaved products must fit in one row pitch
    st, _ = bplan(4, 64, 128, 96, ldc=3 * 128, sc=128)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_one_launch_counts_tiles_of_every_product():
    st1, p1 = single(1024, 1024, 1024, path=tg.TG_PATH_TC_PAIR, multicast=1, block_n=256)
    st, p = bplan(16, 1024, 1024, 1024, path=tg.TG_PATH_TC_PAIR, multicast=1, block_n=256)
    assert st == st1 == tg.TG_OK
    assert p["per_batch"] == 0 and p["kernels"] == 1 and p["workspace_bytes"] == 0
    assert p["tiles"] == 16 * p1["tiles"]
    assert p["splits"] == 1
    assert p["ctas"] == 152                           # every pair resident


def test_batch_of_one_plans_as_one_product():
    st, p = bplan(1, 300, 520, 200)
    st1, p1 = tg.tg_plan_gemm(300, 520, 200, A, 200, B, 520, C, 520, "f16", "f16", 152, None)
    assert st == st1 == tg.TG_OK
    assert p == p1


def test_no_k_split_across_kernels_with_a_batch():
    # one 256x256 tile per product would be split over K alone; a batch fills the GPU
    st1, p1 = single(256, 256, 16384)
    assert p1["splits"] > 1
    st, p = bplan(64, 256, 256, 16384)
    assert st == tg.TG_OK and p["splits"] == 1 and p["workspace_bytes"] == 0


def test_shared_operands():
    st, p = bplan(8, 512, 512, 512, sa=0)
    assert st == tg.TG_OK and p["per_batch"] == 0
    st, p = bplan(8, 512, 512, 512, sb=0)
    assert st == tg.TG_OK and p["per_batch"] == 0


@pytest.mark.parametrize("kw", [dict(din="f32"), dict(sa=512 * 512 + 1), dict(sb=3),
                                dict(a=A + 2)])
def test_one_call_per_product(kw):
    # TF32 operands, or a batch stride / base that is not 16-byte aligned
    args = dict(batch=5, M=512, N=512, K=512)
    args.update(kw)
    st, p = bplan(**args)
    st1, p1 = tg.tg_plan_gemm(512, 512, 512, args.get("a", A), 512, B, 512, C, 512,
                              args.get("din", "f16"), args.get("din", "f16"), 152, None)
    assert st == st1 == tg.TG_OK
    assert p["per_batch"] == 1
    assert p["kernels"] == 5 * p1["kernels"]
    assert p["tiles"] == 5 * p1["tiles"]


def test_small_m_batch_uses_the_skinny_kernel():
    st, p = bplan(32, 64, 8192, 8192)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY
    # 64 columns tiles x 32 products: more CTAs than SMs, no K split
    assert p["splits"] == 1 and p["ctas"] == 64 * 32 and p["tiles"] == 64 * 32
    # a short batch still splits K on chip to fill the GPU
    st, p = bplan(2, 16, 2048, 8192)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY and p["splits"] > 1
    assert p["tiles"] * p["splits"] <= 2 * 152
    # forced on-chip split with a batch
    st, p = bplan(3, 64, 512, 2048, path=tg.TG_PATH_SKINNY, splits=4)
    assert st == tg.TG_OK and p["splits"] == 4 and p["ctas"] == 3 * 4 * 4


def test_skinny_grid_rows_limit():
    st, p = bplan(70000, 16, 128, 64)
    assert st == tg.TG_OK and p["path"] != tg.TG_PATH_SKINNY
    st, p = bplan(65535, 16, 128, 64)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY


def test_empty_batches_plan_no_kernels():
    for args in [(0, 64, 64, 64), (4, 0, 64, 64), (4, 64, 0, 64), (4, 64, 64, 0)]:
        st, p = bplan(*args, sc=max(args[1] * 64, 64))
        assert st == tg.TG_OK and p["kernels"] == 0 and p["workspace_bytes"] == 0


def test_too_many_tiles():
    st, _ = bplan(2 ** 24, 1024, 2048, 64, sa=0, sb=0)   # 2^31 tiles of 128 x 128
    assert st == tg.TG_ERR_UNSUPPORTED
