"""Host-only rules of the FP8 operand types (no GPU): accepted type pairs,
the 128-element K block, packing of pitches that are not 16-byte multiples,
and the small-M streaming kernel's K blocks for FP8."""
from __future__ import annotations

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

A, B, C = 0x10000, 0x100000000, 0x200000000


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    return tg.load()


def plan(M, N, K, din, dout, lda=None, ldb=None, **opts):
    o = tg.make_options(**opts) if opts else None
    return tg.tg_plan_gemm(M, N, K, A, K if lda is None else lda, B, N if ldb is None else ldb,
                           C, N, din, dout, 152, o)


@pytest.mark.parametrize("din", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dout,ok", [("f16", True), ("bf16", True), ("f32", True),
                                     ("e4m3", False), ("e5m2", False)])
def test_type_pairs(din, dout, ok):
    st, p = plan(512, 512, 512, din, dout)
    assert st == (tg.TG_OK if ok else tg.TG_ERR_UNSUPPORTED)
    if ok:
        assert p["block_k"] == 128 and p["pack_b"] == 0


def test_mixed_fp8_and_16bit_is_not_a_type_pair():
    # one dtype_in for both operands: nothing to mix; 16-bit in with FP8 out is refused
    st, _ = plan(64, 64, 64, "f16", "e4m3")
    assert st == tg.TG_ERR_UNSUPPORTED


def test_pitch_packing_rule():
    st, p = plan(300, 300, 300, "e4m3", "f16", lda=304, ldb=320)
    assert st == tg.TG_OK and p["pack_a"] == 0 and p["pack_b"] == 0
    st, p = plan(300, 300, 300, "e4m3", "f16", lda=301, ldb=310)
    assert st == tg.TG_OK and p["pack_a"] == 1 and p["pack_b"] == 1


def test_small_m_uses_the_streaming_kernel():
    st, p = plan(16, 8192, 8192, "e4m3", "f16")
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY and p["block_k"] == 128
    st, p = plan(16, 8192, 8192, "e4m3", "f16", path=tg.TG_PATH_SKINNY, splits=8)
    assert st == tg.TG_OK and p["splits"] == 8
    # 8 K ranges of 128-element tiles need K > 7 * 128
    st, _ = plan(16, 8192, 896, "e4m3", "f16", path=tg.TG_PATH_SKINNY, splits=8)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_bench_shape_plan():
    st, p = plan(4096, 4096, 4096, "e4m3", "f16")
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC_PAIR and p["kernels"] == 1
