"""Host-only rules of the 3xTF32 mode (tg_options.f32_mode): validation and
the plan (split operands in workspace, kernel over K' = 3K).  No GPU."""
from __future__ import annotations

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

A, B, C = 0x10000, 0x100000000, 0x200000000


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    return tg.load()


def plan(M, N, K, din="f32", dout="f32", **opts):
    o = tg.make_options(**opts)
    return tg.tg_plan_gemm(M, N, K, A, K, B, N, C, N, din, dout, 152, o)


def test_split_operands_and_three_k():
    st, p = plan(2048, 2048, 2048, f32_mode=tg.TG_F32_3XTF32)
    st1, p1 = plan(2048, 2048, 2048)
    assert st == st1 == tg.TG_OK
    assert p["pack_a"] == 3 and p["pack_b"] == 3 and p["kernels"] == 3
    assert p1["pack_a"] == 0 and p1["pack_b"] == 0
    # A' [M, 3K] and B' [3K, N] in FP32
    assert p["workspace_bytes"] >= (2048 + 2048) * 3 * 2048 * 4


def test_ragged_k_pitch():
    st, p = plan(1000, 1999, 777, f32_mode=tg.TG_F32_3XTF32)
    assert st == tg.TG_OK and p["workspace_bytes"] >= (1000 + 1999) * 2332 * 4


@pytest.mark.parametrize("din,dout", [("f16", "f16"), ("bf16", "f32"), ("e4m3", "f16")])
def test_other_operand_types_unsupported(din, dout):
    st, _ = plan(64, 64, 64, din, dout, f32_mode=tg.TG_F32_3XTF32)
    assert st == tg.TG_ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", [-1, 2])
def test_bad_mode(mode):
    st, _ = plan(64, 64, 64, f32_mode=mode)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_reserved_field():
    o = tg.make_options()
    o.reserved = 7
    st, _ = tg.tg_plan_gemm(64, 64, 64, A, 64, B, 64, C, 64, "f32", "f32", 152, o)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_k_limit():
    st, _ = plan(16, 16, 2 ** 30, f32_mode=tg.TG_F32_3XTF32)
    assert st == tg.TG_ERR_UNSUPPORTED
