"""Argument rules of tg_gemm_fused that are decided on the host before any
device call (so these run without a GPU): each rejected call returns its
status and enqueues nothing."""
from __future__ import annotations

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

A, B, C = 0x10000, 0x100000000, 0x200000000
M, N, K = 64, 128, 96


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    return tg.load()


def call(ep, c=C, ldc=N, dout="f16", m=M, n=N):
    return tg.tg_gemm_fused(m, n, K, A, K, B, n, c, ldc, "f16", dout, ep, 0)


@pytest.mark.parametrize("kw", [
    dict(activation=4), dict(activation=-1),
    dict(residual=0x300000000, ldr=N - 1),                 # ldr < N
    dict(residual=0x300000001, ldr=N),                     # misaligned for f16
    dict(residual=C + 2 * 10, ldr=N),                      # overlaps C, not in place
    dict(residual=C, ldr=N + 8),                           # same base, other pitch
    dict(scale=0x300000002),                               # not 4-byte aligned
    dict(bias=0x300000001),
    dict(bias=C + 64),                                     # bias inside C
    dict(scale=C + M * N * 2 - 8),                         # scale runs into the end of C
])
def test_rejected(kw):
    assert call(tg.make_epilogue(**kw)) == tg.TG_ERR_INVALID_VALUE


def test_reserved_must_be_zero():
    e = tg.make_epilogue()
    e.reserved = 1
    assert call(e) == tg.TG_ERR_INVALID_VALUE


def test_product_rules_still_apply():
    assert tg.tg_gemm_fused(-1, N, K, A, K, B, N, C, N, "f16", "f16", tg.make_epilogue(), 0) \
        == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm_fused(M, N, K, A, K, B, N, C, N, "f16", "bf16", tg.make_epilogue(), 0) \
        == tg.TG_ERR_UNSUPPORTED


def test_empty_output_is_ok_without_device():
    # M == 0: nothing to do, decided on the host
    assert tg.tg_gemm_fused(0, N, K, A, K, B, N, C, N, "f16", "f16",
                            tg.make_epilogue(activation="silu"), 0) == tg.TG_OK


def test_struct_layout_matches_header():
    import ctypes
    assert ctypes.sizeof(tg.tg_epilogue) == 48
    assert tg.tg_epilogue.ldr.offset == 32 and tg.tg_epilogue.activation.offset == 40


# ---- tg_gemm_strided_batched_fused: the same rules over a batch of products ----

BATCH = 3
SC = M * N            # stacked C blocks


def bcall(ep, sr=0, c=C, sc=SC, batch=BATCH):
    return tg.tg_gemm_strided_batched_fused(batch, M, N, K, A, K, M * K, B, N, K * N, c, N, sc,
                                            "f16", "f16", ep, sr, 0)


@pytest.mark.parametrize("kw,sr", [
    (dict(residual=C + (BATCH - 1) * SC * 2, ldr=N), SC),   # inside the last product's C
    (dict(residual=C - SC * 2, ldr=N), SC // 2),             # runs into the first C block
    (dict(residual=C, ldr=N), SC // 2),                       # same base, other batch stride
    (dict(residual=C, ldr=N), 0),                             # one shared residual that is C
    (dict(residual=0x300000000, ldr=N), -1),                  # negative stride
    (dict(), SC),                                             # stride without a residual
    (dict(bias=C + (BATCH - 1) * SC * 2 + 64), 0),            # bias inside the last C block
])
def test_batched_rejected(kw, sr):
    assert bcall(tg.make_epilogue(**kw), sr) == tg.TG_ERR_INVALID_VALUE


def test_batched_stride_without_epilogue():
    assert bcall(None, sr=SC) == tg.TG_ERR_INVALID_VALUE


def test_batched_accepted_without_device():
    # batch == 0 and M == 0 are decided on the host; in place and a shared
    # residual block pass validation
    ep = tg.make_epilogue(residual=C, ldr=N, beta=1.0)
    assert bcall(ep, sr=SC, batch=0) == tg.TG_OK
    assert tg.tg_gemm_strided_batched_fused(BATCH, 0, N, K, A, K, M * K, B, N, K * N, C, N, SC,
                                            "f16", "f16", ep, SC, 0) == tg.TG_OK
    shared = tg.make_epilogue(residual=0x300000000, ldr=N, beta=0.5)
    assert tg.tg_gemm_strided_batched_fused(BATCH, 0, N, K, A, K, M * K, B, N, K * N, C, N, SC,
                                            "f16", "f16", shared, 0, 0) == tg.TG_OK


def test_batched_product_rules_still_apply():
    ep = tg.make_epilogue()
    # C blocks of the products overlap
    assert bcall(ep, sc=N) == tg.TG_ERR_INVALID_VALUE
    # K split across kernels is not available with a batch
    opt = tg.make_options(splits=2, path=tg.TG_PATH_TC)
    assert tg.tg_gemm_strided_batched_fused(BATCH, M, N, K, A, K, M * K, B, N, K * N, C, N, SC,
                                            "f16", "f16", ep, 0, 0, opt) == tg.TG_ERR_UNSUPPORTED
