"""GPU parity of the FP8 path (E4M3 / E5M2 operands through kind::f8f6f4,
FP32 accumulate, FP16 / BF16 / FP32 output) against the oracle: bit-exact on
small-integer operands, within the tolerance on uniform ones, on every
tensor-core variant and the small-M streaming kernel, with ragged sizes,
padded and packed operands, the 4096^3 problem (sampled rows), strided
batches and the fused epilogue."""
from __future__ import annotations

import numpy as np
import pytest

import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare, padding_untouched, run_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

VARIANTS = {
    "auto": {},
    "single_cta": dict(path=tg.TG_PATH_TC, block_n=128),
    "single_cta_256": dict(path=tg.TG_PATH_TC, block_n=256),
    "pair_192": dict(path=tg.TG_PATH_TC_PAIR, block_n=192, multicast=1),
    "pair_256": dict(path=tg.TG_PATH_TC_PAIR, block_n=256, multicast=1),
    "pair_multicast": dict(path=tg.TG_PATH_TC_PAIR, block_n=256, multicast=2),
    "pair_multicast_224": dict(path=tg.TG_PATH_TC_PAIR, block_n=224, multicast=2),
    "split_k": dict(path=tg.TG_PATH_TC_PAIR, splits=3, multicast=1),
    "pair_512": dict(path=tg.TG_PATH_TC_PAIR, block_n=512),
}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_integer_operands_bit_exact(fmt, variant):
    M, N, K = 520, 600, 700          # ragged in every dimension, several K tiles
    a, b, c = run_gemm(M, N, K, fmt, "f16", dist="int", **VARIANTS[variant])
    compare(a, b, c, M, N, K, fmt, "f16", exact=True)


@pytest.mark.parametrize("fmt,dout", [("e4m3", "f16"), ("e4m3", "bf16"), ("e4m3", "f32"),
                                      ("e5m2", "f16"), ("e5m2", "f32")])
def test_uniform_within_tolerance(fmt, dout):
    M, N, K = 300, 520, 1000
    a, b, c = run_gemm(M, N, K, fmt, dout, ldc=N + 8)
    compare(a, b, c, M, N, K, fmt, dout)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("lda,ldb", [(720, 608), (701, 603)])
def test_padded_and_packed_operands(lda, ldb):
    # pitches that are multiples of 16 bytes are read in place; others packed
    M, N, K = 257, 600, 700
    p = tg.plan(M, N, K, "e4m3", "f32", num_sms=152, lda=lda, ldb=ldb)
    assert bool(p["pack_a"]) == (lda % 16 != 0) and bool(p["pack_b"]) == (ldb % 16 != 0)
    a, b, c = run_gemm(M, N, K, "e4m3", "f32", dist="int", lda=lda, ldb=ldb)
    compare(a, b, c, M, N, K, "e4m3", "f32", exact=True)


def test_wide_tiles_small_grid():
    M, N, K = 1000, 1000, 2200
    opts = dict(path=tg.TG_PATH_TC_PAIR, block_n=512, max_ctas=4)
    a, b, c = run_gemm(M, N, K, "e4m3", "f16", dist="int", **opts)
    compare(a, b, c, M, N, K, "e4m3", "f16", exact=True)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_small_m_kernel_exact(fmt, M):
    # the transposed streaming kernel with FP8 operands (kind::f8f6f4 with an
    # N-major B^T as the MMA's A operand), K split over a 4-CTA cluster
    p = tg.plan(M, 8192, 8192, fmt, "f16", num_sms=152, path=tg.TG_PATH_SKINNY)
    assert p["path"] == tg.TG_PATH_SKINNY and p["block_k"] == 128
    a, b, c = run_gemm(M, 8192, 8192, fmt, "f16", dist="int", path=tg.TG_PATH_SKINNY)
    compare(a, b, c, M, 8192, 8192, fmt, "f16", exact=True)
    if M > 32:   # what the planner picks for these rows: single-CTA tiles, K split
        a, b, c = run_gemm(M, 8192, 8192, fmt, "f16", dist="int")
        compare(a, b, c, M, 8192, 8192, fmt, "f16", exact=True)


@pytest.mark.parametrize("M,N,K,opts", [
    (37, 1000, 700, {}),
    (64, 512, 2048, dict(path=tg.TG_PATH_SKINNY, splits=8)),
    (100, 1536, 640, dict(path=tg.TG_PATH_SKINNY, block_n=256, splits=2)),
    (16, 2048, 1024, dict(path=tg.TG_PATH_SKINNY, block_n=512, splits=1)),
])
def test_small_m_kernel_uniform(M, N, K, opts):
    a, b, c = run_gemm(M, N, K, "e4m3", "bf16", ldc=N + 8, **opts)
    compare(a, b, c, M, N, K, "e4m3", "bf16")
    assert padding_untouched(c, N, "bf16")


def test_k_zero_and_tiny():
    a, b, c = run_gemm(33, 47, 0, "e4m3", "f32")
    assert np.all(c[:, :47] == 0)
    a, b, c = run_gemm(3, 5, 7, "e5m2", "f32", dist="int")
    compare(a, b, c, 3, 5, 7, "e5m2", "f32", exact=True)


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_square_4096(dist):
    n = 4096
    a, b, c = run_gemm(n, n, n, "e4m3", "f16", dist=dist)
    rows = np.unique(np.concatenate([np.random.default_rng(8).choice(n, 48, replace=False),
                                     [0, n - 1]]))
    compare(a, b, c, n, n, n, "e4m3", "f16", exact=(dist == "int"), rows=rows)


def test_batched_fp8():
    from tests.test_batched_gpu import check_all
    check_all(3, 300, 520, 256, "e4m3", "bf16")
    check_all(4, 256, 256, 512, "e5m2", "f16", exact=True, dist="int")
    check_all(40, 16, 1024, 512, "e4m3", "f32")          # small-M kernel, two CTAs per SM


def test_fused_epilogue_fp8():
    from tests.test_epilogue_gpu import run_fused
    run_fused(300, 520, 640, "e4m3", "bf16", act="silu", alpha=0.5, beta=1.0)
