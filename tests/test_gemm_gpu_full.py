"""GPU parity at the full sizes of the named workloads, in the launch
configuration the library picks by itself (the one bench.py times).  The
oracle checks every element of small problems and a seeded sample of output
rows (and, for the largest, columns) of the big ones.

Workloads: the 127x255x65 FP16->FP32 problem; square 4096^3 FP16 (the bench
workload); the transformer-prefill set in BF16 with N(0, 0.02) inputs; FP32
operands at TF32 (2048^3 and the ragged 1000x1999x777); the square sweep
256 .. 16384; the skinny decode shapes M in {1, 16, 64, 128} x 8192 x 8192.
"""
from __future__ import annotations

import numpy as np
import pytest

from tests.conftest import cuda_ok
from tests.gemm_util import compare, run_gemm

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


def sample(n: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    idx = rng.choice(n, size=min(k, n), replace=False)
    # always include the first and last row/column (edge tiles)
    return np.unique(np.concatenate([idx, [0, n - 1]]))


def test_small_fp16_to_fp32_every_element():
    a, b, c = run_gemm(127, 255, 65, "f16", "f32")
    compare(a, b, c, 127, 255, 65, "f16", "f32")


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_square_4096_fp16(dist):
    M = N = K = 4096
    a, b, c = run_gemm(M, N, K, "f16", "f16", dist=dist)
    compare(a, b, c, M, N, K, "f16", "f16", exact=(dist == "int"), rows=sample(M, 96, 1))


@pytest.mark.parametrize("M,N,K", [(8192, 6144, 4096), (8192, 4096, 4096), (8192, 14336, 4096),
                                   (8192, 4096, 14336)])
def test_prefill_bf16(M, N, K):
    a, b, c = run_gemm(M, N, K, "bf16", "bf16", dist="normal")
    compare(a, b, c, M, N, K, "bf16", "bf16", rows=sample(M, 48, M + N))


def test_tf32_square_2048():
    a, b, c = run_gemm(2048, 2048, 2048, "f32", "f32")
    compare(a, b, c, 2048, 2048, 2048, "f32", "f32", rows=sample(2048, 128, 3))


def test_tf32_ragged_every_element():
    a, b, c = run_gemm(1000, 1999, 777, "f32", "f32")
    compare(a, b, c, 1000, 1999, 777, "f32", "f32")


@pytest.mark.parametrize("n", [256, 512, 1024, 2048])
def test_square_sweep_every_element(n):
    a, b, c = run_gemm(n, n, n, "f16", "f16")
    compare(a, b, c, n, n, n, "f16", "f16")


@pytest.mark.parametrize("n", [8192, 16384])
def test_square_sweep_large_sampled(n):
    a, b, c = run_gemm(n, n, n, "f16", "f16")
    compare(a, b, c, n, n, n, "f16", "f16", rows=sample(n, 24, n), cols=sample(n, 2048, n + 1))


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_skinny_every_element(M):
    a, b, c = run_gemm(M, 8192, 8192, "f16", "f16")
    compare(a, b, c, M, 8192, 8192, "f16", "f16")


@pytest.mark.parametrize("M", [1, 64])
def test_skinny_integer_exact(M):
    a, b, c = run_gemm(M, 8192, 8192, "f16", "f16", dist="int")
    compare(a, b, c, M, 8192, 8192, "f16", "f16", exact=True)
