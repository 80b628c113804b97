"""GPU parity on degenerate and extreme shapes: single rows, columns and
inner dimensions, the M = 128 / 129 boundary between the small-M kernel and
the tile kernel, a very long K, a very wide N, tall-and-thin products, and
every output type -- each element checked against the oracle."""
from __future__ import annotations

import pytest

from tests.conftest import cuda_ok
from tests.gemm_util import compare, padding_untouched, run_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 1), (1, 1, 4096), (1, 8, 1), (7, 1, 300), (5000, 1, 300), (3, 3, 3),
    (128, 64, 64), (129, 64, 64), (128, 1000, 513), (129, 1000, 513),
    (16, 16, 100_000),          # one output tile, 1563 K tiles
    (2, 70_000, 16),            # very wide, tiny K
    (40_000, 8, 64),            # tall and thin
    (257, 257, 257),
])
@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("bf16", "bf16")])
def test_shapes_exact(M, N, K, din, dout):
    a, b, c = run_gemm(M, N, K, din, dout, dist="int")
    compare(a, b, c, M, N, K, din, dout, exact=True)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 64, 64), (16, 16, 20_000), (3000, 9, 50)])
@pytest.mark.parametrize("din,dout", [("f32", "f32"), ("e4m3", "f16"), ("e5m2", "bf16")])
def test_shapes_other_types(M, N, K, din, dout):
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", ldc=N + 5)
    compare(a, b, c, M, N, K, din, dout, exact=True)
    assert padding_untouched(c, N, dout)


def test_long_k_uniform_tolerance():
    # the error bound grows with K: 2e-3 * sum|ab| still holds at K = 65536
    a, b, c = run_gemm(64, 256, 65536, "f16", "f32")
    compare(a, b, c, 64, 256, 65536, "f16", "f32")
