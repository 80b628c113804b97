"""Pins for the tiled model and the closed forms the measurement uses.  CPU only."""
from __future__ import annotations

import itertools

import numpy as np
import pytest

from oracle import tiled_model as tm
from tests.conftest import parse_numbers, read_golden


def test_tile_ranges_printed():
    g = read_golden("tile_ranges.txt")
    want = [tuple(int(v) for v in r.split()) for r in g["ranges"].split(";")]
    assert tm.tile_ranges(int(g["n"]), int(g["t"])) == want


def test_tile_ranges_cover_exactly():
    for n, t in itertools.product(range(0, 40), range(1, 9)):
        r = tm.tile_ranges(n, t)
        covered = [i for a, b in r for i in range(a, b)]
        assert covered == list(range(n))
        assert all(0 < b - a <= t for a, b in r)


def test_exit_check():
    g = read_golden("exit_check.txt")
    M, N, K, BM, BN, BK = (int(g[k]) for k in ("M", "N", "K", "BM", "BN", "BK"))
    programs, k_steps, masked = tm.exit_check(M, N, K, BM, BN, BK)
    assert programs == int(g["programs"]) and k_steps == int(g["k_steps"])
    assert masked == tuple(g["masked"].split())
    # the executed model agrees with the closed form
    A = np.arange(M * K, dtype=np.float64).reshape(M, K)
    B = np.arange(K * N, dtype=np.float64).reshape(K, N)
    run = tm.tiled_gemm(A, B, BM, BN, BK)
    assert (run.programs, run.k_steps, run.masked_dims) == (programs, k_steps, masked)
    assert np.array_equal(run.C, A @ B)


def test_tiled_traffic_law_64():
    g = read_golden("tiled_traffic.txt")
    A = np.random.default_rng(0).standard_normal((64, 64))
    B = np.random.default_rng(1).standard_normal((64, 64))
    naive = tm.naive_loads(64, 64, 64)
    for T in (int(t) for t in parse_numbers(g["square_64_tiles"])):
        run = tm.tiled_gemm(A, B, T)
        assert run.loads * T == naive, T                 # exactly 1/T of naive
        assert run.loads == tm.tiled_loads(64, 64, 64, T)
        np.testing.assert_allclose(run.C, A @ B, rtol=1e-12, atol=1e-12)


def test_tiled_traffic_sweep_256():
    g = read_golden("tiled_traffic.txt")
    A = np.random.default_rng(2).standard_normal((256, 256))
    B = np.random.default_rng(3).standard_normal((256, 256))
    for T in (int(t) for t in parse_numbers(g["square_256_tiles"])):
        run = tm.tiled_gemm(A, B, T)
        assert run.loads == 2 * 256 ** 3 // T


@pytest.mark.parametrize("M,N,K,T", [(64, 64, 64, 5), (64, 64, 64, 24), (50, 70, 30, 16),
                                     (7, 5, 3, 4), (33, 1, 17, 8)])
def test_tiled_traffic_general_form(M, N, K, T):
    """Edge tiles are clipped, so for T not dividing M, N the count is
    K*(M*ceil(N/T) + N*ceil(M/T)) rather than 2MNK/T."""
    A = np.ones((M, K))
    B = np.ones((K, N))
    run = tm.tiled_gemm(A, B, T)
    assert run.loads == tm.tiled_loads(M, N, K, T)
    assert np.array_equal(run.C, np.full((M, N), float(K)))


def test_closed_forms_printed():
    g = read_golden("closed_forms.txt")
    ai = tm.matmul_intensity(4096, 4096, 4096, 2)
    assert round(ai) == int(g["intensity_4096_f16"]) and ai > float(g["intensity_threshold"])
    assert abs(ai - 4096 / 3) < 1e-9
    elems, nbytes, flops, ratio = tm.tile_reuse(32, 64, 32, 2)
    assert (elems, nbytes, flops) == (int(g["tile_reuse_elems"]), int(g["tile_reuse_bytes"]),
                                      int(g["tile_reuse_flops"]))
    assert round(ratio, 2) == float(g["tile_reuse_ratio"])
    n = 4096
    assert round(tm.naive_loads(n, n, n) / 1e9) == int(g["naive_loads_4096_billion"])
    assert round(n * n / 1e6, 1) == float(g["naive_outputs_4096_million"])
    assert round(3 * n * n / 1e6) == int(g["naive_distinct_4096_million"])
    # every A element is used by N outputs and every B element by M: 2MNK / (MK + KN) = n
    assert tm.naive_loads(n, n, n) // (2 * n * n) == int(g["naive_refetch_4096"])
    assert tm.phase_intensity(16, 4) == float(g["phase_intensity_T16"])
    assert tm.phase_intensity(1, 4) == float(g["phase_intensity_naive"])


@pytest.mark.parametrize("variant", ["in_group", "global"])
def test_grouped_raster_is_bijection(variant):
    rng = np.random.default_rng(7)
    for _ in range(200):
        tiles_m, tiles_n, G = (int(x) for x in rng.integers(1, 23, size=3))
        seen = {tm.grouped_tile(p, tiles_m, tiles_n, G, variant) for p in range(tiles_m * tiles_n)}
        assert seen == {(i, j) for i in range(tiles_m) for j in range(tiles_n)}


def test_grouped_raster_walks_rows_first():
    # GROUP_M=8 walks eight tile rows down before moving right (lesson 6)
    order = [tm.grouped_tile(p, 16, 4, 8) for p in range(10)]
    assert order[:8] == [(i, 0) for i in range(8)]
    assert order[8:10] == [(0, 1), (1, 1)]
    # GROUP_M=1 is plain row-major order (p // tiles_n, p % tiles_n)
    assert [tm.grouped_tile(p, 3, 5, 1) for p in range(15)] == [(p // 5, p % 5) for p in range(15)]
