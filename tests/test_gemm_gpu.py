"""GPU parity of the tensor-core GEMM against the CPU oracle on small and
ragged problems: several tiles, partial tiles in M, N and K, strided and
misaligned operands, split K, the degenerate sizes."""
from __future__ import annotations

import numpy as np
import pytest

from tests.conftest import cuda_ok
from tests.gemm_util import compare, padding_untouched, run_gemm

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

PAIRS = [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")]
SHAPES = [(1, 1, 1), (5, 7, 5), (128, 256, 64), (127, 255, 65), (129, 257, 129),
          (256, 512, 1000), (300, 130, 70), (64, 1000, 48), (1000, 64, 300)]


@pytest.mark.parametrize("din,dout", PAIRS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_integer_inputs_bit_exact(M, N, K, din, dout):
    a, b, c = run_gemm(M, N, K, din, dout, dist="int")
    compare(a, b, c, M, N, K, din, dout, exact=True)


@pytest.mark.parametrize("din,dout", PAIRS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_uniform_inputs_within_tolerance(M, N, K, din, dout):
    a, b, c = run_gemm(M, N, K, din, dout, dist="uniform")
    compare(a, b, c, M, N, K, din, dout)


def test_config_small_fp16_to_fp32():
    """127 x 255 x 65, FP16 in, FP32 out, U[-1,1]: the oracle checks every element."""
    a, b, c = run_gemm(127, 255, 65, "f16", "f32")
    compare(a, b, c, 127, 255, 65, "f16", "f32")


@pytest.mark.parametrize("din,dout", PAIRS)
@pytest.mark.parametrize("lda_pad,ldb_pad,ldc_pad", [(8, 64, 8), (3, 5, 1), (0, 0, 24)])
def test_strided_operands(din, dout, lda_pad, ldb_pad, ldc_pad):
    """Leading dimensions above the logical width, aligned and not; the padding
    of A and B holds NaN (so reading it would poison C) and C's padding must
    come back untouched."""
    M, N, K = 200, 300, 150
    a, b, c = run_gemm(M, N, K, din, dout, dist="uniform", lda=K + lda_pad, ldb=N + ldb_pad,
                       ldc=N + ldc_pad)
    compare(a, b, c, M, N, K, din, dout)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("din,dout", [("f16", "f16"), ("bf16", "f32"), ("f32", "f32")])
def test_forced_split_k(splits, din, dout):
    M, N, K = 256, 384, 1000
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", splits=splits)
    compare(a, b, c, M, N, K, din, dout, exact=True)
    a, b, c = run_gemm(M, N, K, din, dout, dist="uniform", splits=splits, ldc=N + 8)
    compare(a, b, c, M, N, K, din, dout)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("group_m,max_ctas", [(1, 0), (8, 3), (3, 1)])
def test_tile_width_raster_and_grid(block_n, group_m, max_ctas):
    """Every tile is produced once whatever the tile width, raster height and
    persistent-grid size (a grid of 1 CTA walks all tiles itself)."""
    M, N, K = 700, 900, 256
    a, b, c = run_gemm(M, N, K, "f16", "f16", dist="int", block_n=block_n, group_m=group_m,
                       max_ctas=max_ctas)
    compare(a, b, c, M, N, K, "f16", "f16", exact=True)


def test_k_zero_gives_zeros():
    a, b, c = run_gemm(33, 17, 0, "f16", "f32", ldc=20)
    assert np.all(c[:, :17] == 0)
    assert padding_untouched(c, 17, "f32")


def test_empty_output_is_noop():
    run_gemm(0, 16, 16, "bf16", "bf16")
    run_gemm(16, 0, 16, "bf16", "bf16")


def test_identity_and_permutation_exact():
    """B = I gives C = A; a permutation matrix permutes A's columns."""
    import oracle
    from tiled_matrix_multiplication_gb300 import inputs
    M, K = 300, 256
    a = inputs.matrix_bits(M, K, "bf16", "uniform", 5)
    eye = oracle.encode(np.eye(K), "bf16")
    _, _, c = run_gemm(M, K, K, "bf16", "bf16", a_bits=a, b_bits=eye)
    assert np.array_equal(c, a)
    perm = np.random.default_rng(1).permutation(K)
    P = np.zeros((K, K))
    P[perm, np.arange(K)] = 1.0
    _, _, c = run_gemm(M, K, K, "bf16", "f32", a_bits=a, b_bits=oracle.encode(P, "bf16"))
    assert np.array_equal(oracle.decode(c, "f32"), oracle.decode(a, "bf16")[:, perm])


PATHS = {"tc": 1, "pair": 2}


@pytest.mark.parametrize("path", ["tc", "pair"])
@pytest.mark.parametrize("block_n", [128, 192, 224, 256, 512])
@pytest.mark.parametrize("din,dout", [("f16", "f16"), ("bf16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("M,N,K", [(100, 300, 200), (300, 520, 333), (513, 257, 1000),
                                   (1024, 1024, 64)])
def test_forced_paths_exact(path, block_n, din, dout, M, N, K):
    """Each kernel variant on its own, with ragged tiles: for a pair, M = 100 leaves
    the peer CTA's rows entirely out of range and M = 300 leaves a partial peer.
    FP32 operands (TF32) read B N-major like the others."""
    if path == "tc" and block_n == 512:   # pairs only: refused on the host
        import tiled_matrix_multiplication_gb300 as tg
        with pytest.raises(tg.TgError):
            tg.plan(M, N, K, din, dout, num_sms=152, path=1, block_n=512)
        return
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", path=PATHS[path], block_n=block_n)
    compare(a, b, c, M, N, K, din, dout, exact=True)


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("max_ctas", [0, 2, 6])
def test_pair_split_and_grid(splits, max_ctas):
    M, N, K = 700, 900, 640
    a, b, c = run_gemm(M, N, K, "bf16", "bf16", dist="uniform", path=PATHS["pair"], splits=splits,
                       max_ctas=max_ctas, ldc=N + 8)
    compare(a, b, c, M, N, K, "bf16", "bf16")
    assert padding_untouched(c, N, "bf16")


@pytest.mark.parametrize("din,dout", [("f16", "f16"), ("f16", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 64, 100, 128])
@pytest.mark.parametrize("N,K,splits", [(1000, 777, 1), (128, 64, 1), (1, 300, 2), (520, 2000, 4),
                                        (4096, 1024, 0), (300, 4100, 8)])
def test_skinny_path_exact(din, dout, M, N, K, splits):
    """The small-M kernel (C^T = B^T A^T) for every row-count bucket, ragged N and K,
    without a K split and with K split over clusters of 2, 4 and 8 CTAs."""
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", path=3, splits=splits)
    compare(a, b, c, M, N, K, din, dout, exact=True)


@pytest.mark.parametrize("M", [1, 16, 40, 64, 128])
@pytest.mark.parametrize("block_n", [128, 256, 512])
@pytest.mark.parametrize("splits", [1, 4])
def test_skinny_tile_widths_exact(M, block_n, splits):
    """Each column-tile width (1, 2 or 4 MMAs per k step), ragged N."""
    if M > 64 and block_n == 512:
        # a 128 x 512 FP32 partial tile does not fit shared memory: the
        # combination is refused on the host, before any device work
        import tiled_matrix_multiplication_gb300 as tg
        with pytest.raises(tg.TgError) as err:
            tg.plan(M, 1300, 1000, "f16", "f32", num_sms=152, path=3, block_n=512,
                    splits=splits)
        assert err.value.status == tg.TG_ERR_UNSUPPORTED
        return
    N, K = 1300, 1000
    a, b, c = run_gemm(M, N, K, "f16", "f32", dist="int", path=3, block_n=block_n, splits=splits)
    compare(a, b, c, M, N, K, "f16", "f32", exact=True)


@pytest.mark.parametrize("M", [1, 16, 128])
def test_skinny_path_strided_uniform(M):
    N, K = 700, 900
    a, b, c = run_gemm(M, N, K, "bf16", "bf16", dist="uniform", path=3, lda=K + 8, ldb=N + 36,
                       ldc=N + 8, splits=2)
    compare(a, b, c, M, N, K, "bf16", "bf16")
    assert padding_untouched(c, N, "bf16")


@pytest.mark.parametrize("dout,ldc", [("f16", 1008), ("f32", 1004), ("bf16", 1001)])
@pytest.mark.parametrize("M", [3, 64, 128])
def test_skinny_split_store_pieces(M, dout, ldc):
    """The K-split owner writes C in 16-byte pieces where C allows them: a
    padded C whose last piece straddles column N (ldc 1008 / 1004: aligned rows,
    the piece at N = 1001 partly outside), and an unaligned row pitch (1001:
    element stores throughout).  Padding columns must keep their poison."""
    N, K = 1001, 1500
    din = "bf16" if dout == "bf16" else "f16"
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", path=3, splits=4, ldc=ldc)
    compare(a, b, c, M, N, K, din, dout, exact=True)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_skinny_two_ctas_per_sm_exact(M):
    """The half-ring variant (two CTAs per SM), forced by a small CTA budget."""
    N, K = 4100, 2000
    a, b, c = run_gemm(M, N, K, "bf16", "bf16", dist="int", path=3, block_n=128, splits=4,
                       max_ctas=16)
    compare(a, b, c, M, N, K, "bf16", "bf16", exact=True)



@pytest.mark.parametrize("din,dout", [("f16", "f16"), ("bf16", "f32"), ("f32", "f32"),
                                      ("e4m3", "bf16")])
@pytest.mark.parametrize("M,N,K,max_ctas", [(256, 512, 192, 0), (300, 1100, 700, 0),
                                            (1000, 1500, 1000, 4), (2048, 2048, 256, 2),
                                            (600, 300, 2000, 0)])
def test_wide_tiles_exact(din, dout, M, N, K, max_ctas):
    """512-wide pair tiles (two N = 256 MMAs per K step into one 512-column
    accumulator): ragged M, N and K, a tile whose second MMA's columns lie
    wholly beyond N (N = 300), and grids of 1-2 pairs that reuse the single
    accumulator buffer for many tiles."""
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", path=2, block_n=512, max_ctas=max_ctas)
    compare(a, b, c, M, N, K, din, dout, exact=True)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32")])
def test_wide_tiles_uniform(din, dout):
    M, N, K = 1536, 2560, 1200
    a, b, c = run_gemm(M, N, K, din, dout, dist="uniform", path=2, block_n=512, ldc=N + 8)
    compare(a, b, c, M, N, K, din, dout)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("path,block_n", [(1, 128), (1, 224), (2, 256), (2, 512)])
@pytest.mark.parametrize("dout", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("M,N,ldc_pad", [(200, 300, 8), (257, 1001, 7), (129, 33, 31),
                                         (513, 700, 0)])
def test_tma_store_epilogue_edges(path, block_n, dout, M, N, ldc_pad):
    """C leaves through TMA stores of 32-row boxes when its base, pitch and
    row length are 16-byte multiples, else through the warps' own stores: both
    give the oracle's bits on ragged M and N, boxes partly or wholly outside C
    (the store clips them), and C's padding (poisoned) is never written --
    also where a row of C ends inside a 16-byte piece (N = 1001, 33), which a
    TMA store would overwrite up to the next 16-byte boundary."""
    import tiled_matrix_multiplication_gb300 as tg
    din = "bf16" if dout == "bf16" else "f16"
    K = 300
    ldc = N + ldc_pad
    eo = 4 if dout == "f32" else 2
    p = tg.plan(M, N, K, din, dout, num_sms=152, path=path, block_n=block_n, ldc=ldc)
    assert p["c_vector"] == int((ldc * eo) % 16 == 0), p
    a, b, c = run_gemm(M, N, K, din, dout, dist="int", path=path, block_n=block_n, ldc=ldc)
    compare(a, b, c, M, N, K, din, dout, exact=True)
    assert padding_untouched(c, N, dout)


@pytest.mark.parametrize("block_n", [192, 224, 256])
@pytest.mark.parametrize("M,N,K,max_ctas", [(1024, 1024, 1024, 0), (1000, 1500, 700, 0),
                                            (700, 300, 2000, 8), (2048, 2048, 512, 8),
                                            (300, 5000, 300, 12)])
def test_multicast_pairs_exact(block_n, M, N, K, max_ctas):
    """Clusters of two CTA pairs sharing A tiles by TMA multicast: ragged M, an odd
    number of column tiles (the second tile of the last unit lies beyond N), and
    small grids that walk many units."""
    a, b, c = run_gemm(M, N, K, "f16", "f16", dist="int", path=2, block_n=block_n, multicast=2,
                       max_ctas=max_ctas)
    compare(a, b, c, M, N, K, "f16", "f16", exact=True)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32")])
def test_multicast_pairs_uniform(din, dout):
    M, N, K = 1536, 2560, 1200
    a, b, c = run_gemm(M, N, K, din, dout, dist="uniform", path=2, block_n=256, multicast=2,
                       ldc=N + 8)
    compare(a, b, c, M, N, K, din, dout)
    assert padding_untouched(c, N, dout)
