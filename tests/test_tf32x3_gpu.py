"""GPU parity and accuracy of the 3xTF32 mode: every element within the
3xTF32 bound of the FP64 oracle (oracle.rel_tol_3xtf32) on ragged, padded,
split-K and batched problems and with the fused epilogue; integer operands
bit-exact; and, on the same uniform operands, an error at least 30 times
smaller than the one-pass TF32 result's."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare, padding_untouched, run_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

X3 = dict(f32_mode=tg.TG_F32_3XTF32)


def check_x3(a, b, c, M, N, K, rows=None):
    rows = np.arange(M) if rows is None else np.asarray(rows)
    C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a[rows]), b, K=K, N=N, fmt="f32")
    got = oracle.decode(np.ascontiguousarray(c[rows][:, :N]), "f32")
    ok, rep = oracle.check_close(got, C_ref, S, "f32", "f32", rel=oracle.rel_tol_3xtf32(K))
    assert ok, rep
    return np.abs(got - C_ref) / np.where(S > 0, S, 1.0)


@pytest.mark.parametrize("M,N,K", [(1000, 1999, 777), (130, 70, 50), (1, 300, 2000),
                                   (257, 513, 1)])
def test_ragged(M, N, K):
    a, b, c = run_gemm(M, N, K, "f32", "f32", ldc=N + 3, **X3)
    check_x3(a, b, c, M, N, K)
    assert padding_untouched(c, N, "f32")


def test_padded_operands():
    a, b, c = run_gemm(300, 200, 500, "f32", "f32", lda=503, ldb=205, **X3)
    check_x3(a, b, c, 300, 200, 500)


def test_integer_operands_exact():
    a, b, c = run_gemm(300, 520, 700, "f32", "f32", dist="int", **X3)
    compare(a, b, c, 300, 520, 700, "f32", "f32", exact=True)


@pytest.mark.parametrize("variant", [dict(path=tg.TG_PATH_TC, block_n=128),
                                     dict(path=tg.TG_PATH_TC_PAIR, splits=3, multicast=1)])
def test_variants(variant):
    a, b, c = run_gemm(520, 600, 900, "f32", "f32", **X3, **variant)
    check_x3(a, b, c, 520, 600, 900)


def test_accuracy_against_one_pass_tf32():
    M = N = K = 1024
    a, b, c3 = run_gemm(M, N, K, "f32", "f32", **X3)
    _, _, c1 = run_gemm(M, N, K, "f32", "f32")
    rows = np.arange(0, M, 16)
    e3 = check_x3(a, b, c3, M, N, K, rows=rows)
    C_ref, S = oracle.gemm_ref_bits(np.ascontiguousarray(a[rows]), b, K=K, N=N, fmt="f32")
    e1 = np.abs(oracle.decode(np.ascontiguousarray(c1[rows][:, :N]), "f32") - C_ref) / S
    assert np.sqrt(np.mean(e3 ** 2)) * 30 < np.sqrt(np.mean(e1 ** 2)), (e3.max(), e1.max())
    assert e3.max() * 30 < e1.max()


def test_square_2048_sampled():
    n = 2048
    a, b, c = run_gemm(n, n, n, "f32", "f32", **X3)
    rows = np.unique(np.concatenate([np.random.default_rng(4).choice(n, 32, replace=False),
                                     [0, n - 1]]))
    check_x3(a, b, c, n, n, n, rows=rows)


def test_batched_per_product():
    import torch
    from tests.gemm_util import to_bits, to_device
    from tiled_matrix_multiplication_gb300 import inputs
    batch, M, N, K = 3, 130, 70, 96
    a_bits = [inputs.matrix_bits(M, K, "f32", "uniform", 100 + z) for z in range(batch)]
    b_bits = [inputs.matrix_bits(K, N, "f32", "uniform", 200 + z) for z in range(batch)]
    a = torch.stack([to_device(x, "f32") for x in a_bits])
    b = torch.stack([to_device(x, "f32") for x in b_bits])
    c = tg.bmm(a, b, **X3)
    torch.cuda.synchronize()
    for z in range(batch):
        check_x3(a_bits[z], b_bits[z], to_bits(c[z], "f32"), M, N, K)


def test_fused_epilogue():
    import torch
    from tests.gemm_util import to_device
    from tiled_matrix_multiplication_gb300 import inputs
    M, N, K = 200, 300, 400
    a_bits = inputs.matrix_bits(M, K, "f32", "uniform", 5)
    b_bits = inputs.matrix_bits(K, N, "f32", "uniform", 6)
    bias = torch.linspace(-1, 1, N, device="cuda", dtype=torch.float32)
    out = tg.gemm_fused(to_device(a_bits, "f32"), to_device(b_bits, "f32"), bias=bias,
                        activation="relu", **X3)
    torch.cuda.synchronize()
    C_ref, S = oracle.gemm_ref_bits(a_bits, b_bits, K=K, N=N, fmt="f32")
    D_ref, _ = oracle.epilogue.epilogue_ref(C_ref, bias=bias.cpu().numpy(), act="relu")
    err = np.abs(out.cpu().numpy().astype(np.float64) - D_ref)
    assert np.all(err <= oracle.rel_tol_3xtf32(K) * S + oracle.ulp(D_ref, "f32") +
                  2.0 ** -20 * (np.abs(C_ref) + 1.0))


def test_bench_shape_4096_sampled():
    n = 4096
    a, b, c = run_gemm(n, n, n, "f32", "f32", **X3)
    rows = np.unique(np.concatenate([np.random.default_rng(14).choice(n, 16, replace=False),
                                     [0, n - 1]]))
    check_x3(a, b, c, n, n, n, rows=rows)


def test_multicast_pairs():
    # TF32 on clusters of two CTA pairs sharing A (one pass and three)
    a, b, c = run_gemm(1000, 1999, 777, "f32", "f32", path=tg.TG_PATH_TC_PAIR, multicast=2)
    compare(a, b, c, 1000, 1999, 777, "f32", "f32")
    a, b, c = run_gemm(1000, 1999, 777, "f32", "f32", path=tg.TG_PATH_TC_PAIR, multicast=2, **X3)
    check_x3(a, b, c, 1000, 1999, 777)
