"""tg_gemm_splitk_noalloc: the split-K GEMM for callers that cannot let the
library allocate device memory (their memory is all held by their own
allocator, or the call sits on a path that must not allocate).  Its partial
tiles live in a fixed array owned by the library instead of workspace.

Checked through the C ABI against the existing entry point (tg_gemm_ex with the
same path and split) within the tests' tolerance rule, on two calls in a row
with different operands, so a stale array from the first call would show up in
the second.  This file is collected last and is also meant to pass on its own
in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

from tests.conftest import cuda_ok

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


@pytest.fixture(scope="module")
def tg():
    from tiled_matrix_multiplication_gb300 import build
    import tiled_matrix_multiplication_gb300 as tgmod
    build.build()
    tgmod.load()
    return tgmod


def _operands(M, N, K, din, seed):
    import torch
    from tiled_matrix_multiplication_gb300 import inputs
    a = inputs.matrix_bits(M, K, din, "uniform", seed)
    b = inputs.matrix_bits(K, N, din, "uniform", seed + 1)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[din]
    ta = torch.from_numpy(a.view(np.int16)).view(tdt).cuda()
    tb = torch.from_numpy(b.view(np.int16)).view(tdt).cuda()
    return a, b, ta, tb


def _bits(t, dout):
    import torch
    ints = {"f16": torch.int16, "bf16": torch.int16, "f32": torch.int32}[dout]
    npt = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}[dout]
    return t.contiguous().view(ints).cpu().numpy().view(npt)


@pytest.mark.parametrize("M,N,K,din,dout,splits", [
    (64, 8192, 4096, "f16", "f16", 4),
    (128, 4096, 2048, "bf16", "f32", 3),
    (100, 1000, 777 + 7, "bf16", "bf16", 5),
    # more than 128 rows: the planner picks 224-wide tiles, whose B boxes are
    # 64-byte swizzled (112 of them are 448 bytes per K row); ragged N
    (896, 2000, 1024, "bf16", "bf16", 2),
    (1024, 2048, 1024, "f16", "f16", 2),   # 256-wide tiles; the array exactly full
])
def test_noalloc_matches_existing_entry_point(tg, M, N, K, din, dout, splits):
    import torch
    import oracle
    if M > 128:
        p = tg.plan(M, N, K, din, dout, num_sms=torch.cuda.get_device_properties(0).multi_processor_count,
                    path=tg.TG_PATH_TC, splits=splits)
        assert p["block_n"] != 128 and p["splits"] == splits, p
        assert splits * M * N * 4 <= tg.NOALLOC_SCRATCH_BYTES
    tdo = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dout]
    stream = torch.cuda.current_stream().cuda_stream
    opt = tg.make_options(path=tg.TG_PATH_TC, splits=splits)
    for call, seed in enumerate((101, 202)):           # two calls in a row
        a_bits, b_bits, a, b = _operands(M, N, K, din, seed)
        c_new = torch.full((M, N), float("nan"), dtype=tdo, device="cuda")
        c_old = torch.full((M, N), float("nan"), dtype=tdo, device="cuda")
        st = tg.tg_gemm_splitk_noalloc(M, N, K, a.data_ptr(), K, b.data_ptr(), N,
                                       c_new.data_ptr(), N, din, dout, splits, stream)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        st = tg.tg_gemm_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_old.data_ptr(), N,
                           din, dout, stream, opt)
        assert st == tg.TG_OK, tg.tg_status_string(st)
        torch.cuda.synchronize()
        assert tg.tg_last_device_error(stream) == tg.TG_OK
        new = oracle.decode(_bits(c_new, dout), dout)
        old = oracle.decode(_bits(c_old, dout), dout)
        C_ref, S = oracle.gemm_ref_bits(a_bits, b_bits, K=K, N=N, fmt=din)
        tol = oracle.tolerance(old, S, din, dout)
        err = np.abs(new - old)
        assert np.all(err <= tol), f"call {call}: max err/tol {np.max(err / tol):.3g}"
        ok, report = oracle.check_close(new, C_ref, S, din, dout)
        assert ok, f"call {call}: {report}"


def test_noalloc_rejects_sizes_beyond_its_array(tg):
    import torch
    a = torch.zeros((128, 4096), dtype=torch.float16, device="cuda")
    b = torch.zeros((4096, 8192), dtype=torch.float16, device="cuda")
    c = torch.zeros((128, 8192), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # 8 splits x 128 x 8192 x 4 bytes = 32 MiB > the 16 MiB array
    assert 8 * 128 * 8192 * 4 > tg.NOALLOC_SCRATCH_BYTES
    st = tg.tg_gemm_splitk_noalloc(128, 8192, 4096, a.data_ptr(), 4096, b.data_ptr(), 8192,
                                   c.data_ptr(), 8192, "f16", "f16", 8, stream)
    assert st == tg.TG_ERR_UNSUPPORTED
    st = tg.tg_gemm_splitk_noalloc(128, 8192, 4096, a.data_ptr(), 4096, b.data_ptr(), 8192,
                                   c.data_ptr(), 8192, "f32", "f32", 2, stream)
    assert st == tg.TG_ERR_UNSUPPORTED
    torch.cuda.synchronize()
