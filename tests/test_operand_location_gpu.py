"""Operands that are not device memory of the calling GPU are refused.

The tile kernels read A through TMA loads multicast to the CTAs of a cluster
of this GPU, and no kernel of the library is meant to reach host memory or a
peer GPU's memory over the interconnect.  Every launching entry point checks,
before it enqueues anything, that A, B, C and the epilogue's vectors and
residual are device memory of the current device; host memory (page-locked or
pageable) returns TG_ERR_INVALID_VALUE and leaves C untouched.  (This pool has
one GPU per call, so a peer GPU's memory cannot be passed here; the rule that
refuses host memory is the same one that refuses it.)"""
from __future__ import annotations

import numpy as np
import pytest

from tests.conftest import cuda_ok

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

M, N, K = 256, 256, 128


@pytest.fixture(scope="module")
def tg():
    from tiled_matrix_multiplication_gb300 import build
    import tiled_matrix_multiplication_gb300 as tgmod
    build.build()
    tgmod.load()
    return tgmod


@pytest.fixture(scope="module")
def bufs():
    import torch
    dev = dict(a=torch.ones((M, K), dtype=torch.float16, device="cuda"),
               b=torch.ones((K, N), dtype=torch.float16, device="cuda"),
               c=torch.full((M, N), 7.0, dtype=torch.float16, device="cuda"),
               v=torch.ones(N, dtype=torch.float32, device="cuda"))
    pinned = {k: t.cpu().pin_memory() for k, t in dev.items()}
    pageable = {k: np.ascontiguousarray(t.cpu().numpy()) for k, t in dev.items()}
    return dev, pinned, pageable


def _ptr(x):
    return x.data_ptr() if hasattr(x, "data_ptr") else x.ctypes.data


@pytest.mark.parametrize("where", ["pinned", "pageable"])
@pytest.mark.parametrize("which", ["a", "b", "c"])
def test_host_operand_is_refused(tg, bufs, where, which):
    import torch
    dev, pinned, pageable = bufs
    host = pinned if where == "pinned" else pageable
    p = {k: _ptr(dev[k]) for k in "abc"}
    p[which] = _ptr(host[which])
    s = torch.cuda.current_stream().cuda_stream
    calls = {
        "tg_gemm": lambda: tg.tg_gemm(M, N, K, p["a"], K, p["b"], N, p["c"], N, "f16", "f16", s),
        "tg_gemm_fused": lambda: tg.tg_gemm_fused(
            M, N, K, p["a"], K, p["b"], N, p["c"], N, "f16", "f16",
            tg.make_epilogue(activation="relu"), s, None),
        "tg_gemm_strided_batched": lambda: tg.tg_gemm_strided_batched(
            1, M, N, K, p["a"], K, 0, p["b"], N, 0, p["c"], N, 0, "f16", "f16", s, None),
        "tg_gemm_strided_batched_fused": lambda: tg.tg_gemm_strided_batched_fused(
            2, M // 2, N, K, p["a"], K, (M // 2) * K, p["b"], N, 0, p["c"], N, (M // 2) * N,
            "f16", "f16", tg.make_epilogue(activation="relu"), 0, s, None),
        "tg_gemm_splitk_noalloc": lambda: tg.tg_gemm_splitk_noalloc(
            M, N, K, p["a"], K, p["b"], N, p["c"], N, "f16", "f16", 2, s),
    }
    for name, call in calls.items():
        assert call() == tg.TG_ERR_INVALID_VALUE, name
    torch.cuda.synchronize()
    assert tg.tg_last_device_error(s) == tg.TG_OK
    assert bool((dev["c"] == 7.0).all())
    if which == "c":
        assert bool((torch.as_tensor(host["c"]) == 7.0).all())


@pytest.mark.parametrize("field", ["bias", "scale", "residual"])
def test_host_epilogue_operand_is_refused(tg, bufs, field):
    import torch
    dev, pinned, _ = bufs
    s = torch.cuda.current_stream().cuda_stream
    kw = {"activation": "silu", field: pinned["v"].data_ptr() if field != "residual"
          else pinned["c"].data_ptr()}
    if field == "residual":
        kw["ldr"] = N
        kw["beta"] = 1.0
    epi = tg.make_epilogue(**kw)
    st = tg.tg_gemm_fused(M, N, K, dev["a"].data_ptr(), K, dev["b"].data_ptr(), N,
                          dev["c"].data_ptr(), N, "f16", "f16", epi, s, None)
    assert st == tg.TG_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert bool((dev["c"] == 7.0).all())


def test_device_operands_still_run(tg, bufs):
    import torch
    dev, _, _ = bufs
    s = torch.cuda.current_stream().cuda_stream
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    st = tg.tg_gemm(M, N, K, dev["a"].data_ptr(), K, dev["b"].data_ptr(), N, c.data_ptr(), N,
                    "f16", "f16", s)
    assert st == tg.TG_OK
    torch.cuda.synchronize()
    assert tg.tg_last_device_error(s) == tg.TG_OK
    assert bool((c == float(K)).all())
