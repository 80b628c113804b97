"""Failure detection on the GPU without a fault: a kernel's bounded wait on a
barrier that nothing arrives on runs out, the kernel records TG_ERR_TIMEOUT
in the device status word and exits; the host reads the status, it is then
cleared, and the context keeps working (a GEMM afterwards matches the
oracle)."""
from __future__ import annotations

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tests.conftest import cuda_ok
from tests.gemm_util import compare, run_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]


def test_timeout_is_reported_and_cleared():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_last_device_error(s) == tg.TG_OK          # nothing pending
    assert tg.tg_selftest_timeout(20, s) == tg.TG_OK
    assert tg.tg_last_device_error(s) == tg.TG_ERR_TIMEOUT
    assert tg.tg_last_device_error(s) == tg.TG_OK          # read clears it


def test_context_usable_after_timeout():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    assert tg.tg_selftest_timeout(5, s) == tg.TG_OK
    assert tg.tg_last_device_error(s) == tg.TG_ERR_TIMEOUT
    a, b, c = run_gemm(300, 520, 200, "f16", "f16", dist="int")
    compare(a, b, c, 300, 520, 200, "f16", "f16", exact=True)


def test_first_failure_is_kept():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        assert tg.tg_selftest_timeout(2, s) == tg.TG_OK
    assert tg.tg_last_device_error(s) == tg.TG_ERR_TIMEOUT
    assert tg.tg_last_device_error(s) == tg.TG_OK
