"""The checked build (device-side bounds and alignment checks compiled in,
``libtg_gemm_checked.so``): built here, then every kernel choice is run
through it in a child process (``tests/checked_cases.py``) and compared with
the oracle; no check may fail, and the check mechanism itself must catch an
out-of-range index without touching memory."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

from tests.conftest import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.timeout(1200)
def test_checked_build_runs_every_kernel_choice_clean():
    from tiled_matrix_multiplication_gb300 import build
    build.build(checked=True)
    r = subprocess.run([sys.executable, "-m", "tests.checked_cases"], cwd=ROOT,
                       capture_output=True, text=True, timeout=1100,
                       env={**os.environ, "TG_CHECKED": "1"})
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "every case clean" in r.stdout
