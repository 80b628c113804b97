"""bench.py's launch rules on CPU.

The GPU arm runs on one GPU only: the library's tile kernels share A tiles
inside a thread-block cluster by TMA multicast, which is used only in
single-GPU processes, so ``--gpus N`` with N > 1 and a torchrun launch with
WORLD_SIZE > 1 are refused before any GPU work.  The reference arm (the CPU
oracle) still runs under torchrun: rank 0 prints exactly one JSON line and the
other ranks exit 0 without work."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_refusal_rule():
    import bench
    assert bench.refuse_multi_gpu(1, 1) is None
    assert "--gpus 2" in bench.refuse_multi_gpu(2, 1)
    assert "WORLD_SIZE=4" in bench.refuse_multi_gpu(1, 4)
    assert "multicast" in bench.refuse_multi_gpu(8, 8)


@pytest.mark.parametrize("argv,env", [
    (["--gpus", "2"], {}),
    (["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}),
])
def test_gpu_arm_refuses_more_than_one_gpu(argv, env):
    # refused before torch, the library or a GPU is touched: exit code 2 and
    # the reason on stderr, no JSON line
    r = subprocess.run([sys.executable, "bench.py", *argv, "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120,
                       env={**os.environ, **env})
    assert r.returncode == 2, (r.returncode, r.stderr[-2000:])
    assert "one GPU only" in r.stderr
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--workload",
           "small127_f16"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=280,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
