"""Shared test configuration.

Markers:
  gpu -- needs a CUDA device (a GB300, sm_103); everything else runs on CPU.
"""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GB300 device")


def read_golden(name: str) -> dict:
    """Parse a ``key = value`` fixture; '#' lines are the citation."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition("=")
            out[key.strip()] = val.strip()
    return out


def parse_matrix(text: str):
    return [[float(x) for x in row.split()] for row in text.split(";")]


def parse_numbers(text: str):
    return [float(x) for x in text.split()]


def cuda_ok() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001
        return False


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle
