"""Cases run against the checked build (``TG_CHECKED=1``): one or more calls of
every kernel choice -- the tile kernel on single-CTA tiles, CTA pairs, pairs
sharing A by multicast and 512-wide pairs, split K, TF32, 3xTF32, FP8, packed
operands, the fused epilogue and a strided batch; the small-M kernel with and
without its on-chip K split, two CTAs per SM and one -- each compared with the
oracle, with the device status word read after every call (a failed
device-side check raises TG_ERR_BOUNDS there).  Run by
tests/test_checked_build_gpu.py in a subprocess, since a process loads one
variant of the library:

    TG_CHECKED=1 python -m tests.checked_cases
"""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import tiled_matrix_multiplication_gb300 as tg  # noqa: E402
from tests.gemm_util import compare, run_gemm  # noqa: E402

P1, P2, SK = tg.TG_PATH_TC, tg.TG_PATH_TC_PAIR, tg.TG_PATH_SKINNY

# (M, N, K, din, dout, options), integer inputs: the oracle's result exactly
CASES = [
    (300, 520, 200, "f16", "f16", dict(path=P1, block_n=128)),
    (300, 520, 200, "bf16", "f32", dict(path=P1, block_n=192)),
    (300, 520, 200, "f16", "f16", dict(path=P1, block_n=224)),
    (300, 520, 200, "f16", "f32", dict(path=P1, block_n=256)),
    (600, 1100, 300, "f16", "f16", dict(path=P2, block_n=256, multicast=1)),
    (600, 1100, 300, "bf16", "bf16", dict(path=P2, block_n=224, multicast=1)),
    (600, 1100, 300, "f16", "f16", dict(path=P2, block_n=256, multicast=2)),
    (600, 1100, 300, "f16", "f16", dict(path=P2, block_n=512)),
    (256, 384, 1000, "f16", "f16", dict(path=P1, splits=3)),
    (200, 300, 130, "f32", "f32", {}),
    (200, 300, 130, "f32", "f32", dict(f32_mode=1)),
    (300, 520, 256, "e4m3", "f16", {}),
    (127, 255, 65, "f16", "f32", {}),                       # both operands packed
    (1, 1000, 777, "f16", "f16", dict(path=SK)),
    (37, 1000, 700, "bf16", "bf16", dict(path=SK, splits=1, multicast=1)),
    (64, 4100, 2000, "f16", "f16", dict(path=SK, splits=4, block_n=128, max_ctas=16)),
    (128, 8192, 2048, "f16", "f16", dict(path=SK)),          # split of 2, one CTA per SM
    (128, 1300, 1000, "f16", "f32", dict(path=SK, block_n=256, splits=4)),
    (100, 2048, 1024, "e4m3", "bf16", dict(path=SK)),
    (1000, 1999, 777, "f32", "f32", {}),                    # TF32, packed, C row by row
    (2048, 4096, 1024, "f16", "f16", {}),                   # the planner's pairs sharing A, many tiles
]


def main() -> int:
    import torch
    assert tg.CHECKED and tg.tg_checked_build() == 1, "the checked library is not loaded"
    s = torch.cuda.current_stream().cuda_stream
    # the mechanism itself: an index inside the array passes, one outside is
    # caught and its store skipped
    assert tg.tg_selftest_bounds(5, s) == tg.TG_OK
    assert tg.tg_last_device_error(s) == tg.TG_OK
    assert tg.tg_selftest_bounds(40, s) == tg.TG_OK
    assert tg.tg_last_device_error(s) == tg.TG_ERR_BOUNDS
    assert tg.tg_last_device_error(s) == tg.TG_OK          # read and cleared
    for M, N, K, din, dout, opts in CASES:
        a, b, c = run_gemm(M, N, K, din, dout, dist="int", **opts)   # raises on a device error
        rows = np.arange(M) if M <= 300 else np.r_[0:64, M - 64:M]
        compare(a, b, c, M, N, K, din, dout, exact=True, rows=rows)
        print("ok", M, N, K, din, dout, opts, flush=True)
    # the fused epilogue and a strided batch
    from tests.test_epilogue_gpu import run_fused
    run_fused(300, 520, 200, "f16", "f16", act="silu", alpha=0.75, beta=-0.5)
    run_fused(40, 1000, 700, "bf16", "bf16", act="gelu_tanh", beta=1.0, path=SK)
    from tests.test_batched_gpu import check_all
    check_all(3, 130, 200, 96, "f16", "f16")
    check_all(3, 64, 512, 2048, "bf16", "bf16", path=SK, splits=4)
    print("checked build: every case clean", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
