"""CPU model of the tiled computation and its traffic (test infrastructure).

Nothing here is used to produce reference values for the GPU comparison; the
FP64 three-loop GEMM in ``gemm_ref.c`` does that.  This module restates, from
the pages, the tiled schedule itself so that its facts can be pinned:

* ``tile_ranges`` -- "Matrix multiplication: reuse the inputs" (triton-cuda-lab
  lesson 6), section "Tiles are small rectangles of work": half-open tile
  intervals, the last one clipped at the edge.
* ``tiled_gemm`` -- "Fast matrix multiplication" (inference.shantanugoel.com
  ch. 12), section "Tiling: load once, use many times": the output is computed
  one BM x BN tile at a time, walking K in BK-wide phases; every element of an
  A or B tile copied to "shared memory" is counted as one global load.  The
  accumulator of a tile starts at zero and survives every phase (lesson 6, the
  BK = 2 walk-through of C[0,0]).  The per-phase tile product is a library
  matmul on float64 values.
* ``grouped_tile`` -- the grouped program ordering of the three tile kernels
  (teenygrad "Matrix Multiplication"; llm-systems-cookbook "Triton tiled
  matmul", section "The kernel"; ch. 12 "The CUDA kernel"): a 1-D program id
  walks GROUP_M tile rows down before moving one tile column right.
* closed forms -- naive and tiled load counts (ch. 12 "Counting the waste" and
  its tiled-traffic equation), arithmetic intensity of a whole GEMM
  (cookbook, "Correctness check" pre-check) and of one tile (lesson 6, "Why
  tiling can improve throughput").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def tile_ranges(n: int, t: int):
    """Half-open ``(start, stop)`` intervals of width ``t`` covering ``0..n``."""
    if t <= 0:
        raise ValueError("tile width must be positive")
    return [(s, min(s + t, n)) for s in range(0, n, t)]


@dataclass
class TiledRun:
    C: np.ndarray
    loads: int = 0              # elements of A and B copied into "shared memory"
    programs: int = 0           # output tiles (one program / thread block each)
    k_steps: int = 0            # K phases walked by each program
    masked_dims: tuple = ()     # dimensions whose last tile is partial
    trace: list = field(default_factory=list)  # per-phase contributions to one element


def tiled_gemm(A: np.ndarray, B: np.ndarray, bm: int, bn: int | None = None,
               bk: int | None = None, trace=None) -> TiledRun:
    """Compute C = A @ B tile by tile (float64) and count global loads.

    ``trace=(i, j)`` records the contribution of each K phase to C[i, j].
    """
    bn = bm if bn is None else bn
    bk = bm if bk is None else bk
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    run = TiledRun(C=np.zeros((M, N), dtype=np.float64))
    mr, nr, kr = tile_ranges(M, bm), tile_ranges(N, bn), tile_ranges(K, bk)
    run.programs = len(mr) * len(nr)
    run.k_steps = len(kr)
    run.masked_dims = tuple(d for d, (n, t) in zip("MNK", ((M, bm), (N, bn), (K, bk))) if n % t)
    for (r0, r1) in mr:
        for (c0, c1) in nr:
            acc = np.zeros((r1 - r0, c1 - c0), dtype=np.float64)
            for (k0, k1) in kr:
                a_tile = A[r0:r1, k0:k1]
                b_tile = B[k0:k1, c0:c1]
                run.loads += a_tile.size + b_tile.size
                part = a_tile @ b_tile
                if trace is not None and r0 <= trace[0] < r1 and c0 <= trace[1] < c1:
                    run.trace.append(float(part[trace[0] - r0, trace[1] - c0]))
                acc += part
            run.C[r0:r1, c0:c1] = acc
    return run


def grouped_tile(pid: int, tiles_m: int, tiles_n: int, group_m: int, variant: str = "in_group"):
    """Map a 1-D program id to ``(pid_m, pid_n)`` in grouped order.

    ``variant="in_group"`` takes the row offset from the id's position inside
    its group (teenygrad kernel); ``variant="global"`` takes it from the global
    id (cookbook and ch. 12 kernels).  Both visit every tile exactly once; they
    differ only inside a final, shorter group.
    """
    per_group = group_m * tiles_n
    g = pid // per_group
    first_m = g * group_m
    size_m = min(tiles_m - first_m, group_m)
    q = pid % per_group
    off = (q if variant == "in_group" else pid) % size_m
    return first_m + off, q // size_m


# ---------------------------------------------------------------- closed forms

def naive_loads(M: int, N: int, K: int) -> int:
    """One output element per program: K loads of A and K of B each."""
    return 2 * M * N * K


def tiled_loads(M: int, N: int, K: int, T: int) -> int:
    """Loads of the T x T tiled schedule with clipped edge tiles.

    Each output tile of r rows and c columns loads r*K elements of A and K*c of
    B over its phases; summing over the tile grid gives
    K * (M * ceil(N/T) + N * ceil(M/T)), which is 2MNK/T when T divides M and N.
    """
    return K * (M * cdiv(N, T) + N * cdiv(M, T))


def matmul_intensity(m: int, k: int, n: int, dtype_bytes: int = 2) -> float:
    """FLOPs per byte of compulsory traffic (read A and B, write C once)."""
    return 2 * m * k * n / (dtype_bytes * (m * k + k * n + m * n))


def tile_reuse(bm: int, bn: int, bk: int, dtype_bytes: int = 2):
    """One tile step: (input elements, input bytes, FLOPs, FLOPs per input byte)."""
    elems = bm * bk + bk * bn
    nbytes = elems * dtype_bytes
    flops = 2 * bm * bn * bk
    return elems, nbytes, flops, flops / nbytes


def phase_intensity(T: int, dtype_bytes: int = 4) -> float:
    """One T x T phase: 2T^3 FLOPs over 2T^2 loaded values."""
    return 2 * T ** 3 / (2 * T * T * dtype_bytes)


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def exit_check(M: int, N: int, K: int, bm: int, bn: int, bk: int):
    """(programs, K steps, dimensions needing masks) of one tiled launch."""
    return (cdiv(M, bm) * cdiv(N, bn), cdiv(K, bk),
            tuple(d for d, (n, t) in zip("MNK", ((M, bm), (N, bn), (K, bk))) if n % t))

