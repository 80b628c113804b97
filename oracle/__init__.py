"""CPU oracle for the dense GEMM C[m,n] = sum_k A[m,k]*B[k,n].

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` leg may import this
package.  The CUDA library never calls it, and it imports nothing from the
library: both sides receive the same seeded bit patterns and nothing else.

Contents:
  * ``ref``         -- ctypes front-end to ``gemm_ref.c`` (FP64 three-loop GEMM,
                       format decoders and round-to-nearest-even encoders).
  * ``tiled_model`` -- the pages' CPU tiled model: tile ranges, grouped raster,
                       per-K-chunk partial sums and the global-load counter.
  * ``compare``     -- the tolerance rule and ulp of the output format.
  * ``epilogue``    -- the fused epilogue act(alpha*scale*C + bias) + beta*R in
                       FP64 and its tolerance.

Every pin that ties these functions to the pages or to mathematics lives in
``tests/test_oracle_*.py``.
"""
from .ref import (F16, BF16, F32, FORMATS, build, decode, encode, gemm_ref,
                  gemm_ref_bits, num_threads, lib_path)
from .compare import ulp, tolerance, check_close, rel_tol_for, rel_tol_3xtf32
from . import epilogue, tiled_model

__all__ = [
    "F16", "BF16", "F32", "FORMATS", "build", "decode", "encode", "gemm_ref",
    "gemm_ref_bits", "num_threads", "lib_path", "ulp", "tolerance", "check_close",
    "rel_tol_for", "rel_tol_3xtf32", "tiled_model", "epilogue",
]
