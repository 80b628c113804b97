"""Builds the CUDA library ``libtg_gemm.so`` in-tree for sm_103a.

Each translation unit in ``csrc/`` is compiled with nvcc in parallel into
``_build/``, then linked into ``libtg_gemm.so`` next to this file.  A rebuild
happens only when a source or header is newer than the library.  ``--checked``
builds ``libtg_gemm_checked.so`` (objects in ``_build_checked/``) with the
device-side bounds and alignment checks compiled in (``-DTG_CHECKED``).

    python -m tiled_matrix_multiplication_gb300.build [--force] [--ptxas-info] [--checked]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtg_gemm.so")
LIB_CHECKED = os.path.join(PKG, "libtg_gemm_checked.so")

SOURCES = ["tg_api.cu", "tg_plan.cu", "tg_host.cu", "gemm_tc.cu", "gemm_tc_f16.cu",
           "gemm_tc_tf32.cu", "gemm_tc_fp8.cu", "gemm_skinny.cu", "gemm_skinny_fp8.cu",
           "aux_kernels.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtg_gemm.so")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    """Compile and link the library (the checked variant if ``checked``) if
    needed; returns its path."""
    lib, bdir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checked:
        extra.append("-DTG_CHECKED")

    def compile_one(src):
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        out = _run([cc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj])
        return obj, out

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    if verbose or ptxas_info:
        for _, out in results:
            if out.strip():
                print(out, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    _run([cc, *ARCH, "-shared", *objs, "-o", tmp])
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / smem / spills")
    ap.add_argument("--checked", action="store_true",
                    help="build libtg_gemm_checked.so with the device-side checks")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=True, ptxas_info=args.ptxas_info, checked=args.checked))


if __name__ == "__main__":
    main()
