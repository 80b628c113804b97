"""The C-ABI library: builds, loads, exports what the header declares, and its
host-only logic (validation and planning).  No compute call is made here, so
these run without a GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg_gemm.h")

A, B, C = 0x10000, 0x100000000, 0x200000000   # aligned, disjoint placeholder addresses


@pytest.fixture(scope="module")
def lib():
    tgbuild.build()
    return tg.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert names == sorted(tg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(tg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_abi_version_and_status_strings(lib):
    assert tg.tg_abi_version() == 10
    assert tg.tg_status_string(tg.TG_OK) == "TG_OK"
    assert tg.tg_status_string(tg.TG_ERR_TIMEOUT) == "TG_ERR_TIMEOUT"
    assert tg.tg_status_string(tg.TG_ERR_BOUNDS) == "TG_ERR_BOUNDS"
    assert tg.tg_status_string(99) == "TG_ERR_UNKNOWN"


def test_normal_build_has_no_device_checks(lib):
    # the device-side checks exist only in the checked build; the normal one
    # says so without touching the device
    assert tg.tg_checked_build() == 0 and not tg.CHECKED
    assert tg.tg_selftest_bounds(40, 0) == tg.TG_ERR_NOT_IMPLEMENTED
    assert tg.tg_selftest_bounds(-1, 0) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_selftest_bounds(1025, 0) == tg.TG_ERR_INVALID_VALUE


def plan(M, N, K, din="f16", dout=None, lda=None, ldb=None, ldc=None, a=A, b=B, c=C, sms=148,
         **opts):
    dout = din if dout is None else dout
    o = tg.make_options(**opts) if opts else None
    return tg.tg_plan_gemm(M, N, K, a, K if lda is None else lda, b, N if ldb is None else ldb,
                           c, N if ldc is None else ldc, din, dout, sms, o)


@pytest.mark.parametrize("args,status", [
    (dict(M=-1, N=4, K=4), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, lda=3), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, ldb=3), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, ldc=3), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, a=0), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, c=0), tg.TG_ERR_INVALID_VALUE),
    (dict(M=4, N=4, K=4, a=A + 1), tg.TG_ERR_INVALID_VALUE),          # not element aligned
    (dict(M=4, N=4, K=4, c=A + 8), tg.TG_ERR_INVALID_VALUE),          # C overlaps A
    (dict(M=4, N=4, K=4, c=B), tg.TG_ERR_INVALID_VALUE),              # C overlaps B
    (dict(M=4, N=4, K=4, din="f16", dout="bf16"), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, din="bf16", dout="f16"), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, din="f32", dout="f16"), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, din=7), tg.TG_ERR_INVALID_VALUE),
    (dict(M=1 << 31, N=4, K=4), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, block_n=96), tg.TG_ERR_UNSUPPORTED),
    (dict(M=4, N=4, K=4, splits=-2), tg.TG_ERR_INVALID_VALUE),
])
def test_validation(lib, args, status):
    st, _ = plan(**args)
    assert st == status


def test_gemm_rejects_before_touching_the_device(lib):
    # argument errors come back before any CUDA call, so they work without a GPU
    assert tg.tg_gemm(-1, 4, 4, A, 4, B, 4, C, 4, "f16", "f16", 0) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm(4, 4, 4, A, 4, B, 4, C, 4, "f16", "bf16", 0) == tg.TG_ERR_UNSUPPORTED
    assert tg.tg_gemm(4, 4, 4, A, 4, B, 4, A, 4, "f16", "f16", 0) == tg.TG_ERR_INVALID_VALUE
    # empty output: nothing to do
    assert tg.tg_gemm(0, 4, 4, 0, 4, 0, 4, 0, 4, "f16", "f16", 0) == tg.TG_OK
    assert tg.tg_gemm(4, 0, 4, 0, 4, 0, 0, 0, 0, "f16", "f16", 0) == tg.TG_OK


def test_plan_square_4096(lib):
    st, p = plan(4096, 4096, 4096, sms=148)
    assert st == tg.TG_OK
    assert p["path"] == tg.TG_PATH_TC_PAIR and p["block_m"] == 256 and p["block_k"] == 64
    # work units: tiles, or pairs of adjacent tiles sharing A by multicast
    assert p["tiles"] == (4096 // 256) * -(-(4096 // p["block_n"]) // p["multicast"])
    assert p["splits"] == 1
    # the resident grid: 74 pairs, or 35 four-CTA clusters when two pairs share A
    assert p["ctas"] == (148 if p["multicast"] == 1 else 4 * (148 * 19 // 80))
    assert p["pack_a"] == 0 and p["pack_b"] == 0 and p["c_vector"] == 1
    assert p["kernels"] == 1 and p["workspace_bytes"] == 0


def test_plan_wide_tiles(lib):
    # 512-wide tiles: CTA pairs only (two N = 256 MMAs per K step), every
    # operand type, no A multicast
    for din, dout in (("f16", "f16"), ("bf16", "f32"), ("e4m3", "f16"), ("f32", "f32")):
        st, p = plan(4096, 4096, 4096, din, dout, sms=148, path=tg.TG_PATH_TC_PAIR, block_n=512)
        assert st == tg.TG_OK and p["block_n"] == 512 and p["block_m"] == 256, (din, p)
        assert p["multicast"] == 1 and p["tiles"] == 16 * 8 and p["stages"] == 4
    st, p = plan(4096, 4096, 4096, block_n=512, sms=148)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC_PAIR
    for bad in (dict(path=tg.TG_PATH_TC, block_n=512), dict(block_n=512, multicast=2)):
        st, _ = plan(4096, 4096, 4096, sms=148, **bad)
        assert st == tg.TG_ERR_UNSUPPORTED, bad


def test_plan_tf32_reads_b_in_place(lib):
    # B is read N-major by the TF32 MMA (32-byte-atom swizzle): no transposed copy
    st, p = plan(2048, 2048, 2048, "f32", "f32", sms=148)
    assert st == tg.TG_OK and p["pack_a"] == 0 and p["pack_b"] == 0 and p["kernels"] == 1
    assert p["workspace_bytes"] == 0


def test_plan_config1_needs_pack(lib):
    # 127x255x65 FP16 -> FP32: lda = 65 halves = 130 bytes, ldb = 255 halves = 510 bytes
    st, p = plan(127, 255, 65, "f16", "f32")
    assert st == tg.TG_OK
    assert p["pack_a"] == 1 and p["pack_b"] == 1
    assert p["c_vector"] == 0            # ldc = 255 floats = 1020 bytes
    assert p["workspace_bytes"] >= 127 * 72 * 2 + 65 * 256 * 2


def test_plan_tf32(lib):
    st, p = plan(2048, 2048, 2048, "f32", "f32")
    assert st == tg.TG_OK and p["block_k"] == 32
    assert p["pack_a"] == 0 and p["pack_b"] == 0          # B read in place, N-major
    assert p["workspace_bytes"] == 0 and p["kernels"] == 1
    # 777 and 1999 floats are not 16-byte pitches: both operands are packed
    st, p = plan(1000, 1999, 777, "f32", "f32")
    assert st == tg.TG_OK and p["pack_a"] == 1 and p["pack_b"] == 1
    assert p["workspace_bytes"] >= 1000 * 780 * 4 + 777 * 2000 * 4


@pytest.mark.parametrize("M", [1, 16, 64])
def test_plan_skinny_splits_k(lib, M):
    st, p = plan(M, 8192, 8192, sms=148)
    assert st == tg.TG_OK
    assert p["path"] == tg.TG_PATH_SKINNY and p["block_n"] in (128, 256, 512)
    assert p["block_m"] == {1: 16, 16: 16, 64: 64}[M]
    assert p["tiles"] == 8192 // p["block_n"] and p["splits"] in (2, 4, 8)
    # one CTA per unit, all resident at once (two per SM when there are more
    # units than SMs), with the largest cluster that allows that
    assert p["ctas"] == p["tiles"] * p["splits"] <= 2 * 148
    assert p["ctas"] * 2 > 2 * 148 or p["splits"] == 8
    assert p["workspace_bytes"] == 0 and p["kernels"] == 1  # partials summed on chip


def test_plan_skinny_tile_widths(lib):
    for bn in (128, 256, 512):
        st, p = plan(16, 4096, 4096, path=tg.TG_PATH_SKINNY, block_n=bn)
        assert st == tg.TG_OK and p["block_n"] == bn and p["tiles"] == 4096 // bn
    st, _ = plan(128, 4096, 4096, path=tg.TG_PATH_SKINNY, block_n=512)   # 128x512 FP32 partial
    assert st == tg.TG_ERR_UNSUPPORTED
    st, _ = plan(16, 4096, 4096, path=tg.TG_PATH_SKINNY, block_n=192)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_plan_skinny_cluster_limits(lib):
    st, p = plan(16, 4096, 4096, path=tg.TG_PATH_SKINNY, splits=8)
    assert st == tg.TG_OK and p["splits"] == 8
    for s in (3, 5, 16):
        st, _ = plan(16, 4096, 4096, path=tg.TG_PATH_SKINNY, splits=s)
        assert st == tg.TG_ERR_UNSUPPORTED
    st, _ = plan(16, 4096, 64, path=tg.TG_PATH_SKINNY, splits=2)   # one K tile: empty range
    assert st == tg.TG_ERR_UNSUPPORTED
    st, p = plan(16, 4096, 64, sms=148)                           # planner keeps 1 range
    assert st == tg.TG_OK and p["splits"] == 1


def test_plan_forced_options(lib):
    st, p = plan(512, 512, 512, splits=3, block_n=128, group_m=4, max_ctas=7, path=tg.TG_PATH_TC)
    assert st == tg.TG_OK
    assert (p["splits"], p["block_n"], p["group_m"], p["ctas"]) == (3, 128, 4, 7)
    st, p = plan(512, 512, 512, max_ctas=1)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC and p["ctas"] == 1
    st, p = plan(1024, 1024, 512, path=tg.TG_PATH_TC_PAIR, block_n=128, max_ctas=10)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC_PAIR and p["block_m"] == 256
    assert p["ctas"] == 10 and p["tiles"] == 4 * 8


def test_plan_multicast_rules(lib):
    st, p = plan(4096, 4096, 4096, multicast=2, block_n=256, sms=148)
    assert st == tg.TG_OK and p["multicast"] == 2 and p["ctas"] % 4 == 0
    st, p = plan(4096, 4096, 4096, multicast=1, sms=148)
    assert st == tg.TG_OK and p["multicast"] == 1
    # pairs share A in clusters of two pairs (192, 224, 256) and may split K;
    # a few-row product asked to share A goes to the pair kernel
    st, p = plan(4096, 4096, 4096, multicast=2, splits=2, sms=148)
    assert st == tg.TG_OK and p["splits"] == 2 and p["multicast"] == 2
    st, p = plan(64, 8192, 8192, multicast=2, sms=148)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC_PAIR and p["multicast"] == 2
    for bad in (dict(multicast=2, path=tg.TG_PATH_TC), dict(multicast=2, path=tg.TG_PATH_TC,
                                                             block_n=128),
                dict(multicast=2, path=tg.TG_PATH_TC_PAIR, block_n=128),
                dict(multicast=2, block_n=512), dict(multicast=2, path=tg.TG_PATH_SKINNY)):
        st, _ = plan(4096, 4096, 4096, **bad)
        assert st == tg.TG_ERR_UNSUPPORTED, bad
    st, _ = plan(4096, 4096, 4096, multicast=3)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_plan_width_limits(lib):
    for bn in (128, 192, 224, 256, 512):
        st, p = plan(512, 512, 512, path=tg.TG_PATH_TC_PAIR, block_n=bn)
        assert st == tg.TG_OK and p["block_n"] == bn
    st, _ = plan(512, 512, 512, path=tg.TG_PATH_TC_PAIR, block_n=160)
    assert st == tg.TG_ERR_UNSUPPORTED
    st, _ = plan(512, 512, 512, path=tg.TG_PATH_SKINNY)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_plan_prefers_pairs_for_large_and_single_ctas_for_skinny(lib):
    for M, N, K in [(8192, 8192, 8192), (8192, 14336, 4096), (8192, 4096, 14336)]:
        st, p = plan(M, N, K, "bf16", sms=148)
        assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC_PAIR
    st, p = plan(16, 8192, 8192, sms=148)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY
    st, p = plan(16, 8192, 8192, "f32", sms=148)          # TF32: no small-M kernel
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC
    st, _ = plan(129, 512, 512, path=tg.TG_PATH_SKINNY)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_plan_zero_sizes(lib):
    st, p = plan(0, 5, 5)
    assert st == tg.TG_OK and p["kernels"] == 0
    st, p = plan(5, 5, 0, lda=0)
    assert st == tg.TG_OK and p["kernels"] == 0


def test_python_gemm_checks_shapes():
    torch = pytest.importorskip("torch")
    a = torch.zeros(3, 4, dtype=torch.float16)
    b = torch.zeros(5, 2, dtype=torch.float16)
    with pytest.raises(ValueError):
        tg.gemm(a, b)
    with pytest.raises(ValueError):   # CPU tensors are refused: no CPU path exists
        tg.gemm(a, torch.zeros(4, 2, dtype=torch.float16))


def test_selftest_timeout_argument_range(lib):
    # rejected on the host, before any device call
    assert tg.tg_selftest_timeout(0, 0) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_selftest_timeout(10001, 0) == tg.TG_ERR_INVALID_VALUE


@pytest.mark.parametrize("opts", [dict(path=tg.TG_PATH_TC_PAIR, max_ctas=1),
                                  dict(multicast=2, max_ctas=1),
                                  dict(path=tg.TG_PATH_TC_PAIR, block_n=256, multicast=2,
                                       max_ctas=2)])
def test_options_that_exclude_every_variant(lib, opts):
    # no kernel variant fits: refused on the host, nothing planned or launched
    st, _ = plan(2048, 2048, 2048, **opts)
    assert st == tg.TG_ERR_UNSUPPORTED
    o = tg.make_options(**opts)
    st, _ = tg.tg_plan_gemm_strided_batched(4, 1024, 1024, 1024, A, 1024, 1024 * 1024, B, 1024,
                                             1024 * 1024, C, 1024, 1024 * 1024, "f16", "f16",
                                             148, o)
    assert st == tg.TG_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,din", [(65, "f16"), (128, "f16"), (128, "bf16"), (33, "e4m3"),
                                   (128, "e4m3")])
def test_plan_small_m_up_to_128_rows(lib, M, din):
    # up to 128 rows, 16-bit and FP8 alike: the transposed streaming kernel,
    # 128 columns per CTA, a cluster K split summed on chip
    st, p = plan(M, 8192, 8192, din, "f16" if din == "e4m3" else din, sms=148)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_SKINNY
    assert p["block_n"] == 128 and p["splits"] >= 2 and p["workspace_bytes"] == 0
    assert p["block_m"] == (64 if M <= 64 else 128)
    # the tile kernel can still be forced
    st, p = plan(M, 8192, 8192, din, "f16" if din == "e4m3" else din, sms=148,
                 path=tg.TG_PATH_TC)
    assert st == tg.TG_OK and p["path"] == tg.TG_PATH_TC
    # 129 rows: no longer the small-M kernel
    st, p = plan(129, 8192, 8192, din, "f16" if din == "e4m3" else din, sms=148)
    assert st == tg.TG_OK and p["path"] != tg.TG_PATH_SKINNY


def test_noalloc_argument_errors_on_the_host(lib):
    """tg_gemm_splitk_noalloc rejects bad arguments before it touches a device
    (the device array's set-up comes after these checks), and an empty output
    is a no-op.  Only calls that stop before any device work are made here."""
    call = tg.tg_gemm_splitk_noalloc
    ok = dict(M=256, N=512, K=1024, lda=1024, ldb=512, ldc=512)

    def st(splits=2, din="f16", dout="f16", a=A, b=B, c=C, **kw):
        d = dict(ok, **kw)
        return call(d["M"], d["N"], d["K"], a, d["lda"], b, d["ldb"], c, d["ldc"], din, dout,
                    splits, 0)

    assert st(splits=0) == tg.TG_ERR_INVALID_VALUE
    assert st(splits=129) == tg.TG_ERR_INVALID_VALUE
    assert st(din="f32", dout="f32") == tg.TG_ERR_UNSUPPORTED        # TF32 needs B^T
    assert st(din="e4m3", dout="f16") == tg.TG_ERR_UNSUPPORTED
    assert st(din="f16", dout="bf16") == tg.TG_ERR_UNSUPPORTED       # not a type pair
    assert st(M=-1) == tg.TG_ERR_INVALID_VALUE
    assert st(lda=1000) == tg.TG_ERR_INVALID_VALUE                   # lda < K
    assert st(ldc=500) == tg.TG_ERR_INVALID_VALUE                    # ldc < N
    assert st(a=0) == tg.TG_ERR_INVALID_VALUE
    assert st(c=A + 64) == tg.TG_ERR_INVALID_VALUE                   # C overlaps A
    assert st(M=0) == tg.TG_OK and st(N=0) == tg.TG_OK               # nothing to do


def test_host_operand_call_argument_errors_on_the_host(lib):
    """tg_gemm_host applies tg_gemm's argument rules to its host pointers
    before it stages anything, and an empty output is a no-op.  Only calls
    that stop before any device work are made here."""
    call = tg.tg_gemm_host

    def st(M=300, N=200, K=100, lda=100, ldb=200, ldc=200, din="f16", dout="f16", a=A, b=B,
           c=C, options=None):
        return call(M, N, K, a, lda, b, ldb, c, ldc, din, dout, 0, options)

    assert st(K=-1) == tg.TG_ERR_INVALID_VALUE
    assert st(ldb=199) == tg.TG_ERR_INVALID_VALUE
    assert st(din="bf16", dout="f16") == tg.TG_ERR_UNSUPPORTED
    assert st(b=0) == tg.TG_ERR_INVALID_VALUE
    assert st(c=B + 16) == tg.TG_ERR_INVALID_VALUE                   # C overlaps B
    assert st(options=tg.make_options(multicast=3)) == tg.TG_ERR_INVALID_VALUE
    assert st(M=0) == tg.TG_OK and st(N=0) == tg.TG_OK


def test_every_declaration_cites_its_passage_or_says_it_has_none():
    """Each entry point's comment in the header names the page passage that
    defines what it computes, or states that the pages have no counterpart."""
    text = open(HEADER).read()
    pages = ("teenygrad", "llm-systems-cookbook", "triton-cuda-lab", "Fast matrix multiplication")
    for name in declared_functions():
        decl = re.search(r"\n(?:tg_status\s+|const char\s*\*\s*|int32_t\s+)" + name + r"\s*\(", text)
        assert decl, name
        comment = text[:decl.start()].rsplit("/*", 1)[1]
        assert "*/" in comment and text[:decl.start()].rstrip().endswith("*/"), name
        assert any(p in comment for p in pages) or \
            ("counterpart" in comment and "pages" in comment), name
