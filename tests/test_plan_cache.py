"""The planner keeps the plans of recent calls (16, replaced round-robin):
repeating a query in any order, with entries evicted and recomputed in
between, must give exactly the plan of its first computation -- and queries
that differ only in an operand's 16-byte alignment, a pitch, a batch stride
or an option field must not share a plan.  Host only."""
from __future__ import annotations

import random

import pytest

import tiled_matrix_multiplication_gb300 as tg
from tiled_matrix_multiplication_gb300 import build as tgbuild

A, B, C = 0x10000, 0x100000000, 0x200000000


@pytest.fixture(scope="module")
def lib():
    tgbuild.build()
    return tg.load()


def query(M, N, K, din="f16", dout=None, a=A, b=B, c=C, lda=None, ldb=None, ldc=None, sms=148,
          **opts):
    dout = din if dout is None else dout
    o = tg.make_options(**opts) if opts else None
    st, p = tg.tg_plan_gemm(M, N, K, a, K if lda is None else lda, b, N if ldb is None else ldb,
                            c, N if ldc is None else ldc, din, dout, sms, o)
    assert st == tg.TG_OK
    return p


QUERIES = [
    dict(M=4096, N=4096, K=4096), dict(M=4096, N=4096, K=4096, sms=152),
    dict(M=4096, N=4096, K=4096, multicast=1), dict(M=4096, N=4096, K=4096, block_n=512),
    dict(M=4096, N=4096, K=4096, a=A + 8), dict(M=4096, N=4096, K=4096, c=C + 2),
    dict(M=4096, N=4096, K=4096, lda=4100), dict(M=4096, N=4096, K=4096, ldb=4097),
    dict(M=127, N=255, K=65, dout="f32"), dict(M=127, N=255, K=65, dout="f32", splits=2),
    dict(M=1, N=8192, K=8192), dict(M=64, N=8192, K=8192), dict(M=128, N=8192, K=8192),
    dict(M=128, N=8192, K=8192, multicast=1), dict(M=128, N=8192, K=8192, splits=4),
    dict(M=2048, N=2048, K=2048, din="f32"), dict(M=2048, N=2048, K=2048, din="f32", f32_mode=1),
    dict(M=1000, N=1999, K=777, din="f32"), dict(M=4096, N=4096, K=4096, din="e4m3", dout="f16"),
    dict(M=8192, N=14336, K=4096, din="bf16"), dict(M=300, N=520, K=200, path=tg.TG_PATH_TC),
    dict(M=300, N=520, K=200, path=tg.TG_PATH_TC_PAIR), dict(M=300, N=520, K=200, max_ctas=4),
    dict(M=300, N=520, K=200, group_m=4), dict(M=300, N=520, K=200, timeout_ms=100),
    dict(M=512, N=512, K=512, splits=3, path=tg.TG_PATH_TC),
    dict(M=1024, N=4096, K=4096), dict(M=16, N=1024, K=512), dict(M=37, N=1000, K=700),
]


def test_plans_do_not_depend_on_the_order_of_queries(lib):
    first = [query(**q) for q in QUERIES]   # more distinct queries than cache entries
    rng = random.Random(7)
    for _ in range(3):
        order = list(range(len(QUERIES)))
        rng.shuffle(order)
        for i in order:
            assert query(**QUERIES[i]) == first[i], QUERIES[i]


def test_queries_that_differ_get_their_own_plan(lib):
    base = query(4096, 4096, 4096)
    assert query(4096, 4096, 4096, a=A + 8)["pack_a"] == 1 and base["pack_a"] == 0
    assert query(4096, 4096, 4096, b=B + 4)["pack_b"] == 1 and base["pack_b"] == 0
    assert query(4096, 4096, 4096, c=C + 2)["c_vector"] == 0 and base["c_vector"] == 1
    assert query(4096, 4096, 4096, multicast=1)["multicast"] == 1
    assert query(4096, 4096, 4096, group_m=4)["group_m"] == 4 and base["group_m"] == 8
    assert query(4096, 4096, 4096)["group_m"] == 8
