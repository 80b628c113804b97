"""Host-side logic of bench.py that needs no GPU: the key under which the
committed DRAM-traffic figures are stored (the kernel code, comments
stripped) and the lookup that drops a figure once that code has changed."""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_strips_comments_but_not_literals():
    src = ('int a = 1; // trailing\n'
           '/* a block\n   over two lines */ int b = 2;\n'
           'const char *s = "// kept: inside a string";\n'
           "char q = '/';\n"
           '\n'
           'int c; /* inline */ int d;\n')
    got = bench._code_only(src)
    assert "trailing" not in got and "block" not in got and "inline" not in got
    assert '"// kept: inside a string"' in got and "'/'" in got
    assert got.splitlines() == ["int a = 1;", " int b = 2;",
                                'const char *s = "// kept: inside a string";',
                                "char q = '/';", "int c;  int d;"]


def test_code_only_escapes_in_literals():
    src = 'const char *s = "a \\" // b"; int x; // gone\n'
    assert bench._code_only(src) == 'const char *s = "a \\" // b"; int x;'


def test_traffic_lookup_follows_the_code_hash(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "w_same": {"source_sha": sha, "dram_bytes_per_launch": 123},
        "w_old": {"source_sha": "0" * 16, "dram_bytes_per_launch": 456}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the kernel sources are read from the package next to ROOT: point back
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    assert bench.profiled_traffic("w_same") == 123
    assert bench.profiled_traffic("w_old") is None
    assert bench.profiled_traffic("missing") is None


def test_every_bench_workload_plans_on_the_host():
    """Each workload bench.py can time gets a valid plan from the host-only
    planner (152 SMs): the small-M kernel at most 128 rows, the tile kernel
    otherwise, one launch per batch where the batch allows it, and no
    operand packing except where a row pitch is not a 16-byte multiple."""
    import tiled_matrix_multiplication_gb300 as tg
    from tiled_matrix_multiplication_gb300 import build as tgbuild
    tgbuild.build()
    tg.load()
    for name, (M, N, K, din, dout, _dist, _desc) in bench.WORKLOADS.items():
        opts = dict(bench.WORKLOAD_OPTS.get(name, {}))
        batch = bench.BATCH.get(name, 1)
        if batch > 1:
            p = tg.plan_batched(batch, M, N, K, din, dout, num_sms=152, **opts)
            assert p["per_batch"] == 0, name
        else:
            p = tg.plan(M, N, K, din, dout, num_sms=152, **opts)
        want_skinny = M <= 128
        assert (p["path"] == tg.TG_PATH_SKINNY) == want_skinny, (name, p)
        aligned = (K * bench.ESIZE[din]) % 16 == 0 and (N * bench.ESIZE[din]) % 16 == 0
        if aligned and not opts.get("f32_mode"):
            assert p["pack_a"] == 0 and p["pack_b"] == 0, (name, p)
        assert p["ctas"] >= 1 and p["tiles"] >= 1, (name, p)
    # the default workload is the A-multicast pair kernel the profiles describe
    M, N, K, din, dout = bench.WORKLOADS[bench.DEFAULT_WORKLOAD][:5]
    p = tg.plan(M, N, K, din, dout, num_sms=152)
    assert (p["path"], p["block_n"], p["multicast"]) == (tg.TG_PATH_TC_PAIR, 256, 2)
