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
