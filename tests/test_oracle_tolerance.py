"""Pins of the comparison rule (``oracle/compare.py``) and a battery of planted
mistakes in it.  CPU only.

The rule's constants are fixed two ways:
  * exactly, against the rule stated in ``tests/golden/tolerance_rule.txt``;
  * by what the arithmetic requires of any usable rule -- a correct FP32
    accumulation of exact products at the largest K, a TF32 operand
    conversion that truncates, and a correctly rounded BF16 or subnormal
    FP16 result must all pass; a kernel that drops one K tile of the
    tile kernel's ring (64 K elements of a 16-bit operand, 32 of TF32, 128
    of FP8) must fail, as must an FP32 result off by 2.5e-3 S.
A copy of compare.py with one plausible mistake planted (a looser or tighter
constant, the ulp term dropped or taken in the wrong format, the relative
term keyed by the output type) must fail at least one of these pins.
"""
from __future__ import annotations

import importlib.util
import os
import types

import numpy as np
import pytest

import oracle
from tests.conftest import read_golden

SRC = os.path.join(os.path.dirname(oracle.__file__), "compare.py")
RULE = read_golden("tolerance_rule.txt")
IN_TYPES = ("f16", "bf16", "e4m3", "e5m2", "f32")
OUT_OF = {"f16": ("f16", "f32"), "bf16": ("bf16", "f32"), "e4m3": ("f16", "bf16", "f32"),
          "e5m2": ("f16", "bf16", "f32"), "f32": ("f32",)}
# K elements in one 128-byte K row of a ring stage of the tile kernel
BK = {"f16": 64, "bf16": 64, "e4m3": 128, "e5m2": 128, "f32": 32}
K_MAX = int(RULE["k_max"])


def _passes(m, c, c_ref, s, din, dout) -> bool:
    ok, _ = m.check_close(np.array([[c]]), np.array([[c_ref]]), np.array([[s]]), din, dout)
    return ok


def pins(m: types.ModuleType) -> list[str]:
    """Runs every pin against the comparison module ``m``; returns the names
    of those that fail."""
    failed = []
    rng = np.random.default_rng(5)
    # 1. the exact form stated in the fixture, on random magnitudes
    for din in IN_TYPES:
        rel = float(RULE[f"rel_{din}"])
        for dout in OUT_OF[din]:
            c_ref = rng.standard_normal(64) * 10.0 ** rng.integers(-6, 4, 64)
            s = np.abs(c_ref) * (1.0 + rng.random(64) * 50)
            want = rel * s + float(RULE["ulp_coeff"]) * m.ulp(c_ref, dout)
            if not np.array_equal(m.tolerance(c_ref, s, din, dout), want):
                failed.append(f"exact_form_{din}_{dout}")
    # 2. accept: FP32 accumulation of K_MAX exact products, worst case, FP32 out
    for din in ("f16", "bf16", "e4m3", "e5m2"):
        if not _passes(m, 1.0 + K_MAX * 2.0 ** -24, 1.0, 1.0, din, "f32"):
            failed.append(f"accept_fp32_accumulation_{din}")
    # 3. accept: TF32 truncation of both operands (2^-10 each) plus accumulation
    if not _passes(m, 1.0 + 2 * 2.0 ** -10 + K_MAX * 2.0 ** -24, 1.0, 1.0, "f32", "f32"):
        failed.append("accept_tf32_truncation")
    # 4. accept: a correctly rounded BF16 result more than 2e-3 S from C_ref
    #    (C_ref just above the midpoint of 1 and 1 + 2^-7 rounds up)
    c_ref = 1.0 + 2.0 ** -8 + 2.0 ** -12
    for din in ("bf16", "e4m3", "e5m2"):
        if not _passes(m, 1.0 + 2.0 ** -7, c_ref, c_ref, din, "bf16"):
            failed.append(f"accept_rounded_bf16_{din}")
    # 5. accept: a result below FP16's subnormal spacing rounds to zero
    if not _passes(m, 0.0, 3 * 2.0 ** -26, 3 * 2.0 ** -26, "f16", "f16"):
        failed.append("accept_f16_subnormal_rounding")
    # 6. reject: one K tile of 64 dropped (all products positive, S = C_ref)
    for din in IN_TYPES:
        k = 64 * BK[din]
        for dout in OUT_OF[din]:
            if _passes(m, 1.0 - 1.0 / 64, 1.0, 1.0, din, dout):
                failed.append(f"reject_dropped_k_tile_{din}_{dout}")
        assert k >= BK[din]
    # 7. reject: TF32 with one of 32 K tiles dropped (3.1 % of S)
    if _passes(m, 1.0 - 1.0 / 32, 1.0, 1.0, "f32", "f32"):
        failed.append("reject_dropped_k_tile_tf32_of_32")
    # 8. reject: FP32 output off by 2.5e-3 S for 16-bit and 8-bit operands
    for din in ("f16", "bf16", "e4m3", "e5m2"):
        if _passes(m, 1.0 + 2.5e-3, 1.0, 1.0, din, "f32"):
            failed.append(f"reject_fp32_out_{din}")
    # 9. NaN never passes
    if _passes(m, float("nan"), 1.0, 1.0, "f16", "f16"):
        failed.append("reject_nan")
    # 10. the ulp term at textbook points of each format: the spacing of IEEE
    #     binary16 (10 fraction bits, smallest normal 2^-14, largest finite
    #     65504), bfloat16 (7 fraction bits, FP32's exponent range) and
    #     binary32 (23 fraction bits)
    textbook = [("f16", 1.0, 2.0 ** -10), ("f16", 1.999, 2.0 ** -10), ("f16", 65504.0, 32.0),
                ("f16", 2.0 ** -14, 2.0 ** -24), ("f16", 2.0 ** -20, 2.0 ** -24),
                ("f16", 0.0, 2.0 ** -24), ("bf16", 1.0, 2.0 ** -7), ("bf16", 3.0, 2.0 ** -6),
                ("bf16", 2.0 ** -126, 2.0 ** -133), ("bf16", 2.0 ** -130, 2.0 ** -133),
                ("f32", 1.0, 2.0 ** -23), ("f32", 1000.0, 2.0 ** -14),
                ("f32", 2.0 ** -140, 2.0 ** -149)]
    for fmt, x, want in textbook:
        if float(m.ulp(np.array([x]), fmt)[0]) != want:
            failed.append(f"ulp_{fmt}_{x}")
    return failed


def test_the_rule_passes_every_pin():
    assert pins(oracle.compare) == []


def test_fixture_values_are_consistent_with_the_arithmetic():
    # the accumulation bound at the largest K sits inside the 16-bit term,
    # truncated TF32 plus accumulation inside the TF32 term
    assert K_MAX * 2.0 ** -24 < float(RULE["rel_f16"])
    assert 2 * 2.0 ** -10 + K_MAX * 2.0 ** -24 < float(RULE["rel_f32"])
    assert all(float(RULE[f"rel_{t}"]) == float(RULE["rel_f16"]) for t in ("bf16", "e4m3", "e5m2"))


MUTANTS = {
    "tf32_loose": ('"f32": 1e-2', '"f32": 1e-1'),
    "tf32_tight": ('"f32": 1e-2', '"f32": 2e-3'),
    "bf16_loose": ('"bf16": 2e-3', '"bf16": 2e-2'),
    "f16_tight": ('"f16": 2e-3', '"f16": 5e-4'),
    "e4m3_loose": ('"e4m3": 2e-3', '"e4m3": 2e-2'),
    "e5m2_loose": ('"e5m2": 2e-3', '"e5m2": 1e-2'),
    "ulp_dropped": ("return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_out)",
                    "return REL_TOL[dtype_in] * S"),
    "ulp_of_input_type": ("return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_out)",
                          "return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_in if dtype_in in _FORMAT else dtype_out)"),
    "rel_keyed_by_output": ("return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_out)",
                            "return REL_TOL[dtype_out] * S + ulp(C_ref, dtype_out)"),
    "ulp_doubled": ("return REL_TOL[dtype_in] * S + ulp(C_ref, dtype_out)",
                    "return REL_TOL[dtype_in] * S + 2 * ulp(C_ref, dtype_out)"),
    "no_subnormal_clamp": ("e = np.where(ax > 0, np.maximum(e, emin), emin)",
                           "e = np.where(ax > 0, e, emin)"),
    "bf16_fraction_bits": ('"bf16": (-126, 7)', '"bf16": (-126, 8)'),
    "nan_passes": ("bad = ~(err <= tol)", "bad = err > tol"),
}


def _load_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the planted line is not in compare.py"
    path = tmp_path / f"compare_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"compare_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new, tmp_path)
    assert pins(mod), f"mutant {name} passes every pin"
