"""Pins for the fused-epilogue reference (oracle/epilogue.py), each tying it to
mathematics or to an independent library routine, never to itself; and a
mutant battery: plausible mistakes planted in a copy of its source must each
fail at least one pin.  CPU only.

* the activations: values at a few points worked by hand; the odd-part
  identity act(x) - act(-x) = x that relu, silu and the GELU share; silu
  against scipy's logistic function; the tanh-form GELU within 5e-4 of the
  exact x * Phi(x) (math.erf), which a 10 % change of its cubic coefficient
  breaks; the tolerance's Lipschitz bounds against finite differences;
* the order of the steps on the pages' 2 x 2 worked example, with the
  epilogue's expected values worked by hand;
* special cases: the identity epilogue returns C unchanged; C = 0 leaves
  act(bias) + beta * R.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest

from oracle import epilogue as ep
from tests.conftest import parse_matrix, read_golden

SRC = ep.__file__


def worked_C():
    g = read_golden("worked_example.txt")
    return np.array(parse_matrix(g["C"]), dtype=np.float64)   # [[58, 64], [139, 154]]


def pin_hand_values(mod) -> bool:
    x = np.array([-2.0, -0.0, 0.0, 3.0])
    relu_ok = np.array_equal(mod.activation(x, "relu"), [0.0, 0.0, 0.0, 3.0])
    # silu(0) = 0, silu(ln 3) = ln 3 * 3/4 (sigmoid(ln 3) = 3/4)
    s = mod.activation(np.array([0.0, math.log(3.0)]), "silu")
    silu_ok = s[0] == 0.0 and abs(s[1] - 0.75 * math.log(3.0)) < 1e-15
    # GELU(0) = 0 and GELU'(0) = 1/2 (central difference)
    h = 1e-6
    g = mod.activation(np.array([0.0, h, -h]), "gelu_tanh")
    gelu_ok = g[0] == 0.0 and abs((g[1] - g[2]) / (2 * h) - 0.5) < 1e-9
    return relu_ok and silu_ok and gelu_ok and np.array_equal(mod.activation(x, "none"), x)


def pin_odd_part(mod) -> bool:
    x = np.linspace(-9.0, 9.0, 1801)
    return all(np.allclose(mod.activation(x, a) - mod.activation(-x, a), x, rtol=0, atol=1e-12)
               for a in ("relu", "silu", "gelu_tanh"))


def pin_library_forms(mod) -> bool:
    from scipy.special import expit
    x = np.linspace(-30.0, 30.0, 6001)
    silu_ok = np.allclose(mod.activation(x, "silu"), x * expit(x), rtol=1e-14, atol=1e-300)
    exact = 0.5 * x * (1.0 + np.array([math.erf(v / math.sqrt(2.0)) for v in x]))
    gelu_ok = float(np.max(np.abs(mod.activation(x, "gelu_tanh") - exact))) < 5e-4
    return silu_ok and gelu_ok


def pin_lipschitz(mod) -> bool:
    x = np.linspace(-12.0, 12.0, 240001)
    ok = True
    for a in mod.ACTIVATIONS:
        d = np.max(np.abs(np.diff(mod.activation(x, a)) / np.diff(x)))
        ok &= bool(d <= mod.LIPSCHITZ[a] and d >= 0.97 * mod.LIPSCHITZ[a])
    return ok


def pin_worked_example(mod) -> bool:
    # alpha = 1/2, bias = (1, -100), relu, beta = 2, R = [[1, 2], [3, 4]]:
    #   pre = [[30, -68], [70.5, -23]] -> relu -> [[30, 0], [70.5, 0]] -> + 2R
    C = worked_C()
    D, pre = mod.epilogue_ref(C, alpha=0.5, bias=[1.0, -100.0], act="relu", beta=2.0,
                              R=np.array([[1.0, 2.0], [3.0, 4.0]]))
    ok = np.array_equal(pre, [[30.0, -68.0], [70.5, -23.0]])
    ok &= np.array_equal(D, [[32.0, 4.0], [76.5, 8.0]])
    # per-column scale (2, -1) with bias 0: [[116, -64], [278, -154]] -> relu
    D2, _ = mod.epilogue_ref(C, scale=[2.0, -1.0], act="relu")
    ok &= np.array_equal(D2, [[116.0, 0.0], [278.0, 0.0]])
    return bool(ok)


def pin_special_cases(mod) -> bool:
    rng = np.random.default_rng(3)
    C = rng.standard_normal((5, 7))
    D, _ = mod.epilogue_ref(C)
    ok = np.array_equal(D, C)
    bias = rng.standard_normal(7)
    R = rng.standard_normal((5, 7))
    D0, _ = mod.epilogue_ref(np.zeros((5, 7)), alpha=3.0, scale=rng.standard_normal(7),
                             bias=bias, act="silu", beta=-0.5, R=R)
    want = bias / (1.0 + np.exp(-bias))
    ok &= np.allclose(D0, want[None, :] - 0.5 * R, rtol=1e-15, atol=1e-15)
    return bool(ok)


def pin_tolerance_scale(mod) -> bool:
    # the bound grows with |alpha * scale| and with the activation's slope, and
    # reduces to about the GEMM rule for the identity epilogue
    C = np.array([[100.0]])
    S = np.array([[200.0]])
    t1 = mod.epilogue_tolerance(C, S, "f16", "f32")
    t2 = mod.epilogue_tolerance(C, S, "f16", "f32", alpha=4.0)
    t3 = mod.epilogue_tolerance(C, S, "f16", "f32", act="gelu_tanh")
    gemm = 2e-3 * 200.0
    return bool(gemm <= t1[0, 0] <= gemm * 1.01 and t2[0, 0] > 3.9 * gemm
                and t3[0, 0] > 1.1 * gemm)


PINS = [pin_hand_values, pin_odd_part, pin_library_forms, pin_lipschitz, pin_worked_example,
        pin_special_cases, pin_tolerance_scale]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin(ep)


def _mutant(old: str, new: str):
    text = open(SRC).read()
    assert text.count(old) == 1, old
    mod = types.ModuleType("epilogue_mutant")
    mod.__package__ = "oracle"
    mod.__file__ = os.path.join(os.path.dirname(SRC), "epilogue_mutant.py")
    exec(compile(text.replace(old, new), mod.__file__, "exec"), mod.__dict__)
    return mod


MUTANTS = {
    "relu_keeps_negatives": ('np.where(x > 0, x, 0.0)', 'np.where(x > 0, x, 0.1 * x)'),
    "silu_sign": ("x / (1.0 + np.exp(-x))", "x / (1.0 + np.exp(x))"),
    "gelu_no_half": ("return 0.5 * x * (1.0 + np.tanh(", "return x * (1.0 + np.tanh("),
    "gelu_cubic_coeff": ("0.044715 * x ** 3", "0.04 * x ** 3"),
    "gelu_sqrt_pi": ("math.sqrt(2.0 / math.pi)", "math.sqrt(1.0 / math.pi)"),
    "bias_after_activation": (
        "    D = activation(pre, act)\n",
        "    D = activation(pre - (np.asarray(bias, dtype=np.float64)[None, :] if bias is not None "
        "else 0.0), act) + (np.asarray(bias, dtype=np.float64)[None, :] if bias is not None "
        "else 0.0)\n"),
    "residual_before_activation": (
        "    D = activation(pre, act)\n    if R is not None:\n"
        "        D = D + float(beta) * np.asarray(R, dtype=np.float64)\n",
        "    if R is not None:\n        pre = pre + float(beta) * np.asarray(R, dtype=np.float64)\n"
        "    D = activation(pre, act)\n"),
    "scale_ignored": ("        pre = pre * np.asarray(scale, dtype=np.float64)[None, :]\n",
                      "        pass\n"),
    "alpha_ignored": ("    pre = float(alpha) * C_ref\n", "    pre = 1.0 * C_ref\n"),
    "beta_ignored": ("        D = D + float(beta) * np.asarray(R, dtype=np.float64)\n",
                     "        D = D + np.asarray(R, dtype=np.float64)\n"),
    "lipschitz_too_small": ('"gelu_tanh": 1.13}', '"gelu_tanh": 1.0}'),
    "tolerance_without_gain": ("    return (LIPSCHITZ[act] * gain * REL_TOL",
                               "    return (LIPSCHITZ[act] * REL_TOL"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = [p.__name__ for p in PINS if not p(mod)]
    assert failed, f"mutant {name} passes every pin"
