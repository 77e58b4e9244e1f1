"""Plant plausible slips in a copy of the oracle and check the pins catch them.

The copy is built from the oracle's source text with one replacement, loaded
as a separate module, and the pin battery of test_oracle_pins.py runs against
it.  Every mutant must fail at least one pin.  Nothing here touches the CUDA
path.
"""
import importlib.util
import os
import sys
import types

import pytest

import tests.test_oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "evo_oracle.py")).read()

MUTANTS = {
    "dropped_scale": ("x = s * (q @ k.T) + bias", "x = (q @ k.T) + bias"),
    "transposed_bias": ("x = s * (q @ k.T) + bias", "x = s * (q @ k.T) + bias.T"),
    "dropped_delta": ("ds = p * (dp - delta[:, None])", "ds = p * dp"),
    "dq_sign": ("dq = s * (ds @ k)", "dq = -s * (ds @ k)"),
    "dk_transposed": ("dk = s * (ds.T @ q)", "dk = s * (ds @ q)"),
    "dv_transposed": ("dv = p.T @ do", "dv = p @ do"),
    "dq_unscaled": ("dq = s * (ds @ k)", "dq = (ds @ k)"),
    "bias2_wrong_head": ("out = out + bias2[b, 0, h, :, :]", "out = out + bias2[b, 0, 0, :, :]"),
    "bias1_on_queries": ("out = out + bias1[b, n, 0, 0, :][None, :]",
                         "out = out + bias1[b, n, 0, 0, :][:, None]"),
    "lse_without_max": ("m_safe + np.log(np.where(empty, 1.0, l))", "np.log(np.where(empty, 1.0, l))"),
    "dbias1_wrong_axis": ('dbias1[b, n, 0, 0, :] += g["ds"].sum(axis=0)',
                          'dbias1[b, n, 0, 0, :] += g["ds"].sum(axis=1)'),
    "sample_dropped_delta": ("out += p * (dp - delta[:, None])", "out += p * dp"),
    "scale_sqrt_missing": ("return 1.0 / math.sqrt(D)", "return 1.0 / D"),
}


def load_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, name
    src = SRC.replace(old, new)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def battery():
    yield P.test_hand_derived_example
    yield lambda: P.test_torch_sdpa((1, 3, 16, 2, 8), True, True)
    yield lambda: P.test_finite_differences((1, 2, 5, 2, 3))
    yield P.test_sampled_helpers_match_full_oracle
    yield lambda: P.test_brute_force((2, 2, 4, 1, 3))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    mod = load_mutant(name)
    monkeypatch.setattr(P, "O", mod)
    caught = []
    for pin in battery():
        try:
            pin()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_copy_passes():
    mod = types.ModuleType("oracle_copy")
    exec(compile(SRC, "<copy>", "exec"), mod.__dict__)
    saved = P.O
    P.O = mod
    try:
        for pin in battery():
            pin()
    finally:
        P.O = saved
