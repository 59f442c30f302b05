"""The oracle's discretisation variants (zero-order hold, Euler, trapezoid)
against their pins, and planted mistakes in them that some pin must catch
(CPU only)."""
import os

import pytest

import oracle
from tests import pins

SRC = open(oracle.SRC).read()

MUTATIONS = {
    "trapezoid_without_decay_on_previous": [("0.5 * dt * (qt + abar * q[n])", "0.5 * dt * (qt + q[n])")],
    "trapezoid_full_weight": [("0.5 * dt * (qt + abar * q[n])", "dt * (qt + abar * q[n])")],
    "trapezoid_previous_never_kept": [("            q[n] = qt;\n", "")],
    "euler_as_zoh": [("h[n] = abar * h[n] + dt * qt;", "h[n] = abar * h[n] + expm1(dt * a) / a * qt;")],
    "euler_previous_input": [("h[n] = abar * h[n] + dt * qt;", "h[n] = abar * h[n] + dt * q[n];")],
}


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.DISC_PINS, ids=lambda f: f.__name__)
def test_disc_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_disc_mistake_is_caught(tmp_path, name):
    src = SRC
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation {name}: pattern not unique: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(str(tmp_path), f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    mlib = oracle.load(oracle.build(src=path, out=os.path.join(str(tmp_path), f"lib_{name}.so")))
    caught = []
    for pin in pins.DISC_PINS:
        try:
            pin(mlib)
        except (AssertionError, ValueError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every discretisation pin"
