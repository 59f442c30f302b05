"""The oracle's convolution prologue against its pins, and planted mistakes in
it that some pin must catch (CPU only)."""
import os

import pytest

import oracle
from tests import pins

SRC = open(oracle.SRC).read()

MUTATIONS = {
    "anti_causal": [("int64_t ts = t - 3 + k;", "int64_t ts = t + k;")],
    "weights_reversed": [("(double)conv_w[d * 4 + k] * load_elem(x,", "(double)conv_w[d * 4 + 3 - k] * load_elem(x,")],
    "silu_dropped": [("const double ut = act ? v / (1.0 + exp(-v)) : v;", "const double ut = v;")],
    "bias_ignored": [("const double cb = conv_b ? (double)conv_b[d] : 0.0;", "const double cb = 0.0;")],
    "history_off_by_one": [("int64_t ts = t - 3 + k;", "int64_t ts = t - 4 + k;")],
}


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.CONV_PINS, ids=lambda f: f.__name__)
def test_conv_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_conv_mistake_is_caught(tmp_path, name):
    src = SRC
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation {name}: pattern not unique: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(str(tmp_path), f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    mlib = oracle.load(oracle.build(src=path, out=os.path.join(str(tmp_path), f"lib_{name}.so")))
    caught = []
    for pin in pins.CONV_PINS:
        try:
            pin(mlib)
        except (AssertionError, ValueError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every convolution pin"
