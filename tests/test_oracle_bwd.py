"""The oracle's backward pass against its pins (finite differences of the
pinned forward, exact linearity identities, torch.autograd), and planted
mistakes in it that some pin must catch (CPU only)."""
import os

import pytest

import oracle
from tests import pins

SRC = open(oracle.SRC).read()

MUTATIONS = {
    "dA_series_term_sign": [("(dt * abar * hp + dq_da(dt, a) * bt * ut)", "(dt * abar * hp - dq_da(dt, a) * bt * ut)")],
    "adjoint_not_decayed": [("lam[n] *= abar;", "lam[n] *= 1.0;")],
    "dC_from_previous_state": [("dC[r] += ds * ht;", "dC[r] += ds * hp;")],
    "softplus_derivative_dropped": [("const double dd = ddt * sigmoid_of(pre);", "const double dd = ddt;")],
    "silu_derivative_wrong": [("sg * (1.0 + zt * (1.0 - sg))", "sg")],
    "dt_input_term_dropped": [("ddt += lam[n] * abar * (a * hp + bt * ut);", "ddt += lam[n] * abar * (a * hp);")],
    "dq_da_small_limit_wrong": [("return dt * dt * (0.5 + x *", "return dt * dt * (1.0 + x *")],
    "dB_without_coefficient": [("dB[r] += lam[n] * q * ut;", "dB[r] += lam[n] * ut;")],
    "readout_not_added_to_adjoint": [("lam[n] += ds * load_elem(C, r, dtype);\n", "")],
}


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.BWD_PINS, ids=lambda f: f.__name__)
def test_bwd_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_bwd_mistake_is_caught(tmp_path, name):
    src = SRC
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation {name}: pattern not unique: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(str(tmp_path), f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    mlib = oracle.load(oracle.build(src=path, out=os.path.join(str(tmp_path), f"lib_{name}.so")))
    caught = []
    for pin in pins.BWD_PINS:
        try:
            pin(mlib)
        except (AssertionError, ValueError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every backward pin"
