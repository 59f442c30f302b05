"""The SSD (Mamba-2) form of the oracle against its pins, and planted mistakes
in its channel mapping that some pin must catch (CPU only)."""
import inspect

import numpy as np
import pytest

import oracle
from tests import pins

MUTATIONS = {
    "heads_tiled_not_repeated": [("np.repeat(np.asarray(A, np.float32), P)", "np.tile(np.asarray(A, np.float32), P)")],
    "bias_tiled_not_repeated": [("np.repeat(np.asarray(dt_bias, np.float32), P)", "np.tile(np.asarray(dt_bias, np.float32), P)")],
    "skip_dropped": [("skip = None if Dskip is None else", "skip = None if True else")],
    "zero_order_hold_instead_of_euler": [("None, EULER, dtype=dtype", "None, ZOH, dtype=dtype")],
}


def _mutant(name):
    src = inspect.getsource(oracle.ssd_fwd)
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation {name}: pattern not unique: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(oracle))
    exec(compile(src, f"<mutant {name}>", "exec"), ns)
    return ns["ssd_fwd"]


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.SSD_PINS, ids=lambda f: f.__name__)
def test_ssd_pin(lib, pin):
    pin(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_ssd_mistake_is_caught(lib, name):
    fn = _mutant(name)
    caught = []
    for pin in pins.SSD_PINS:
        try:
            pin(lib, ssd=fn)
        except (AssertionError, ValueError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every SSD pin"
