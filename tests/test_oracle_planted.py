"""Planted mistakes: each plausible error in the oracle must fail some pin.

Each case patches a copy of ``oracle/ssm_oracle.c`` (text substitution, in a
temporary directory), builds it with gcc and runs every pin against it.  A
mutation that no pin notices would mean the pins leave that part of the
oracle unpinned.  CPU only; the shipped oracle is never modified.
"""
import os

import pytest

import oracle
from tests import pins

SRC = open(oracle.SRC).read()

MUTATIONS = {
    "euler_input_matrix": [("*bcoef = (a == 0.0) ? dt : expm1(dt * a) / a;", "*bcoef = dt;")],
    "decay_sign": [("*abar = exp(dt * a);", "*abar = exp(-dt * a);")],
    "skip_dropped": [("        acc += dsk * ut;\n", "\n")],
    "skip_outside_gate": [(
        "        acc += dsk * ut;\n        if (z)\n            acc *= silu(load_elem(z, i_btd, dtype));\n",
        "        if (z)\n            acc *= silu(load_elem(z, i_btd, dtype));\n        acc += dsk * ut;\n")],
    "sigmoid_gate": [("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));")],
    "softplus_is_exp": [("return fmax(x, 0.0) + log1p(exp(-fabs(x)));", "return exp(x);")],
    "softplus_sign": [("log1p(exp(-fabs(x)))", "log1p(exp(fabs(x)))")],
    "readout_before_update": [(
        "            h[n] = abar * h[n] + bcoef * bt * ut;\n            acc += ct * h[n];\n",
        "            acc += ct * h[n];\n            h[n] = abar * h[n] + bcoef * bt * ut;\n")],
    "A_transposed": [("zoh(dt, (double)A[d * N + n], &abar, &bcoef);",
                      "zoh(dt, (double)A[n * D + d], &abar, &bcoef);", 2)],
    "B_previous_step": [("double bt = load_elem(B, (b * L + t) * N + n, dtype);",
                         "double bt = load_elem(B, (b * L + (t > 0 ? t - 1 : 0)) * N + n, dtype);")],
    "B_C_swapped": [("double bt = load_elem(B, (b * L + t) * N + n, dtype);\n"
                     "            double ct = load_elem(C, (b * L + t) * N + n, dtype);",
                     "double bt = load_elem(C, (b * L + t) * N + n, dtype);\n"
                     "            double ct = load_elem(B, (b * L + t) * N + n, dtype);")],
    "bf16_decode_shift": [("(uint32_t)bits16 << 16", "(uint32_t)bits16 << 15")],
    "dt_bias_ignored": [("double bias = dt_bias ? (double)dt_bias[d] : 0.0;\n    double dsk",
                         "double bias = 0.0;\n    double dsk")],
    "state_not_reset_per_channel": [("    for (int64_t n = 0; n < N; n++)\n        h[n] = 0.0;\n", "")],
    "y_wrong_time_index": [("        y[i_btd] = acc;",
                            "        y[(b * L + (t + 1) % L) * D + d] = acc;")],
    "h_last_wrong_layout": [("h_last[(b * D + d) * N + n] = h[n];",
                             "h_last[(d * (int64_t)0 + b * D * N) + n * D + d] = h[n];")],
    "step_state_index": [("double *hp = &state[i_bd * N + n];", "double *hp = &state[d * N + n];")],
    "step_bias_ignored": [("double bias = dt_bias ? (double)dt_bias[d] : 0.0;\n            double dt",
                           "double bias = 0.0;\n            double dt")],
    "step_gate_dropped": [("            if (z)\n                acc *= silu(load_elem(z, i_bd, dtype));\n", "")],
    "zero_A_limit_wrong": [("(a == 0.0) ? dt :", "(a == 0.0) ? 0.0 :")],
}


def _build(tmp_path, name, edits):
    src = SRC
    for old, new, *count in edits:
        want = count[0] if count else 1
        assert src.count(old) == want, f"mutation {name}: pattern count != {want}: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    return oracle.build(src=path, out=os.path.join(tmp_path, f"lib_{name}.so"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = oracle.load(_build(str(tmp_path), name, MUTATIONS[name]))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, RuntimeError, FloatingPointError) as e:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
