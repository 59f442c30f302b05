"""Full-size parity of the variants on the Mamba-2.8B-shaped layer (batch 4,
L 4096, D 5120, N 16, bf16), the workload and launch plan (chained) the
benchmark times them on: the Euler and trapezoidal input terms and the
convolution prologue with SiLU, on sampled channels against the oracle."""
import pytest
import torch

from selective_state_space_113_b300 import workloads as wl
from tests import parity
from tests import test_gpu_conv as gc
from tests import test_gpu_disc as gd

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _channels(inp, b, idx):
    return {k: (None if v is None else
                (v[b:b + 1].index_select(2, idx) if k in ("u", "delta", "z") else
                 v[b:b + 1] if k in ("B", "C") else v.index_select(0, idx)))
            for k, v in inp.items()}


def _check(y, h, inp, oracle_of, what):
    batch, L, D = inp["u"].shape
    chans = parity.sample_channels(batch, D, 16, seed=5)
    tol = parity.TOL[inp["u"].dtype]
    for b in sorted({c[0] for c in chans}):
        idx = torch.tensor(sorted({c[1] for c in chans if c[0] == b}), device=DEV)
        y_ref, h_ref = oracle_of(_channels(inp, b, idx))
        parity.check(parity.to_f64(y[b].index_select(1, idx)), y_ref[0], tol, f"{what} y b={b}")
        parity.check(parity.to_f64(h[b].index_select(0, idx)), h_ref[0], tol, f"{what} h b={b}")


@pytest.mark.parametrize("disc", ["euler", "trapezoid"])
def test_disc_mamba2p8b_sampled(disc):
    inp = wl.make_scan_inputs(wl.MAMBA_2P8B, device=DEV)
    y, h = gd.run_disc(inp, gd.DISCS[disc])
    _check(y, h, inp, lambda q: gd.oracle_disc(q, gd.DISCS[disc]), disc)


def test_conv_silu_mamba2p8b_sampled():
    inp = gc.inputs(wl.MAMBA_2P8B)
    y, h = gc.run_conv(inp, 1)
    _check(y, h, inp, lambda q: gc.oracle_conv(q, 1), "conv+silu")
