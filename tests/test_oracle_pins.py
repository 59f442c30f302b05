"""The float64 oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_tiny_workload_time_invariant_matches_convolution(lib):
    """The tiny fp32 workload's time-invariant variant (2x256x64, N=16, the
    workload generator's own inputs) equals its convolution form
    y_t = silu(z_t) (sum_k K_k[d] u_{t-k} + D u_t), K_k[d] = sum_n C_n Abar^k Bbar."""
    import numpy as np
    from selective_state_space_113_b300 import workloads as wl
    inp = wl.make_scan_inputs(wl.TINY_F32_LTI, device="cpu")
    p = {k: (None if v is None else oracle.bits_of(v)) for k, v in inp.items()}
    y, _ = oracle.scan_fwd(p["u"], p["delta"], p["dt_bias"], p["A"], p["B"], p["C"],
                           p["Dskip"], p["z"], dtype=oracle.F32, lib=lib)
    batch, L, D = p["u"].shape
    k = np.arange(L)
    for b in range(batch):
        for d in range(D):
            dt = float(pins.softplus_ref(np.float64(p["delta"][b, 0, d]) + np.float64(p["dt_bias"][d])))
            K = np.zeros(L)
            for n in range(p["A"].shape[1]):
                ad, bd = pins.zoh_ref(float(p["A"][d, n]), dt)
                K += float(p["C"][b, 0, n]) * ad ** k * bd * float(p["B"][b, 0, n])
            us = p["u"][b, :, d].astype(np.float64)
            conv = np.convolve(K, us)[:L]
            want = (conv + float(p["Dskip"][d]) * us) * pins.silu_ref(p["z"][b, :, d])
            pins._close(y[b, :, d], want, 1e-9, 1e-11, f"tiny LTI b={b} d={d}")
