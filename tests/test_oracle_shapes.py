"""The oracle over random small shapes, including the degenerate ones
(L = 1, N = 1, D = 1, batch = 1): the forward and its Euler and trapezoid
variants against brute-force unrolling, the backward against torch.autograd,
the SSD form against its masked matrix products, the convolution against
numpy.convolve and the decode step against library routines (CPU only)."""
import numpy as np
import pytest
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@settings(max_examples=40, deadline=None)
@given(batch=st.integers(1, 3), L=st.integers(1, 12), D=st.integers(1, 5), N=st.integers(1, 9),
       seed=st.integers(0, 2**31 - 1))
def test_forward_against_unrolling(lib, batch, L, D, N, seed):
    pins.bruteforce_check(lib, np.random.default_rng(seed), batch, L, D, N)


@settings(max_examples=20, deadline=None)
@given(batch=st.integers(1, 2), L=st.integers(1, 8), D=st.integers(1, 4), N=st.integers(1, 7),
       seed=st.integers(0, 2**31 - 1))
def test_backward_against_autograd(lib, batch, L, D, N, seed):
    pins.bwd_against_autograd(lib, batch, L, D, N, seed)


def _variant_unrolled(p, disc):
    """y and h_last of the Euler (disc 1) or trapezoidal (disc 2) input term
    by the brute-force sum h_t = sum_{s<=t} (prod_{r=s+1..t} Abar_r) v_s, with
    Abar_r = exp(dt_r a) from scipy's ZOH and v_s = dt_s B_s u_s (Euler) or
    dt_s / 2 (B_s u_s + Abar_s B_{s-1} u_{s-1}) (trapezoid, 0 before step 0)."""
    batch, L, D = p["u"].shape
    N = p["A"].shape[1]
    y = np.zeros((batch, L, D))
    h_last = np.zeros((batch, D, N))
    for b in range(batch):
        for d in range(D):
            dts = pins.softplus_ref(p["delta"][b, :, d].astype(np.float64)
                                    + np.float64(p["dt_bias"][d]))
            u = p["u"][b, :, d].astype(np.float64)
            hs = np.zeros((L, N))
            for n in range(N):
                ab = [pins.zoh_ref(float(p["A"][d, n]), float(dt))[0] for dt in dts]
                bu = p["B"][b, :, n].astype(np.float64) * u
                v = [dts[s] * bu[s] if disc == 1 else
                     dts[s] / 2 * (bu[s] + (ab[s] * bu[s - 1] if s > 0 else 0.0))
                     for s in range(L)]
                for t in range(L):
                    hs[t, n] = sum(np.prod(ab[s + 1:t + 1]) * v[s] for s in range(t + 1))
            y[b, :, d] = ((p["C"][b].astype(np.float64) * hs).sum(1)
                          + float(p["Dskip"][d]) * u) * pins.silu_ref(p["z"][b, :, d])
            h_last[b, d] = hs[-1]
    return y, h_last


@settings(max_examples=30, deadline=None)
@given(disc=st.sampled_from([oracle.EULER, oracle.TRAPEZOID]), batch=st.integers(1, 2),
       L=st.integers(1, 10), D=st.integers(1, 4), N=st.integers(1, 6),
       seed=st.integers(0, 2**31 - 1))
def test_variants_against_unrolling(lib, disc, batch, L, D, N, seed):
    p = pins.random_problem(np.random.default_rng(seed), batch, L, D, N)
    y, h = oracle.scan_fwd_disc(p["u"], p["delta"], p["dt_bias"], p["A"], p["B"], p["C"],
                                p["Dskip"], p["z"], disc, dtype=oracle.F32, lib=lib)
    want_y, want_h = _variant_unrolled(p, disc)
    pins._close(y, want_y, 1e-10, 1e-12, f"disc {disc} y")
    pins._close(h, want_h, 1e-10, 1e-12, f"disc {disc} h_last")


@settings(max_examples=25, deadline=None)
@given(batch=st.integers(1, 2), L=st.integers(1, 20), H=st.integers(1, 3), P=st.integers(1, 5),
       N=st.integers(1, 9), seed=st.integers(0, 2**31 - 1))
def test_ssd_against_masked_matmul(lib, batch, L, H, P, N, seed):
    pins.ssd_masked_matmul_check(lib, np.random.default_rng(seed), batch=batch, L=L, H=H, P=P,
                                 N=N)


@settings(max_examples=25, deadline=None)
@given(batch=st.integers(1, 2), L=st.integers(1, 12), D=st.integers(1, 5), N=st.integers(1, 4),
       seed=st.integers(0, 2**31 - 1))
def test_conv_against_numpy(lib, batch, L, D, N, seed):
    """Including sequences shorter than the width-4 filter."""
    pins.conv_numpy_check(lib, np.random.default_rng(seed), batch, L, D, N)


@settings(max_examples=30, deadline=None)
@given(batch=st.integers(1, 3), D=st.integers(1, 6), N=st.integers(1, 12),
       seed=st.integers(0, 2**31 - 1))
def test_step_against_library_pipeline(lib, batch, D, N, seed):
    pins.step_pipeline_check(lib, np.random.default_rng(seed), batch, D, N)
