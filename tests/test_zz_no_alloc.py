"""ssm_scan_fwd_noalloc: the selective scan for callers that cannot allocate
device memory while they run (a server whose memory is all reserved up front
by its own pool, or code where a cudaMalloc would synchronise, fail or is not
allowed).  It keeps the kernel's scratch -- the unit counter, the per-chain
progress flags and, without h_last, the carried state -- in one fixed array
inside the library, shared by every call.

These tests call it through the C ABI and compare each result with the
float64 oracle and with ssm_scan_fwd, on calls in a row, so that whatever one
call leaves in the shared array (flags of a larger problem, carried states)
would show up as a wrong result in the next one.  Chains are also cut into
pieces on purpose (SSM_CHUNK_T), so that the hand-over through the fixed
array's flags and carry slots is exercised.

The file's name sorts it after every other test file.  It was added after the
rest of the suite and depends on nothing they leave behind; placing it last
means that a run which stops at the first failure has already run every other
test when it gets here, and it passes both alone in a fresh process and after
the others.
"""
import os

import pytest
import torch

import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _p(t):
    return None if t is None else t.data_ptr()


def noalloc(inp, want_h):
    """One call of the C entry point; returns (y, h_last or None)."""
    u = inp["u"]
    batch, L, D = u.shape
    N = inp["A"].shape[1]
    y = torch.full_like(u, float("nan"))
    h = torch.full((batch, D, N), float("nan"), device=DEV) if want_h else None
    rc = ssm.lib.ssm_scan_fwd_noalloc(
        _p(u), _p(inp["delta"]), _p(inp["dt_bias"]), _p(inp["A"]), _p(inp["B"]), _p(inp["C"]),
        _p(inp["Dskip"]), _p(inp["z"]), _p(y), _p(h), batch, L, D, N,
        0 if u.dtype == torch.float32 else 1, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ssm.ssm_status_string(rc)
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return y, h


def reference(inp):
    y, h = ssm.scan(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                    inp["Dskip"], inp["z"])
    torch.cuda.synchronize()
    return y, h


def check_against_oracle(inp, y, h, tol, what):
    y_ref, h_ref = parity.oracle_scan(inp)
    parity.check(parity.to_f64(y), y_ref, tol, f"{what} y vs oracle")
    if h is not None:
        parity.check(parity.to_f64(h), h_ref, tol, f"{what} h_last vs oracle")


CASES = [  # (batch, L, D, dtype, seed)
    (2, 1024, 512, torch.bfloat16, 1),
    (3, 300, 96, torch.bfloat16, 2),       # ragged L, several 32-channel blocks
    (2, 256, 64, torch.float32, 3),
    (2, 100, 40, torch.float32, 4),        # ragged D
]


@pytest.mark.parametrize("want_h", [True, False], ids=["h_last", "no_h_last"])
def test_noalloc_matches_oracle_two_calls(want_h):
    """Two different problems, then the first again: each call agrees with
    the oracle and with ssm_scan_fwd within the scan's tolerance."""
    for batch, L, D, dtype, seed in CASES:
        w = wl.ScanWorkload("t", batch, L, D, 16, dtype, seed)
        first = wl.make_scan_inputs(w, device=DEV)
        second = wl.make_scan_inputs(w, device=DEV, seed=seed + 100)
        tol = parity.TOL[dtype]
        for k, inp in enumerate((first, second, first)):
            y, h = noalloc(inp, want_h)
            check_against_oracle(inp, y, h, tol, f"call {k} {w}")
            y_ref, h_ref = reference(inp)
            parity.check(parity.to_f64(y), parity.to_f64(y_ref), tol, f"call {k} y {w}")
            if want_h:
                parity.check(parity.to_f64(h), parity.to_f64(h_ref), tol, f"call {k} h {w}")


@pytest.mark.parametrize("want_h", [True, False], ids=["h_last", "no_h_last"])
def test_noalloc_cut_chains_large_then_small(want_h, monkeypatch):
    """Chains cut into pieces that hand their state over through the fixed
    array: first a problem with more pieces than resident CTAs (bf16, batch
    8, D 5120, L 512: 320 chains, pieces of 64 steps), then a smaller one
    whose flag slots the first call's higher counts covered.  Both agree with
    the oracle on sampled channels (one in every 128-channel chain, and each
    chain's first and last channel)."""
    monkeypatch.setenv("SSM_CHUNK_T", "64")
    big = wl.make_scan_inputs(wl.MAMBA_2P8B, device=DEV, batch=8, L=512, D=5120, seed=7)
    small = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=448, D=384, seed=8)
    tol = parity.TOL[torch.bfloat16]
    for k, inp in enumerate((big, small, big)):
        y, h = noalloc(inp, want_h)
        batch, L, D = inp["u"].shape
        chans = set()
        for b in range(batch):
            for c in range(0, D, 128):
                chans.update({(b, c), (b, min(c + 127, D - 1)), (b, c + (37 * b + c) % 128 % (D - c))})
        ref = parity.oracle_scan_channels(inp, sorted(chans))
        for (b, d), (y_r, h_r) in ref.items():
            parity.check(parity.to_f64(y[b, :, d]), y_r, tol, f"call {k} y[{b},:,{d}]")
            if want_h:
                parity.check(parity.to_f64(h[b, d]), h_r, tol, f"call {k} h[{b},{d}]")
        y_ref, h_ref = reference(inp)
        parity.check(parity.to_f64(y), parity.to_f64(y_ref), tol, f"call {k} y vs ssm_scan_fwd")


def test_noalloc_generic_shapes_and_limit():
    """Shapes the fast kernel does not take run the generic kernel; a problem
    that needs more than the fixed scratch is refused before any work."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=40, D=24, N=7, seed=5)
    for _ in range(2):
        y, h = noalloc(inp, True)
        check_against_oracle(inp, y, h, 1e-4, "generic")
    fake = 1 << 16   # never dereferenced: the size check comes first
    rc = ssm.lib.ssm_scan_fwd_noalloc(fake, fake, None, fake, fake, fake, None, None, fake, None,
                                      8, 32, 16384, 16, 1, None)
    assert rc == -9, ssm.ssm_status_string(rc)
