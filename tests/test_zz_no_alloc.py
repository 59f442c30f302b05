"""ssm_scan_fwd_noalloc: the selective scan for callers that cannot allocate
device memory (a server whose memory is all reserved up front by its own pool,
or code where cudaMalloc would synchronise, fail or is not allowed).  It keeps
the kernel's scratch in a fixed array inside the library; these tests call it
through the C ABI and check it against ssm_scan_fwd, on two calls in a row so
that what the first call leaves in the shared array cannot leak into the
second.  This file is collected last on purpose."""
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


CASES = [  # (batch, L, D, dtype, seed)
    (2, 1024, 512, torch.bfloat16, 1),
    (3, 300, 96, torch.bfloat16, 2),       # ragged L, several 32-channel blocks
    (2, 256, 64, torch.float32, 3),
    (2, 100, 40, torch.float32, 4),        # ragged D
]


@pytest.mark.parametrize("want_h", [True, False], ids=["h_last", "no_h_last"])
def test_noalloc_matches_scan_two_calls(want_h):
    """Two different problems, then the first again: each call agrees with
    ssm_scan_fwd within the scan's tolerance."""
    for batch, L, D, dtype, seed in CASES:
        w = wl.ScanWorkload("t", batch, L, D, 16, dtype, seed)
        first = wl.make_scan_inputs(w, device=DEV)
        second = wl.make_scan_inputs(w, device=DEV, seed=seed + 100)
        tol = parity.TOL[dtype]
        for k, inp in enumerate((first, second, first)):
            y, h = noalloc(inp, want_h)
            y_ref, h_ref = reference(inp)
            parity.check(parity.to_f64(y), parity.to_f64(y_ref), tol, f"call {k} y {w}")
            if want_h:
                parity.check(parity.to_f64(h), parity.to_f64(h_ref), tol, f"call {k} h {w}")


def test_noalloc_generic_shapes_and_limit():
    """Shapes the fast kernel does not take run the generic kernel; a problem
    that needs more than the fixed scratch is refused before any work."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=40, D=24, N=7, seed=5)
    for _ in range(2):
        y, h = noalloc(inp, True)
        y_ref, h_ref = reference(inp)
        parity.check(parity.to_f64(y), parity.to_f64(y_ref), 1e-4, "generic y")
        parity.check(parity.to_f64(h), parity.to_f64(h_ref), 1e-4, "generic h")
    fake = 1 << 16   # never dereferenced: the size check comes first
    rc = ssm.lib.ssm_scan_fwd_noalloc(fake, fake, None, fake, fake, fake, None, None, fake, None,
                                      8, 32, 16384, 16, 1, None)
    assert rc == -9, ssm.ssm_status_string(rc)
