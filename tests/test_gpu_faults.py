"""Error propagation, with the failures injected on the host
(SSM_FAULT_INJECT=alloc|launch): the stream-ordered workspace allocation or
the kernel launch fails before anything runs on the device, each entry point
returns SSM_ERR_NOMEM or SSM_ERR_CUDA, the device reports no error, and the
next call without injection gives the oracle's result.  Nothing faults, traps
or hangs on the GPU."""
import os

import pytest
import torch

import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
NOMEM, CUDA_ERR = -7, -6


class env:
    """Sets environment variables for the duration of a with-block."""

    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        os.environ.update(self.kv)

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def status_of(fn):
    try:
        fn()
    except ssm.SsmError as e:
        return e.status
    return 0


def scan_call(inp, h_last=True):
    y = torch.empty_like(inp["u"])
    b, L, D = inp["u"].shape
    h = torch.empty((b, D, 16), device=DEV) if h_last else None
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                     inp["Dskip"], inp["z"], y, h)
    torch.cuda.synchronize()
    return y, h


def check_scan(inp, tol):
    y, h = scan_call(inp)
    y_ref, h_ref = parity.oracle_scan(inp)
    parity.check(parity.to_f64(y), y_ref, tol, "y after injection")
    parity.check(parity.to_f64(h), h_ref, tol, "h_last after injection")


@pytest.mark.parametrize("plan", ["chained", "narrow", "generic"])
@pytest.mark.parametrize("kind,want", [("alloc", NOMEM), ("launch", CUDA_ERR)])
def test_scan_reports_injected_failure_then_recovers(plan, kind, want):
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=512, D=256, seed=41)
    with env(SSM_FORCE_PLAN=plan):
        with env(SSM_FAULT_INJECT=kind):
            st = status_of(lambda: scan_call(inp, h_last=False))
        if plan == "generic" and kind == "alloc":
            want = 0   # the generic kernel takes no workspace
        assert st == want, (plan, kind, st)
        assert ssm.ssm_device_status() == 0
        check_scan(inp, parity.TOL[torch.bfloat16])


@pytest.mark.parametrize("n_state", [16, 7], ids=["unit_kernels", "generic"])
@pytest.mark.parametrize("kind,want", [("alloc", NOMEM), ("launch", CUDA_ERR)])
def test_backward_reports_injected_failure_then_recovers(n_state, kind, want):
    batch, L, D = 2, 96, 128
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=batch, L=L, D=D, N=n_state, seed=42)
    dy, dh = wl.grad_inputs(batch, L, D, n_state, torch.float32, 43, DEV)
    u = inp["u"]
    g = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u), dz=torch.empty_like(u),
             dB=torch.empty((batch, L, n_state), device=DEV),
             dC=torch.empty((batch, L, n_state), device=DEV),
             dA=torch.empty((D, n_state), device=DEV), ddt_bias=torch.empty(D, device=DEV),
             dDskip=torch.empty(D, device=DEV))

    def call():
        ssm.ssm_scan_bwd(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                         inp["Dskip"], inp["z"], dy, dh, g["du"], g["ddelta"], g["ddt_bias"],
                         g["dA"], g["dB"], g["dC"], g["dDskip"], g["dz"])
        torch.cuda.synchronize()

    with env(SSM_FAULT_INJECT=kind):
        assert status_of(call) == want
    assert ssm.ssm_device_status() == 0
    call()
    import oracle
    ref = oracle.scan_bwd(*(parity.host(inp[k]) for k in
                            ("u", "delta", "dt_bias", "A", "B", "C", "Dskip", "z")),
                          parity.host(dy), parity.host(dh), dtype=oracle.F32, threads=8)
    for k in g:
        parity.check(parity.to_f64(g[k]), ref[k], 1e-4, f"{k} after injection")


def test_launch_injection_covers_step_ssd_and_noalloc():
    """The decode step, the SSD form and the allocation-free scan allocate
    nothing, so only a refused launch can fail them; each reports it and the
    next call runs."""
    w = wl.StepWorkload("t", 4, 64, 16, 1, torch.float32, 44)
    s = wl.make_step_inputs(w, device=DEV)
    st = s["state"].clone()

    def step():
        return ssm.step(st, s["u"][0], s["delta"][0], s["dt_bias"], s["A"], s["B"][0],
                        s["C"][0], s["Dskip"], s["z"][0])

    q = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=1, L=64, H=2, N=64)
    ys = torch.empty_like(q["x"])

    def ssd():
        ssm.ssm_ssd_fwd(q["x"], q["dt"], q["dt_bias"], q["A"], q["B"], q["C"], q["Dskip"], ys,
                        None)

    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=1, L=128, D=128, seed=45)
    yn = torch.empty_like(inp["u"])

    def noalloc():
        ssm.ssm_scan_fwd_noalloc(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"],
                                 inp["C"], inp["Dskip"], inp["z"], yn, None)

    with env(SSM_FAULT_INJECT="launch"):
        for fn in (step, ssd, noalloc):
            assert status_of(fn) == CUDA_ERR, fn.__name__
    with env(SSM_FAULT_INJECT="alloc"):
        for fn in (step, ssd, noalloc):
            assert status_of(fn) == 0, fn.__name__
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    for fn in (step, ssd, noalloc):
        assert status_of(fn) == 0
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0


def test_ssd_ticket_walk_reports_injected_failure_then_recovers():
    """The SSD kernel's ticket walk takes a workspace (its ticket, the
    per-head counters and states): a failed allocation or launch is reported
    and the next call gives the oracle's result."""
    from tests.test_gpu_ssd import oracle_ssd
    q = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=2, L=300, H=3, N=128)
    y = torch.empty_like(q["x"])
    h = torch.empty((2, 3, 64, 128), device=DEV)

    def ssd():
        ssm.ssm_ssd_fwd(q["x"], q["dt"], q["dt_bias"], q["A"], q["B"], q["C"], q["Dskip"], y, h)

    with env(SSM_SSD_SEG="1", SSM_SSD_CTAS="4"):
        with env(SSM_FAULT_INJECT="alloc"):
            assert status_of(ssd) == NOMEM
        with env(SSM_FAULT_INJECT="launch"):
            assert status_of(ssd) == CUDA_ERR
        torch.cuda.synchronize()
        assert ssm.ssm_device_status() == 0
        assert status_of(ssd) == 0
        torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    y_ref, h_ref = oracle_ssd(q)
    parity.check(parity.to_f64(y), y_ref, 2e-2, "ssd y after injection")
    parity.check(parity.to_f64(h), h_ref, 2e-2, "ssd h_last after injection")
