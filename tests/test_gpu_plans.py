"""Every launch plan of ssm_scan_fwd against the oracle, forced through the
SSM_FORCE_PLAN / SSM_CHUNK_T development switches (read at each call), plus
the bounded-wait failure path of the chained plan."""
import pytest
import torch

import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [  # (batch, L, D, dtype, chunk)
    (2, 256, 64, torch.float32, 32),
    (2, 300, 96, torch.bfloat16, 64),     # ragged L (300 = 9*32 + 12), three 32-channel blocks
    (3, 97, 40, torch.bfloat16, 32),      # ragged D (40 = 32 + 8), ragged L
    (1, 1, 64, torch.bfloat16, 32),       # L = 1
    (2, 33, 8, torch.float32, 32),        # D < 32
    (1, 1000, 128, torch.bfloat16, 96),   # many chunks
]


def run(inp, monkeypatch, plan, chunk=None):
    monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    if chunk:
        monkeypatch.setenv("SSM_CHUNK_T", str(chunk))
    else:
        monkeypatch.delenv("SSM_CHUNK_T", raising=False)
    y, h = ssm.scan(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                    inp["Dskip"], inp["z"])
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return y, h


@pytest.mark.parametrize("plan", ["generic", "chained", "narrow"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}_{s[3]}_T{s[4]}")
def test_plan_parity(monkeypatch, plan, shape):
    batch, L, D, dtype, chunk = shape
    w = wl.ScanWorkload("t", batch, L, D, 16, dtype, 17)
    inp = wl.make_scan_inputs(w, device=DEV)
    y, h = run(inp, monkeypatch, plan, chunk)
    y_ref, h_ref = parity.oracle_scan(inp)
    tol = parity.TOL[dtype]
    parity.check(parity.to_f64(y), y_ref, tol, f"{plan} y")
    parity.check(parity.to_f64(h), h_ref, tol, f"{plan} h_last")


@pytest.mark.parametrize("plan", ["chained", "narrow"])
def test_plan_general_A_and_options(monkeypatch, plan):
    """Non-geometric A (per-state path, including A = 0 channels) and the
    optional NULL inputs on the fast kernel."""
    w = wl.ScanWorkload("t", 2, 200, 96, 16, torch.bfloat16, 23)
    inp = wl.make_scan_inputs(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(3)
    inp["A"][:40] = -torch.rand((40, 16), generator=g, device=DEV) * 4 - 0.05
    inp["A"][40:44] = 0.0
    inp["A"][44, 3] = 0.0
    for drop in (None, "z", "Dskip", "dt_bias"):
        q = dict(inp)
        if drop:
            q[drop] = None
        y, h = run(q, monkeypatch, plan, 64)
        y_ref, h_ref = parity.oracle_scan(q)
        parity.check(parity.to_f64(y), y_ref, 2e-2, f"{plan} drop={drop} y")
        parity.check(parity.to_f64(h), h_ref, 2e-2, f"{plan} drop={drop} h")


def test_plans_agree_with_each_other(monkeypatch):
    """The three plans compute the same function: bf16 outputs within one
    rounding of each other, states within float32 noise."""
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=512, D=256, seed=41)
    outs = {p: run(inp, monkeypatch, p, 64) for p in ("generic", "chained", "narrow")}
    for p in ("chained", "narrow"):
        parity.check(parity.to_f64(outs[p][1]), parity.to_f64(outs["generic"][1]), 1e-3,
                     f"{p} vs generic h")
        parity.check(parity.to_f64(outs[p][0]), parity.to_f64(outs["generic"][0]), 2e-2,
                     f"{p} vs generic y")


def test_chained_wait_times_out_and_recovers(monkeypatch):
    """Failure detection without a GPU fault: with chunk states never
    published, the successors' bounded wait (20 ms) gives up, the kernel drains
    and returns, the device status reports SSM_ERR_TIMEOUT, and the context
    stays usable for a correct run afterwards."""
    w = wl.ScanWorkload("t", 1, 512, 64, 16, torch.bfloat16, 5)
    inp = wl.make_scan_inputs(w, device=DEV)
    monkeypatch.setenv("SSM_TEST_STALL_CHAIN", "1")
    monkeypatch.setenv("SSM_WAIT_LIMIT_NS", "20000000")
    monkeypatch.setenv("SSM_FORCE_PLAN", "chained")
    monkeypatch.setenv("SSM_CHUNK_T", "64")
    y = torch.empty_like(inp["u"])
    h = torch.empty((1, 64, 16), device=DEV)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                     inp["Dskip"], inp["z"], y, h)
    assert ssm.ssm_device_status() == -8
    assert ssm.ssm_device_status() == 0          # cleared
    monkeypatch.delenv("SSM_TEST_STALL_CHAIN")
    monkeypatch.delenv("SSM_WAIT_LIMIT_NS")
    y, h = run(inp, monkeypatch, "chained", 64)
    y_ref, h_ref = parity.oracle_scan(inp)
    parity.check(parity.to_f64(y), y_ref, 2e-2, "after recovery y")
    parity.check(parity.to_f64(h), h_ref, 2e-2, "after recovery h")
