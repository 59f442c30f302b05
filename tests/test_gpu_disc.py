"""GPU parity of ssm_scan_fwd_disc (Euler and trapezoidal discretisations, and
the zero-order hold through the same entry point) against the float64
oracle's variants, through the C ABI, on every launch plan."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
DISCS = {"zoh": 0, "euler": 1, "trapezoid": 2}


def run_disc(inp, disc):
    u = inp["u"]
    y = torch.empty_like(u)
    h = torch.empty((u.shape[0], u.shape[2], inp["A"].shape[1]), device=DEV)
    ssm.ssm_scan_fwd_disc(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                          inp["Dskip"], inp["z"], y, h, disc)
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return y, h


def oracle_disc(inp, disc):
    dt = parity.dtype_code(inp["u"].dtype)
    h = parity.host
    return oracle.scan_fwd_disc(h(inp["u"]), h(inp["delta"]), h(inp["dt_bias"]), h(inp["A"]),
                                h(inp["B"]), h(inp["C"]), h(inp["Dskip"]), h(inp.get("z")),
                                disc, dtype=dt, threads=8)


def full_parity(inp, disc, what):
    y, h = run_disc(inp, disc)
    y_ref, h_ref = oracle_disc(inp, disc)
    tol = parity.TOL[inp["u"].dtype]
    parity.check(parity.to_f64(y), y_ref, tol, what + " y")
    parity.check(parity.to_f64(h), h_ref, tol, what + " h_last")


SHAPES = [  # (batch, L, D, dtype, plan, chunk)
    (2, 256, 64, torch.float32, None, None),
    (2, 300, 96, torch.bfloat16, None, None),          # ragged L
    (3, 97, 40, torch.bfloat16, "chained", 32),        # ragged D, chains cut into pieces
    (1, 1000, 128, torch.bfloat16, "chained", 96),
    (1, 1000, 128, torch.bfloat16, "narrow", 96),
    (2, 33, 8, torch.float32, "narrow", 32),
    (2, 200, 72, torch.bfloat16, "generic", None),
]


@pytest.mark.parametrize("disc", ["euler", "trapezoid", "zoh"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}_{s[3]}_{s[4]}")
def test_disc_parity(monkeypatch, disc, shape):
    batch, L, D, dtype, plan, chunk = shape
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    if chunk:
        monkeypatch.setenv("SSM_CHUNK_T", str(chunk))
    inp = wl.make_scan_inputs(wl.ScanWorkload("t", batch, L, D, 16, dtype, 51))
    inp = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    full_parity(inp, DISCS[disc], f"{disc} {shape}")


@pytest.mark.parametrize("disc", ["euler", "trapezoid"])
def test_disc_general_A_and_nulls(monkeypatch, disc):
    """Non-geometric A rows (per-state path, A = 0 channels) and optional NULL
    inputs on the fast kernel, chained pieces."""
    monkeypatch.setenv("SSM_FORCE_PLAN", "chained")
    monkeypatch.setenv("SSM_CHUNK_T", "64")
    w = wl.ScanWorkload("t", 2, 200, 96, 16, torch.bfloat16, 23)
    inp = wl.make_scan_inputs(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(3)
    inp["A"][:40] = -torch.rand((40, 16), generator=g, device=DEV) * 4 - 0.05
    inp["A"][40:44] = 0.0
    for drop in (None, "z", "Dskip", "dt_bias"):
        q = dict(inp)
        if drop:
            q[drop] = None
        full_parity(q, DISCS[disc], f"{disc} drop={drop}")


@pytest.mark.parametrize("disc", ["euler", "trapezoid"])
@pytest.mark.parametrize("N", [7, 33])
def test_disc_other_state_sizes(disc, N):
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=40, D=24, N=N, seed=N)
    full_parity(inp, DISCS[disc], f"{disc} N={N}")


@pytest.mark.parametrize("disc", ["euler", "trapezoid"])
def test_disc_mamba130m_sampled(disc):
    """Full-size Mamba-130M-shaped layer; sampled channels against the oracle."""
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV)
    y, h = run_disc(inp, DISCS[disc])
    batch, L, D = inp["u"].shape
    chans = parity.sample_channels(batch, D, 24)
    tol = parity.TOL[inp["u"].dtype]
    for b in sorted({c[0] for c in chans}):
        ds = sorted({c[1] for c in chans if c[0] == b})
        idx = torch.tensor(ds, device=DEV)
        sub = {k: (None if v is None else
                   (v[b:b + 1].index_select(2, idx) if k in ("u", "delta", "z") else
                    v[b:b + 1] if k in ("B", "C") else v.index_select(0, idx)))
               for k, v in inp.items()}
        y_ref, h_ref = oracle_disc(sub, DISCS[disc])
        parity.check(parity.to_f64(y[b].index_select(1, idx)), y_ref[0], tol, f"{disc} y b={b}")
        parity.check(parity.to_f64(h[b].index_select(0, idx)), h_ref[0], tol, f"{disc} h b={b}")


def test_disc_rejects_unknown():
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=1, L=4, D=8, seed=1)
    with pytest.raises(ssm.SsmError):
        run_disc(inp, 3)


@pytest.mark.parametrize("disc", ["euler", "trapezoid"])
def test_disc_huge_and_tiny_dt(disc):
    """delta + bias far above 88 (where 2^(v log2 e) overflows float32) and far
    below: dt must stay finite and follow the oracle, on geometric rows, an
    A = 0 row and per-state rows.  With these input terms a huge dt makes the
    state itself huge (dt B u), and the outputs of later steps would then be
    small differences of huge terms, beyond float32; so the huge steps are
    the last ones, where y and h_last are large themselves."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=64, D=32, seed=13)
    inp["delta"][0, -1] = 1e4
    inp["delta"][1, -1] = 300.0
    inp["delta"][1, ::4] = -1e4
    inp["A"][3] = 0.0
    g = torch.Generator(device=DEV).manual_seed(2)
    inp["A"][4:8] = -torch.rand((4, 16), generator=g, device=DEV) * 5
    full_parity(inp, DISCS[disc], f"{disc} huge/tiny dt")

