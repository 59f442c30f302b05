"""GPU parity of ssm_conv_scan_fwd (causal depthwise width-4 convolution, with
and without SiLU, feeding the zero-order-hold scan) against the float64
oracle, through the C ABI, on every launch plan."""
import pytest
import torch

import oracle
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def inputs(w, seed=None, **kw):
    inp = wl.make_scan_inputs(w, device=DEV, seed=seed, **kw)
    cw, cb = wl.conv_params(inp["u"].shape[2], 1000 + (w.seed if seed is None else seed), DEV)
    inp["conv_w"], inp["conv_b"] = cw, cb
    return inp


def run_conv(inp, act):
    x = inp["u"]
    y = torch.empty_like(x)
    h = torch.empty((x.shape[0], x.shape[2], inp["A"].shape[1]), device=DEV)
    ssm.ssm_conv_scan_fwd(x, inp["conv_w"], inp["conv_b"], act, inp["delta"], inp["dt_bias"],
                          inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"], y, h)
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return y, h


def oracle_conv(inp, act):
    dt = parity.dtype_code(inp["u"].dtype)
    h = parity.host
    return oracle.conv_scan_fwd(h(inp["u"]), h(inp["conv_w"]), h(inp.get("conv_b")), act,
                                h(inp["delta"]), h(inp["dt_bias"]), h(inp["A"]), h(inp["B"]),
                                h(inp["C"]), h(inp["Dskip"]), h(inp.get("z")), dtype=dt,
                                threads=8)


def full_parity(inp, act, what):
    y, h = run_conv(inp, act)
    y_ref, h_ref = oracle_conv(inp, act)
    tol = parity.TOL[inp["u"].dtype]
    parity.check(parity.to_f64(y), y_ref, tol, what + " y")
    parity.check(parity.to_f64(h), h_ref, tol, what + " h_last")


SHAPES = [  # (batch, L, D, dtype, plan, chunk)
    (2, 256, 64, torch.float32, None, None),
    (2, 300, 96, torch.bfloat16, None, None),          # ragged L
    (3, 97, 40, torch.bfloat16, "chained", 32),        # ragged D, chains cut into pieces
    (1, 1000, 128, torch.bfloat16, "chained", 96),     # pieces start mid-sequence
    (1, 1000, 128, torch.float32, "narrow", 96),
    (2, 33, 8, torch.float32, "narrow", 32),
    (2, 200, 72, torch.bfloat16, "generic", None),
    (1, 2, 16, torch.float32, None, None),             # shorter than the filter
]


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}_{s[3]}_{s[4]}")
def test_conv_parity(monkeypatch, act, shape):
    batch, L, D, dtype, plan, chunk = shape
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    if chunk:
        monkeypatch.setenv("SSM_CHUNK_T", str(chunk))
    w = wl.ScanWorkload("t", batch, L, D, 16, dtype, 61)
    full_parity(inputs(w), act, f"act={act} {shape}")


def test_conv_general_A_and_nulls(monkeypatch):
    """Non-geometric A rows and optional NULL inputs (conv_b, z, Dskip,
    dt_bias) on the fast kernel, chained pieces."""
    monkeypatch.setenv("SSM_FORCE_PLAN", "chained")
    monkeypatch.setenv("SSM_CHUNK_T", "64")
    w = wl.ScanWorkload("t", 2, 200, 96, 16, torch.bfloat16, 29)
    inp = inputs(w)
    g = torch.Generator(device=DEV).manual_seed(5)
    inp["A"][:40] = -torch.rand((40, 16), generator=g, device=DEV) * 4 - 0.05
    inp["A"][40:44] = 0.0
    for drop in (None, "conv_b", "z", "Dskip", "dt_bias"):
        q = dict(inp)
        if drop:
            q[drop] = None
        full_parity(q, 1, f"drop={drop}")


@pytest.mark.parametrize("N", [7, 33])
def test_conv_other_state_sizes(N):
    full_parity(inputs(wl.TINY_F32, batch=2, L=40, D=24, N=N, seed=N), 1, f"N={N}")


def test_conv_identity_filter_is_the_scan():
    """conv_w = (0, 0, 0, 1), no bias, no activation: the plain scan."""
    inp = inputs(wl.TINY_F32, batch=2, L=300, D=64, seed=7)
    inp["conv_w"].zero_()
    inp["conv_w"][:, 3] = 1.0
    y, h = run_conv(dict(inp, conv_b=None), 0)
    y2 = torch.empty_like(y)
    h2 = torch.empty_like(h)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                     inp["Dskip"], inp["z"], y2, h2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(h, h2)


def test_conv_mamba130m_sampled():
    """Full-size Mamba-130M-shaped layer with SiLU; sampled channels against
    the oracle."""
    inp = inputs(wl.MAMBA_130M)
    y, h = run_conv(inp, 1)
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
        y_ref, h_ref = oracle_conv(sub, 1)
        parity.check(parity.to_f64(y[b].index_select(1, idx)), y_ref[0], tol, f"y b={b}")
        parity.check(parity.to_f64(h[b].index_select(0, idx)), h_ref[0], tol, f"h b={b}")


def test_conv_rejects_bad_arguments():
    inp = inputs(wl.TINY_F32, batch=1, L=4, D=8, seed=1)
    with pytest.raises(ssm.SsmError):
        run_conv(inp, 2)
    with pytest.raises(ssm.SsmError):
        run_conv(dict(inp, conv_w=None), 1)
