"""GPU parity of ssm_ssd_fwd (the Mamba-2 SSD form: scalar A per head, head
dimension P, Euler input term) against the float64 oracle through the C ABI:
the tcgen05 chunked kernel (bf16, P = 64, N = 64 or 128, 128-step chunks)
on shapes with exact and ragged last chunks, the one-thread-per-channel kernel for the rest, and the
Mamba-2 2.7B-shaped layer on sampled heads."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_ssd(inp):
    x = inp["x"]
    b, L, H, P = x.shape
    N = inp["B"].shape[-1]
    y = torch.empty_like(x)
    h = torch.empty((b, H, P, N), device=DEV)
    ssm.ssm_ssd_fwd(x, inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["Dskip"], y, h)
    torch.cuda.synchronize()
    return y, h


def oracle_ssd(inp, threads=8):
    hst = parity.host
    return oracle.ssd_fwd(hst(inp["x"]), hst(inp["dt"]), hst(inp["dt_bias"]), hst(inp["A"]),
                          hst(inp["B"]), hst(inp["C"]), hst(inp["Dskip"]),
                          dtype=parity.dtype_code(inp["x"].dtype), threads=threads)


SHAPES = [  # (batch, L, H, P, N, dtype, plan)
    (2, 64, 3, 64, 64, torch.bfloat16, None),
    (1, 200, 2, 64, 128, torch.bfloat16, None),     # ragged last chunk
    (2, 130, 4, 64, 128, torch.bfloat16, None),
    (1, 1, 2, 64, 64, torch.bfloat16, None),
    (1, 128, 2, 64, 128, torch.bfloat16, None),     # exactly one 128-step chunk
    (1, 129, 2, 64, 64, torch.bfloat16, None),      # a one-step second chunk
    (2, 383, 3, 64, 128, torch.bfloat16, None),     # three chunks, ragged
    (2, 70, 2, 64, 128, torch.bfloat16, "generic"),
    (2, 50, 3, 32, 16, torch.float32, None),        # one thread per channel
    (1, 70, 2, 64, 128, torch.float32, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"_{s[5]}_{s[6]}")
def test_ssd_parity(monkeypatch, shape):
    b, L, H, P, N, dtype, plan = shape
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    inp = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=b, L=L, H=H, P=P, N=N, dtype=dtype)
    y, h = run_ssd(inp)
    y_ref, h_ref = oracle_ssd(inp)
    tol = parity.TOL[dtype]
    parity.check(parity.to_f64(y), y_ref, tol, f"{shape} y")
    parity.check(parity.to_f64(h), h_ref, tol, f"{shape} h_last")


# The ticket walk (heads cut into segments, persistent CTAs taking them from a
# counter, each head's state passed between segments through global memory),
# forced on small shapes: (batch, L, H, N, chunks per segment, CTAs).
TICKET_SHAPES = [
    (2, 640, 4, 128, 1, 0),     # every chunk its own segment, one per CTA
    (2, 640, 4, 128, 2, 3),     # 24 units on 3 CTAs
    (2, 383, 3, 64, 1, 4),      # ragged last chunk, N = 64
    (1, 1000, 5, 128, 3, 2),    # segments of 3 chunks, the last one short
    (3, 300, 7, 128, 0, 5),     # whole heads, 21 units on 5 CTAs
    (1, 128, 1, 128, 1, 1),     # one chunk, one unit
]


@pytest.mark.parametrize("shape", TICKET_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ssd_ticket_walk_parity(monkeypatch, shape):
    b, L, H, N, seg, ctas = shape
    if seg:
        monkeypatch.setenv("SSM_SSD_SEG", str(seg))
    if ctas:
        monkeypatch.setenv("SSM_SSD_CTAS", str(ctas))
    inp = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=b, L=L, H=H, P=64, N=N,
                             dtype=torch.bfloat16)
    y, h = run_ssd(inp)
    assert ssm.ssm_device_status() == 0
    y_ref, h_ref = oracle_ssd(inp)
    parity.check(parity.to_f64(y), y_ref, 2e-2, f"{shape} y")
    parity.check(parity.to_f64(h), h_ref, 2e-2, f"{shape} h_last")
    # the same bits as one head per CTA
    monkeypatch.delenv("SSM_SSD_SEG", raising=False)
    monkeypatch.delenv("SSM_SSD_CTAS", raising=False)
    y1, h1 = run_ssd(inp)
    assert torch.equal(y1, y) and torch.equal(h1, h)


def test_ssd_nulls_and_empty():
    inp = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=1, L=100, H=2)
    q = dict(inp, dt_bias=None, Dskip=None)
    y, h = run_ssd(q)
    y_ref, h_ref = oracle_ssd(q)
    parity.check(parity.to_f64(y), y_ref, 2e-2, "nulls y")
    parity.check(parity.to_f64(h), h_ref, 2e-2, "nulls h_last")
    e = wl.make_ssd_inputs(wl.SSD_SMALL, device=DEV, batch=1, L=0, H=2)
    _, h0 = run_ssd(e)
    assert torch.count_nonzero(h0) == 0


def test_ssd_mamba2_2p7b_sampled_heads():
    """The 4 x 4096 x (80 heads x 64) layer with N = 128 on the tensor-core
    kernel (the ticket walk: 320 heads on the SMs of a B300 would leave a last
    wave of 24 CTAs, so every head runs as segments on several CTAs); every
    output of sampled heads against the oracle.  The sample
    always holds the six most slowly decaying heads (smallest |A|), whose long
    memories make the largest states and the most cancellation in y: rounding
    the bf16 operands of the products once (without a low part) put y 4.6% off
    on such a head."""
    w = wl.SSD_2P7B
    inp = wl.make_ssd_inputs(w, device=DEV)
    y, h = run_ssd(inp)
    heads = sorted(set(torch.argsort(inp["A"].abs())[:6].tolist()) | {0, 37, w.H - 1})
    idx = torch.tensor(heads, device=DEV)
    sub = dict(inp, x=inp["x"].index_select(2, idx), dt=inp["dt"].index_select(2, idx),
               dt_bias=inp["dt_bias"].index_select(0, idx), A=inp["A"].index_select(0, idx),
               Dskip=inp["Dskip"].index_select(0, idx))
    y_ref, h_ref = oracle_ssd(sub, threads=16)
    parity.check(parity.to_f64(y.index_select(2, idx)), y_ref, 2e-2, "2.7B y")
    parity.check(parity.to_f64(h.index_select(1, idx)), h_ref, 2e-2, "2.7B h_last")
