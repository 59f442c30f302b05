"""GPU parity of ssm_step (decode) against the float64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_steps(inp, steps):
    state = inp["state"].clone()
    ys = []
    for s in range(steps):
        ys.append(ssm.step(state, inp["u"][s], inp["delta"][s], inp["dt_bias"], inp["A"],
                           inp["B"][s], inp["C"][s], inp["Dskip"],
                           None if inp["z"] is None else inp["z"][s]))
    torch.cuda.synchronize()
    return state, torch.stack(ys)


def oracle_steps(inp, steps, chans):
    """Oracle decode on sampled (b, d) channels; returns {(b,d): (state [N], y [steps])}."""
    dt = parity.dtype_code(inp["u"].dtype)
    by_b = {}
    for b, d in chans:
        by_b.setdefault(b, []).append(d)
    out = {}
    for b, ds in by_b.items():
        ds = sorted(set(ds))
        idx = torch.tensor(ds, device=DEV)
        st = parity.to_f64(inp["state"][b:b + 1].index_select(1, idx))
        A = parity.host(inp["A"].index_select(0, idx))
        bias = parity.host(None if inp["dt_bias"] is None else inp["dt_bias"].index_select(0, idx))
        dsk = parity.host(None if inp["Dskip"] is None else inp["Dskip"].index_select(0, idx))
        ys = []
        for s in range(steps):
            sub = lambda t: None if t is None else parity.host(t[s, b:b + 1].index_select(1, idx))  # noqa: E731
            st, y = oracle.step(st, sub(inp["u"]), sub(inp["delta"]), bias, A,
                                parity.host(inp["B"][s, b:b + 1]), parity.host(inp["C"][s, b:b + 1]),
                                dsk, sub(inp["z"]), dtype=dt)
            ys.append(y[0])
        ys = np.stack(ys)  # [steps, len(ds)]
        for j, d in enumerate(ds):
            out[(b, d)] = (st[0, j], ys[:, j])
    return out


def check_steps(inp, steps, chans, what):
    state, ys = gpu_steps(inp, steps)
    ref = oracle_steps(inp, steps, chans)
    tol = parity.TOL[inp["u"].dtype]
    for (b, d) in chans:
        parity.check(parity.to_f64(state[b, d]), ref[(b, d)][0], tol, f"{what} state b={b} d={d}")
        parity.check(parity.to_f64(ys[:, b, d]), ref[(b, d)][1], tol, f"{what} y b={b} d={d}")


def test_decode_full_size_64_steps_sampled():
    """The 256 x 5120 decode, 64 steps: 320 channels, d and d + D/2 (the pair
    one thread group of the one-pass kernel handles) with every batch row's
    first and last channel among them."""
    inp = wl.make_step_inputs(wl.DECODE, device=DEV)
    half = wl.DECODE.D // 2
    base = parity.sample_channels(wl.DECODE.batch, half, 160, seed=5)
    chans = sorted({c for b, d in base for c in ((b, d), (b, d + half))})
    check_steps(inp, wl.DECODE.steps, chans, "decode")


def test_decode_full_size_tiled_matches_one_pass(monkeypatch):
    """At 256 x 5120, the tiled kernel (what the benchmark times) and the
    one-pass kernel agree over 4 steps: the state to 2e-6 relative (they
    round the B_bar coefficient differently) and y to one bf16 unit."""
    inp = wl.make_step_inputs(wl.DECODE, device=DEV)
    st, y = gpu_steps(inp, 4)
    monkeypatch.setenv("SSM_STEP_KERNEL", "threads")
    st_ref, y_ref = gpu_steps(inp, 4)
    parity.check(parity.to_f64(st), parity.to_f64(st_ref), 2e-6, "tiled vs one-pass state")
    parity.check(parity.to_f64(y), parity.to_f64(y_ref), 8e-3, "tiled vs one-pass y")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_full_size_tiled_repeatable(dtype):
    """The tiled kernel's result does not depend on timing: the 256 x 5120
    decode, 64 steps, gives bit-identical states and outputs as plain
    launches, with L2 flushed before every step (copies landing out of
    order), and replayed as one CUDA graph.  A ring whose stages were read by
    alternating groups failed this, a group passing its wait on a stage whose
    previous copy had not landed."""
    w = wl.DECODE if dtype == torch.bfloat16 else wl.StepWorkload(
        "decode f32", wl.DECODE.batch, wl.DECODE.D, 16, wl.DECODE.steps, torch.float32, 41)
    inp = wl.make_step_inputs(w, device=DEV)
    state = inp["state"].clone()
    ys = torch.empty((w.steps, w.batch, w.D), device=DEV, dtype=w.dtype)
    flush = torch.empty(64 << 20, device=DEV, dtype=torch.float32)

    def run(flushed=False):
        for s in range(w.steps):
            if flushed:
                flush.zero_()
            ssm.ssm_step(state, inp["u"][s], inp["delta"][s], inp["dt_bias"], inp["A"],
                         inp["B"][s], inp["C"][s], inp["Dskip"], inp["z"][s], ys[s])

    results = []
    for flushed in (False, False, True, True):
        state.copy_(inp["state"])
        run(flushed)
        torch.cuda.synchronize()
        results.append((state.clone(), ys.clone()))
    state.copy_(inp["state"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        state.copy_(inp["state"])
        g.replay()
        torch.cuda.synchronize()
        results.append((state.clone(), ys.clone()))
    assert ssm.ssm_device_status() == 0
    st0, y0 = results[0]
    for i, (st, y) in enumerate(results[1:], 1):
        assert torch.equal(st, st0), f"run {i}: state differs"
        assert torch.equal(y, y0), f"run {i}: y differs"


@pytest.mark.parametrize("N", [1, 5, 16, 32, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_step_small_full(N, dtype):
    w = wl.StepWorkload("small", 3, 70, N, 5, dtype, 100 + N)
    inp = wl.make_step_inputs(w, device=DEV)
    chans = [(b, d) for b in range(3) for d in range(70)]
    check_steps(inp, 5, chans, f"step N={N} {dtype}")


def test_step_optional_null_and_empty():
    w = wl.StepWorkload("small", 2, 40, 16, 3, torch.bfloat16, 7)
    for drop in ("z", "Dskip", "dt_bias"):
        inp = wl.make_step_inputs(w, device=DEV)
        inp[drop] = None
        check_steps(inp, 3, [(b, d) for b in range(2) for d in range(40)], f"{drop}=NULL")
    inp = wl.make_step_inputs(w, device=DEV, batch=0)
    gpu_steps(inp, 1)


def test_step_small_dt_and_pure_decay():
    """dt -> 0 leaves the state unchanged; B = 0 gives state * exp(dt A)."""
    w = wl.StepWorkload("small", 2, 64, 16, 1, torch.float32, 8)
    inp = wl.make_step_inputs(w, device=DEV)
    inp["delta"][:] = -60.0
    inp["dt_bias"] = None
    st0 = inp["state"].clone()
    state, _ = gpu_steps(inp, 1)
    assert torch.equal(state, st0)
    inp = wl.make_step_inputs(w, device=DEV)
    inp["B"][:] = 0.0
    st0 = inp["state"].clone()
    state, _ = gpu_steps(inp, 1)
    dt = torch.nn.functional.softplus(inp["delta"][0].double() + inp["dt_bias"].double())
    want = st0.double() * torch.exp(dt[:, :, None] * inp["A"].double()[None])
    parity.check(parity.to_f64(state), want.cpu().numpy(), 1e-5, "pure decay")


@pytest.mark.parametrize("per_group", ["1", "2", "4"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fast_step_matches_generic(monkeypatch, dtype, per_group):
    """The N == 16 decode kernel (four threads per channel, one, two or four
    channels per thread group) and the generic one-thread-per-channel kernel
    agree step by step; a ragged channel count leaves a partly filled last
    warp."""
    w = wl.StepWorkload("small", 3, 203, 16, 4, dtype, 11)
    inp = wl.make_step_inputs(w, device=DEV)
    monkeypatch.delenv("SSM_FORCE_GENERIC_STEP", raising=False)
    monkeypatch.setenv("SSM_STEP_KERNEL", "threads")
    monkeypatch.setenv("SSM_STEP_J", per_group)
    st_fast, y_fast = gpu_steps(inp, 4)
    monkeypatch.setenv("SSM_FORCE_GENERIC_STEP", "1")
    st_gen, y_gen = gpu_steps(inp, 4)
    tol = parity.TOL[dtype]
    parity.check(parity.to_f64(st_fast), parity.to_f64(st_gen), 1e-5, "fast vs generic state")
    parity.check(parity.to_f64(y_fast), parity.to_f64(y_gen), tol, "fast vs generic y")


TILED_CASES = [  # (batch, D, steps): D % 8 == 0 takes the tiled kernel (128 channels x 4 entries)
    (3, 200, 3),     # a full and a ragged (72-channel) block; 3 of a tile's 4 entries
    (64, 1024, 2),   # 128 tiles: CTAs cross channel blocks
    (1, 8, 2),       # one 8-channel, 1-entry tile
    (5, 136, 2),     # 4 + 1 entries, 128 + 8 channels
    (9, 384, 2),
]


@pytest.mark.parametrize("batch,D,steps", TILED_CASES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiled_step_matches_oracle_and_one_pass(monkeypatch, batch, D, steps, dtype):
    """The tiled decode kernel (persistent CTAs, tensor copies of whole
    tiles, out-of-range channels and entries read as zeros and not stored)
    against the oracle on every channel, and against the one-pass kernel."""
    w = wl.StepWorkload("small", batch, D, 16, steps, dtype, 200 + D)
    inp = wl.make_step_inputs(w, device=DEV)
    monkeypatch.delenv("SSM_FORCE_GENERIC_STEP", raising=False)
    monkeypatch.delenv("SSM_STEP_KERNEL", raising=False)
    chans = [(b, d) for b in range(batch) for d in range(D)]
    if len(chans) > 600:
        chans = parity.sample_channels(batch, D, 600, seed=D)
    check_steps(inp, steps, chans, f"tiled {batch}x{D} {dtype}")
    assert ssm.ssm_device_status() == 0
    st, y = gpu_steps(inp, steps)
    monkeypatch.setenv("SSM_STEP_KERNEL", "threads")
    st_ref, y_ref = gpu_steps(inp, steps)
    parity.check(parity.to_f64(st), parity.to_f64(st_ref), 2e-6, "tiled vs one-pass state")
    parity.check(parity.to_f64(y), parity.to_f64(y_ref), parity.TOL[dtype], "tiled vs one-pass y")


def test_tiled_step_optional_null_and_zero_A():
    """z, D and dt_bias absent (the z copy is skipped, the others read as
    zero), and A with zero entries, where B_bar = dt B (the limit the oracle
    takes)."""
    w = wl.StepWorkload("small", 4, 256, 16, 2, torch.bfloat16, 17)
    chans = [(b, d) for b in range(4) for d in range(0, 256, 3)]
    for drop in ("z", "Dskip", "dt_bias"):
        inp = wl.make_step_inputs(w, device=DEV)
        inp[drop] = None
        check_steps(inp, 2, chans, f"tiled {drop}=NULL")
    inp = wl.make_step_inputs(w, device=DEV)
    inp["A"][::3, ::2] = 0.0
    check_steps(inp, 2, chans, "tiled A with zeros")
