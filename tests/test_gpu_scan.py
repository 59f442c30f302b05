"""GPU parity of ssm_scan_fwd against the float64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_gpu(inp, want_h=True):
    y, h = ssm.scan(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                    inp["Dskip"], inp["z"], want_h_last=want_h)
    torch.cuda.synchronize()
    return y, h


def full_parity(inp, what):
    y, h = run_gpu(inp)
    y_ref, h_ref = parity.oracle_scan(inp)
    tol = parity.TOL[inp["u"].dtype]
    parity.check(parity.to_f64(y), y_ref, tol, what + " y")
    parity.check(parity.to_f64(h), h_ref, tol, what + " h_last")


def sampled_parity(inp, what, count=None, threads=8, chans=None):
    y, h = run_gpu(inp)
    batch, L, D = inp["u"].shape
    if chans is None:
        chans = parity.sample_channels(batch, D, count)
    ref = parity.oracle_scan_channels(inp, chans, threads=threads)
    tol = parity.TOL[inp["u"].dtype]
    idx_b = torch.tensor([c[0] for c in chans], device=DEV)
    idx_d = torch.tensor([c[1] for c in chans], device=DEV)
    ys = parity.to_f64(y[idx_b, :, idx_d])          # [n_chan, L]
    hs = parity.to_f64(h[idx_b, idx_d])             # [n_chan, N]
    y_ref = np.stack([ref[c][0] for c in chans])
    h_ref = np.stack([ref[c][1] for c in chans])
    parity.check(ys, y_ref, tol, what + " y")
    parity.check(hs, h_ref, tol, what + " h_last")
    assert torch.isfinite(y.float()).all(), what + ": non-finite y"


def test_tiny_f32_full():
    full_parity(wl.make_scan_inputs(wl.TINY_F32, device=DEV), "tiny f32")


def test_tiny_f32_time_invariant_full():
    full_parity(wl.make_scan_inputs(wl.TINY_F32_LTI, device=DEV), "tiny f32 LTI")


@pytest.mark.parametrize("L,D", [(300, 96), (1, 64), (17, 37), (513, 200)])
def test_bf16_ragged_full(L, D):
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=L, D=D, seed=7)
    full_parity(inp, f"bf16 L={L} D={D}")


@pytest.mark.parametrize("N", [1, 4, 7, 16, 33, 64, 256])
def test_state_sizes(N):
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=40, D=24, N=N, seed=N)
    full_parity(inp, f"f32 N={N}")


def test_mamba130m_full_size_sampled():
    """Every one of the 96 chains (8 x 12 blocks of 128 channels): its first
    and last channel and one more."""
    w = wl.MAMBA_130M
    chans = parity.chain_channels(w.batch, w.D, per_chain=3, seed=1)
    assert len({(b, d // 128) for b, d in chans}) == 96
    sampled_parity(wl.make_scan_inputs(w, device=DEV), "mamba130m", chans=chans, threads=16)


def test_mamba2p8b_full_size_sampled():
    """Every one of the 160 chains (4 x 40 blocks of 128 channels), at the
    bench's launch configuration: first, last and one more channel each."""
    w = wl.MAMBA_2P8B
    chans = parity.chain_channels(w.batch, w.D, per_chain=3, seed=2)
    assert len({(b, d // 128) for b, d in chans}) == 160
    sampled_parity(wl.make_scan_inputs(w, device=DEV), "mamba2.8b", chans=chans, threads=16)


@pytest.mark.slow
def test_longseq_full_size_sampled():
    """64 channels spanning all 12 chains of the 1 x 1,048,576 x 1536
    sequence (each chain's first and last channel and 3-4 more), through
    the narrow plan's three launches."""
    w = wl.LONG_SEQ
    chans = parity.chain_channels(w.batch, w.D, per_chain=5, seed=3)
    rng = np.random.default_rng(4)
    while len(chans) < 64:
        chans = sorted(set(chans) | {(0, int(rng.integers(w.D)))})
    assert len({d // 128 for _, d in chans}) == 12
    inp = wl.make_scan_inputs(w, device=DEV)
    sampled_parity(inp, "longseq", chans=chans, threads=16)


def test_optional_inputs_null():
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=64, D=64, seed=3)
    for drop in ("z", "Dskip", "dt_bias"):
        q = dict(inp)
        q[drop] = None
        full_parity(q, f"{drop}=NULL")


def test_h_last_null_and_empty():
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=64, D=64, seed=4)
    y1, _ = run_gpu(inp, want_h=False)
    y2, _ = run_gpu(inp, want_h=True)
    assert torch.equal(y1, y2)
    # L == 0: the state after zero steps is 0
    q = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=0, D=64, seed=4)
    h = torch.full((2, 64, 16), 7.0, device=DEV)
    y = torch.empty_like(q["u"])
    ssm.ssm_scan_fwd(q["u"], q["delta"], q["dt_bias"], q["A"], q["B"], q["C"], q["Dskip"],
                     q["z"], y, h)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h) == 0
    # batch == 0 / D == 0: nothing to do, no error
    q = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=0, L=8, D=64, seed=4)
    run_gpu(q)


def test_edge_values():
    """Huge |delta| (dt -> 0 and dt -> huge), z = 0 (gate closes), A = 0
    (integrator) and a generic A: finite and matching the oracle."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=64, D=32, seed=9)
    inp["delta"][0, ::3, 8:] = 1e4
    inp["delta"][1, ::5, 8:] = -1e4
    inp["delta"][0, 1::7, :8] = 1e4     # huge dt on the A = 0 and per-state channels too
    inp["delta"][1, 2::9, :8] = 300.0
    inp["z"][0, 10:20] = 0.0
    inp["A"][3] = 0.0
    g = torch.Generator(device=DEV).manual_seed(1)
    inp["A"][4:8] = -torch.rand((4, 16), generator=g, device=DEV) * 5
    full_parity(inp, "edge values")
    y, _ = run_gpu(inp)
    assert torch.count_nonzero(y[0, 10:20]) == 0


def test_bf16_roundtrip_exact_inputs():
    """Inputs that are exact in bf16: the oracle sees the same numbers, and y
    is the float32 result rounded once (within one bf16 ulp of the oracle)."""
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=1, L=32, D=64, seed=12)
    y, _ = run_gpu(inp)
    y_ref, _ = parity.oracle_scan(inp)
    err = np.abs(parity.to_f64(y) - y_ref)
    assert (err <= 2.0 ** -7 * np.abs(y_ref) + 1e-6).mean() > 0.99


def test_consistency_scan_then_steps():
    """scan(L) followed by K decode steps equals scan(L + K) (training form
    and inference form of the same model)."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=48, D=40, seed=21)
    Lh = 40
    head = {k: (v[:, :Lh].contiguous() if k in ("u", "delta", "z", "B", "C") else v)
            for k, v in inp.items()}
    _, state = run_gpu(head)
    y_full, h_full = run_gpu(inp)
    for t in range(Lh, 48):
        y_t = ssm.step(state, inp["u"][:, t].contiguous(), inp["delta"][:, t].contiguous(),
                       inp["dt_bias"], inp["A"], inp["B"][:, t].contiguous(),
                       inp["C"][:, t].contiguous(), inp["Dskip"], inp["z"][:, t].contiguous())
        torch.cuda.synchronize()
        parity.check(parity.to_f64(y_t), parity.to_f64(y_full[:, t]), 1e-4, f"step t={t}")
    parity.check(parity.to_f64(state), parity.to_f64(h_full), 1e-4, "state after steps")


def test_misaligned_and_strided_inputs():
    """Element-aligned but not 16-byte-aligned tensors take the generic kernel;
    pointers that are not element-aligned are rejected."""
    inp = wl.make_scan_inputs(wl.MAMBA_130M, device=DEV, batch=2, L=50, D=65, seed=5)
    big = {k: (torch.cat([torch.zeros(1, dtype=v.dtype, device=DEV), v.flatten()])
               if v is not None else None) for k, v in inp.items()}
    off = {k: (big[k][1:].view(inp[k].shape) if inp[k] is not None else None) for k in inp}
    full_parity(off, "element-aligned offset")
    raw = torch.zeros(inp["u"].numel() * 2 + 2, dtype=torch.uint8, device=DEV)
    y = torch.empty_like(inp["u"])
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    rc = ssm.lib.ssm_scan_fwd(raw.data_ptr() + 1, p(inp["delta"]), p(inp["dt_bias"]),
                              p(inp["A"]), p(inp["B"]), p(inp["C"]), p(inp["Dskip"]),
                              p(inp["z"]), p(y), None, 2, 50, 65, 16, 1, None)
    assert rc == -4


def test_fp32_mamba_shape_sampled():
    """float32 inputs at a Mamba-130M-like shape (multi-tile, long L)."""
    inp = wl.make_scan_inputs(wl.TINY_F32, device=DEV, batch=2, L=2048, D=512, seed=31)
    sampled_parity(inp, "f32 2x2048x512", 32)


@pytest.mark.parametrize("plan", [None, "narrow"])
def test_small_dt_times_a_f32(monkeypatch, plan):
    """fp32 inputs with |dt A| far below 1: geometric rows with a tiny a0,
    non-geometric tiny rows, and ordinary rows, all at the fp32 tolerance.
    exp(dt A) - 1 must not be formed by subtracting 1 from a number near 1
    there (a few surviving bits), on either path of the kernel."""
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
        monkeypatch.setenv("SSM_CHUNK_T", "64")
    inp = wl.make_scan_inputs(wl.TINY_F32, device="cuda", batch=2, L=300, D=64, seed=17)
    n1 = torch.arange(1, 17, device="cuda", dtype=torch.float32)
    inp["A"][0:16] = -1e-4 * n1                    # geometric, tiny a0
    inp["A"][16:32] = -1e-4                        # not geometric, tiny
    inp["A"][32:48] = -3e-3 * n1                   # geometric, small
    full_parity(inp, f"small dt*A plan={plan}")
