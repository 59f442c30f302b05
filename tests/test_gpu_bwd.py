"""GPU parity of ssm_scan_bwd (the backward pass of the zero-order-hold scan)
against the float64 oracle's adjoint, through the C ABI: every output element
by element on shapes that span several 32-step units, a ragged last unit and
a ragged channel block; the generic kernel; other state sizes; empty inputs;
the Mamba-130M layer in full and the Mamba-2.8B layer on sampled channels plus
linearity identities that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"
OUTS = ("du", "ddelta", "dz", "dB", "dC", "dA", "ddt_bias", "dDskip")


def inputs(batch, L, D, N, dtype, seed, with_dh=True):
    w = wl.ScanWorkload("t", batch, L, D, N, dtype, seed)
    inp = wl.make_scan_inputs(w, device=DEV)
    dy, dh = wl.grad_inputs(batch, L, D, N, dtype, seed + 500, DEV)
    inp["dy"], inp["dh_last"] = dy, (dh if with_dh else None)
    return inp


def run_bwd(inp, want=OUTS):
    u = inp["u"]
    batch, L, D = u.shape
    N = inp["A"].shape[1]
    out = {
        "du": torch.empty_like(u), "ddelta": torch.empty_like(u),
        "dz": torch.empty_like(u) if inp["z"] is not None else None,
        "dB": torch.empty((batch, L, N), device=DEV), "dC": torch.empty((batch, L, N), device=DEV),
        "dA": torch.empty((D, N), device=DEV), "ddt_bias": torch.empty(D, device=DEV),
        "dDskip": torch.empty(D, device=DEV),
    }
    for k in OUTS:
        if k not in want and k not in ("du", "ddelta", "dA"):
            out[k] = None
    ssm.ssm_scan_bwd(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"], inp["Dskip"],
                     inp["z"], inp["dy"], inp["dh_last"], out["du"], out["ddelta"],
                     out["ddt_bias"], out["dA"], out["dB"], out["dC"], out["dDskip"], out["dz"])
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return out


def oracle_bwd(inp, threads=8):
    h = parity.host
    return oracle.scan_bwd(h(inp["u"]), h(inp["delta"]), h(inp["dt_bias"]), h(inp["A"]),
                           h(inp["B"]), h(inp["C"]), h(inp["Dskip"]), h(inp["z"]), h(inp["dy"]),
                           h(inp["dh_last"]), dtype=parity.dtype_code(inp["u"].dtype),
                           threads=threads)


def compare(out, ref, tol, what, keys=OUTS):
    for k in keys:
        if out.get(k) is None:
            continue
        parity.check(parity.to_f64(out[k]), ref[k], tol, f"{what} {k}")


SHAPES = [  # (batch, L, D, dtype, plan)
    (2, 64, 128, torch.float32, None),
    (2, 100, 96, torch.bfloat16, None),       # ragged last unit
    (3, 97, 40, torch.bfloat16, None),        # ragged channel block
    (1, 300, 256, torch.float32, None),       # ten units, two blocks
    (2, 33, 8, torch.float32, None),          # last unit of one step
    (2, 31, 32, torch.bfloat16, None),        # a single unit
    (1, 1, 16, torch.float32, None),
    (2, 200, 72, torch.bfloat16, "generic"),
    # the states entering the units from the forward scan's chained plan
    # (taken unforced when the chains fill the GPU, as at full size)
    (2, 100, 96, torch.bfloat16, "chained"),
    (1, 300, 256, torch.float32, "chained"),
    (3, 97, 40, torch.bfloat16, "chained"),
    # and from the unit summaries with their carry
    (1, 300, 256, torch.float32, "narrow"),
]


@pytest.mark.parametrize("with_dh", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}_{s[3]}_{s[4]}")
def test_bwd_parity(monkeypatch, shape, with_dh):
    batch, L, D, dtype, plan = shape
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    inp = inputs(batch, L, D, 16, dtype, 71, with_dh)
    compare(run_bwd(inp), oracle_bwd(inp), parity.TOL[dtype], f"{shape} dh={with_dh}")


@pytest.mark.parametrize("plan", [None, "generic"])
def test_bwd_general_A_and_nulls(monkeypatch, plan):
    """Non-geometric A rows (per-state path), A = 0 entries, tiny A, and every
    optional input and output left out in turn."""
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    inp = inputs(2, 150, 96, 16, torch.float32, 33)
    g = torch.Generator(device=DEV).manual_seed(9)
    inp["A"][:40] = -torch.rand((40, 16), generator=g, device=DEV) * 4 - 0.05
    inp["A"][40:44] = 0.0
    inp["A"][44:46] = -1e-4
    for drop in (None, "z", "Dskip", "dt_bias", "dh_last"):
        q = dict(inp)
        if drop:
            q[drop] = None
        compare(run_bwd(q), oracle_bwd(q), 1e-4, f"drop={drop}")
    # outputs that may be left out
    out = run_bwd(inp, want=("du", "ddelta", "dz", "dA"))
    compare(out, oracle_bwd(inp), 1e-4, "outputs left out")


def _shifted(t):
    """A copy of t whose data starts one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0
    return v


@pytest.mark.parametrize("which", ["dy", "u", "z"])
def test_bwd_unaligned_operand(which):
    """An operand that is element-aligned but not 16-byte aligned sends the call
    to the generic kernel (the fast kernels copy 16-byte pieces); the result
    still follows the oracle."""
    inp = inputs(2, 90, 64, 16, torch.bfloat16, 17)
    inp[which] = _shifted(inp[which])
    compare(run_bwd(inp), oracle_bwd(inp), parity.TOL[torch.bfloat16], f"unaligned {which}")


@pytest.mark.parametrize("N", [7, 20, 33, 100])
def test_bwd_other_state_sizes(N):
    """The generic backward's four instantiations: N <= 16, <= 32, <= 64 and
    <= 256."""
    inp = inputs(2, 40, 24, N, torch.float32, N)
    compare(run_bwd(inp), oracle_bwd(inp), 1e-4, f"N={N}")


def test_bwd_empty_inputs():
    inp = inputs(2, 0, 32, 16, torch.float32, 3)
    out = run_bwd(inp)
    for k in ("dA", "ddt_bias", "dDskip"):
        assert torch.count_nonzero(out[k]) == 0
    inp = inputs(0, 16, 32, 16, torch.float32, 3)
    out = run_bwd(inp)
    assert torch.count_nonzero(out["dA"]) == 0


def test_bwd_rejects_missing_dz():
    inp = inputs(1, 8, 16, 16, torch.float32, 1)
    u = inp["u"]
    with pytest.raises(ssm.SsmError):
        ssm.ssm_scan_bwd(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                         inp["Dskip"], inp["z"], inp["dy"], None, torch.empty_like(u),
                         torch.empty_like(u), None, torch.empty((16, 16), device=DEV), None, None,
                         None, None)


def test_bwd_mamba130m_full():
    """The Mamba-130M-shaped layer (8 x 2048 x 1536, bf16): every output
    against the oracle's adjoint."""
    w = wl.MAMBA_130M
    inp = inputs(w.batch, w.L, w.D, w.N, w.dtype, w.seed)
    out = run_bwd(inp)
    compare(out, oracle_bwd(inp, threads=16), parity.TOL[w.dtype], "130M")


def test_bwd_mamba2p8b_sampled_and_identities():
    """The Mamba-2.8B-shaped layer (4 x 4096 x 5120, bf16) in the bench's
    configuration: du, ddelta, dz, dA, ddt_bias and dDskip of sampled channels
    (all batch entries) against the oracle; dB and dC, which sum over all
    5120 channels, through identities of linearity that hold at any size:
    <dC, C> = <dy, y0> and <dB, B> = <dy, y0> + <dh_last, h_last>, with y0
    the output at Dskip = 0 (z fixed)."""
    w = wl.MAMBA_2P8B
    inp = inputs(w.batch, w.L, w.D, w.N, w.dtype, w.seed)
    out = run_bwd(inp)
    tol = parity.TOL[w.dtype]
    ds = sorted({int(x) for x in np.random.default_rng(5).choice(w.D, 12, replace=False)} |
                {0, w.D - 1})
    idx = torch.tensor(ds, device=DEV)
    sub = {k: (None if v is None else
               v.index_select(2, idx) if k in ("u", "delta", "z", "dy") else
               v.index_select(1, idx) if k == "dh_last" else
               v if k in ("B", "C") else v.index_select(0, idx))
           for k, v in inp.items()}
    ref = oracle_bwd(sub, threads=16)
    for k in ("du", "ddelta", "dz"):
        parity.check(parity.to_f64(out[k].index_select(2, idx)), ref[k], tol, f"2.8B {k}")
    for k in ("dA", "ddt_bias", "dDskip"):
        parity.check(parity.to_f64(out[k].index_select(0, idx)), ref[k], tol, f"2.8B {k}")
    # identities for the channel sums, against a float32 forward of the same
    # values (bf16 widens exactly) so that y0 carries no bf16 rounding
    f = {k: (None if v is None else v.float()) for k, v in inp.items()}
    y0 = torch.empty_like(f["u"])
    hl = torch.empty((w.batch, w.D, w.N), device=DEV)
    ssm.ssm_scan_fwd(f["u"], f["delta"], f["dt_bias"], f["A"], f["B"], f["C"], None, f["z"], y0, hl)
    torch.cuda.synchronize()
    dyy = f["dy"].double() * y0.double()                     # [b, L, D]
    dcc = out["dC"].double() * inp["C"].double()             # [b, L, N]
    # per row (b, t): C_t reaches only y_t
    lhs, rhs = dcc.sum(-1), dyy.sum(-1)
    scale = dcc.abs().sum(-1) + dyy.abs().sum(-1)
    bad = (lhs - rhs).abs() > 1e-4 * scale
    assert not bool(bad.any()), f"{int(bad.sum())} rows break <dC, C> = <dy, y0>"
    # per batch entry: B reaches every later h and h_last
    dbb = (out["dB"].double() * inp["B"].double()).sum((1, 2))
    dhh = (f["dh_last"].double() * hl.double()).sum((1, 2))
    rhs_b = dyy.sum((1, 2)) + dhh
    scale_b = (out["dB"].double() * inp["B"].double()).abs().sum((1, 2)) + dyy.abs().sum((1, 2)) \
        + (f["dh_last"].double() * hl.double()).abs().sum((1, 2))
    assert bool(((dbb - rhs_b).abs() <= 3e-6 * scale_b).all()), (dbb, rhs_b, scale_b)


def run_ckpt(inp, plan=None, monkeypatch=None):
    """ssm_scan_fwd_ckpt then ssm_scan_bwd_ckpt; returns (y, h_last, outputs)."""
    u = inp["u"]
    batch, L, D = u.shape
    N = inp["A"].shape[1]
    ckpt = torch.full(((L + 31) // 32, batch, D, N), float("nan"), device=DEV)
    y = torch.empty_like(u)
    h = torch.empty((batch, D, N), device=DEV)
    ssm.ssm_scan_fwd_ckpt(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                          inp["Dskip"], inp["z"], y, h, ckpt)
    out = {
        "du": torch.empty_like(u), "ddelta": torch.empty_like(u),
        "dz": torch.empty_like(u) if inp["z"] is not None else None,
        "dB": torch.empty((batch, L, N), device=DEV), "dC": torch.empty((batch, L, N), device=DEV),
        "dA": torch.empty((D, N), device=DEV), "ddt_bias": torch.empty(D, device=DEV),
        "dDskip": torch.empty(D, device=DEV),
    }
    ssm.ssm_scan_bwd_ckpt(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                          inp["Dskip"], inp["z"], inp["dy"], inp["dh_last"], ckpt, out["du"],
                          out["ddelta"], out["ddt_bias"], out["dA"], out["dB"], out["dC"],
                          out["dDskip"], out["dz"])
    torch.cuda.synchronize()
    assert ssm.ssm_device_status() == 0
    return y, h, ckpt, out


CKPT_SHAPES = [  # (batch, L, D, dtype, plan)
    (2, 100, 96, torch.bfloat16, None),       # ragged last unit
    (1, 300, 256, torch.float32, None),       # 16-step stages: every other one writes
    (2, 1000, 128, torch.bfloat16, "narrow"), # the narrow plan's output pass writes them
    (2, 31, 32, torch.bfloat16, None),        # one unit: nothing to write
    (3, 64, 40, torch.bfloat16, None),        # a ragged channel block, L a multiple of 32
]


@pytest.mark.parametrize("shape", CKPT_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}_{s[3]}_{s[4]}")
def test_bwd_with_forward_checkpoints(monkeypatch, shape):
    """The forward pass that writes the unit states gives y and h_last
    bit-identical to ssm_scan_fwd; its checkpoints equal the oracle's states
    at the unit boundaries; the backward that reads them matches the oracle
    and ssm_scan_bwd."""
    batch, L, D, dtype, plan = shape
    if plan:
        monkeypatch.setenv("SSM_FORCE_PLAN", plan)
    inp = inputs(batch, L, D, 16, dtype, 60 + L)
    y, h, ckpt, out = run_ckpt(inp)
    y_ref, h_ref = ssm.scan(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                            inp["Dskip"], inp["z"])
    assert torch.equal(y, y_ref) and torch.equal(h, h_ref)
    tol = parity.TOL[dtype]
    # the states at the unit boundaries, from the oracle's scan of the first 32 k steps
    for k in range(1, (L + 31) // 32):
        sub = {n: (t[:, :32 * k] if t is not None and t.dim() == 3 and n in ("u", "delta", "z", "B", "C")
                   else t) for n, t in inp.items()}
        _, hk = parity.oracle_scan(sub)
        parity.check(parity.to_f64(ckpt[k]), hk, tol, f"checkpoint {k}")
        if k >= 3:
            break
    ref = oracle_bwd(inp)
    compare(out, ref, 1e-4 if dtype == torch.float32 else 2e-2, f"ckpt {shape}")
    plain = run_bwd(inp)
    for k in OUTS:
        if out[k] is not None:
            parity.check(parity.to_f64(out[k]), parity.to_f64(plain[k]),
                         2e-5 if dtype == torch.float32 else 1e-2, f"ckpt vs ssm_scan_bwd {k}")


def test_checkpoints_refuse_other_state_sizes():
    """N != 16 has no unit kernels: both calls refuse before any work."""
    inp = inputs(1, 64, 32, 8, torch.float32, 3)
    ckpt = torch.empty((2, 1, 32, 8), device=DEV)
    y, h = torch.empty_like(inp["u"]), torch.empty((1, 32, 8), device=DEV)
    with pytest.raises(ssm.SsmError) as e:
        ssm.ssm_scan_fwd_ckpt(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"],
                              inp["C"], inp["Dskip"], inp["z"], y, h, ckpt)
    assert e.value.status == -5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bwd_checkpoint_only_walk_matches_forward_checkpoints(monkeypatch, dtype):
    """ssm_scan_bwd, on the chained plan, takes its unit states from the
    forward recurrence's checkpoint-only walk (no readout, no y); the
    training pair takes them from the forward scan proper.  The recurrence is
    the same arithmetic, so every per-element output agrees bit for bit (the
    sums formed with atomic adds, dA, ddt_bias and dDskip, to rounding), on a
    shape with several chains cut into pieces and a ragged last unit."""
    monkeypatch.setenv("SSM_FORCE_PLAN", "chained")
    monkeypatch.setenv("SSM_CHUNK_T", "96")
    inp = inputs(2, 500, 384, 16, dtype, 77)
    _, _, _, pair = run_ckpt(inp)
    own = run_bwd(inp)
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        assert torch.equal(own[k], pair[k]), k
    for k in ("dA", "ddt_bias", "dDskip"):
        parity.check(parity.to_f64(own[k]), parity.to_f64(pair[k]), 1e-5, f"{k}")
