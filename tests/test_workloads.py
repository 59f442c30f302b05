"""The seeded input generators follow their stated recipe (CPU only):
deterministic per seed, the workloads' shapes and dtypes, and the value
distributions (N(0, 1) tensors, softplus(dt_bias) log-uniform in
[1e-3, 1e-1], A = -(n+1), the time-invariant variant, the convolution's,
the backward's and the SSD form's parameters)."""
import math

import torch

from selective_state_space_113_b300 import workloads as wl


def _same(a, b):
    assert a.keys() == b.keys()
    for k in a:
        assert (a[k] is None and b[k] is None) or torch.equal(a[k], b[k]), k


def _moments(t, what):
    x = t.float().flatten()
    assert abs(x.mean().item()) < 0.02, what
    assert abs(x.std().item() - 1.0) < 0.02, what


def test_workload_table():
    assert (wl.TINY_F32.batch, wl.TINY_F32.L, wl.TINY_F32.D, wl.TINY_F32.N) == (2, 256, 64, 16)
    assert (wl.MAMBA_130M.batch, wl.MAMBA_130M.L, wl.MAMBA_130M.D) == (8, 2048, 1536)
    assert (wl.MAMBA_2P8B.batch, wl.MAMBA_2P8B.L, wl.MAMBA_2P8B.D) == (4, 4096, 5120)
    assert (wl.LONG_SEQ.batch, wl.LONG_SEQ.L, wl.LONG_SEQ.D) == (1, 1 << 20, 1536)
    assert (wl.DECODE.batch, wl.DECODE.D, wl.DECODE.N, wl.DECODE.steps) == (256, 5120, 16, 64)
    assert wl.TINY_F32.dtype == torch.float32 and wl.TINY_F32_LTI.time_invariant
    for w in (wl.MAMBA_130M, wl.MAMBA_2P8B, wl.LONG_SEQ, wl.DECODE):
        assert w.dtype == torch.bfloat16 and w.N == 16
    # seed = the workload's index
    assert [w.seed for w in (wl.TINY_F32, wl.MAMBA_130M, wl.MAMBA_2P8B, wl.LONG_SEQ,
                             wl.DECODE)] == [0, 1, 2, 3, 4]
    assert wl.MAMBA_2P8B.elements == 4 * 4096 * 5120


def test_scan_inputs_seeded_and_shaped():
    kw = dict(batch=2, L=256, D=256)
    a = wl.make_scan_inputs(wl.MAMBA_130M, **kw)
    _same(a, wl.make_scan_inputs(wl.MAMBA_130M, **kw))
    b = wl.make_scan_inputs(wl.MAMBA_130M, seed=99, **kw)
    assert not torch.equal(a["u"], b["u"])
    for k in ("u", "delta", "z"):
        assert a[k].shape == (2, 256, 256) and a[k].dtype == torch.bfloat16
    for k in ("B", "C"):
        assert a[k].shape == (2, 256, 16) and a[k].dtype == torch.bfloat16
    assert a["A"].shape == (256, 16) and a["dt_bias"].shape == (256,)
    for k in ("A", "dt_bias", "Dskip"):
        assert a[k].dtype == torch.float32
    for k in ("u", "delta", "z", "B", "C"):
        _moments(a[k], k)
    f = wl.make_scan_inputs(wl.TINY_F32)
    assert f["u"].dtype == torch.float32 and f["u"].shape == (2, 256, 64)


def test_channel_parameters_follow_the_recipe():
    p = wl.make_scan_inputs(wl.MAMBA_130M, batch=1, L=2, D=4096)
    n = torch.arange(16, dtype=torch.float32)
    assert torch.equal(p["A"], (-(n + 1)).repeat(4096, 1))
    dt0 = torch.nn.functional.softplus(p["dt_bias"].double())
    assert dt0.min().item() >= 1e-3 * (1 - 1e-5) and dt0.max().item() <= 1e-1 * (1 + 1e-5)
    # log-uniform: log dt0 is uniform on [log 1e-3, log 1e-1]
    ld = torch.log(dt0)
    mid = (math.log(1e-3) + math.log(1e-1)) / 2
    assert abs(ld.mean().item() - mid) < 0.1
    assert abs(ld.std().item() - (math.log(1e-1) - math.log(1e-3)) / math.sqrt(12)) < 0.05
    assert abs(p["Dskip"].mean().item()) < 0.05 and abs(p["Dskip"].std().item() - 1) < 0.05


def test_time_invariant_variant():
    p = wl.make_scan_inputs(wl.TINY_F32_LTI)
    for k in ("delta", "B", "C"):
        assert torch.equal(p[k], p[k][:, :1].expand_as(p[k])), k
    for k in ("u", "z"):
        assert not torch.equal(p[k], p[k][:, :1].expand_as(p[k])), k


def test_step_inputs():
    s = wl.make_step_inputs(wl.DECODE, batch=8, D=64, steps=5)
    _same(s, wl.make_step_inputs(wl.DECODE, batch=8, D=64, steps=5))
    assert s["state"].shape == (8, 64, 16) and s["state"].dtype == torch.float32
    assert s["u"].shape == (5, 8, 64) and s["u"].dtype == torch.bfloat16
    assert s["B"].shape == (5, 8, 16)


def test_conv_and_gradient_inputs():
    w, b = wl.conv_params(4096, 5)
    assert w.shape == (4096, 4) and b.shape == (4096,)
    assert w.min().item() >= -0.5 and w.max().item() < 0.5
    assert abs(w.mean().item()) < 0.02 and abs(w.var().item() - 1 / 12) < 0.005
    dy, dh = wl.grad_inputs(2, 128, 256, 16, torch.bfloat16, 7)
    assert dy.shape == (2, 128, 256) and dy.dtype == torch.bfloat16
    assert dh.shape == (2, 256, 16) and dh.dtype == torch.float32
    _moments(dy, "dy")
    dy2, _ = wl.grad_inputs(2, 128, 256, 16, torch.bfloat16, 7)
    assert torch.equal(dy, dy2)


def test_ssd_inputs():
    s = wl.make_ssd_inputs(wl.SSD_2P7B, batch=1, L=64, H=80)
    assert s["x"].shape == (1, 64, 80, 64) and s["dt"].shape == (1, 64, 80)
    assert s["B"].shape == (1, 64, 128) and s["x"].dtype == torch.bfloat16
    assert s["A"].shape == (80,) and s["A"].min().item() >= -16 and s["A"].max().item() <= -1
    dt0 = torch.nn.functional.softplus(s["dt_bias"].double())
    assert dt0.min().item() >= 1e-3 * (1 - 1e-5) and dt0.max().item() <= 1e-1 * (1 + 1e-5)
    _same(s, wl.make_ssd_inputs(wl.SSD_2P7B, batch=1, L=64, H=80))
    assert (wl.SSD_2P7B.batch, wl.SSD_2P7B.L, wl.SSD_2P7B.H, wl.SSD_2P7B.P,
            wl.SSD_2P7B.N) == (4, 4096, 80, 64, 128)
