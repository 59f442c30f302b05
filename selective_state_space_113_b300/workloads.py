"""Seeded synthetic inputs for the selective scan and the decode step.

This module only draws random inputs; it holds none of the scan's arithmetic.
Both the CUDA library's tests/benchmarks and the float64 oracle consume what it
produces, so the two sides always see bit-identical inputs.

Recipe (the shapes are Mamba layers; the distributions are the ones the
workload definitions fix):
  u, delta, z ~ N(0, 1)   [batch, L, D]      (cast to the workload dtype)
  B, C        ~ N(0, 1)   [batch, L, N]      (cast to the workload dtype)
  dt0         = exp(U(log 1e-3, log 1e-1))   per channel, float32
  dt_bias     = log(expm1(dt0))              per channel, float32
                (so softplus(dt_bias) = dt0: the usual Mamba dt initialisation)
  Dskip       ~ N(0, 1)   [D]                float32
  A[d, n]     = -(n + 1)                     float32 (S4D-real / Mamba init)
  decode state ~ N(0, 1)  [batch, D, N]      float32
  conv_w, conv_b ~ U(-1/2, 1/2)  [D, 4], [D]  float32 (the default init of a
                depthwise width-4 Conv1d, bound 1/sqrt(fan_in) = 1/2), drawn
                by ``conv_params`` from a generator of their own
  backward: dy ~ N(0, 1) [batch, L, D] (workload dtype), dh_last ~ N(0, 1)
                [batch, D, N] float32, by ``grad_inputs`` from a generator of
                their own
Draws happen in float32 from one torch.Generator seeded with the workload's
seed, in the order listed, then are rounded to bf16 where the workload is bf16.
The time-invariant variant repeats the t = 0 draws of delta, B and C along t.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    L: int
    D: int
    N: int
    dtype: torch.dtype
    seed: int
    time_invariant: bool = False

    @property
    def elements(self) -> int:
        return self.batch * self.L * self.D


@dataclasses.dataclass(frozen=True)
class StepWorkload:
    name: str
    batch: int
    D: int
    N: int
    steps: int
    dtype: torch.dtype
    seed: int

    @property
    def elements_per_step(self) -> int:
        return self.batch * self.D


# The five workloads: a tiny fp32 scan (plus its time-invariant variant), the
# Mamba-130M and Mamba-2.8B shaped layer scans, a 2^20-step scan and a
# 64-token decode of 256 sequences.
TINY_F32 = ScanWorkload("tiny_f32_2x256x64_n16", 2, 256, 64, 16, torch.float32, 0)
TINY_F32_LTI = ScanWorkload("tiny_f32_lti_2x256x64_n16", 2, 256, 64, 16,
                            torch.float32, 0, time_invariant=True)
MAMBA_130M = ScanWorkload("mamba130m_8x2048x1536_n16_bf16", 8, 2048, 1536, 16,
                          torch.bfloat16, 1)
MAMBA_2P8B = ScanWorkload("mamba2.8b_4x4096x5120_n16_bf16", 4, 4096, 5120, 16,
                          torch.bfloat16, 2)
LONG_SEQ = ScanWorkload("longseq_1x1048576x1536_n16_bf16", 1, 1 << 20, 1536, 16,
                        torch.bfloat16, 3)
DECODE = StepWorkload("decode_256x5120_n16_bf16_64steps", 256, 5120, 16, 64,
                      torch.bfloat16, 4)

SCAN_WORKLOADS = {w.name: w for w in (TINY_F32, TINY_F32_LTI, MAMBA_130M,
                                      MAMBA_2P8B, LONG_SEQ)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, dtype):
    return torch.randn(shape, generator=g, device=device,
                       dtype=torch.float32).to(dtype)


def channel_params(D: int, N: int, g: torch.Generator, device):
    """dt_bias, Dskip and A for D channels (all float32)."""
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt0 = torch.exp(torch.rand(D, generator=g, device=device) * (hi - lo) + lo)
    dt_bias = torch.log(torch.expm1(dt0)).to(torch.float32)
    Dskip = torch.randn(D, generator=g, device=device, dtype=torch.float32)
    A = -(torch.arange(N, device=device, dtype=torch.float32) + 1.0)
    A = A.unsqueeze(0).repeat(D, 1).contiguous()
    return dt_bias, Dskip, A


def make_scan_inputs(w: ScanWorkload, device="cpu", seed: int | None = None,
                     batch: int | None = None, L: int | None = None,
                     D: int | None = None, N: int | None = None):
    """All inputs of one scan workload as a dict of tensors on ``device``.

    ``batch``/``L``/``D``/``N``/``seed`` override the workload's values (used
    for smaller parity cases with the same distributions).
    """
    batch = w.batch if batch is None else batch
    L = w.L if L is None else L
    D = w.D if D is None else D
    N = w.N if N is None else N
    g = _gen(w.seed if seed is None else seed, device)
    dt = w.dtype
    if w.time_invariant:
        u = _randn((batch, L, D), g, device, dt)
        delta = _randn((batch, 1, D), g, device, dt).expand(batch, L, D).contiguous()
        z = _randn((batch, L, D), g, device, dt)
        B = _randn((batch, 1, N), g, device, dt).expand(batch, L, N).contiguous()
        C = _randn((batch, 1, N), g, device, dt).expand(batch, L, N).contiguous()
    else:
        u = _randn((batch, L, D), g, device, dt)
        delta = _randn((batch, L, D), g, device, dt)
        z = _randn((batch, L, D), g, device, dt)
        B = _randn((batch, L, N), g, device, dt)
        C = _randn((batch, L, N), g, device, dt)
    dt_bias, Dskip, A = channel_params(D, N, g, device)
    return dict(u=u, delta=delta, dt_bias=dt_bias, A=A, B=B, C=C, Dskip=Dskip, z=z)


def conv_params(D: int, seed: int, device="cpu"):
    """conv_w [D, 4] and conv_b [D], float32, U(-1/2, 1/2), for the causal
    convolution in front of the scan (x takes the place of u)."""
    g = _gen(seed, device)
    w = (torch.rand((D, 4), generator=g, device=device) - 0.5).contiguous()
    b = torch.rand(D, generator=g, device=device) - 0.5
    return w, b


def grad_inputs(batch: int, L: int, D: int, N: int, dtype, seed: int, device="cpu"):
    """Upstream derivatives for the backward pass: dy [batch, L, D] ~ N(0, 1)
    in the workload dtype and dh_last [batch, D, N] ~ N(0, 1) float32, from a
    generator of their own."""
    g = _gen(seed, device)
    dy = _randn((batch, L, D), g, device, dtype)
    dh = torch.randn((batch, D, N), generator=g, device=device, dtype=torch.float32)
    return dy, dh


@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    """A Mamba-2 (SSD) layer: H heads of dimension P, one B/C group of state N."""
    name: str
    batch: int
    L: int
    H: int
    P: int
    N: int
    dtype: torch.dtype
    seed: int

    @property
    def elements(self) -> int:
        return self.batch * self.L * self.H * self.P


SSD_SMALL = SsdWorkload("ssd_small_2x256_h4_p64_n128_bf16", 2, 256, 4, 64, 128, torch.bfloat16, 7)
SSD_2P7B = SsdWorkload("mamba2_2.7b_4x4096_h80_p64_n128_bf16", 4, 4096, 80, 64, 128,
                       torch.bfloat16, 8)


def make_ssd_inputs(w: SsdWorkload, device="cpu", seed: int | None = None, **over):
    """Inputs of the SSD form, drawn in this order from one generator:
    x ~ N(0,1) [batch,L,H,P], dt ~ N(0,1) [batch,L,H] (before the softplus),
    B, C ~ N(0,1) [batch,L,N] (input dtype); dt_bias = log(expm1(dt0)) with
    dt0 log-uniform in [1e-3, 1e-1], A = -U(1, 16), Dskip ~ N(0,1) per head
    (float32) -- the Mamba-2 initialisation ranges.  ``over`` replaces
    batch/L/H/P/N."""
    v = {k: over.get(k, getattr(w, k)) for k in ("batch", "L", "H", "P", "N")}
    dtype = over.get("dtype", w.dtype)
    g = _gen(w.seed if seed is None else seed, device)
    b, L, H, P, N = v["batch"], v["L"], v["H"], v["P"], v["N"]
    x = _randn((b, L, H, P), g, device, dtype)
    dt = _randn((b, L, H), g, device, dtype)
    B = _randn((b, L, N), g, device, dtype)
    C = _randn((b, L, N), g, device, dtype)
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt0 = torch.exp(torch.rand(H, generator=g, device=device) * (hi - lo) + lo)
    dt_bias = torch.log(torch.expm1(dt0)).to(torch.float32)
    A = -(1.0 + 15.0 * torch.rand(H, generator=g, device=device))
    Dskip = torch.randn(H, generator=g, device=device, dtype=torch.float32)
    return dict(x=x, dt=dt, dt_bias=dt_bias, A=A, B=B, C=C, Dskip=Dskip)


def make_step_inputs(w: StepWorkload, device="cpu", seed: int | None = None,
                     batch: int | None = None, D: int | None = None,
                     N: int | None = None, steps: int | None = None):
    """Decode inputs: per-step tensors stacked on a leading ``steps`` axis.

    Returns dict with state [batch,D,N] f32, u/delta/z [steps,batch,D],
    B/C [steps,batch,N] (workload dtype) and dt_bias/Dskip/A.
    """
    batch = w.batch if batch is None else batch
    D = w.D if D is None else D
    N = w.N if N is None else N
    steps = w.steps if steps is None else steps
    g = _gen(w.seed if seed is None else seed, device)
    dt = w.dtype
    state = torch.randn((batch, D, N), generator=g, device=device,
                        dtype=torch.float32)
    u = _randn((steps, batch, D), g, device, dt)
    delta = _randn((steps, batch, D), g, device, dt)
    z = _randn((steps, batch, D), g, device, dt)
    B = _randn((steps, batch, N), g, device, dt)
    C = _randn((steps, batch, N), g, device, dt)
    dt_bias, Dskip, A = channel_params(D, N, g, device)
    return dict(state=state, u=u, delta=delta, dt_bias=dt_bias, A=A, B=B, C=C,
                Dskip=Dskip, z=z)
