"""Pins for the float64 oracle: checks against values fixed by the pages and by
mathematics, each independent of the oracle's own code.

Every pin takes an oracle library handle (``oracle.load()`` or a build with a
planted mistake) and raises AssertionError when the oracle disagrees.  The
references here use library routines (scipy's zero-order-hold discretisation,
scipy's IIR filter, an adaptive ODE solver, numpy/torch softplus and SiLU) or
closed forms, never a retyped copy of the oracle's recurrence.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.integrate
import scipy.signal
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers
def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def softplus_ref(x):
    """softplus via numpy's log-add-exp: log(exp(0) + exp(x))."""
    return np.logaddexp(0.0, np.asarray(x, np.float64))


def silu_ref(z):
    """SiLU via scipy's logistic function."""
    z = np.asarray(z, np.float64)
    return z * scipy.special.expit(z)


def zoh_ref(a: float, dt: float):
    """(Abar, Bbar/B) of the scalar system h' = a h + 1*x, by scipy's ZOH."""
    Ad, Bd, _, _, _ = scipy.signal.cont2discrete(
        (np.array([[a]]), np.array([[1.0]]), np.array([[1.0]]), np.array([[0.0]])),
        dt, method="zoh")
    return float(Ad[0, 0]), float(Bd[0, 0])


def random_problem(rng, batch, L, D, N, gate=True, skip=True, bias=True):
    """Small random float32 selective-scan problem (time-varying everything)."""
    u = _f32(rng.standard_normal((batch, L, D)))
    delta = _f32(rng.standard_normal((batch, L, D)))
    z = _f32(rng.standard_normal((batch, L, D))) if gate else None
    B = _f32(rng.standard_normal((batch, L, N)))
    C = _f32(rng.standard_normal((batch, L, N)))
    # distinct, negative A entries (a generic diagonal A, not the -(n+1) init)
    A = _f32(-(0.2 + 2.0 * rng.random((D, N))))
    dt_bias = _f32(np.log(np.expm1(np.exp(rng.uniform(np.log(1e-2), np.log(0.5), D)))))
    Dskip = _f32(rng.standard_normal(D)) if skip else None
    return dict(u=u, delta=delta, dt_bias=dt_bias if bias else None, A=A, B=B,
                C=C, Dskip=Dskip, z=z)


def scan(lib, p, dtype=oracle.F32):
    return oracle.scan_fwd(p["u"], p["delta"], p["dt_bias"], p["A"], p["B"],
                           p["C"], p["Dskip"], p["z"], dtype=dtype, lib=lib)


def _close_scaled(got, want, scale, rtol, what):
    """|got - want| <= rtol * scale, scale the size of the terms summed."""
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bad = ~(err <= rtol * np.asarray(scale))
    assert not bad.any(), (f"{what}: {int(bad.sum())} mismatches, max err "
                           f"{float(np.nanmax(err)):.3e}")


def _close(got, want, rtol, atol, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} mismatches, max err "
                           f"{float(np.nanmax(err)):.3e}")


# ------------------------------------------------------------------- pins
def pin_p2_worked_example(lib):
    """Ultralytics page, 'SSMの仕組み' listing: recurrent form == convolution form.

    Same inputs as the listing (torch seed 0, L=64, N=16, A = -(U+0.5),
    delta = 0.1); the page prints only 'Same outputs: True' at atol 1e-5.
    The convolution kernel K_k = C . (Abar^k * Bbar) is evaluated directly.
    """
    with open(os.path.join(GOLDEN, "p2_worked_example.json")) as f:
        gold = json.load(f)
    L, N = gold["L"], gold["N"]
    torch.manual_seed(gold["seed"])
    x = torch.randn(L)
    A = -(torch.rand(N) + 0.5)
    Bv, Cv = torch.randn(N), torch.randn(N)
    dt_target = gold["delta"]
    dt_bias = _f32([math.log(math.expm1(dt_target))])
    dt = float(softplus_ref(dt_bias.astype(np.float64))[0])  # what the oracle sees
    p = dict(u=_f32(x.numpy().reshape(1, L, 1)),
             delta=_f32(np.zeros((1, L, 1))), dt_bias=dt_bias,
             A=_f32(A.numpy().reshape(1, N)),
             B=_f32(np.tile(Bv.numpy(), (1, L, 1))),
             C=_f32(np.tile(Cv.numpy(), (1, L, 1))), Dskip=None, z=None)
    y, _ = scan(lib, p)
    a = A.numpy().astype(np.float64)
    abar = np.exp(dt * a)
    bbar = (abar - 1.0) / a * Bv.numpy().astype(np.float64)
    K = np.array([Cv.numpy().astype(np.float64) @ (abar ** k * bbar) for k in range(L)])
    xs = x.numpy().astype(np.float64)
    y_conv = np.array([K[: t + 1][::-1] @ xs[: t + 1] for t in range(L)])
    same = bool(np.allclose(y[0, :, 0], y_conv, atol=gold["atol"]))
    assert same == gold["expected_same_outputs"], "page's identity does not hold"
    _close(y[0, :, 0], y_conv, 1e-11, 1e-12, "recurrent vs convolution")


def pin_lti_convolution_with_skip_and_gate(lib):
    """Time-invariant variant (dt, B, C constant in t): y_t = silu(z_t) *
    (sum_k K_k[d] u_{t-k} + D u_t), K_k[d] = sum_n C_n Abar^k Bbar B_n, with
    Abar/Bbar from scipy's ZOH (several channels, batch 2)."""
    rng = np.random.default_rng(11)
    batch, L, D, N = 2, 40, 3, 5
    p = random_problem(rng, batch, L, D, N)
    for key in ("delta", "B", "C"):
        p[key] = _f32(np.repeat(p[key][:, :1, :], L, axis=1))
    y, h = scan(lib, p)
    for b in range(batch):
        for d in range(D):
            dt = float(softplus_ref(p["delta"][b, 0, d] + np.float64(p["dt_bias"][d])))
            K = np.zeros(L)
            for n in range(N):
                ad, bd = zoh_ref(float(p["A"][d, n]), dt)
                K += float(p["C"][b, 0, n]) * ad ** np.arange(L) * bd * float(p["B"][b, 0, n])
            us = p["u"][b, :, d].astype(np.float64)
            conv = np.array([K[: t + 1][::-1] @ us[: t + 1] for t in range(L)])
            want = (conv + float(p["Dskip"][d]) * us) * silu_ref(p["z"][b, :, d])
            _close(y[b, :, d], want, 1e-10, 1e-12, f"LTI conv b={b} d={d}")


def bruteforce_check(lib, rng, batch, L, D, N):
    """The oracle's scan on a random problem of the given shape against the
    brute-force sum h_t = sum_{s<=t} (prod_{r=s+1..t} Abar_r) Bbar_s B_s u_s,
    with no recurrence; ZOH from scipy, softplus from numpy, SiLU from scipy."""
    p = random_problem(rng, batch, L, D, N)
    y, h = scan(lib, p)
    for b in range(batch):
        for d in range(D):
            dts = softplus_ref(p["delta"][b, :, d].astype(np.float64)
                               + np.float64(p["dt_bias"][d]))
            hs = np.zeros((L, N))
            for n in range(N):
                pairs = [zoh_ref(float(p["A"][d, n]), float(dt)) for dt in dts]
                for t in range(L):
                    tot = 0.0
                    for s in range(t + 1):
                        prod = 1.0
                        for r in range(s + 1, t + 1):
                            prod *= pairs[r][0]
                        tot += prod * pairs[s][1] * float(p["B"][b, s, n]) * float(p["u"][b, s, d])
                    hs[t, n] = tot
            Ct = p["C"][b].astype(np.float64)
            want = ((Ct * hs).sum(1) + float(p["Dskip"][d]) * p["u"][b, :, d].astype(np.float64)) \
                * silu_ref(p["z"][b, :, d])
            _close(y[b, :, d], want, 1e-10, 1e-12, f"unrolled y b={b} d={d}")
            _close(h[b, d], hs[-1], 1e-10, 1e-12, f"unrolled h_last b={b} d={d}")


def pin_bruteforce_unrolled(lib):
    """Selective (time-varying) case by brute force (see bruteforce_check)."""
    bruteforce_check(lib, np.random.default_rng(5), 2, 12, 3, 4)


def pin_continuous_time_ode(lib):
    """Zero-order hold is exact for input held constant over each step
    (ta-paperlens page, 仕組み: 'その区間では入力が一定だとみなす'): integrate
    h' = A h + B_t u_t over consecutive intervals of length dt_t with an
    adaptive ODE solver and compare the state and the readout."""
    rng = np.random.default_rng(7)
    batch, L, D, N = 1, 10, 2, 3
    p = random_problem(rng, batch, L, D, N, gate=False)
    y, h = scan(lib, p)
    for d in range(D):
        a = p["A"][d].astype(np.float64)
        dts = softplus_ref(p["delta"][0, :, d].astype(np.float64) + np.float64(p["dt_bias"][d]))
        state = np.zeros(N)
        for t in range(L):
            drive = p["B"][0, t].astype(np.float64) * float(p["u"][0, t, d])
            sol = scipy.integrate.solve_ivp(lambda _s, x: a * x + drive, (0.0, dts[t]),
                                            state, method="DOP853", rtol=1e-12, atol=1e-15)
            state = sol.y[:, -1]
            want_y = float(p["C"][0, t].astype(np.float64) @ state) \
                + float(p["Dskip"][d]) * float(p["u"][0, t, d])
            _close(y[0, t, d], want_y, 1e-8, 1e-10, f"ODE y t={t} d={d}")
        _close(h[0, d], state, 1e-8, 1e-10, f"ODE h_last d={d}")


def pin_constant_input_closed_form(lib):
    """dt, B, u constant: h_t = (B u / -A) (1 - Abar^(t+1)) -> -B u / A."""
    rng = np.random.default_rng(3)
    batch, L, D, N = 1, 60, 2, 4
    p = random_problem(rng, batch, L, D, N, gate=False, skip=False)
    for key in ("delta", "B", "C", "u"):
        p[key] = _f32(np.repeat(p[key][:, :1, :], L, axis=1))
    y, h = scan(lib, p)
    t = np.arange(L, dtype=np.float64)
    for d in range(D):
        dt = float(softplus_ref(p["delta"][0, 0, d] + np.float64(p["dt_bias"][d])))
        uu = float(p["u"][0, 0, d])
        hs = np.zeros((L, N))
        for n in range(N):
            a = float(p["A"][d, n])
            hs[:, n] = (float(p["B"][0, 0, n]) * uu / -a) * (1.0 - np.exp(dt * a * (t + 1)))
        _close(h[0, d], hs[-1], 1e-11, 1e-13, f"closed-form h d={d}")
        _close(y[0, :, d], hs @ p["C"][0, 0].astype(np.float64), 1e-10, 1e-12,
               f"closed-form y d={d}")


def pin_small_dt_keeps_state(lib):
    """dt -> 0 (delta + dt_bias = -40): the state keeps its value (ta-paperlens
    page: a small Delta ignores the input) so h stays 0 and y = D u silu(z);
    the decode step leaves a stored state unchanged."""
    rng = np.random.default_rng(9)
    batch, L, D, N = 2, 20, 3, 4
    p = random_problem(rng, batch, L, D, N, bias=False)
    p["delta"] = _f32(np.full((batch, L, D), -40.0))
    y, h = scan(lib, p)
    assert np.abs(h).max() < 1e-15, "state moved although dt ~ 4e-18"
    want = p["Dskip"][None, None, :].astype(np.float64) * p["u"] \
        * torch.nn.functional.silu(torch.from_numpy(p["z"].astype(np.float64))).numpy()
    _close(y, want, 1e-12, 1e-14, "dt->0 readout")
    st0 = rng.standard_normal((batch, D, N))
    st1, _ = oracle.step(st0, p["u"][:, 0], p["delta"][:, 0], None, p["A"], p["B"][:, 0],
                         p["C"][:, 0], p["Dskip"], p["z"][:, 0], lib=lib)
    _close(st1, st0, 1e-15, 1e-15, "dt->0 step state")


def pin_pure_decay(lib):
    """B = 0 (eigenvalue argument of the ta-paperlens page): the step does
    state <- exp(dt A) * state; the scan's impulse at t = 0 decays as
    Bbar_0 u_0 exp(A sum_{s=1..t} dt_s)."""
    rng = np.random.default_rng(4)
    batch, D, N = 2, 3, 5
    A = _f32(-(0.1 + 3 * rng.random((D, N))))
    dt_bias = _f32(rng.standard_normal(D) - 2)
    u = _f32(rng.standard_normal((batch, D)))
    delta = _f32(rng.standard_normal((batch, D)))
    z = _f32(rng.standard_normal((batch, D)))
    C = _f32(rng.standard_normal((batch, N)))
    Dskip = _f32(rng.standard_normal(D))
    st0 = rng.standard_normal((batch, D, N))
    st1, y1 = oracle.step(st0, u, delta, dt_bias, A, _f32(np.zeros((batch, N))), C,
                          Dskip, z, lib=lib)
    dt = softplus_ref(delta.astype(np.float64) + dt_bias[None, :])
    decay = np.exp(dt[:, :, None] * A[None].astype(np.float64))
    _close(st1, decay * st0, 1e-13, 1e-15, "step decay")
    want_y = ((st1 * C[:, None, :]).sum(-1) + Dskip.astype(np.float64) * u) * silu_ref(z)
    _close(y1, want_y, 1e-12, 1e-14, "step readout")
    # scan impulse
    L = 30
    p = random_problem(rng, 1, L, D, N, gate=False, skip=False)
    p["B"][:, 1:, :] = 0.0
    y, h = scan(lib, p)
    for d in range(D):
        dts = softplus_ref(p["delta"][0, :, d].astype(np.float64) + np.float64(p["dt_bias"][d]))
        for n in range(N):
            a = float(p["A"][d, n])
            _, bd0 = zoh_ref(a, float(dts[0]))
            want = bd0 * float(p["B"][0, 0, n]) * float(p["u"][0, 0, d]) * math.exp(a * dts[1:].sum())
            _close(h[0, d, n], want, 1e-11, 1e-15, f"impulse decay d={d} n={n}")


def pin_ema_special_case(lib):
    """N=1, A=-1, B=C=1, constant dt: h_t = e^-dt h + (1 - e^-dt) u_t, i.e. the
    first-order IIR filter y = lfilter([alpha], [1, alpha-1], u)."""
    rng = np.random.default_rng(2)
    L = 200
    dtb = 0.3
    p = dict(u=_f32(rng.standard_normal((1, L, 1))), delta=_f32(np.zeros((1, L, 1))),
             dt_bias=_f32([dtb]), A=_f32([[-1.0]]), B=_f32(np.ones((1, L, 1))),
             C=_f32(np.ones((1, L, 1))), Dskip=None, z=None)
    y, h = scan(lib, p)
    dt = float(softplus_ref(np.float64(np.float32(dtb))))
    alpha = -math.expm1(-dt)
    want = scipy.signal.lfilter([alpha], [1.0, alpha - 1.0], p["u"][0, :, 0].astype(np.float64))
    _close(y[0, :, 0], want, 1e-12, 1e-14, "EMA")


def pin_zero_A_integrator(lib):
    """A = 0: the ZOH input matrix tends to dt*B and the state integrates,
    h_t = sum_{s<=t} dt_s B_s u_s (cumulative sum)."""
    rng = np.random.default_rng(8)
    L, N = 25, 3
    p = random_problem(rng, 1, L, 1, N, gate=False, skip=False)
    p["A"] = _f32(np.zeros((1, N)))
    y, h = scan(lib, p)
    dts = softplus_ref(p["delta"][0, :, 0].astype(np.float64) + np.float64(p["dt_bias"][0]))
    hs = np.cumsum(dts[:, None] * p["B"][0].astype(np.float64) * p["u"][0, :, :1], axis=0)
    _close(h[0, 0], hs[-1], 1e-12, 1e-14, "integrator h")
    _close(y[0, :, 0], (hs * p["C"][0]).sum(1), 1e-11, 1e-13, "integrator y")


def pin_scan_step_consistency(lib):
    """Training form == inference form: L decode steps from a zero state give
    the scan's y and h_last; scan(L1) + K steps == scan(L1 + K)."""
    rng = np.random.default_rng(6)
    batch, L, D, N = 2, 16, 3, 4
    p = random_problem(rng, batch, L, D, N)
    y, h = scan(lib, p)
    st = np.zeros((batch, D, N))
    ys = []
    for t in range(L):
        st, yt = oracle.step(st, p["u"][:, t], p["delta"][:, t], p["dt_bias"], p["A"],
                             p["B"][:, t], p["C"][:, t], p["Dskip"], p["z"][:, t], lib=lib)
        ys.append(yt)
    _close(np.stack(ys, 1), y, 1e-13, 1e-15, "steps vs scan y")
    _close(st, h, 1e-13, 1e-15, "steps vs scan h_last")
    L1 = 9
    q = {k: (v[:, :L1] if k in ("u", "delta", "z", "B", "C") else v) for k, v in p.items()}
    _, h1 = scan(lib, q)
    st = h1
    for t in range(L1, L):
        st, yt = oracle.step(st, p["u"][:, t], p["delta"][:, t], p["dt_bias"], p["A"],
                             p["B"][:, t], p["C"][:, t], p["Dskip"], p["z"][:, t], lib=lib)
        _close(yt, y[:, t], 1e-13, 1e-15, f"scan+step y t={t}")
    _close(st, h, 1e-13, 1e-15, "scan+step h_last")


def pin_channels_independent(lib):
    """Each (b, d) channel is its own scan: running a channel alone (batch 1,
    D 1, its own A row and parameters) reproduces the full run, and permuting
    channels permutes outputs."""
    rng = np.random.default_rng(12)
    batch, L, D, N = 3, 10, 4, 3
    p = random_problem(rng, batch, L, D, N)
    y, h = scan(lib, p)
    for b in range(batch):
        for d in range(D):
            q = dict(u=p["u"][b:b + 1, :, d:d + 1], delta=p["delta"][b:b + 1, :, d:d + 1],
                     dt_bias=p["dt_bias"][d:d + 1], A=p["A"][d:d + 1],
                     B=p["B"][b:b + 1], C=p["C"][b:b + 1], Dskip=p["Dskip"][d:d + 1],
                     z=p["z"][b:b + 1, :, d:d + 1])
            y1, h1 = scan(lib, q)
            _close(y1[0, :, 0], y[b, :, d], 0, 0, f"channel alone b={b} d={d}")
            _close(h1[0, 0], h[b, d], 0, 0, f"channel alone h b={b} d={d}")
    perm = rng.permutation(D)
    q = dict(p)
    for k in ("u", "delta", "z"):
        q[k] = _f32(p[k][:, :, perm])
    for k in ("dt_bias", "Dskip"):
        q[k] = _f32(p[k][perm])
    q["A"] = _f32(p["A"][perm])
    yp, hp = scan(lib, q)
    _close(yp, y[:, :, perm], 0, 0, "permuted channels y")
    _close(hp, h[:, perm], 0, 0, "permuted channels h")


def pin_optional_inputs(lib):
    """dt_bias = NULL is 0, Dskip = NULL is 0, z = NULL disables the gate
    (then y * silu(z) equals the gated output)."""
    rng = np.random.default_rng(13)
    batch, L, D, N = 2, 8, 3, 4
    p = random_problem(rng, batch, L, D, N)
    y, h = scan(lib, p)
    r = dict(p, dt_bias=_f32(np.zeros(D)))
    _close(scan(lib, dict(p, dt_bias=None))[0], scan(lib, r)[0], 0, 0, "dt_bias NULL")
    r = dict(p, Dskip=_f32(np.zeros(D)))
    _close(scan(lib, dict(p, Dskip=None))[0], scan(lib, r)[0], 0, 0, "Dskip NULL")
    yg, hg = scan(lib, dict(p, z=None))
    _close(yg * silu_ref(p["z"]), y, 1e-13, 1e-15, "z NULL then gate")
    _close(hg, h, 0, 0, "gate does not touch the state")


def pin_bf16_decode(lib):
    """bf16 inputs decode exactly: the bf16 run equals the float32 run on
    torch's own bf16 -> float32 conversion of the same tensors."""
    g = torch.Generator().manual_seed(21)
    batch, L, D, N = 2, 12, 5, 4
    bf = {k: torch.randn(s, generator=g).to(torch.bfloat16)
          for k, s in (("u", (batch, L, D)), ("delta", (batch, L, D)),
                       ("z", (batch, L, D)), ("B", (batch, L, N)), ("C", (batch, L, N)))}
    rng = np.random.default_rng(21)
    A = _f32(-(0.5 + rng.random((D, N))))
    dt_bias = _f32(rng.standard_normal(D) - 2)
    Dskip = _f32(rng.standard_normal(D))
    pb = dict({k: oracle.bits_of(v) for k, v in bf.items()}, A=A, dt_bias=dt_bias, Dskip=Dskip)
    pf = dict({k: v.to(torch.float32).numpy() for k, v in bf.items()}, A=A,
              dt_bias=dt_bias, Dskip=Dskip)
    yb, hb = scan(lib, pb, dtype=oracle.BF16)
    yf, hf = scan(lib, pf, dtype=oracle.F32)
    _close(yb, yf, 0, 0, "bf16 vs f32 decode y")
    _close(hb, hf, 0, 0, "bf16 vs f32 decode h")
    sb, ysb = oracle.step(np.ones((batch, D, N)), pb["u"][:, 0], pb["delta"][:, 0], dt_bias,
                          A, pb["B"][:, 0], pb["C"][:, 0], Dskip, pb["z"][:, 0],
                          dtype=oracle.BF16, lib=lib)
    sf, ysf = oracle.step(np.ones((batch, D, N)), pf["u"][:, 0], pf["delta"][:, 0], dt_bias,
                          A, pf["B"][:, 0], pf["C"][:, 0], Dskip, pf["z"][:, 0],
                          dtype=oracle.F32, lib=lib)
    _close(sb, sf, 0, 0, "bf16 step state")
    _close(ysb, ysf, 0, 0, "bf16 step y")


def step_pipeline_check(lib, rng, batch, D, N):
    """One decode step from a random state, every stage from a library
    routine: softplus (torch), ZOH (scipy), SiLU (torch)."""
    A = _f32(-(0.2 + 2 * rng.random((D, N))))
    dt_bias = _f32(rng.standard_normal(D) - 1)
    u, delta, z = (_f32(rng.standard_normal((batch, D))) for _ in range(3))
    B, C = (_f32(rng.standard_normal((batch, N))) for _ in range(2))
    Dskip = _f32(rng.standard_normal(D))
    st0 = rng.standard_normal((batch, D, N))
    st1, y1 = oracle.step(st0, u, delta, dt_bias, A, B, C, Dskip, z, lib=lib)
    v = torch.from_numpy(delta.astype(np.float64) + dt_bias.astype(np.float64)[None])
    dt = torch.nn.functional.softplus(v, beta=1.0, threshold=1e9).numpy()
    silu = torch.nn.functional.silu(torch.from_numpy(z.astype(np.float64))).numpy()
    want_s = np.zeros_like(st0)
    want_y = np.zeros((batch, D))
    # the size of the terms each result sums: two float64 evaluations of the
    # same sum differ by rounding relative to its terms, not to the sum
    # (which can cancel to near zero)
    scale_s = np.zeros_like(st0)
    scale_y = np.zeros((batch, D))
    for b in range(batch):
        for d in range(D):
            for n in range(N):
                ad, bd = zoh_ref(float(A[d, n]), float(dt[b, d]))
                t1, t2 = ad * st0[b, d, n], bd * float(B[b, n]) * float(u[b, d])
                want_s[b, d, n] = t1 + t2
                scale_s[b, d, n] = abs(t1) + abs(t2)
            cs = C[b].astype(np.float64)
            want_y[b, d] = (want_s[b, d] @ cs + float(Dskip[d]) * float(u[b, d])) * silu[b, d]
            scale_y[b, d] = (np.abs(want_s[b, d]) @ np.abs(cs)
                             + abs(float(Dskip[d]) * float(u[b, d]))) * abs(silu[b, d])
    _close_scaled(st1, want_s, scale_s, 1e-12, "library step state")
    _close_scaled(y1, want_y, scale_y, 1e-12, "library step y")


def pin_step_matches_library_pipeline(lib):
    """One decode step against library routines (see step_pipeline_check)."""
    step_pipeline_check(lib, np.random.default_rng(17), 2, 3, 4)


ALL_PINS = [
    pin_p2_worked_example,
    pin_lti_convolution_with_skip_and_gate,
    pin_bruteforce_unrolled,
    pin_continuous_time_ode,
    pin_constant_input_closed_form,
    pin_small_dt_keeps_state,
    pin_pure_decay,
    pin_ema_special_case,
    pin_zero_A_integrator,
    pin_scan_step_consistency,
    pin_channels_independent,
    pin_optional_inputs,
    pin_bf16_decode,
    pin_step_matches_library_pipeline,
]


# ------------------------------------------------- discretisation variants
def _disc(lib, p, disc):
    return oracle.scan_fwd_disc(p["u"], p["delta"], p["dt_bias"], p["A"], p["B"], p["C"],
                                p["Dskip"], p["z"], disc, dtype=oracle.F32, lib=lib)


def _constant_problem(L, a_vals, dt, b, u):
    """batch 1, D 1, N = len(a_vals): dt, B, u constant in t; C = 1, no gate,
    no skip; dt_bias 0 and delta = softplus^-1(dt) (float32)."""
    N = len(a_vals)
    delta = np.float32(np.log(np.expm1(dt)))
    dt_used = float(softplus_ref(np.float64(delta)))
    return dict(u=_f32(np.full((1, L, 1), u)), delta=_f32(np.full((1, L, 1), delta)),
                dt_bias=None, A=_f32(np.array([a_vals])), B=_f32(np.full((1, L, N), b)),
                C=_f32(np.ones((1, L, N))), Dskip=None, z=None), dt_used


def pin_disc_zoh_is_the_scan(lib):
    """Variant 0 is the zero-order hold of oracle_scan_fwd (same inputs, same
    results up to the order of two float64 products)."""
    rng = np.random.default_rng(40)
    p = random_problem(rng, 2, 24, 5, 6)
    y0, h0 = scan(lib, p)
    y1, h1 = _disc(lib, p, oracle.ZOH)
    _close(y1, y0, 1e-13, 1e-15, "disc 0 y")
    _close(h1, h0, 1e-13, 1e-15, "disc 0 h")


def pin_disc_euler_constant_input(lib):
    """Euler with constant dt, B, u: h_t = dt B u sum_{k<=t} Abar^k
    = dt B u (1 - Abar^(t+1)) / (1 - Abar)  (ta-paperlens pseudocode update)."""
    a_vals, L = [-0.3, -1.1, -2.5], 40
    p, dt = _constant_problem(L, a_vals, 0.07, 0.8, -1.3)
    _, h = _disc(lib, p, oracle.EULER)
    q = np.float64(np.float32(0.8)) * np.float64(np.float32(-1.3))
    ab = np.exp(dt * np.float64(np.float32(a_vals)))
    want = dt * q * (1 - ab ** L) / (1 - ab)
    _close(h[0, 0], want, 1e-12, 1e-14, "Euler constant input")


def pin_disc_trapezoid_constant_input(lib):
    """Trapezoid with constant dt, B, u: h_0 = dt/2 q, then
    h_t = Abar h_{t-1} + dt/2 q (1 + Abar), so
    h_t = Abar^t h_0 + dt/2 q (1 + Abar) (1 - Abar^t) / (1 - Abar)."""
    a_vals, L = [-0.4, -1.7], 33
    p, dt = _constant_problem(L, a_vals, 0.11, -0.6, 0.9)
    _, h = _disc(lib, p, oracle.TRAPEZOID)
    q = np.float64(np.float32(-0.6)) * np.float64(np.float32(0.9))
    ab = np.exp(dt * np.float64(np.float32(a_vals)))
    t = L - 1
    want = ab ** t * (dt / 2 * q) + dt / 2 * q * (1 + ab) * (1 - ab ** t) / (1 - ab)
    _close(h[0, 0], want, 1e-12, 1e-14, "trapezoid constant input")


def pin_disc_orders_against_ode(lib):
    """The error against the continuous system h' = a h + x(s) (ta-paperlens,
    "仕組み: 連続時間の線形システム"), sampled at t_k = k dt from h(-dt) = 0,
    falls with the order the news.han.ihouse.idv.tw page states: O(dt^2) per
    step for Euler (so O(dt) over a fixed span), O(dt^3) per step for the
    trapezoid (O(dt^2) over the span); the zero-order hold of a smooth input
    is first order as well.  Halving dt must divide the error by ~2, ~2, ~4.
    The input is zero up to s = 0 and continuous there (x(0) = 0), which is
    what the trapezoid's start, B_{-1} u_{-1} = 0, assumes."""
    a = -0.7
    x = lambda s: np.where(s > 0, np.sin(1.3 * s) + 0.5 * np.sin(2.1 * s), 0.0)  # noqa: E731
    span = 3.0
    errs = {oracle.ZOH: [], oracle.EULER: [], oracle.TRAPEZOID: []}
    for target in (0.02, 0.01):
        delta = np.float32(np.log(np.expm1(target)))
        dt = float(softplus_ref(np.float64(delta)))
        L = int(round(span / dt)) + 1
        tk = np.arange(L) * dt
        p = dict(u=_f32(x(tk).reshape(1, L, 1)), delta=_f32(np.full((1, L, 1), delta)),
                 dt_bias=None, A=_f32([[a]]), B=_f32(np.ones((1, L, 1))),
                 C=_f32(np.ones((1, L, 1))), Dskip=None, z=None)
        # the float32 samples differ from x by < 1e-7, far below the
        # discretisation errors measured here
        af = float(np.float32(a))
        sol = scipy.integrate.solve_ivp(lambda s, h: af * h + x(s), (-dt, tk[-1]), [0.0],
                                        rtol=1e-12, atol=1e-14)
        exact = sol.y[0, -1]
        for disc in errs:
            _, h = _disc(lib, p, disc)
            errs[disc].append(abs(h[0, 0, 0] - exact))
    for disc, lo, hi in ((oracle.ZOH, 1.7, 2.4), (oracle.EULER, 1.7, 2.4),
                         (oracle.TRAPEZOID, 3.3, 4.8)):
        ratio = errs[disc][0] / errs[disc][1]
        assert lo < ratio < hi, f"disc {disc}: error ratio {ratio:.2f} ({errs[disc]})"


DISC_PINS = [pin_disc_zoh_is_the_scan, pin_disc_euler_constant_input,
             pin_disc_trapezoid_constant_input, pin_disc_orders_against_ode]


# ------------------------------------------------ convolution before the SSM
def _conv(lib, p, w, cb, act):
    return oracle.conv_scan_fwd(p["u"], _f32(w), None if cb is None else _f32(cb), act,
                                p["delta"], p["dt_bias"], p["A"], p["B"], p["C"], p["Dskip"],
                                p["z"], dtype=oracle.F32, lib=lib)


def conv_numpy_check(lib, rng, batch, L, D, N):
    """With B = 0 the state stays 0 and y = Dskip u: with Dskip = 1 and no gate
    y is the convolution output itself, checked against numpy.convolve (causal,
    width 4, w[d, 3] on the current input) plus bias, and SiLU via scipy's
    logistic function for act = 1."""
    p = random_problem(rng, batch, L, D, N, gate=False)
    p["B"] = _f32(np.zeros_like(p["B"]))
    p["Dskip"] = _f32(np.ones(D))
    w = rng.standard_normal((D, 4))
    cb = rng.standard_normal(D)
    for act in (0, 1):
        y, _ = _conv(lib, p, w, cb, act)
        x = np.float64(p["u"])
        wf, cbf = np.float64(np.float32(w)), np.float64(np.float32(cb))
        for b in range(batch):
            for d in range(D):
                v = np.convolve(x[b, :, d], wf[d][::-1])[:L] + cbf[d]
                want = v * scipy.special.expit(v) if act else v
                _close(y[b, :, d], want, 1e-12, 1e-13, f"conv act={act} b={b} d={d}")


def pin_conv_against_numpy(lib):
    """The convolution against numpy.convolve (see conv_numpy_check)."""
    conv_numpy_check(lib, np.random.default_rng(60), 2, 30, 5, 4)


def pin_conv_identity_is_the_scan(lib):
    """Kernel (0, 0, 0, 1), no bias, no activation: u = x, so the result is the
    plain scan of x."""
    rng = np.random.default_rng(61)
    p = random_problem(rng, 2, 20, 4, 6)
    w = np.tile([0.0, 0.0, 0.0, 1.0], (4, 1))
    y, h = _conv(lib, p, w, None, 0)
    y0, h0 = scan(lib, p)
    _close(y, y0, 1e-13, 1e-15, "identity kernel y")
    _close(h, h0, 1e-13, 1e-15, "identity kernel h")


def pin_conv_shift_is_a_delay(lib):
    """Kernel (0, 0, 1, 0): u_t = x_{t-1} (0 at t = 0), the plain scan of the
    delayed input."""
    rng = np.random.default_rng(62)
    p = random_problem(rng, 1, 25, 3, 5)
    w = np.tile([0.0, 0.0, 1.0, 0.0], (3, 1))
    y, h = _conv(lib, p, w, None, 0)
    q = dict(p)
    shifted = np.zeros_like(p["u"])
    shifted[:, 1:] = p["u"][:, :-1]
    q["u"] = _f32(shifted)
    y0, h0 = scan(lib, q)
    # the skip term uses the (delayed) u as well
    _close(y, y0, 1e-13, 1e-15, "delay kernel y")
    _close(h, h0, 1e-13, 1e-15, "delay kernel h")


CONV_PINS = [pin_conv_against_numpy, pin_conv_identity_is_the_scan, pin_conv_shift_is_a_delay]


# ------------------------------------------------- backward-pass pins
def _bwd(lib, p, dy, dh, dtype=oracle.F32):
    return oracle.scan_bwd(p["u"], p["delta"], p["dt_bias"], p["A"], p["B"], p["C"], p["Dskip"],
                           p["z"], dy, dh, dtype=dtype, lib=lib)


def _loss(lib, p, dy, dh):
    """The scalar whose derivatives the backward pass returns:
    sum(dy * y) + sum(dh * h_last), from the (separately pinned) forward."""
    y, h = scan(lib, p)
    out = float(np.sum(dy.astype(np.float64) * y))
    if dh is not None:
        out += float(np.sum(dh.astype(np.float64) * h))
    return out


GRAD_OF = {"u": "du", "delta": "ddelta", "z": "dz", "B": "dB", "C": "dC", "A": "dA",
           "dt_bias": "ddt_bias", "Dskip": "dDskip"}


def pin_bwd_finite_differences(lib):
    """Every gradient element against a central difference of the forward
    scan: (loss(x + e) - loss(x - e)) / (x+ - x-), with the perturbed values
    rounded to float32 first and the actual step used.  One channel has tiny
    and zero A entries (the small-x series and the a == 0 limit)."""
    rng = np.random.default_rng(11)
    p = random_problem(rng, 2, 10, 4, 5)
    p["A"][3] = _f32([-1e-4, -3e-6, 0.0, -2e-3, -1.0])
    dy = _f32(rng.standard_normal(p["u"].shape))
    dh = _f32(rng.standard_normal((2, 4, 5)))
    g = _bwd(lib, p, dy, dh)
    for key, gname in GRAD_OF.items():
        x0 = p[key]
        fd = np.zeros(x0.shape)
        for idx in np.ndindex(x0.shape):
            step = 1e-4 * max(abs(float(x0[idx])), 0.1)
            xp, xm = x0.copy(), x0.copy()
            xp[idx] = np.float32(float(x0[idx]) + step)
            xm[idx] = np.float32(float(x0[idx]) - step)
            lp = _loss(lib, dict(p, **{key: xp}), dy, dh)
            lm = _loss(lib, dict(p, **{key: xm}), dy, dh)
            fd[idx] = (lp - lm) / (float(xp[idx]) - float(xm[idx]))
        _close(g[gname], fd, 1e-6, 1e-6, f"finite differences, {gname}")


def pin_bwd_homogeneity(lib):
    """Exact identities from linearity (Euler's theorem for functions of
    degree 1): with the others fixed, y is linear in C, in u, in B (through
    h) and in Dskip, and the gate depends on none of them.  So, with y0 the
    output at Dskip = 0:  <dC, C> = <dy, y0>;  <du, u> = <dy, y> + <dh, h>;
    <dB, B> = <dy, y0> + <dh, h>;  <dDskip, Dskip> = <dy, y - y0>."""
    rng = np.random.default_rng(12)
    p = random_problem(rng, 2, 30, 6, 4)
    dy = _f32(rng.standard_normal(p["u"].shape))
    dh = _f32(rng.standard_normal((2, 6, 4)))
    g = _bwd(lib, p, dy, dh)
    y, h = scan(lib, p)
    y0, _ = scan(lib, dict(p, Dskip=None))            # the C h part of y (gated)
    dy64, dh64 = dy.astype(np.float64), dh.astype(np.float64)
    pairs = [
        ("C", np.sum(dy64 * y0)),                      # h_last does not depend on C
        ("u", np.sum(dy64 * y) + np.sum(dh64 * h)),
        ("B", np.sum(dy64 * y0) + np.sum(dh64 * h)),
        ("Dskip", np.sum(dy64 * (y - y0))),
    ]
    for key, want in pairs:
        got = float(np.sum(g[GRAD_OF[key]] * p[key].astype(np.float64)))
        _close(got, want, 1e-10, 1e-10, f"homogeneity in {key}")


def bwd_against_autograd(lib, batch, L, D, N, seed):
    rng = np.random.default_rng(seed)
    p = random_problem(rng, batch, L, D, N)
    dy = _f32(rng.standard_normal(p["u"].shape))
    dh = _f32(rng.standard_normal((batch, D, N)))
    g = _bwd(lib, p, dy, dh)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    dt = torch.nn.functional.softplus(t["delta"] + t["dt_bias"])       # [b, L, D]
    a = t["A"]                                                          # [D, N]
    h = torch.zeros((batch, D, N), dtype=torch.float64)
    ys = []
    for step in range(L):
        x = dt[:, step, :, None] * a                                    # [b, D, N]
        h = torch.exp(x) * h + torch.expm1(x) / a * t["B"][:, step, None, :] * t["u"][:, step, :, None]
        s = (h * t["C"][:, step, None, :]).sum(-1) + t["Dskip"] * t["u"][:, step]
        ys.append(s * torch.nn.functional.silu(t["z"][:, step]))
    y = torch.stack(ys, 1)
    loss = (y * torch.tensor(dy, dtype=torch.float64)).sum() + \
        (h * torch.tensor(dh, dtype=torch.float64)).sum()
    grads = torch.autograd.grad(loss, [t[k] for k in GRAD_OF])
    for key, gr in zip(GRAD_OF, grads):
        _close(g[GRAD_OF[key]], gr.numpy(), 1e-9, 1e-9, f"autograd N={N}, {GRAD_OF[key]}")


def pin_bwd_matches_autograd(lib):
    """All gradients against torch.autograd of a float64 torch statement of
    the forward (the derivative is the library's, not a hand derivation)."""
    bwd_against_autograd(lib, 2, 9, 3, 4, 13)


def pin_bwd_largest_state(lib):
    """The same comparison at the largest state size the library takes
    (N = 256, D != N), where a state-index stride or a per-state buffer
    mistake would show."""
    bwd_against_autograd(lib, 1, 6, 3, 256, 15)


def pin_bwd_optional_inputs(lib):
    """NULL gate, skip and bias: the gradients equal those of the explicit
    neutral values (z -> SiLU gate absent, Dskip = 0, dt_bias = 0), and no
    dh_last equals dh_last = 0."""
    rng = np.random.default_rng(14)
    p = random_problem(rng, 1, 12, 3, 4, gate=False, skip=False, bias=False)
    dy = _f32(rng.standard_normal(p["u"].shape))
    g = _bwd(lib, p, dy, None)
    q = dict(p, Dskip=np.zeros(3, np.float32), dt_bias=np.zeros(3, np.float32))
    g2 = _bwd(lib, q, dy, np.zeros((1, 3, 4), np.float32))
    for k in ("du", "ddelta", "dB", "dC", "dA"):
        _close(g[k], g2[k], 0.0, 0.0, f"optional inputs, {k}")
    assert g["dz"] is None


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_homogeneity, pin_bwd_matches_autograd,
            pin_bwd_largest_state, pin_bwd_optional_inputs]


# ------------------------------------------------------ SSD (Mamba-2) pins
def _ssd_problem(rng, batch=2, L=24, H=3, P=4, N=8):
    x = _f32(rng.standard_normal((batch, L, H, P)))
    dt = _f32(rng.standard_normal((batch, L, H)))
    dt_bias = _f32(np.log(np.expm1(np.exp(rng.uniform(np.log(1e-2), np.log(0.5), H)))))
    A = _f32(-(0.1 + 2.0 * rng.random(H)))
    B = _f32(rng.standard_normal((batch, L, N)))
    C = _f32(rng.standard_normal((batch, L, N)))
    Dskip = _f32(rng.standard_normal(H))
    return dict(x=x, dt=dt, dt_bias=dt_bias, A=A, B=B, C=C, Dskip=Dskip)


def _ssd_run(ssd, lib, p):
    return ssd(p["x"], p["dt"], p["dt_bias"], p["A"], p["B"], p["C"], p["Dskip"], lib=lib)


def ssd_masked_matmul_check(lib, rng, ssd=oracle.ssd_fwd, **shape):
    """The pages' duality statement written out: per head, y = (L o C B^T) X
    with the decay mask L[t, s] = exp(a sum_{r=s+1..t} dt_r) dt_s for s <= t
    (0 above the diagonal), plus D x; the final state is
    sum_s exp(a sum_{r>s} dt_r) dt_s B_s^T x_s.  numpy matmuls, float64."""
    p = _ssd_problem(rng, **shape)
    y, h = _ssd_run(ssd, lib, p)
    batch, L, H, P = p["x"].shape
    for b in range(batch):
        CB = p["C"][b].astype(np.float64) @ p["B"][b].astype(np.float64).T      # [t, s]
        for hh in range(H):
            dt = softplus_ref(p["dt"][b, :, hh].astype(np.float64) + float(p["dt_bias"][hh]))
            cum = np.cumsum(dt) * float(p["A"][hh])                              # a sum_{r<=t} dt
            seg = np.exp(np.tril(cum[:, None] - cum[None, :]))                    # exp(a sum_{s<r<=t})
            mask = np.tril(seg * dt[None, :])
            xh = p["x"][b, :, hh, :].astype(np.float64)
            want = (mask * CB) @ xh + float(p["Dskip"][hh]) * xh
            _close(y[b, :, hh, :], want, 1e-10, 1e-10, f"SSD masked matmul b={b} h={hh}")
            wlast = np.exp(cum[-1] - cum) * dt                                     # [s]
            hw = (p["B"][b].astype(np.float64) * wlast[:, None]).T @ xh          # [N, P]
            _close(h[b, hh], hw.T, 1e-10, 1e-10, f"SSD final state b={b} h={hh}")


def pin_ssd_masked_matmul(lib, ssd=oracle.ssd_fwd):
    """The duality statement as masked matrix products (see ssd_masked_matmul_check)."""
    ssd_masked_matmul_check(lib, np.random.default_rng(21), ssd)


def pin_ssd_chunked_form(lib, ssd=oracle.ssd_fwd):
    """The chunked form of the duality (the one the tensor-core kernel uses):
    within each chunk the masked matmul from a zero state, across chunks the
    N x P state carried with the chunk's total decay and read out as
    exp(a cum_t) C_t H.  Chunks of 7 steps over L = 24 (a ragged last chunk)."""
    rng = np.random.default_rng(22)
    p = _ssd_problem(rng)
    y, h = _ssd_run(ssd, lib, p)
    batch, L, H, P = p["x"].shape
    N = p["B"].shape[-1]
    Q = 7
    for b in range(batch):
        for hh in range(H):
            a = float(p["A"][hh])
            dt = softplus_ref(p["dt"][b, :, hh].astype(np.float64) + float(p["dt_bias"][hh]))
            Hs = np.zeros((N, P))
            for t0 in range(0, L, Q):
                t1 = min(t0 + Q, L)
                d = dt[t0:t1]
                cum = np.cumsum(d) * a
                Bc = p["B"][b, t0:t1].astype(np.float64)
                Cc = p["C"][b, t0:t1].astype(np.float64)
                xc = p["x"][b, t0:t1, hh, :].astype(np.float64)
                mask = np.tril(np.exp(np.tril(cum[:, None] - cum[None, :])) * d[None, :])
                yc = (mask * (Cc @ Bc.T)) @ xc + np.exp(cum)[:, None] * (Cc @ Hs) \
                    + float(p["Dskip"][hh]) * xc
                _close(y[b, t0:t1, hh, :], yc, 1e-10, 1e-10, f"SSD chunk t0={t0}")
                w = np.exp(cum[-1] - cum) * d
                Hs = np.exp(cum[-1]) * Hs + (Bc * w[:, None]).T @ xc
            _close(h[b, hh], Hs.T, 1e-10, 1e-10, f"SSD chunked final state b={b} h={hh}")


SSD_PINS = [pin_ssd_masked_matmul, pin_ssd_chunked_form]
