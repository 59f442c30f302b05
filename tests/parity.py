"""Helpers for GPU-vs-oracle parity: run the CUDA path through the C ABI and the
float64 oracle on the same (seeded) inputs, and compare element by element.

Tolerances are the ones the scan is specified to: float32 inputs
|err| <= 1e-4 * (1 + |y_ref|); bf16 inputs with a float32 state
|err| <= 2e-2 * (1 + |y_ref|), for y and for h_last alike.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def dtype_code(t: torch.dtype) -> int:
    return oracle.F32 if t == torch.float32 else oracle.BF16


def host(t):
    return None if t is None else oracle.bits_of(t)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check(got, ref, tol, what):
    """Assert |got - ref| <= tol * (1 + |ref|) everywhere; return max err/(1+|ref|)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    rel = np.abs(got - ref) / (1.0 + np.abs(ref))
    bad = ~(rel <= tol)
    if bad.any():
        idx = np.unravel_index(int(np.argmax(np.where(bad, rel, -1))), rel.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{rel.size} outside tol {tol}; "
                             f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")
    return float(rel.max()) if rel.size else 0.0


def oracle_scan(inp: dict, threads: int = 8):
    """Oracle on the full problem (inputs may live on the GPU)."""
    dt = dtype_code(inp["u"].dtype)
    return oracle.scan_fwd(host(inp["u"]), host(inp["delta"]), host(inp["dt_bias"]),
                           host(inp["A"]), host(inp["B"]), host(inp["C"]),
                           host(inp["Dskip"]), host(inp.get("z")), dtype=dt,
                           threads=threads)


def oracle_scan_channels(inp: dict, chans, threads: int = 8):
    """Oracle on sampled channels only.  ``chans`` is a list of (b, d).

    Channels are independent, so each batch entry's sampled channels form a
    sub-problem with the same B/C rows and those channels' parameters.
    Returns {(b, d): (y [L], h_last [N])}.
    """
    dt = dtype_code(inp["u"].dtype)
    by_b = {}
    for b, d in chans:
        by_b.setdefault(int(b), []).append(int(d))
    out = {}
    for b, ds in by_b.items():
        ds = sorted(set(ds))
        idx = torch.tensor(ds, device=inp["u"].device)
        sub = lambda t: None if t is None else t[b:b + 1].index_select(2, idx)  # noqa: E731
        par = lambda t: None if t is None else t.index_select(0, idx)  # noqa: E731
        y, h = oracle.scan_fwd(host(sub(inp["u"])), host(sub(inp["delta"])),
                               host(par(inp["dt_bias"])), host(par(inp["A"])),
                               host(inp["B"][b:b + 1]), host(inp["C"][b:b + 1]),
                               host(par(inp["Dskip"])), host(sub(inp.get("z"))),
                               dtype=dt, threads=threads)
        for j, d in enumerate(ds):
            out[(b, d)] = (y[0, :, j], h[0, j])
    return out


def sample_channels(batch: int, D: int, count: int, seed: int = 0):
    """Deterministic channel sample that always includes the corners."""
    rng = np.random.default_rng(seed)
    chans = {(0, 0), (batch - 1, D - 1), (0, D - 1), (batch - 1, 0)}
    while len(chans) < min(count, batch * D):
        chans.add((int(rng.integers(batch)), int(rng.integers(D))))
    return sorted(chans)


def chain_channels(batch: int, D: int, per_chain: int = 3, block: int = 128, seed: int = 0):
    """Channels that touch every 128-channel chain of the fast kernel: for each
    (batch entry, channel block), its first and last channel plus
    ``per_chain - 2`` others drawn from the block.  A chain is cut only along
    the sequence, so each CTA's static range of chain-major stages starts
    and ends in chains whose first and last channels are all in the sample."""
    rng = np.random.default_rng(seed)
    chans = set()
    for b in range(batch):
        for c0 in range(0, D, block):
            c1 = min(c0 + block, D) - 1
            chans.update({(b, c0), (b, c1)})
            for _ in range(max(0, per_chain - 2)):
                chans.add((b, int(rng.integers(c0, c1 + 1))))
    return sorted(chans)
