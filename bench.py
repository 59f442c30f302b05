#!/usr/bin/env python3
"""Benchmark of the selective-scan forward (ssm_scan_fwd) on the Mamba-2.8B
shaped layer: batch 4, L 4096, D 5120, N 16, bf16 inputs, float32 state.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ssm_scan_fwd call over the whole workload (softplus, ZOH
discretisation, recurrence, readout, D skip and SiLU gate, y and h_last
written).  Inputs are synthetic and seeded (selective_state_space_113_b300.
workloads), generated on the device, 674 MB per step (larger than the 126 MB
L2, so no flush is needed between steps).  Rank 0 prints one JSON line.

--impl reference times the float64 CPU oracle (the only other program this
file runs) on the host cores, on a bounded channel sample of the same
workload per step.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan fwd elements/s (B·L·D) and achieved HBM GB/s vs B300 peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
# Work per element of the scan at N = 16, counted by unit.  fp32 multiply-adds:
# 4 per (element, state) -- the decay's exp(dt A) - 1 (the kernel forms it by
# a multiply-add recurrence over n in place of 15 of the 16 exponentials), the
# two of the state update h + e (h + B u / A), and the readout -- 64 in all.
# Special-function results: 5 (softplus: 2^x and log2; exp(dt A[d,0]); the
# SiLU gate: 2^x and 1/x); 20 with the 16 exponentials of the zero-order hold
# taken one by one as written.
FMA_PER_ELEMENT_N16 = 64
SFU_PER_ELEMENT = 5
SFU_PER_ELEMENT_AS_WRITTEN = 20
# The method's own multiply-adds per element as written, without the kernel's
# stand-in for the exponentials: per (element, state) the input term B_bar u,
# the update A_bar h + B_bar u and the readout C h -- 48 in all (the 16
# exponentials themselves are special-function work, counted in
# SFU_PER_ELEMENT_AS_WRITTEN).
FMA_PER_ELEMENT_METHOD = 48


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--workload", default="mamba2.8b", choices=sorted(WORKLOADS),
                    help="scan shape (default: the Mamba-2.8B layer; the others are the "
                         "smaller cases used for ncu captures)")
    ap.add_argument("--L", type=int, default=None,
                    help="override the workload's sequence length (shorter ncu captures)")
    ap.add_argument("--D", type=int, default=None,
                    help="override the workload's channel count (for experiments)")
    return ap.parse_args()


def _workloads():
    from selective_state_space_113_b300 import workloads as wl
    return {"mamba2.8b": wl.MAMBA_2P8B, "mamba130m": wl.MAMBA_130M, "longseq": wl.LONG_SEQ}


def workload(args):
    import dataclasses
    w = _workloads()[args.workload]
    if args.L is not None:
        w = dataclasses.replace(w, name=f"{w.name}_L{args.L}", L=args.L)
    if args.D is not None:
        w = dataclasses.replace(w, name=f"{w.name}_D{args.D}", D=args.D)
    return w


WORKLOADS = ("mamba2.8b", "mamba130m", "longseq")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of the ranks' values (each rank times its own replica; the
    job's time is the slowest rank's).  world == 1 returns the value as is."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _find_key(d, key):
    """The first positive number stored under ``key`` anywhere in a JSON value."""
    if isinstance(d, dict):
        v = d.get(key)
        if isinstance(v, (int, float)) and not isinstance(v, bool) and v > 0:
            return float(v)
        items = d.values()
    elif isinstance(d, list):
        items = d
    else:
        return None
    for v in items:
        got = _find_key(v, key)
        if got is not None:
            return got
    return None


def measured_peaks(path=None):
    """HBM copy bandwidth (GB/s) from MEASURED_PEAKS.json ("measured"), else
    the stated fallback; a file that cannot be read or holds no positive
    ``hbm_gbs`` falls back too, and the kind says so."""
    p = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(p):
        return FALLBACK_HBM_GBS, "fallback"
    try:
        with open(p) as f:
            v = _find_key(json.load(f), "hbm_gbs")
    except (OSError, ValueError):
        v = None
    if v is None:
        return FALLBACK_HBM_GBS, "fallback (MEASURED_PEAKS.json has no usable hbm_gbs)"
    return v, "measured"


def algorithmic_bytes(w) -> int:
    """Bytes the method must move once: u, delta, z read, y written (dtype);
    B, C read; A, dt_bias, Dskip read; h_last written (float32)."""
    es = 2 if "bf16" in w.name else 4
    elems = w.batch * w.L * w.D
    return (4 * elems * es + 2 * w.batch * w.L * w.N * es + w.D * w.N * 4 + 2 * w.D * 4
            + w.batch * w.D * w.N * 4)


# Sources of the timed scan kernel: a recorded DRAM-traffic figure is used only
# while these, and the library's compile flags, are unchanged since it was
# measured.
SCAN_KERNEL_SOURCES = ("scan_tile.cuh", "scan_tile_host.cuh", "ptx.cuh", "common.cuh")


L2_MB = 126.0


def bench_config(w, world: int) -> dict:
    """The workload as both arms' lines name it."""
    io = {"torch.bfloat16": "bf16", "torch.float32": "f32"}[str(w.dtype)]
    mb = algorithmic_bytes(w) / 1e6
    l2 = (f"inputs {mb:.0f} MB per step > 126 MB L2; no flush" if mb > L2_MB else
          f"inputs {mb:.0f} MB per step fit the 126 MB L2; not flushed")
    return {"workload": w.name, "batch": w.batch, "L": w.L, "D": w.D, "N": w.N,
            "io": io, "state": "fp32", "arith": "fp32", "l2": l2,
            "parallelism": f"replicas x{world} (independent workloads per GPU)"}


def csrc_digest() -> str:
    from selective_state_space_113_b300 import build as libbuild
    h = hashlib.sha256()
    h.update("\0".join(libbuild.FLAGS).encode())
    for name in SCAN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "selective_state_space_113_b300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_metric(key: str):
    """A per-launch figure ``key: <number> csrc_sha256: <digest>`` recorded
    under profiles/ from an ncu capture, if the scan kernel's sources have not
    changed since it was taken (else (None, None))."""
    dig = csrc_digest()
    pat = re.compile(re.escape(key) + r":\s*([0-9.eE+]+)\s+csrc_sha256:\s*([0-9a-f]+)")
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for line in open(f):
            m = pat.match(line.strip())
            if m and m.group(2) == dig:
                return float(m.group(1)), os.path.basename(f)
    return None, None


def recorded_traffic():
    """ncu DRAM bytes (read + write) per launch of the scan kernel."""
    v, src = recorded_metric("traffic_bytes_per_launch")
    return (int(v) if v is not None else None), src


def scan_ceilings(rates: dict, hbm_gbs: float, bytes_per_element: float,
                  warp_inst_per_element) -> dict:
    """Elements/s each unit allows the scan: HBM at the measured copy
    bandwidth, the FMA pipes, the special-function unit and instruction issue
    at the rates measured in this process (``rates`` from ssm_unit_ceilings);
    issue only when the kernel's instruction count per element is recorded."""
    c = {"hbm": hbm_gbs * 1e9 / bytes_per_element,
         "fma": rates["fma_per_s"] / FMA_PER_ELEMENT_N16,
         "sfu": rates["ex2_per_s"] / SFU_PER_ELEMENT,
         "issue": (rates["warp_inst_per_s"] / warp_inst_per_element
                   if warp_inst_per_element else None)}
    binding = min((k for k in c if c[k]), key=lambda k: c[k])
    c["sfu_as_written"] = rates["ex2_per_s"] / SFU_PER_ELEMENT_AS_WRITTEN
    c["fma_method"] = rates["fma_per_s"] / FMA_PER_ELEMENT_METHOD
    c["binding"] = binding
    c["unit"] = "elements/s"
    return c


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            self.proc.wait()
            self.t.join(timeout=1)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def bench_ours(args, rank, world, local):
    import torch
    import selective_state_space_113_b300 as ssm
    from selective_state_space_113_b300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = workload(args)
    inp = wl.make_scan_inputs(w, device=dev, seed=w.seed + rank)
    y = torch.empty_like(inp["u"])
    h = torch.empty((w.batch, w.D, w.N), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)

    def call():
        ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                         inp["Dskip"], inp["z"], y, h, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # unit rates of this GPU, measured before (not inside) the timed region
    rates = ssm.ssm_unit_ceilings(reps=5, stream=stream)
    for _ in range(args.warmup):
        call()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        barrier()
        start.record(stream)
        for e0, e1 in ev:
            e0.record(stream)
            call()
            e1.record(stream)
        stop.record(stream)
        barrier()
    total_ms = start.elapsed_time(stop)
    launch_ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
    status = ssm.ssm_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = max_over_ranks(total_ms, world, dev)

    elems = w.elements * world
    value = elems * args.steps / (total_ms / 1e3)
    alg = algorithmic_bytes(w)
    avg_launch_s = sum(launch_ms) / len(launch_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved_gbs = alg / avg_launch_s / 1e9
    achieved_tflops = 2 * FMA_PER_ELEMENT_METHOD * w.elements / avg_launch_s / 1e12
    fma_peak_tflops = 2 * rates["fma_per_s"] / 1e12
    traffic, traffic_src = recorded_traffic()
    inst_pe, inst_src = recorded_metric("warp_inst_per_element")
    ceilings = scan_ceilings(rates, peak, alg / w.elements, inst_pe)
    ceilings["achieved"] = w.elements / avg_launch_s
    ceilings["warp_inst_per_element"] = inst_pe
    ceilings["warp_inst_per_element_source"] = inst_src
    ceilings["measured_rates"] = rates

    variants = None
    if not args.no_variants:
        variants = bench_variants(ssm, inp, w, stream)
    backward = None
    if not args.no_backward:
        backward = bench_backward(ssm, inp, w, stream)
    configs = None
    if not args.no_configs:
        configs = bench_configs(ssm, dev, stream)
    ssd = None
    if not args.no_ssd:
        ssd = bench_ssd(ssm, dev, stream)
    decode = None
    if not args.no_decode:
        decode = bench_decode(ssm, dev, stream)
    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(args, ssm, inp, w, dev, stream, world)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, w)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) u/delta/z/B/C, Mamba dt_bias init, A=-(n+1))",
        "config": bench_config(w, world),
        "hbm_gbs": achieved_gbs,
        "hbm_frac_measured": achieved_gbs / peak,
        "hbm_frac_nominal_8tbs": achieved_gbs / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "traffic": traffic,
                     "peak_source": peak_kind + " HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg,
                     "avg_launch_ms": avg_launch_s * 1e3,
                     "median_launch_ms": launch_ms[len(launch_ms) // 2],
                     "traffic_source": traffic_src,
                     "frac_of_nominal_8tbs": achieved_gbs / NOMINAL_HBM_GBS},
        "alu_roofline": {"bound": "alu", "achieved": achieved_tflops, "peak": fma_peak_tflops,
                         "unit": "TFLOP/s", "frac": achieved_tflops / fma_peak_tflops,
                         "peak_source": "measured in this run: ssm_unit_ceilings, packed fp32 "
                                        "multiply-add stream on all SMs",
                         "flops_per_element": 2 * FMA_PER_ELEMENT_METHOD,
                         "counted": "the method's own work: 3 fp32 multiply-adds per (element, "
                                    "state), the input term, the update and the readout; the "
                                    "16 exponentials are special-function work (ceilings.sfu_"
                                    "as_written); the kernel itself does 4 per state, forming "
                                    "15 of the exponentials by a multiply-add recurrence"},
        "ceilings": ceilings,
        "clocks": clocks.summary(),
        "backward": backward,
        "ssd": ssd,
        "other_configs": configs,
        "decode": decode,
        "discretisation_variants": variants,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_call(w),
        "cpu_baseline": cpu,
    }


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decode step: state read and written (float32),
    u, delta, z read and y written (dtype), B and C rows, A, dt_bias, Dskip."""
    es = 2 if w.dtype == torch_bf16() else 4
    return (2 * w.batch * w.D * w.N * 4 + 4 * w.batch * w.D * es + 2 * w.batch * w.N * es
            + w.D * w.N * 4 + 2 * w.D * 4)


def torch_bf16():
    import torch
    return torch.bfloat16


def bench_decode(ssm, dev, stream, reps: int = 5):
    """The 64-token decode of 256 sequences x D 5120 x N 16 (ssm_step on a
    stored float32 state), as plain launches and replayed as one CUDA graph."""
    import torch
    from selective_state_space_113_b300 import workloads as wl
    w = wl.DECODE
    inp = wl.make_step_inputs(w, device=dev)
    state0 = inp["state"]
    state = state0.clone()
    ys = torch.empty((w.steps, w.batch, w.D), device=dev, dtype=w.dtype)

    def run():
        # torch's current stream: the capturing stream inside torch.cuda.graph
        for s in range(w.steps):
            ssm.ssm_step(state, inp["u"][s], inp["delta"][s], inp["dt_bias"], inp["A"],
                         inp["B"][s], inp["C"][s], inp["Dskip"], inp["z"][s], ys[s])

    def timed(fn):
        best = None
        for _ in range(reps):
            state.copy_(state0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None or ms < best else best
        return best

    for _ in range(2):
        run()
    torch.cuda.synchronize(dev)
    plain_ms = timed(run)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize(dev)
    graph_ms = timed(g.replay)
    # the graph must have done the work: its result equals the plain run's
    state.copy_(state0)
    run()
    ref = state.clone()
    state.copy_(state0)
    g.replay()
    torch.cuda.synchronize(dev)
    if not torch.equal(ref, state):
        raise RuntimeError("decode graph replay differs from plain launches")
    per_step = decode_bytes(w)
    peak, kind = measured_peaks()
    us = graph_ms * 1e3 / w.steps
    gbs = per_step / (us * 1e-6) / 1e9
    # each step with L2 flushed before it, outside the events: a 256 MB
    # buffer (> 126 MB L2) is written and then read back, so the state comes
    # from DRAM and L2 holds only clean lines of the buffer.  A flush that
    # only writes leaves up to 126 MB of the buffer's dirty lines in L2, whose
    # write-back then lands inside the timed step; that figure is reported
    # beside it.
    flush = torch.empty(64 << 20, device=dev, dtype=torch.float32)

    def cold(read_back: bool):
        state.copy_(state0)
        times = []
        for s_ in range(w.steps):
            flush.zero_()
            if read_back:
                flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ssm.ssm_step(state, inp["u"][s_], inp["delta"][s_], inp["dt_bias"], inp["A"],
                         inp["B"][s_], inp["C"][s_], inp["Dskip"], inp["z"][s_], ys[s_])
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return sorted(times)[len(times) // 2] * 1e3

    cold_us = cold(True)
    cold_w_us = cold(False)
    return {"workload": w.name, "steps": w.steps, "bytes_per_step": per_step,
            "us_per_step_graph": us, "us_per_step_launches": plain_ms * 1e3 / w.steps,
            "us_per_step_l2_flushed": cold_us,
            "gbs_l2_flushed": per_step / (cold_us * 1e-6) / 1e9,
            "hbm_frac_l2_flushed": per_step / (cold_us * 1e-6) / 1e9 / peak,
            "us_per_step_l2_write_flushed": cold_w_us,
            "elements_per_s": w.batch * w.D / (us * 1e-6), "gbs": gbs,
            "hbm_frac": gbs / peak, "peak_source": kind, "kernel_launches": w.steps,
            "note": "graph: best of %d replays of the 64 steps (the 84 MB state can stay "
                    "resident in the 126 MB L2 across steps, so GB/s there is algorithmic "
                    "bytes / time, not DRAM traffic); l2_flushed: median step after a "
                    "256 MB write + read-back flush; l2_write_flushed: after a write-only "
                    "flush, which adds the write-back of its dirty lines" % reps}


def bench_configs(ssm, dev, stream, reps: int = 20):
    """The other scan configurations: the tiny fp32 case (time-varying and
    time-invariant), the Mamba-130M layer and the 1M-step sequence (the narrow
    plan; 5 calls), each the median of `reps` calls back to back and the
    median with L2 flushed before each (a 256 MB write outside the events),
    after 5 warm-up calls."""
    import torch
    from selective_state_space_113_b300 import workloads as wl
    flush = torch.empty(64 << 20, device=dev, dtype=torch.float32)
    out = {}
    for w in (wl.TINY_F32, wl.TINY_F32_LTI, wl.MAMBA_130M, wl.LONG_SEQ):
        n_reps = 5 if w is wl.LONG_SEQ else reps
        inp = wl.make_scan_inputs(w, device=dev)
        y = torch.empty_like(inp["u"])
        h = torch.empty((w.batch, w.D, w.N), device=dev)

        def call():
            ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                             inp["Dskip"], inp["z"], y, h, stream=stream)
        for _ in range(5):
            call()
        res = {}
        for tag, cold in (("ms_back_to_back", False), ("ms_l2_flushed", True)):
            # all calls enqueued before one synchronize, so that the GPU never
            # waits for the host between them
            ev = []
            for _ in range(n_reps):
                if cold:
                    with torch.cuda.stream(stream):
                        flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                ev.append((e0, e1))
            stream.synchronize()
            ts = sorted(a.elapsed_time(b) for a, b in ev)
            res[tag] = ts[len(ts) // 2]
        res["elements_per_s"] = w.elements / (res["ms_l2_flushed"] * 1e-3)
        res["hbm_gbs_l2_flushed"] = algorithmic_bytes(w) / (res["ms_l2_flushed"] * 1e-3) / 1e9
        out[w.name] = res
    return out


def bench_variants(ssm, inp, w, stream, reps: int = 5):
    """The Euler and trapezoidal discretisations (ssm_scan_fwd_disc) and the
    convolution in front of the scan (ssm_conv_scan_fwd, SiLU; x in place of u)
    on the same workload, timed like the headline (CUDA events, best of
    `reps`)."""
    import torch
    from selective_state_space_113_b300 import workloads as wl
    y = torch.empty_like(inp["u"])
    h = torch.empty((w.batch, w.D, w.N), device=inp["u"].device, dtype=torch.float32)
    conv_w, conv_b = wl.conv_params(w.D, w.seed + 1000, inp["u"].device)
    out = {}
    for name, disc in (("euler", 1), ("trapezoid", 2), ("conv_silu", None)):
        def call():
            if disc is None:
                ssm.ssm_conv_scan_fwd(inp["u"], conv_w, conv_b, 1, inp["delta"],
                                      inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                                      inp["Dskip"], inp["z"], y, h, stream=stream)
                return
            ssm.ssm_scan_fwd_disc(inp["u"], inp["delta"], inp["dt_bias"], inp["A"], inp["B"],
                                  inp["C"], inp["Dskip"], inp["z"], y, h, disc, stream=stream)
        for _ in range(3):
            call()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None or ms < best else best
        out[name] = {"ms": best, "elements_per_s": w.elements / (best * 1e-3),
                     "hbm_gbs": algorithmic_bytes(w) / (best * 1e-3) / 1e9}
    return out


def bench_backward(ssm, inp, w, stream, reps: int = 5):
    """ssm_scan_bwd on the same workload (dy and dh_last seeded), timed like
    the headline (CUDA events on the launching stream, best of `reps`).
    Algorithmic bytes: u, delta, z, dy read and du, ddelta, dz written (input
    dtype), B, C read and dB, dC written (float32 outputs), the per-channel
    parameters and dA."""
    import torch
    from selective_state_space_113_b300 import workloads as wl
    dev = inp["u"].device
    dy, dh = wl.grad_inputs(w.batch, w.L, w.D, w.N, w.dtype, w.seed + 500, dev)
    u = inp["u"]
    du, ddelta, dz = torch.empty_like(u), torch.empty_like(u), torch.empty_like(u)
    dB = torch.empty((w.batch, w.L, w.N), device=dev)
    dC = torch.empty_like(dB)
    dA = torch.empty((w.D, w.N), device=dev)
    ddt_bias, dDskip = torch.empty(w.D, device=dev), torch.empty(w.D, device=dev)

    def call():
        ssm.ssm_scan_bwd(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                         inp["Dskip"], inp["z"], dy, dh, du, ddelta, ddt_bias, dA, dB, dC, dDskip,
                         dz, stream=stream)
    for _ in range(3):
        call()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None or ms < best else best
    es = 2 if "bf16" in w.name else 4
    nbytes = (7 * es * w.elements + 2 * w.batch * w.L * w.N * (es + 4)
              + w.D * w.N * 8 + w.batch * w.D * w.N * 4 + 6 * w.D * 4)

    # The training pairing: a forward pass that writes the state entering
    # every 32-step unit, and the backward pass that reads them instead of
    # recomputing them (ssm_scan_fwd_ckpt / ssm_scan_bwd_ckpt).
    ckpt = torch.empty(((w.L + 31) // 32, w.batch, w.D, w.N), device=dev)
    y, h = torch.empty_like(u), torch.empty((w.batch, w.D, w.N), device=dev)

    def fwd_ckpt():
        ssm.ssm_scan_fwd_ckpt(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                              inp["Dskip"], inp["z"], y, h, ckpt, stream=stream)

    def bwd_ckpt():
        ssm.ssm_scan_bwd_ckpt(u, inp["delta"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                              inp["Dskip"], inp["z"], dy, dh, ckpt, du, ddelta, ddt_bias, dA, dB,
                              dC, dDskip, dz, stream=stream)

    def best_of(fn):
        for _ in range(3):
            fn()
        b = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            b = ms if b is None or ms < b else b
        return b

    fwd_ckpt_ms = best_of(fwd_ckpt)
    bwd_ckpt_ms = best_of(bwd_ckpt)
    return {"ms": best, "elements_per_s": w.elements / (best * 1e-3),
            "algorithmic_bytes": nbytes, "hbm_gbs": nbytes / (best * 1e-3) / 1e9,
            "kernel_launches": 5 if w.L > 32 else 3,
            "with_forward_checkpoints": {
                "backward_ms": bwd_ckpt_ms, "forward_ms": fwd_ckpt_ms,
                "checkpoint_bytes": ckpt.numel() * 4, "kernel_launches": 4 if w.L > 32 else 3,
                "note": "ssm_scan_bwd_ckpt reading the unit states that ssm_scan_fwd_ckpt "
                        "wrote (no summary pass of its own); forward_ms is that forward "
                        "pass, y and h_last as ssm_scan_fwd plus the states"},
            "note": "one ssm_scan_bwd call: the forward scan's chained walk writing only the "
                    "state entering every 32-step unit, adjoint summaries + carry, the unit "
                    "kernel, the dB/dC reduction; best of %d" % reps}


def bench_ssd(ssm, dev, stream, reps: int = 5):
    """ssm_ssd_fwd (the Mamba-2 form) on a Mamba-2 2.7B-shaped layer (4 x 4096,
    80 heads of 64, N = 128, bf16): one tensor-core launch per call, timed
    like the headline.  Algorithmic FLOPs are those of the chunked form's four
    dense products per 128-step chunk (C B^T, masked scores X, C H, B^T (w x)),
    counted once (the hi + lo operand split, which doubles three of them, is
    not credited)."""
    import torch
    from selective_state_space_113_b300 import workloads as wl
    w = wl.SSD_2P7B
    inp = wl.make_ssd_inputs(w, device=dev)
    y = torch.empty_like(inp["x"])
    h = torch.empty((w.batch, w.H, w.P, w.N), device=dev)

    def call():
        ssm.ssm_ssd_fwd(inp["x"], inp["dt"], inp["dt_bias"], inp["A"], inp["B"], inp["C"],
                        inp["Dskip"], y, h, stream=stream)
    for _ in range(3):
        call()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None or ms < best else best
    Q = 128   # the kernel's chunk length
    chunks = w.batch * w.H * ((w.L + Q - 1) // Q)
    flops = chunks * 2 * (Q * Q * w.N + Q * Q * w.P + 2 * Q * w.N * w.P)
    nbytes = 2 * w.elements * 2 + w.batch * w.L * w.H * 2 + 2 * w.batch * w.L * w.N * 2 \
        + w.batch * w.H * w.P * w.N * 4
    return {"workload": w.name, "ms": best, "elements_per_s": w.elements / (best * 1e-3),
            "algorithmic_flops": flops, "tflops": flops / (best * 1e-3) / 1e12,
            "algorithmic_bytes": nbytes, "hbm_gbs": nbytes / (best * 1e-3) / 1e9,
            "tensor_path": "tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in TMEM), TMA 128B-swizzled "
                           "operand tiles",
            "note": "best of %d; one kernel launch per call (320 heads on 148 SMs: the ticket "
                    "walk, whose workspace counters are cleared by a memset first)" % reps}


def launches_per_call(w) -> int:
    """Kernels of this library one ssm_scan_fwd call launches on ``w``: one for
    the chained plan, three (chunk summaries, carry, output pass) for the plan
    of narrow problems, which the library picks when batch * ceil(D/32) is
    below 0.55 x the resident CTAs (148 SMs x 4)."""
    chains = w.batch * -(-w.D // 32)
    return 3 if chains * 100 < 148 * 4 * 55 else 1


def bench_e2e(args, ssm, inp, w, dev, stream, world):
    """Same metric through the public call with host buffers: every step
    copies its inputs from pinned host memory and reads y and h_last back.
    Steps are pipelined as a user would run them: two sets of device buffers,
    the next step's inputs copied on a second stream while this step's scan
    and read-back run (the two PCIe directions overlap); every copy of every
    timed step lies inside the timed region."""
    import torch
    names = ("u", "delta", "z", "B", "C", "dt_bias", "A", "Dskip")
    host = {k: inp[k].to("cpu").pin_memory() for k in names}
    dbuf = [{k: torch.empty_like(inp[k]) for k in names} for _ in range(2)]
    ys = [torch.empty_like(inp["u"]) for _ in range(2)]
    hs = [torch.empty((w.batch, w.D, w.N), device=dev, dtype=torch.float32) for _ in range(2)]
    y_host = torch.empty(ys[0].shape, dtype=ys[0].dtype).pin_memory()
    h_host = torch.empty(hs[0].shape, dtype=hs[0].dtype).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = y_host.numel() * y_host.element_size() + h_host.numel() * h_host.element_size()
    steps = max(1, min(args.steps, 5))
    copy_in = torch.cuda.Stream(dev)
    landed = [torch.cuda.Event() for _ in range(2)]   # buffer set j holds a step's inputs
    freed = [torch.cuda.Event() for _ in range(2)]    # buffer set j's last scan is done
    for e in freed:
        e.record(stream)

    def one(i):
        j = i & 1
        copy_in.wait_event(freed[j])
        with torch.cuda.stream(copy_in):
            for k in names:
                dbuf[j][k].copy_(host[k], non_blocking=True)
        landed[j].record(copy_in)
        stream.wait_event(landed[j])
        d = dbuf[j]
        ssm.ssm_scan_fwd(d["u"], d["delta"], d["dt_bias"], d["A"], d["B"], d["C"], d["Dskip"],
                         d["z"], ys[j], hs[j], stream=stream)
        with torch.cuda.stream(stream):
            y_host.copy_(ys[j], non_blocking=True)
            h_host.copy_(hs[j], non_blocking=True)
        freed[j].record(stream)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    copy_in.wait_event(s0)
    for i in range(steps):
        one(i)
    s1.record(stream)   # after the last read-back, which waited for every earlier copy
    torch.cuda.synchronize(dev)
    ms = s0.elapsed_time(s1)
    return {"value": w.elements * world * steps / (ms / 1e3), "unit": "elements/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "pipelined": "two buffer sets; inputs of step i+1 copied on a second stream "
                         "during step i's scan and read-back"}


def _oracle_sample(inp, w, channels: int, threads: int):
    """Oracle on the first ``channels`` channels of every batch entry; returns
    (elements, seconds)."""
    import oracle
    host = {k: (None if v is None else oracle.bits_of(v[..., :channels] if k in ("u", "delta", "z")
                                                     else v))
            for k, v in inp.items()}
    host["A"] = oracle.bits_of(inp["A"][:channels])
    host["dt_bias"] = oracle.bits_of(inp["dt_bias"][:channels])
    host["Dskip"] = oracle.bits_of(inp["Dskip"][:channels])
    dt = oracle.BF16 if host["u"].dtype.name == "uint16" else oracle.F32
    t0 = time.perf_counter()
    oracle.scan_fwd(host["u"], host["delta"], host["dt_bias"], host["A"], host["B"], host["C"],
                    host["Dskip"], host["z"], dtype=dt, threads=threads)
    return w.batch * w.L * channels, time.perf_counter() - t0


def cores():
    return len(os.sched_getaffinity(0))


def cpu_baseline(inp, w):
    """The float64 oracle, as it stands, on this host's cores: a channel sample
    of the same workload sized to ~10-30 s of CPU work."""
    n = cores()
    # ~20 core-seconds of work: the oracle runs ~3-4e6 elements/s per core
    channels = min(w.D, max(64, int(20 * 3.5e6 / (w.batch * w.L))))
    channels = max(n, channels - channels % n)
    elems, secs = _oracle_sample(inp, w, channels, n)
    # one core on a sample of the Mamba-130M layer, for scale
    from selective_state_space_113_b300 import workloads as wl
    w1 = wl.MAMBA_130M
    inp1 = wl.make_scan_inputs(w1, device="cpu")
    e1, s1 = _oracle_sample(inp1, w1, 64, 1)
    # the long sequence (1 x 1,048,576 x 1536): every step of a 2n-channel
    # slice drawn with that workload's recipe (the oracle's time depends on
    # the sizes, not on which channels)
    w3 = wl.LONG_SEQ
    ch3 = 2 * n
    inp3 = wl.make_scan_inputs(w3, device="cpu", D=ch3)
    e3, s3 = _oracle_sample(inp3, w3, ch3, n)
    return {"value": elems / secs, "unit": "elements/s", "cores": n, "kind": "oracle",
            "sample": f"all {w.batch}x{w.L} steps of the first {channels} of {w.D} channels "
                      f"({elems} elements, {secs:.1f} s wall, float64)",
            "single_core_mamba130m": {"value": e1 / s1, "unit": "elements/s",
                                      "sample": f"all {w1.batch}x{w1.L} steps of 64 of {w1.D} "
                                                f"channels ({e1} elements, {s1:.1f} s)"},
            "longseq": {"value": e3 / s3, "unit": "elements/s", "cores": n,
                        "sample": f"all {w3.L} steps of {ch3} of {w3.D} channels ({e3} "
                                  f"elements, {s3:.1f} s wall, float64)",
                        "full_workload_s_at_this_rate": w3.elements / (e3 / s3)}}


def bench_reference(args, rank, world):
    """The oracle as the reference arm: each step a channel sample of the workload."""
    if rank != 0:
        return None
    import torch
    from selective_state_space_113_b300 import workloads as wl
    w = workload(args)
    inp = wl.make_scan_inputs(w, device="cpu", seed=w.seed)
    n = cores()
    channels = max(n, min(w.D, 128 * n))
    for _ in range(args.warmup):
        _oracle_sample(inp, w, channels, n)
    tot_e, tot_s = 0, 0.0
    for _ in range(args.steps):
        e, s = _oracle_sample(inp, w, channels, n)
        tot_e += e
        tot_s += s
    value = tot_e / tot_s
    del torch
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": n, "kind": "oracle",
                         "sample": f"per step: all {w.batch}x{w.L} steps of {channels} of "
                                   f"{w.D} channels"},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        out = bench_reference(args, rank, world)
    else:
        out = bench_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
