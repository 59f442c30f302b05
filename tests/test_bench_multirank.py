"""bench.py's multi-GPU bookkeeping on CPU: two gloo ranks, each timing its own
replica, agree on the slowest rank's time (what the bench reports), the
rank/world environment is read as torchrun sets it, and the reference arm
under torchrun prints from rank 0 alone."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    # rank 0 is the faster replica, rank 1 the slower one
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    out.put((r, w, local, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as two torchrun ranks: rank 0 alone
    runs the oracle and prints one JSON line; the other rank exits 0 without
    work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--L", "64"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["e2e"]["h2d_bytes_per_step"] == 0
    assert out["config"]["workload"].endswith("_L64")
