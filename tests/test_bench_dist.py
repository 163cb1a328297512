"""The benchmark's multi-process plumbing on CPU (gloo, world size 2).

The product runs one independent replica per GPU; what the N > 1 path adds is
host logic: the barrier around the timed region, the maximum of the per-rank
times, and rank 0 printing the single JSON line.  These tests run that logic
with the gloo backend on the host, and the CPU reference arm end to end under
torch.distributed.run.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier()
    m = bench.max_over_ranks(float(rank + 1) * 1.5)
    bench.barrier()
    out.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 3.0, 1: 3.0}


def test_max_over_ranks_without_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.5) == 2.5


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched like the driver launches N = 2:
    rank 0 prints one JSON line with impl=reference, rank 1 exits 0 without
    work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "square_256"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["unit"] == "TFLOP/s" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
