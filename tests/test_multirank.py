"""The N > 1 launch path of bench.py on CPU: world_size 2 over gloo.

The decode step does not shard across GPUs here (replicas only: each rank
decodes its own token stream, no exchange step), so what there is to cover
is the plumbing: the barrier around the timed region, the max over ranks of
the timed duration (the slowest rank's time sets the whole job's), and the
reference arm under torchrun, which rank 0 alone runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(1.5 + rank, world)  # rank 1 is the slow one
        bench.barrier(world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(3.25, 1) == 3.25


@pytest.mark.parametrize("workload", ["gemv_q4_k_64x512"])
def test_reference_arm_under_torchrun(workload):
    """torchrun with two ranks: rank 0 prints one JSON line, rank 1 exits 0
    without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", workload, "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
