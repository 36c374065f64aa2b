"""The benchmark's multi-process path on CPU: two gloo ranks (no GPU).

The block has no exchange between GPUs, so `bench.py --gpus N` runs N independent replicas;
the only collectives are the barrier around the timed region and the max / sum reductions of
the timings and token counts. This checks those reductions and that the reference arm does its
work on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_init(world)
    bench.dist_barrier(w)
    got = (r, w, local, bench.dist_max(1.5 + r, w), bench.dist_sum(10 * (r + 1), w))
    dist.destroy_process_group()
    q.put(got)


def test_two_gloo_ranks_reduce_max_and_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    for _, _, _, mx, sm in res:
        assert mx == 2.5 and sm == 30.0  # every rank sees the max time and the total tokens


def test_reference_arm_under_torchrun_prints_one_line():
    # rank 0 times the oracle and prints the JSON line; rank 1 exits 0 without work
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert '"impl": "reference"' in lines[0]
