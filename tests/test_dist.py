"""The multi-GPU path of the bench on CPU: two gloo ranks.

Decode shards with no exchange (independent replicas, one per GPU), so the
only multi-process logic is the bench's own: a barrier around the timed
region, the slowest rank's time (max over ranks) and the whole-job rate, and
the reference arm printing one line from rank 0 while the other ranks exit 0
without work.  These run as real processes over gloo on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + rank, w, "cpu")   # rank 1 is the slow one
    rate = bench.whole_job_rate(w, 64, 10, slowest)
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, slowest, rate))


def test_two_rank_barrier_max_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest rank's time and the same whole-job rate:
    # 2 ranks x 64 requests x 10 steps over 2 s
    assert got == [(0, 2.0, 640.0), (1, 2.0, 640.0)]


def test_reference_arm_under_torchrun_prints_once(orc):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "3", "--warmup", "3"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "tiny"
