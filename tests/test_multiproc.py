"""The bench's multi-rank host logic on CPU with the gloo backend, world size
2: every rank processes its own batch (replicas: requests are independent,
no data-path collective), the step time is the maximum over ranks, and only
rank 0 prints the reference arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_rejection_gb300 import synthetic as S
    w, r, _ = bench.dist_setup()
    # each rank times its own batch; the step time reported is the slowest
    t = bench.max_over_ranks(1.5 + r, w)
    bench.barrier(w)
    # per-rank inputs: the bench offsets the input seed by 7919 per rank
    lb = S.make_linear(1, input_seed=S.INPUT_SEED_BASE + 1 + 7919 * r)
    q.put((r, t, float(lb.target.float().sum())))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_distinct_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert [g[1] for g in got] == [2.5, 2.5]
    assert got[0][2] != got[1][2]


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--config", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
