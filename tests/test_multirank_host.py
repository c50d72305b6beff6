"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The prefill has no exchange step: every rank runs its own replica and the job's
time is the slowest rank's.  These tests run two processes and check the pieces
that make that true without a GPU: the max-over-ranks reduction and barrier, and
that under a 2-rank launch only rank 0 prints the reference arm's line.
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(world)
    mx = bench.max_over_ranks(1.5 + rank, world)      # rank 1 is the slow one
    out[rank] = mx
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(2.5) and out[1] == pytest.approx(2.5)


def test_reference_arm_prints_on_rank_zero_only():
    """bench.py --impl reference under a 2-rank launch: rank 0 prints one JSON line with
    impl = reference, rank 1 exits 0 without output (the oracle runs on rank 0 only)."""
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "0"],
                           env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append([l for l in r.stdout.splitlines() if l.strip()])
    assert len(outs[0]) == 1 and outs[1] == []
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
