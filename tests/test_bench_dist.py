"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks, the
max-over-ranks time and summed bytes that the weak-scaling line reports, and
rank-0-only printing of the reference arm.  No GPU involved."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    t = bench.max_over_ranks(1.5 + rank, world)        # per-rank time
    b = bench.sum_over_ranks(1000.0 * (rank + 1), world)  # per-rank bytes
    out[rank] = (t, b)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_bytes():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.5, 3000.0)


def test_reference_arm_prints_only_on_rank0(tmp_path):
    """Rank 1 of a torchrun launch exits 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
