"""The N > 1 path of the benchmark on CPU: world_size-2 gloo process groups.

On several GPUs the bench runs independent replicas of the emulated data-parallel group (one
per GPU, no collective on the data path); the only cross-rank operations are the barrier, the
max-over-ranks of the timed region and rank 0's report.  Those run here over gloo.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        env = bench.dist_env()
        slowest = bench.max_over_ranks(1.0 + 2.0 * rank, dist)     # rank times 1.0 s, 3.0 s
        value = bench.job_value(1000, 10, world, slowest)
        # the reference arm prints on rank 0 only; the other ranks exit without work
        out = io.StringIO()
        args = type("A", (), dict(config=0, steps=1, warmup=0, cpu_sample_elems=4096))()
        with redirect_stdout(out):
            bench.reference_arm(args, world, rank)
        dist.barrier()
        q.put((rank, env, slowest, value, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, slowest, value, printed in res:
        assert env == (world, rank, rank)
        assert slowest == 3.0                                # every rank sees the slowest
        assert value == pytest.approx(2 * 1000 * 10 / 3.0)  # all replicas' work / slowest time
    line = json.loads(res[0][4])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert res[1][4] == ""


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None) == 2.5
    assert bench.job_value(10, 3, 1, 2.0) == 15.0
