"""Multi-process plumbing of bench.py on CPU: two gloo ranks, barrier, the max
over ranks used for the timed region, and disjoint per-rank input seeds (the
path shards over independent (batch, head) units with no data exchange)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import txl_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    out[rank] = (bench.max_over_ranks(float(10 * rank + 3), world),
                 bench.rank_seed(txl_inputs.WORKLOADS[txl_inputs.HEADLINE].seed, rank))
    dist.destroy_process_group()


def test_two_ranks_max_and_disjoint_seeds():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 13.0
    assert out[0][1] != out[1][1]
