"""The N>1 host path of bench.py on CPU: two gloo ranks (127.0.0.1) reduce their step
times with the same helper the GPU run uses, and get distinct replica batches."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, loc = bench.dist_setup()
    assert (w, r, loc) == (world, rank, rank)
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5], dist)
    dist.barrier()
    out[rank] = (got, bench.replica_seed(rank, 1234))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_use_disjoint_replicas():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    expect = [2.0, 10.0, 0.5]
    assert out[0][0] == expect and out[1][0] == expect
    assert out[0][1] != out[1][1]
