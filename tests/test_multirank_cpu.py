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


# ---------------------------------------------------------------------------- token-range split
def test_token_ranges_tile_every_sequence_page_aligned():
    """Host side of the token-split decode: each sequence's tokens are cut into one contiguous,
    page-aligned run per rank, in rank order, that together cover [0, L) exactly, with the runs'
    page counts differing by at most one."""
    sys.path.insert(0, ROOT)
    import numpy as np

    from compressed_kv_cache_lrkv_gb300.token_split import token_ranges
    rng = np.random.default_rng(5)
    for world in (1, 2, 3, 4, 8):
        lens = np.concatenate([[1, 63, 64, 65, 128, 0], rng.integers(1, 40000, 20)])
        starts, plens = token_ranges(lens, world, 64)
        assert starts.shape == plens.shape == (world, len(lens))
        assert np.all(plens >= 0)
        assert np.all(starts[0] == 0)
        assert np.all(starts[1:] == starts[:-1] + plens[:-1])  # contiguous, in rank order
        assert np.all(starts[-1] + plens[-1] == lens)           # covers [0, L)
        assert np.all(starts % 64 == 0)
        pages = (plens + 63) // 64
        assert np.all(pages.max(0) - pages.min(0) <= 1)


def _split_rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch

    from compressed_kv_cache_lrkv_gb300.token_split import gather_partials
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # this rank's partials [B, H, d_h + r + 2], recognisable by rank
    mine = torch.full((3, 2, 10), float(rank)) + torch.arange(10.0)
    got = gather_partials(mine)
    out[rank] = got.tolist()
    dist.destroy_process_group()


def test_two_gloo_ranks_gather_token_split_partials_in_rank_order():
    """The one exchange of the token-split decode: every rank receives [world, B, H, W], part k
    being rank k's partials."""
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_split_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    import numpy as np
    for r in range(world):
        got = np.asarray(out[r])
        assert got.shape == (world, 3, 2, 10)
        for k in range(world):
            assert np.all(got[k] == k + np.arange(10.0))
