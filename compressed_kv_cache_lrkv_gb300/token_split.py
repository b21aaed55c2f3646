"""Decode of sequences whose cached tokens are split by token range over several GPUs.

One process per GPU.  Each rank holds, in its own paged cache, one contiguous token range of
every sequence, decodes it into partials with ``lrkv_decode_partials`` (per sequence and head:
the aggregate [acc_s | acc_z], its running maximum m and sum l over the rank's tokens), and one
all-gather hands every rank all ranks' partials, which ``lrkv_decode_merge`` combines by
log-sum-exp and projects through B^V.  The online softmax is associative over any split of the
tokens ("Low-Rank Key Value Attention", frame "Compute logits without expanding historical
keys"), and the residual values are aggregated before B^V is applied (Eq. (7)), so the exchange
is only B * H * (d_h + r + 2) floats per step.

Nothing here computes: the partials and the merge run in the library's kernels; this module
chooses the ranges and moves the partials with torch.distributed.
"""
from __future__ import annotations

import numpy as np

from . import binding as b


def token_ranges(seq_lens, world: int, block_size: int = 64):
    """Each sequence's pages cut into ``world`` contiguous runs of nearly equal length, in rank
    order: returns (starts, lens), int64 arrays [world][B] of each rank's first token and token
    count of every sequence (lens may be 0 where a sequence has fewer pages than ranks)."""
    seq_lens = np.asarray(seq_lens, np.int64)
    if world < 1:
        raise ValueError("world must be >= 1")
    pages = (seq_lens + block_size - 1) // block_size
    r = np.arange(world + 1, dtype=np.int64)[:, None]
    p_edge = (r * pages[None, :]) // world                          # [world + 1][B] page boundaries
    t_edge = np.minimum(p_edge * block_size, seq_lens[None, :])      # token boundaries
    return t_edge[:-1], t_edge[1:] - t_edge[:-1]


def gather_partials(partials, group=None):
    """All-gather of every rank's partials [B, H, W] into [world, B, H, W], in rank order."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(partials) for _ in range(world)]
    dist.all_gather(parts, partials.contiguous(), group=group)
    return torch.stack(parts)


def decode_token_split(dims, q, BK, BV, cache, block_table, seq_lens, out, workspace, group=None, status=None):
    """This rank's part of a token-split decode: ``cache``, ``block_table`` and ``seq_lens`` describe
    the rank's own token range of each sequence (``seq_lens`` may hold zeros); q [B, H, d_h] and the
    weights are the same on every rank; every rank receives the full out [B, H, d_h].  Runs on
    torch's current stream."""
    import torch
    B, H = int(q.shape[0]), int(q.shape[1])
    partials = torch.empty((B, H, dims.d_h + dims.r + 2), dtype=torch.float32, device=q.device)
    b.lrkv_decode_partials(dims, q, BK, cache, block_table, seq_lens, partials, workspace, status=status)
    b.lrkv_decode_merge(dims, gather_partials(partials, group), BV, out, status=status)
