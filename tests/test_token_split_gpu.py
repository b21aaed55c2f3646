"""Token-range split of the decode: lrkv_decode_partials over each part of the sequences' tokens
(each part in a cache of its own, as one device would hold it) and lrkv_decode_merge, against
the oracle's decode of the whole sequences.  The parts, one per device in a multi-GPU run, are
run one after another on one GPU here."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402
from compressed_kv_cache_lrkv_gb300.token_split import token_ranges  # noqa: E402

BS = 64


def local_cache(pools, pt, starts, lens):
    """Tokens [starts[b], starts[b] + lens[b]) of every sequence, copied into pools of their own
    (pages numbered from 0, in sequence order) with the block table that addresses them."""
    npg = [(int(n) + BS - 1) // BS for n in lens]
    bt = np.zeros((len(lens), max(1, max(npg))), np.int32)
    nb = sum(npg) + 1
    out = [np.zeros((nb, BS) + p.shape[2:], np.uint16) for p in pools]
    src_flat = [p.reshape((-1,) + p.shape[2:]) for p in pools]
    dst_flat = [o.reshape((-1,) + o.shape[2:]) for o in out]
    nxt = 0
    for bb, n in enumerate(lens):
        n = int(n)
        bt[bb, :npg[bb]] = np.arange(nxt, nxt + npg[bb])
        nxt += npg[bb]
        if n:
            src = S.slots_for(pt, bb, int(starts[bb]), int(starts[bb]) + n).astype(np.int64)
            t = np.arange(n)
            dst = bt[bb, t // BS].astype(np.int64) * BS + t % BS
            for fs, fd in zip(src_flat, dst_flat):
                fd[dst] = fs[src]
    return out, bt


def run_parts(H, d_h, r, pools, pt, lens, q, BK, parts_ranges, status, d_rope=0):
    """Partials of every part, stacked [P, B, H, d_h + r + 2]."""
    dims = b.make_dims(H, d_h, r, H * d_h, d_rope=d_rope)
    qd, bkd = dev_bf16(q), dev_bf16(BK)
    out = []
    for starts, plens in parts_ranges:
        lp, bt = local_cache(pools, pt, starts, plens)
        cache = b.PagedCache(*(dev_bf16(p) for p in lp))
        ws = b.alloc_workspace(b.decode_workspace_bytes(dims, len(lens)))
        part = torch.full((len(lens), H, d_h + r + 2), float("nan"), dtype=torch.float32, device="cuda")
        b.lrkv_decode_partials(dims, qd, bkd, cache, dev_i32(bt), dev_i32(np.asarray(plens, np.int32)), part, ws,
                               status=status)
        out.append(part)
    torch.cuda.synchronize()
    return torch.stack(out)


def merge(H, d_h, r, parts, BV, status, d_rope=0):
    dims = b.make_dims(H, d_h, r, H * d_h, d_rope=d_rope)
    out = torch.empty((parts.shape[1], H, d_h), dtype=torch.bfloat16, device="cuda")
    b.lrkv_decode_merge(dims, parts, dev_bf16(BV), out, status=status)
    torch.cuda.synchronize()
    return out


def split(lens, world):
    starts, plens = token_ranges(lens, world, BS)
    return [(starts[k], plens[k]) for k in range(world)]


CASES = [
    # H, d_h, r, d_rope, sequence lengths, parts -- 128 heads of d_h = 128 take the tcgen05
    # scan; the short sequences leave some parts empty; one case with the positional key
    (8, 64, 16, 0, [700, 150, 64, 1], 3),
    (32, 128, 32, 0, [3000, 1290], 4),
    (128, 128, 16, 0, [2048, 777, 130], 2),
    (4, 64, 8, 0, [1000, 70, 200, 5, 64], 5),
    (16, 128, 16, 64, [1500, 300, 1], 3),
]


@pytest.mark.parametrize("H,d_h,r,d_rope,lens,P", CASES,
                         ids=[f"H{c[0]}_dh{c[1]}_r{c[2]}_rope{c[3]}_P{c[5]}" for c in CASES])
def test_token_split_matches_oracle(H, d_h, r, d_rope, lens, P):
    seed = 900 + H + r + P
    pt = S.page_table(seed, lens, BS, spare_blocks=1)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r, d_rope=d_rope)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(lens), H, d_h + d_rope))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    parts = run_parts(H, d_h, r, pools, pt, lens, q, w.BK, split(lens, P), st, d_rope)
    assert int(st.item()) == 0  # empty parts are not errors
    assert torch.isfinite(parts[..., :-2]).all() and not torch.isnan(parts).any()
    out = merge(H, d_h, r, parts, w.BV, st, d_rope)
    assert int(st.item()) == 0
    ref = oracle.get().decode_cache(pools, pt.block_table, lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"token-split decode H={H} d_h={d_h} r={r} d_rope={d_rope} over {P} parts")


def test_one_part_equals_decode_and_empty_parts_are_neutral():
    """One part merged alone is lrkv_decode (to the rounding of the two normalisation orders);
    a part with no tokens at all (m = -inf, l = 0) changes nothing, bit for bit."""
    H, d_h, r, lens = 16, 128, 16, [900, 65, 300]
    pt = S.page_table(31, lens, BS, spare_blocks=1)
    pools = random_pools(31, pt.num_blocks, H, d_h, r)
    w = weights(31, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(31, "q", (len(lens), H, d_h))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    zeros = np.zeros(len(lens), np.int64)
    parts = run_parts(H, d_h, r, pools, pt, lens, q, w.BK, [(zeros, np.asarray(lens)), (zeros, zeros)], st)
    assert int(st.item()) == 0
    empty = parts[1]
    assert torch.all(empty[..., -2] == float("-inf")) and torch.all(empty[..., -1] == 0)
    assert torch.all(empty[..., :-2] == 0)
    one = merge(H, d_h, r, parts[:1], w.BV, st)
    both = merge(H, d_h, r, parts, w.BV, st)
    assert torch.equal(one, both)
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    ref = torch.empty_like(one)
    b.lrkv_decode(dims, dev_bf16(q), dev_bf16(w.BK), dev_bf16(w.BV), cache, dev_i32(pt.block_table),
                  dev_i32(np.asarray(lens, np.int32)), ref, b.alloc_workspace(b.decode_workspace_bytes(dims, 3)),
                  status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    d = (one.float() - ref.float()).abs()
    ulp = torch.maximum(ref.float().abs(), torch.tensor(2.0 ** -126, device="cuda")) * 2.0 ** -7
    assert torch.all(d <= 2 * ulp), float((d / ulp).max())


def test_merge_flags_a_sequence_no_part_holds():
    H, d_h, r, lens = 4, 64, 8, [200, 0]
    pt = S.page_table(32, [200, 1], BS)
    pools = random_pools(32, pt.num_blocks, H, d_h, r)
    w = weights(32, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(32, "q", (2, H, d_h))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    parts = run_parts(H, d_h, r, pools, pt, lens, q, w.BK, split(lens, 2), st)
    assert int(st.item()) == 0
    out = merge(H, d_h, r, parts, w.BV, st)
    assert int(st.item()) & b.DEV_BAD_SEQLEN
    assert float(out[1].abs().max()) == 0.0
    ref = oracle.get().decode_cache(pools, pt.block_table[:1], [200], w.BK, w.BV, q[:1])
    assert_close(host_f64(out[:1]), ref, "token-split decode next to an empty sequence")
