"""lrkv_decode on the GPU against the fp64 oracle (E2: same cache bits), plus
invariances and device-side error reporting."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def run_decode(H, d_h, r, pools, pt, q, BK, BV, status=None, scale=0.0):
    dims = b.make_dims(H, d_h, r, H * d_h, softmax_scale=scale)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    Bn = q.shape[0]
    out = torch.empty((Bn, H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, Bn))
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_decode(dims, dev_bf16(q), dev_bf16(BK), dev_bf16(BV), cache, dev_i32(pt.block_table),
                  dev_i32(pt.seq_lens), out, ws, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def decode_case(seed, H, d_h, r, seq_lens, spare=2):
    pt = S.page_table(seed, seq_lens, 64, spare_blocks=spare)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(seq_lens), H, d_h))
    return pt, pools, w, q


SHAPES = [
    # H, d_h, r, seq_lens
    (8, 64, 8, [256]),                      # the small single-layer workload
    (8, 64, 16, [2048, 1, 7, 65, 500]),     # backbone head shape, ragged incl. L=1 and a partial granule
    (32, 128, 32, [3000, 129, 64, 1]),      # long-context head shape, shorter lengths
    (128, 128, 16, [700, 64]),              # DeepSeek-V2-scale heads
    (20, 128, 16, [333, 1024]),             # H not a multiple of 16 (padded head rows)
    (3, 64, 32, [95]),                      # few heads
    (32, 128, 8, [513]),
]


@pytest.mark.parametrize("H,d_h,r,lens", SHAPES, ids=[f"H{s[0]}_dh{s[1]}_r{s[2]}" for s in SHAPES])
def test_decode_matches_oracle(H, d_h, r, lens):
    pt, pools, w, q = decode_case(100 + H + r, H, d_h, r, lens)
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert st == 0
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"decode H={H} d_h={d_h} r={r}")


LONG = [
    # splits longer than the shared-memory ring, so stages are refilled while other
    # consumer groups are still busy (the path the long-context workload takes)
    (32, 128, 32, [32768]),
    (32, 128, 32, [20000, 17000, 31000, 16384]),
    (128, 128, 16, [8192]),
    (8, 64, 16, [40000]),
    (8, 64, 8, [25000, 3]),
]


@pytest.mark.parametrize("H,d_h,r,lens", LONG, ids=[f"H{s[0]}_r{s[2]}_{len(s[3])}seq" for s in LONG])
def test_decode_long_splits_match_oracle(H, d_h, r, lens):
    pt, pools, w, q = decode_case(300 + H + r + len(lens), H, d_h, r, lens)
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert st == 0
    # the oracle on a sample of heads (E2 materialises K_h, V_h per head)
    want = np.zeros((len(lens), H), np.uint8)
    want[:, ::max(1, H // 8)] = 1
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q, want=want)
    got = host_f64(out)
    sel = want.astype(bool)
    assert_close(got[sel], ref[sel], f"long decode H={H} r={r}")
    a2, _ = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert torch.equal(out.view(torch.int16), a2.view(torch.int16))


def test_decode_custom_scale():
    H, d_h, r = 8, 64, 16
    pt, pools, w, q = decode_case(7, H, d_h, r, [300, 80])
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV, scale=0.05)
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q, scale=0.05)
    assert_close(host_f64(out), ref, "custom scale")


def test_decode_is_deterministic_and_page_permutation_invariant():
    H, d_h, r = 32, 128, 32
    pt, pools, w, q = decode_case(11, H, d_h, r, [1500, 700, 64, 3000])
    a, _ = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    a2, _ = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert torch.equal(a.view(torch.int16), a2.view(torch.int16))
    perm = S.permutation(12, "pp", pt.num_blocks)
    pools2 = tuple(np.empty_like(p) for p in pools)
    for p_old, p_new in zip(pools, pools2):
        p_new[perm] = p_old
    pt2 = S.PageTable(np.where(pt.block_table >= 0, perm[np.maximum(pt.block_table, 0)], -1).astype(np.int32),
                      pt.seq_lens, pt.num_blocks)
    c, _ = run_decode(H, d_h, r, pools2, pt2, q, w.BK, w.BV)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_decode_batch_composition_changes_only_rounding():
    """A sequence decoded alone or inside a batch gets the same result up to fp32
    summation order (the split boundaries depend on the whole batch)."""
    H, d_h, r = 32, 128, 16
    pt, pools, w, q = decode_case(13, H, d_h, r, [2000, 900, 4000])
    full, _ = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    sub = S.PageTable(pt.block_table[1:2], pt.seq_lens[1:2], pt.num_blocks)
    one, _ = run_decode(H, d_h, r, pools, sub, q[1:2], w.BK, w.BV)
    x, y = host_f64(full[1]), host_f64(one[0])
    assert np.max(np.abs(x - y)) <= 2 ** -7 * max(1.0, np.max(np.abs(y)))


def test_decode_reports_bad_block_and_bad_length_without_faulting():
    H, d_h, r = 8, 64, 8
    pt, pools, w, q = decode_case(17, H, d_h, r, [200, 100, 50])
    bt = pt.block_table.copy()
    bt[0, 1] = pt.num_blocks + 5          # out-of-range page of sequence 0
    lens = pt.seq_lens.copy()
    lens[2] = 0                           # empty sequence
    bad = S.PageTable(bt, lens, pt.num_blocks)
    out, st = run_decode(H, d_h, r, pools, bad, q, w.BK, w.BV)
    assert st & b.DEV_BAD_BLOCK and st & b.DEV_BAD_SEQLEN
    o = host_f64(out)
    assert np.all(o[2] == 0)
    assert np.all(np.isfinite(o))
    # sequence 1 is untouched by the others' problems
    ref = oracle.get().decode_cache(pools, pt.block_table[1:2], pt.seq_lens[1:2], w.BK, w.BV, q[1:2])
    assert_close(o[1:2], ref, "healthy sequence next to bad ones")


def test_decode_nan_in_unused_slots_does_not_leak():
    """Slots past seq_len (inside the last page) may hold any bits, NaN included."""
    H, d_h, r = 32, 128, 32
    pt, pools, w, q = decode_case(19, H, d_h, r, [70, 130])
    pools = tuple(p.copy() for p in pools)
    nan = np.uint16(0x7FC1)
    for bseq, L in enumerate(pt.seq_lens):
        last = pt.block_table[bseq, (L - 1) // 64]
        for p in pools:
            p[last, L % 64:] = nan if L % 64 else p[last, L % 64:]
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, "NaN in unused slots")
