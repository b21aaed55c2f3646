"""lrkv_decode on the GPU against the fp64 oracle (E2: same cache bits), plus
invariances and device-side error reporting."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, errors, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def run_decode(H, d_h, r, pools, pt, q, BK, BV, status=None, scale=0.0, num_splits=0):
    dims = b.make_dims(H, d_h, r, H * d_h, softmax_scale=scale, num_splits=num_splits)
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
    # many heads (up to eight 16-head warp tiles per stage), ragged
    (128, 128, 16, [1500, 9, 300]),
    (128, 64, 32, [900, 130]),
    (96, 128, 32, [600]),
    (64, 128, 32, [1500, 70]),
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
    (128, 128, 32, [9000, 2000]),
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


def _bf16_ulp(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


SPLITS = [1, 2, 7, 0]


def test_split_count_invariance():
    """The number of pieces the batch's tokens are cut into (num_splits; 0 = one per SM) changes
    only the order of the fp32 sums and which running maximum each probability is taken against.
    Every split count meets the oracle bar.  With flat logits (q = 0, so p = 1 exactly for every
    token) every count sums the same exact products, so the fp32 results agree to ~1e-7 relative
    and the bf16 outputs are equal except where the fp32 value lies within that distance of a
    rounding boundary: at most one ulp apart, in well under 1% of the elements.  With Gaussian
    queries the probabilities are rounded to bf16 (for the tensor-core p . s^V product) against
    different running maxima, so counts differ at that rounding level: rel-L2 <= 2e-3."""
    H, d_h, r = 32, 128, 32
    pt, pools, w, q = decode_case(23, H, d_h, r, [3000, 129, 64, 1, 700])
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    outs = {}
    for ns in SPLITS:
        out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV, num_splits=ns)
        assert st == 0
        outs[ns] = host_f64(out)
        rel, mx = assert_close(outs[ns], ref, f"num_splits={ns}")
        print(f"num_splits={ns}: oracle rel_l2={rel:.2e} max_abs={mx:.2e}")
    for ns in SPLITS[:-1]:
        rel, _ = errors(outs[ns], outs[0])
        print(f"num_splits={ns} vs automatic: rel_l2={rel:.2e}")
        assert rel <= 2e-3, (ns, rel)

    q0 = np.zeros_like(q)
    flat = {}
    for ns in SPLITS:
        out, st = run_decode(H, d_h, r, pools, pt, q0, w.BK, w.BV, num_splits=ns)
        assert st == 0
        flat[ns] = host_f64(out)
    ref0 = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q0)
    assert_close(flat[0], ref0, "flat logits")
    for ns in SPLITS[:-1]:
        d = np.abs(flat[ns] - flat[0])
        frac = float((d > 0).mean())
        print(f"flat logits, num_splits={ns} vs automatic: {frac:.2e} of elements one ulp apart")
        assert np.all(d <= _bf16_ulp(flat[0])), ns
        assert frac <= 1e-2, (ns, frac)


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


def test_expired_wait_reports_timeout_and_gpu_stays_usable(monkeypatch):
    """Failure detection without a fault: with the debugging limit LRKV_DEBUG_WAIT_LIMIT_NS=0 the
    split kernel's pipeline waits give up as soon as a stage is not already there.  The kernel
    then stops consuming, waits (with its full limit) for the copies it has in flight, and exits;
    the call reports LRKV_DEV_TIMEOUT through the status word, and the next decode on the same
    context is correct."""
    H, d_h, r = 32, 128, 32
    pt, pools, w, q = decode_case(29, H, d_h, r, [20000, 9000])
    monkeypatch.setenv("LRKV_DEBUG_WAIT_LIMIT_NS", "0")
    seen = 0
    for _ in range(3):  # a wait is only sure to expire if some stage is not ready at once
        _, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
        seen |= st
        if st & b.DEV_TIMEOUT:
            break
    assert seen & b.DEV_TIMEOUT
    assert seen & ~b.DEV_TIMEOUT == 0
    monkeypatch.delenv("LRKV_DEBUG_WAIT_LIMIT_NS")
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert st == 0
    want = np.zeros((2, H), np.uint8)
    want[:, ::4] = 1
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q, want=want)
    sel = want.astype(bool)
    assert_close(host_f64(out)[sel], ref[sel], "decode after an expired wait")


def test_decode_rejects_head_counts_without_a_group_split():
    """With r = 32 and H >= 105 a stage of all heads' latents does not fit twice in shared memory;
    H a multiple of 8 is scanned in head groups, any other H is refused before any launch."""
    for H, ok in [(109, False), (112, True)]:
        pt, pools, w, q = decode_case(31 + H, H, 64, 32, [70])
        if ok:
            out, st = run_decode(H, 64, 32, pools, pt, q, w.BK, w.BV)
            assert st == 0
            ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
            assert_close(host_f64(out), ref, f"decode H={H} r=32")
        else:
            with pytest.raises(b.LrkvError, match="do not fit"):
                run_decode(H, 64, 32, pools, pt, q, w.BK, w.BV)


@pytest.mark.parametrize("ns", [1, 3, 7, 13, 50, 0])
def test_small_stages_with_segment_edges_inside_a_stage(ns):
    """Small-head shapes stream two granules (16 tokens) per stage; with these split counts and
    ragged lengths the pieces and ranges begin and end inside a stage, whose granules outside the
    segment must be skipped."""
    H, d_h, r = 8, 64, 16
    pt, pools, w, q = decode_case(61, H, d_h, r, [2048, 1, 7, 65, 500, 333, 1000])
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV, num_splits=ns)
    assert st == 0
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"decode H={H} num_splits={ns}")
