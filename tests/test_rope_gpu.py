"""Decode, absorbed-weights decode and chunked prefill with the decoupled positional key
(d_rope = 64) on the GPU against the fp64 oracle.

The shared key row is [s^K | k^R] and the query [q | q^R] (q^R rotated by the caller); the
logit of head h is q . (s^K + B_h^K z^K_h) + q^R . k^R, scaled by 1/sqrt(d_h + d_rope) unless
the caller gives a scale ("Low-Rank Key Value Attention", combination with MLA-style latent
caches, whose decoupled rotary key is one vector per token shared by all heads).  Values carry
no positional part, so outputs keep their widths.
"""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import empty_pools, pack_wcat_t, random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402

D_ROPE = 64


def _dims(H, d_h, r, scale=0.0):
    return b.make_dims(H, d_h, r, H * d_h, softmax_scale=scale, d_rope=D_ROPE)


def run_decode(H, d_h, r, pools, pt, q, BK, BV, scale=0.0, seq_lens=None):
    dims = _dims(H, d_h, r, scale)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    Bn = q.shape[0]
    out = torch.empty((Bn, H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, Bn))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = pt.seq_lens if seq_lens is None else seq_lens
    b.lrkv_decode(dims, dev_bf16(q), dev_bf16(BK), dev_bf16(BV), cache, dev_i32(pt.block_table), dev_i32(lens), out,
                  ws, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def rope_case(seed, H, d_h, r, seq_lens):
    pt = S.page_table(seed, seq_lens, 64, spare_blocks=2)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r, d_rope=D_ROPE)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(seq_lens), H, d_h + D_ROPE))
    return pt, pools, w, q


DECODE_SHAPES = [
    # H, d_h, r, seq_lens
    (8, 64, 8, [256]),
    (8, 64, 16, [2048, 1, 7, 65, 500]),
    (32, 128, 32, [3000, 129, 64, 1]),
    (128, 128, 16, [700, 64]),
    (20, 128, 16, [333, 1024]),
    (3, 64, 32, [95]),
    (32, 128, 16, [20000, 9000, 31000, 17000]),  # long contexts: splits longer than the ring
]


@pytest.mark.parametrize("H,d_h,r,lens", DECODE_SHAPES,
                         ids=[f"H{s[0]}_dh{s[1]}_r{s[2]}_n{len(s[3])}" for s in DECODE_SHAPES])
def test_rope_decode_matches_oracle(H, d_h, r, lens):
    pt, pools, w, q = rope_case(400 + H + r + len(lens), H, d_h, r, lens)
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV)
    assert st == 0
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"decode with positional key H={H} d_h={d_h} r={r}")


def test_rope_decode_explicit_scale_and_bad_length():
    H, d_h, r = 8, 128, 16
    pt, pools, w, q = rope_case(411, H, d_h, r, [300, 200])
    lens = pt.seq_lens.copy()
    lens[1] = 0
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV, scale=0.05, seq_lens=lens)
    assert st & b.DEV_BAD_SEQLEN
    got = host_f64(out)
    assert np.all(got[1] == 0)
    ref = oracle.get().decode_cache(pools, pt.block_table[:1], lens[:1], w.BK, w.BV, q[:1], scale=0.05)
    assert_close(got[:1], ref, "decode with positional key, explicit scale")


def test_rope_decode_zero_positional_query_is_plain_decode_over_content():
    """q^R = 0 removes the positional term: every extra product is an exact zero, so with the same
    scale given to both calls the result equals the plain decode over the content columns bit for bit
    (same split plan: the ring holds the same number of stages for both row widths here)."""
    H, d_h, r = 8, 64, 16
    pt, pools, w, q = rope_case(412, H, d_h, r, [500, 77])
    q = q.copy()
    q[..., d_h:] = 0
    scale = float(np.float32(1.0 / np.sqrt(d_h + D_ROPE)))
    out, st = run_decode(H, d_h, r, pools, pt, q, w.BK, w.BV, scale=scale)
    assert st == 0
    plain = b.make_dims(H, d_h, r, H * d_h, softmax_scale=scale)
    cache = b.PagedCache(*(dev_bf16(p) for p in (np.ascontiguousarray(pools[0][..., :d_h]),) + tuple(pools[1:])))
    pout = torch.empty((2, H, d_h), dtype=torch.bfloat16, device="cuda")
    b.lrkv_decode(plain, dev_bf16(np.ascontiguousarray(q[..., :d_h])), dev_bf16(w.BK), dev_bf16(w.BV), cache,
                  dev_i32(pt.block_table), dev_i32(pt.seq_lens), pout,
                  b.alloc_workspace(b.decode_workspace_bytes(plain, 2)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_f64(out), host_f64(pout))


FUSED_SHAPES = [(8, 64, 16, [2048, 1, 7, 65, 500]), (32, 128, 32, [3000, 129, 64, 1]), (128, 128, 16, [700, 64]),
                (32, 128, 16, [20000, 9000])]


@pytest.mark.parametrize("H,d_h,r,lens", FUSED_SHAPES,
                         ids=[f"H{s[0]}_dh{s[1]}_r{s[2]}_n{len(s[3])}" for s in FUSED_SHAPES])
def test_rope_fused_decode_matches_oracle(H, d_h, r, lens):
    pt, pools, _, q = rope_case(420 + H + r, H, d_h, r, lens)
    qt = S.gaussian_bf16(420 + H + r, "qt", (len(lens), H, r))
    dims = _dims(H, d_h, r)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    out = torch.empty((len(lens), H, d_h + r), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_decode_fused(dims, dev_bf16(q), dev_bf16(qt), cache, dev_i32(pt.block_table), dev_i32(pt.seq_lens), out,
                        b.alloc_workspace(b.decode_workspace_bytes(dims, len(lens))), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.get().decode_fused(pools, pt.block_table, pt.seq_lens, q, qt)
    assert_close(host_f64(out), ref, f"fused decode with positional key H={H} d_h={d_h} r={r}")


PREFILL_CASES = [
    # H, d_h, r, Tq, q_starts
    (4, 64, 8, 64, [0, 64]),
    (4, 64, 16, 130, [0, 100]),
    (3, 64, 32, 17, [511, 5]),
    (2, 128, 16, 200, [0, 300]),
    (4, 128, 32, 1, [0, 1000]),
    (8, 128, 16, 96, [256, 0]),
    (2, 128, 8, 70, [63, 1]),
    # d_h = 128, r = 16 runs the tcgen05 kernel (two-stage key ring of [s^K | k^R] rows):
    # ragged query tiles, contexts not aligned to pages or key tiles, a 4096-token prompt's
    # last chunk, one key tile only
    (1, 128, 16, 300, [37, 0]),
    (3, 128, 16, 512, [3584, 1000]),
    (2, 128, 16, 129, [127, 64]),
    (8, 128, 16, 1, [4095, 0]),
    (2, 128, 16, 40, [0, 60]),
]


@pytest.mark.parametrize("H,d_h,r,Tq,qs", PREFILL_CASES,
                         ids=[f"H{c[0]}_dh{c[1]}_r{c[2]}_T{c[3]}" for c in PREFILL_CASES])
def test_rope_prefill_matches_oracle(H, d_h, r, Tq, qs):
    seed = 430 + H + r + Tq
    pt = S.page_table(seed, [s + Tq for s in qs], 64, spare_blocks=1)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r, d_rope=D_ROPE)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(qs), Tq, H, d_h + D_ROPE))
    q_start = np.array(qs, np.int32)
    dims = _dims(H, d_h, r)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    out = torch.empty((len(qs), Tq, H, d_h), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_prefill(dims, dev_bf16(q), dev_bf16(w.BK), dev_bf16(w.BV), cache, dev_i32(pt.block_table),
                   dev_i32(q_start), out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.get().prefill_cache(pools, pt.block_table, q_start, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"prefill with positional key H={H} d_h={d_h} r={r} Tq={Tq}")


def test_rope_append_then_decode_end_to_end():
    """Hidden rows appended at their positions (the positional key rotated in the append kernel),
    then one decode step per sequence: against the oracle's append and decode of the same inputs."""
    H, d_h, r, d = 8, 128, 16, 1024
    lens = [300, 64, 1]
    pt = S.page_table(440, lens, 64, spare_blocks=1)
    w = weights(440, d, d_h, H, r)
    WKR = S.gaussian_bf16(440, "WKR", (d, D_ROPE), d ** -0.5)
    dims = b.make_dims(H, d_h, r, d, d_rope=D_ROPE)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(pt.num_blocks, H, d_h, r, d_rope=D_ROPE)))
    ref_pools = empty_pools(pt.num_blocks, H, d_h, r, d_rope=D_ROPE)
    wcat = dev_bf16(pack_wcat_t(w, WKR))
    for bi, L in enumerate(lens):
        X = S.gaussian_bf16(441 + bi, "X", (L, d))
        pos = np.arange(L, dtype=np.int32)
        slots = S.slots_for(pt, bi, 0, L)
        b.lrkv_append(dims, dev_bf16(X), wcat, dev_i32(slots), cache, positions=dev_i32(pos))
        rows = oracle.get().append(X, w.WsK, w.WsV, w.UK, w.UV, WKR=WKR, positions=pos)
        oracle.scatter_rows(ref_pools, slots, rows)
    q = S.gaussian_bf16(442, "q", (len(lens), H, d_h + D_ROPE))
    out = torch.empty((len(lens), H, d_h), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_decode(dims, dev_bf16(q), dev_bf16(w.BK), dev_bf16(w.BV), cache, dev_i32(pt.block_table),
                  dev_i32(pt.seq_lens), out, b.alloc_workspace(b.decode_workspace_bytes(dims, len(lens))), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.get().decode_cache(ref_pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, "append with positions, then decode")
