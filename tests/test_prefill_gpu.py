"""lrkv_prefill on the GPU against the fp64 oracle, and the end-to-end
append -> decode / append -> prefill paths against the expanded (E1) oracle."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import empty_pools, pack_wcat_t, random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, errors, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def run_prefill(H, d_h, r, pools, pt, q_start, q, BK, BV, status=None):
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    Bn, Tq = q.shape[:2]
    out = torch.empty((Bn, Tq, H, d_h), dtype=torch.bfloat16, device="cuda")
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_prefill(dims, dev_bf16(q), dev_bf16(BK), dev_bf16(BV), cache, dev_i32(pt.block_table),
                   dev_i32(q_start), out, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = [
    # H, d_h, r, Tq, q_starts
    (4, 64, 8, 64, [0, 64]),
    (4, 64, 16, 130, [0, 100]),
    (3, 64, 32, 17, [511, 5]),
    (2, 128, 16, 200, [0, 300]),
    (4, 128, 32, 1, [0, 1000]),
    (32, 128, 16, 96, [256, 0]),
    (2, 128, 8, 70, [63, 1]),
    # d_h = 128 or 64 with r = 16 runs the tcgen05 kernel: ragged query tiles, contexts
    # not aligned to pages or key tiles, the last chunk of a 4096-token prompt
    (1, 128, 16, 300, [37, 0]),
    (3, 128, 16, 512, [3584, 1000]),
    (2, 128, 16, 129, [127, 64]),
    (8, 128, 16, 1, [4095, 0]),
    (1, 64, 16, 300, [37, 0]),
    (3, 64, 16, 512, [3584, 1000]),
    (12, 64, 16, 129, [127, 64]),
    (2, 64, 16, 1, [4095, 0]),
]


@pytest.mark.parametrize("H,d_h,r,Tq,qs", CASES, ids=[f"H{c[0]}_dh{c[1]}_r{c[2]}_T{c[3]}" for c in CASES])
def test_prefill_matches_oracle(H, d_h, r, Tq, qs):
    seed = 200 + H + r + Tq
    ctx = [s + Tq for s in qs]
    pt = S.page_table(seed, ctx, 64, spare_blocks=1)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(qs), Tq, H, d_h))
    q_start = np.array(qs, np.int32)
    out, st = run_prefill(H, d_h, r, pools, pt, q_start, q, w.BK, w.BV)
    assert st == 0
    ref = oracle.get().prefill_cache(pools, pt.block_table, q_start, w.BK, w.BV, q)
    assert_close(host_f64(out), ref, f"prefill H={H} d_h={d_h} r={r} Tq={Tq}")


def test_prefill_last_query_equals_decode():
    H, d_h, r, Tq = 8, 64, 16, 150
    pt = S.page_table(5, [Tq + 40], 64)
    pools = random_pools(5, pt.num_blocks, H, d_h, r)
    w = weights(5, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(5, "q", (1, Tq, H, d_h))
    out, _ = run_prefill(H, d_h, r, pools, pt, np.array([40], np.int32), q, w.BK, w.BV)
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    dout = torch.empty((1, H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, 1))
    b.lrkv_decode(dims, dev_bf16(q[:, -1]), dev_bf16(w.BK), dev_bf16(w.BV), cache, dev_i32(pt.block_table),
                  dev_i32(pt.seq_lens), dout, ws)
    torch.cuda.synchronize()
    assert_close(host_f64(out[:, -1]), host_f64(dout), "prefill last row vs decode")


def test_end_to_end_append_then_decode_small_workload():
    """The small single-layer workload end to end: hidden states through
    lrkv_append into the paged cache, then lrkv_decode, against the oracle that
    forms W_h = W_shared + U_h B_h^T explicitly (E1)."""
    wl = S.WORKLOADS["small"]
    H, d_h, r, d, L = wl.H, wl.d_h, wl.r, wl.d, wl.L
    X = S.gaussian_bf16(wl.seed, "X", (1, L, d))
    w = weights(wl.seed, d, d_h, H, r)
    q = S.gaussian_bf16(wl.seed, "q", (1, H, d_h))
    pt = S.page_table(wl.seed, [L], 64)
    dims = b.make_dims(H, d_h, r, d)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(pt.num_blocks, H, d_h, r)))
    b.lrkv_append(dims, dev_bf16(X[0]), dev_bf16(pack_wcat_t(w)), dev_i32(S.slots_for(pt, 0, 0, L)), cache)
    out = torch.empty((1, H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, 1))
    b.lrkv_decode(dims, dev_bf16(q), dev_bf16(w.BK), dev_bf16(w.BV), cache, dev_i32(pt.block_table),
                  dev_i32(pt.seq_lens), out, ws)
    torch.cuda.synchronize()
    o = oracle.get()
    # end-to-end oracle: reference append (bf16 cache, as the workload fixes) then E2 decode
    ref_pools = empty_pools(pt.num_blocks, H, d_h, r)
    oracle.scatter_rows(ref_pools, S.slots_for(pt, 0, 0, L), o.append(X[0], w.WsK, w.WsV, w.UK, w.UV))
    e2 = o.decode_cache(ref_pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    got = host_f64(out)
    assert_close(got, e2, "append -> decode vs oracle append -> E2")
    # against the pure-math expansion (E1) the bf16 cache storage itself costs some accuracy:
    # the GPU may add at most the tolerance on top of what the storage rounding costs the oracle
    e1 = o.decode_expanded(X, [L], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    inherent = errors(e2, e1)[0]
    assert errors(got, e1)[0] <= inherent + 5e-3


def test_end_to_end_append_then_chunked_prefill():
    H, d_h, r, d, T, chunk = 4, 128, 16, 512, 384, 128
    X = S.gaussian_bf16(9, "X", (2, T, d))
    w = weights(9, d, d_h, H, r)
    q = S.gaussian_bf16(9, "q", (2, T, H, d_h))
    pt = S.page_table(9, [T, T], 64)
    dims = b.make_dims(H, d_h, r, d)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(pt.num_blocks, H, d_h, r)))
    wcat = dev_bf16(pack_wcat_t(w))
    outs = []
    for c0 in range(0, T, chunk):
        xs = np.concatenate([X[0, c0:c0 + chunk], X[1, c0:c0 + chunk]])
        sl = np.concatenate([S.slots_for(pt, 0, c0, c0 + chunk), S.slots_for(pt, 1, c0, c0 + chunk)])
        b.lrkv_append(dims, dev_bf16(xs), wcat, dev_i32(sl), cache)
        o = torch.empty((2, chunk, H, d_h), dtype=torch.bfloat16, device="cuda")
        b.lrkv_prefill(dims, dev_bf16(q[:, c0:c0 + chunk]), dev_bf16(w.BK), dev_bf16(w.BV), cache,
                       dev_i32(pt.block_table), dev_i32([c0, c0]), o)
        outs.append(o)
    torch.cuda.synchronize()
    got = np.concatenate([host_f64(o) for o in outs], axis=1)
    o_ = oracle.get()
    ref_pools = empty_pools(pt.num_blocks, H, d_h, r)
    for bb in range(2):
        oracle.scatter_rows(ref_pools, S.slots_for(pt, bb, 0, T), o_.append(X[bb], w.WsK, w.WsV, w.UK, w.UV))
    e2 = o_.prefill_cache(ref_pools, pt.block_table, [0, 0], w.BK, w.BV, q)
    assert_close(got, e2, "append -> chunked prefill vs oracle append -> E2")
    e1 = o_.prefill_expanded(X, [0, 0], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    assert errors(got, e1)[0] <= errors(e2, e1)[0] + 5e-3


def test_prefill_bad_context_reports_status():
    H, d_h, r, Tq = 2, 64, 8, 32
    pt = S.page_table(3, [64], 64)
    pools = random_pools(3, pt.num_blocks, H, d_h, r)
    w = weights(3, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(3, "q", (1, Tq, H, d_h))
    out, st = run_prefill(H, d_h, r, pools, pt, np.array([40], np.int32), q, w.BK, w.BV)  # 40 + 32 > 64
    assert st & b.DEV_BAD_SEQLEN
    assert np.all(host_f64(out) == 0)


FUSED_CASES = [
    # H, d_h, r, d_rope, Tq, q_starts -- d_h = 128 or 64 with r = 16 and no positional key
    # runs the tcgen05 kernel, the rest the warp-level one
    (2, 128, 16, 0, 300, [37, 1000]),
    (3, 128, 16, 0, 512, [3584, 0]),
    (12, 64, 16, 0, 129, [127, 64]),
    (2, 64, 16, 0, 1, [4095, 0]),
    (4, 64, 8, 0, 130, [0, 100]),
    (3, 64, 32, 0, 17, [511, 5]),
    (2, 128, 16, 64, 96, [256, 0]),
    (4, 128, 32, 64, 1, [0, 1000]),
]


@pytest.mark.parametrize("H,d_h,r,d_rope,Tq,qs", FUSED_CASES,
                         ids=[f"H{c[0]}_dh{c[1]}_r{c[2]}_rope{c[3]}_T{c[4]}" for c in FUSED_CASES])
def test_prefill_fused_matches_oracle(H, d_h, r, d_rope, Tq, qs):
    """lrkv_prefill_fused (q~ given, [o_s | o_z] returned) against the oracle's causal prefill
    with absorbed weights."""
    seed = 610 + H + r + Tq + d_rope
    pt = S.page_table(seed, [s + Tq for s in qs], 64, spare_blocks=1)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r, d_rope=d_rope)
    q = S.gaussian_bf16(seed, "q", (len(qs), Tq, H, d_h + d_rope))
    qt = S.gaussian_bf16(seed, "qt", (len(qs), Tq, H, r))
    q_start = np.array(qs, np.int32)
    dims = b.make_dims(H, d_h, r, H * d_h, d_rope=d_rope)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    out = torch.empty((len(qs), Tq, H, d_h + r), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_prefill_fused(dims, dev_bf16(q), dev_bf16(qt), cache, dev_i32(pt.block_table), dev_i32(q_start), out,
                         status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.get().prefill_fused(pools, pt.block_table, q_start, q, qt)
    assert_close(host_f64(out), ref, f"absorbed prefill H={H} d_h={d_h} r={r} d_rope={d_rope} Tq={Tq}")


@pytest.mark.parametrize("d_h,r", [(128, 16), (64, 8)])
def test_prefill_fused_bad_context_zeroes_rows(d_h, r):
    """A context past the block table: status LRKV_DEV_BAD_SEQLEN and all d_h + r columns zeroed
    (tcgen05 kernel for r = 16, warp-level kernel for r = 8)."""
    H, Tq = 2, 32
    pt = S.page_table(7, [64], 64)
    pools = random_pools(7, pt.num_blocks, H, d_h, r)
    q = S.gaussian_bf16(7, "q", (1, Tq, H, d_h))
    qt = S.gaussian_bf16(7, "qt", (1, Tq, H, r))
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    out = torch.full((1, Tq, H, d_h + r), 1.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_prefill_fused(dims, dev_bf16(q), dev_bf16(qt), cache, dev_i32(pt.block_table),
                         dev_i32(np.array([40], np.int32)), out, status=st)  # 40 + 32 > 64
    torch.cuda.synchronize()
    assert int(st.item()) & b.DEV_BAD_SEQLEN
    assert float(out.abs().max()) == 0.0
