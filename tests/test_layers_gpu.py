"""Layer-batched calls (lrkv_append_layers, lrkv_decode_layers) on the GPU: several layers with
their own weights, cache pools, queries and outputs, sharing the block table and lengths --
the 12-layer backbone of the KVPath experiments page, one decode step per sequence.  Each
layer is checked against the oracle on that layer's own inputs (Eqs. (4)-(7) of the LRKV
slides per layer), and the layered append against the one-layer append bit for bit."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import empty_pools, pack_wcat_t, random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402

CANARY = 0x7E57


def stacked(arrs):
    return dev_bf16(np.stack(arrs))


@pytest.mark.parametrize("L,H,d_h,r,lens,ns", [
    (3, 8, 64, 16, [2048, 1, 77, 500], 0),        # backbone head shape, ragged incl. L=1
    (12, 8, 64, 16, [300] * 16, 0),               # 12 layers x 16 sequences: more sequences than SMs
    (2, 32, 128, 32, [3000, 129], 0),             # long-context head shape
    (4, 8, 64, 8, [640, 64, 1], 5),               # a caller-set number of pieces, segments across layers
])
def test_decode_layers_matches_oracle_per_layer(L, H, d_h, r, lens, ns):
    seed = 40 + L + H + r
    pt = S.page_table(seed, lens, 64, spare_blocks=1)
    nb = pt.num_blocks
    pools = [random_pools(seed + 7 * l, nb, H, d_h, r) for l in range(L)]
    ws_ = [weights(seed + 7 * l, H * d_h, d_h, H, r) for l in range(L)]
    qs = [S.gaussian_bf16(seed + 7 * l, "q", (len(lens), H, d_h)) for l in range(L)]
    dims = b.make_dims(H, d_h, r, H * d_h, num_splits=ns)
    cache = b.LayeredCache(*(stacked([p[i] for p in pools]) for i in range(4)))
    q = stacked(qs)
    BK, BV = stacked([w.BK for w in ws_]), stacked([w.BV for w in ws_])
    out = torch.empty((L, len(lens), H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, L * len(lens)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_decode_layers(dims, q, BK, BV, cache, dev_i32(pt.block_table), dev_i32(pt.seq_lens), out, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host_f64(out)
    o = oracle.get()
    for l in range(L):
        ref = o.decode_cache(pools[l], pt.block_table, pt.seq_lens, ws_[l].BK, ws_[l].BV, qs[l])
        assert_close(got[l], ref, f"layer {l}")
    # run to run bit for bit
    out2 = torch.empty_like(out)
    b.lrkv_decode_layers(dims, q, BK, BV, cache, dev_i32(pt.block_table), dev_i32(pt.seq_lens), out2, ws, status=st)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_decode_layers_bad_length_and_block_reported_per_sequence():
    L, H, d_h, r = 3, 8, 64, 8
    lens = [200, 100, 50]
    pt = S.page_table(5, lens, 64)
    pools = [random_pools(50 + l, pt.num_blocks, H, d_h, r) for l in range(L)]
    ws_ = [weights(50 + l, H * d_h, d_h, H, r) for l in range(L)]
    qs = [S.gaussian_bf16(50 + l, "q", (3, H, d_h)) for l in range(L)]
    bt = pt.block_table.copy()
    bt[0, 1] = pt.num_blocks + 9
    sl = pt.seq_lens.copy()
    sl[2] = 0
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.LayeredCache(*(stacked([p[i] for p in pools]) for i in range(4)))
    out = torch.empty((L, 3, H, d_h), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, L * 3))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_decode_layers(dims, stacked(qs), stacked([w.BK for w in ws_]), stacked([w.BV for w in ws_]), cache,
                         dev_i32(bt), dev_i32(sl), out, ws, status=st)
    torch.cuda.synchronize()
    code = int(st.item())
    assert code & b.DEV_BAD_BLOCK and code & b.DEV_BAD_SEQLEN
    got = host_f64(out)
    assert np.all(got[:, 2] == 0) and np.all(np.isfinite(got))
    o = oracle.get()
    for l in range(L):  # sequence 1 of every layer is untouched by the others' problems
        ref = o.decode_cache(pools[l], pt.block_table[1:2], pt.seq_lens[1:2], ws_[l].BK, ws_[l].BV, qs[l][1:2])
        assert_close(got[l, 1:2], ref, f"healthy sequence, layer {l}")


@pytest.mark.parametrize("n,rope", [(1, False), (16, False), (5, True), (70, False)])
def test_append_layers_equals_single_layer_appends(n, rope):
    """Layer l of the layered append holds exactly what lrkv_append writes with layer l's rows
    and weights (the same kernels and summation order), and only the given slots change."""
    L, H, d_h, r, d = 3, 8, 64, 16, 512
    dr = 64 if rope else 0
    nb = (n + 63) // 64 + 2
    slots = S.permutation(n, "slots", nb * 64)[:n].astype(np.int32)
    pos = S.uniform_int(n, "pos", n, 0, 40000).astype(np.int32) if rope else None
    Xs = [S.gaussian_bf16(60 + l, "X", (n, d)) for l in range(L)]
    wts = []
    for l in range(L):
        w = weights(60 + l, d, d_h, H, r)
        wkr = S.gaussian_bf16(60 + l, "WKR", (d, dr), d ** -0.5) if rope else None
        wts.append(pack_wcat_t(w, wkr))
    dims = b.make_dims(H, d_h, r, d, d_rope=dr)
    layered = b.LayeredCache(*(stacked([p] * L) for p in empty_pools(nb, H, d_h, r, fill=CANARY, d_rope=dr)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    posd = dev_i32(pos) if rope else None
    b.lrkv_append_layers(dims, stacked(Xs), stacked(wts), dev_i32(slots), layered, status=st, positions=posd)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for l in range(L):
        one = b.PagedCache(*(dev_bf16(p) for p in empty_pools(nb, H, d_h, r, fill=CANARY, d_rope=dr)))
        b.lrkv_append(dims, dev_bf16(Xs[l]), dev_bf16(wts[l]), dev_i32(slots), one, status=st, positions=posd)
        torch.cuda.synchronize()
        for a_, b_, nm in zip(layered.layer(l).tensors(), one.tensors(), ("sK", "sV", "zK", "zV")):
            np.testing.assert_array_equal(host_bits(a_), host_bits(b_), err_msg=f"layer {l} {nm}")
