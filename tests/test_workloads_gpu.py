"""Full-size workloads: the exact step the benchmark times, checked against the oracle on samples.

Each benchmark workload is built at full size by the benchmark's own harness:
  - the single-layer small decode;
  - the 12-layer backbone;
  - the DeepSeek-V2-scale layer (H=128);
  - the ragged long-context decode;
  - the chunked prefill with append.
Its step runs once through the public calls, in the launch configuration the benchmark
times. A sample of (layer, sequence, head) outputs is then recomputed by the fp64 oracle,
one sequence at a time. The oracle sees only that sequence's pages and the sampled heads:
a head's output depends only on the shared s-vectors and that head's own z-vectors
("Low-Rank Key Value Attention", Eqs. (6)-(7)).

Every oracle input is one the harness drew from its seeded device generator (copied back),
with one exception: the cache rows that lrkv_append writes during the step. The oracle
recomputes those from X and W_cat itself (Eqs. (4)-(5)), so no oracle input comes from
the kernels under test.
"""
import numpy as np
import pytest
import torch

import bench
import lrkv_synth as S
import oracle
from gpu_util import assert_close, host_bits, host_f64

pytestmark = pytest.mark.gpu


def _unpack_wcat(wcat_t, d_h, H, r, d_rope=0):
    """W_cat^T [N, d] (library layout) -> W_shared^K, W_shared^V [d, d_h], U^K, U^V [H, d, r] and the
    positional-key projection W^KR [d, d_rope] (None without one)."""
    d = wcat_t.shape[1]
    v0 = d_h + d_rope
    z0 = v0 + d_h
    WsK = np.ascontiguousarray(wcat_t[:d_h].T)
    WKR = np.ascontiguousarray(wcat_t[d_h:v0].T) if d_rope else None
    WsV = np.ascontiguousarray(wcat_t[v0:z0].T)
    UK = np.ascontiguousarray(wcat_t[z0:z0 + H * r].reshape(H, r, d).transpose(0, 2, 1))
    UV = np.ascontiguousarray(wcat_t[z0 + H * r:z0 + 2 * H * r].reshape(H, r, d).transpose(0, 2, 1))
    return WsK, WsV, UK, UV, WKR


def _heads(H, n):
    """Up to n heads spread over [0, H), always the first and the last."""
    return sorted(set(int(x) for x in np.linspace(0, H - 1, min(n, H)).round()))


def _seq_pools(cache, blocks, heads):
    """One sequence's pages, in table order, from a layer's device pools; z columns of `heads` only."""
    dev = cache.sK.device
    idx = torch.as_tensor(np.asarray(blocks, np.int64), device=dev)
    hi = torch.as_tensor(np.asarray(heads, np.int64), device=dev)
    return [host_bits(cache.sK.index_select(0, idx)), host_bits(cache.sV.index_select(0, idx)),
            host_bits(cache.zK.index_select(0, idx).index_select(2, hi)),
            host_bits(cache.zV.index_select(0, idx).index_select(2, hi))]


def _run_step(hz):
    hz.status.zero_()
    hz.step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(hz.status.item()) == 0


@pytest.mark.parametrize("key,d_rope,per_layer", [("small", 0, False), ("backbone12", 0, False),
                                                  ("backbone12", 0, True), ("dsv2", 0, False), ("longctx", 0, False),
                                                  ("dsv2", 64, False), ("longctx", 64, False)])
def test_decode_workload_full_size(key, d_rope, per_layer, oracle_lib):
    """(The 12-layer backbone runs through the layer-batched calls, as the benchmark times it,
    and once more layer by layer.)"""
    wl = S.WORKLOADS[key]
    hz = bench.DecodeHarness(wl, 0, d_rope=d_rope, per_layer=per_layer)
    heads = _heads(wl.H, 8)
    layers = sorted({0, wl.layers // 2, wl.layers - 1})
    seqs = sorted({0, wl.B // 2, wl.B - 1})
    # the cache pages the oracle reads, copied back before the step runs
    pages = {}
    for li in layers:
        for b in seqs:
            n = int(hz.seq_lens[b])
            pages[li, b] = _seq_pools(hz.cache.layer(li), hz.pt.block_table[b, :(n + 63) // 64], heads)
    _run_step(hz)

    got, ref = [], []
    for li in layers:
        WsK, WsV, UK, UV, WKR = _unpack_wcat(host_bits(hz.wcat[li]), wl.d_h, wl.H, wl.r, d_rope)
        X, q = host_bits(hz.x[li]), host_bits(hz.q[li])
        BK, BV = host_bits(hz.BK[li])[heads], host_bits(hz.BV[li])[heads]
        out = host_f64(hz.out[li])
        # the step appended each sequence's newest token (position seq_len - 1) before decoding
        pos = (hz.seq_lens[seqs] - 1).astype(np.int32)
        newest = oracle_lib.append(X[seqs], WsK, WsV, UK[heads], UV[heads], WKR=WKR, positions=pos)
        for k, b in enumerate(seqs):
            n = int(hz.seq_lens[b])
            pools = pages[li, b]
            oracle.scatter_rows(pools, [n - 1], [rows[k:k + 1] for rows in newest])
            bt = np.arange(pools[0].shape[0], dtype=np.int32)[None]
            qs = np.ascontiguousarray(q[b:b + 1][:, heads])
            ref.append(oracle_lib.decode_cache(pools, bt, [n], BK, BV, qs)[0])
            got.append(out[b, heads])
    assert_close(np.stack(got), np.stack(ref), f"{key} decode at full size (layers {layers}, sequences {seqs}, "
                                               f"heads {heads})")


@pytest.mark.parametrize("fused,d_rope", [(False, 0), (False, 64), (True, 0)])
def test_prefill_workload_full_size(fused, d_rope, oracle_lib):
    """Also with the positional key (rotated in the append at each row's position) and with
    absorbed weights (lrkv_prefill_fused), as `bench.py --workload prefill --rope / --fused` runs."""
    wl = S.WORKLOADS["prefill"]
    hz = bench.PrefillHarness(wl, 0, fused=fused, d_rope=d_rope)
    _run_step(hz)

    heads = _heads(wl.H, 4)
    C, T = wl.chunk, wl.L
    WsK, WsV, UK, UV, WKR = _unpack_wcat(host_bits(hz.wcat), wl.d_h, wl.H, wl.r, d_rope)
    BK, BV = host_bits(hz.BK)[heads], host_bits(hz.BV)[heads]
    xs = [host_bits(ch["x"]) for ch in hz.chunks]
    got, ref = [], []
    for b in range(wl.B):
        # sequence b's prompt rows in token order (chunk c holds both sequences' rows, b-major)
        X = np.concatenate([x[b * C:(b + 1) * C] for x in xs])
        rows = oracle_lib.append(X, WsK, WsV, UK[heads], UV[heads], WKR=WKR,
                                 positions=np.arange(T, dtype=np.int32) if d_rope else None)
        npg = T // 64
        pools = [np.zeros((npg, 64) + rr.shape[1:], np.uint16) for rr in rows]
        oracle.scatter_rows(pools, np.arange(T), rows)
        bt = np.arange(npg, dtype=np.int32)[None]
        for ci, ch in enumerate(hz.chunks):
            q = np.ascontiguousarray(host_bits(ch["q"])[b:b + 1][:, :, heads])
            if fused:
                qt = np.ascontiguousarray(host_bits(ch["qt"])[b:b + 1][:, :, heads])
                ref.append(oracle_lib.prefill_fused(pools, bt, [ci * C], q, qt)[0])
            else:
                ref.append(oracle_lib.prefill_cache(pools, bt, [ci * C], BK, BV, q)[0])
            got.append(host_f64(ch["out"])[b][:, heads])
    assert_close(np.stack(got), np.stack(ref), f"prefill (absorbed {fused}, d_rope {d_rope}) at full size "
                                               f"(both sequences, all chunks, heads {heads})")
