"""lrkv_append with the decoupled positional key (d_rope = 64) on the GPU against the oracle.

The key row grows to [s^K | k^R]: k^R = RoPE(x W^KR, pos) is one d_rope-vector per token shared
by all heads (the decoupled rotary key of MLA-style latent caches, which "Low-Rank Key Value
Attention" names as a combination with LRKV).  The kernels accumulate x W^KR in fp32. They turn
each pair at the row's position with the angle in double, and sine and cosine in fp32 corrected to
first order in double (error ~1e-7 of the pair's magnitude), then round to fp32 and to bf16. The
oracle rotates its fp64 sum in double.  On integer-grid inputs the fp32 sums are exact, so every
content column must match bit for bit. A rotated column can differ by one ulp only where that
small error moves a rounding boundary (a few in 10^5 values).
"""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import empty_pools, f64, pack_wcat_t, weights
from gpu_util import dev_bf16, dev_i32, host_bits
from test_append_gpu import CANARY, _bf16_ulp, int_weights

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402

D_ROPE = 64


def run_append_rope(H, d_h, r, d, X, w, WKR, slots, positions, num_blocks, rope_base=0.0):
    dims = b.make_dims(H, d_h, r, d, d_rope=D_ROPE, rope_base=rope_base)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(num_blocks, H, d_h, r, fill=CANARY, d_rope=D_ROPE)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_append(dims, dev_bf16(X), dev_bf16(pack_wcat_t(w, WKR)), dev_i32(slots), cache, status=st,
                  positions=dev_i32(positions))
    torch.cuda.synchronize()
    return tuple(host_bits(t) for t in cache.tensors()), int(st.item())


def oracle_rows(X, w, WKR, positions, rope_base):
    return oracle.get().append(X, w.WsK, w.WsV, w.UK, w.UV, WKR=WKR, positions=positions,
                               rope_base=10000.0 if rope_base == 0.0 else rope_base)


def _positions(seed, n):
    """Mix of position 0, small positions and long-context ones (up to 2^17 - 1)."""
    p = S.uniform_int(seed, "pos", n, 0, 1 << 17).astype(np.int32)
    p[0] = 0
    if n > 2:
        p[1] = 1
        p[2] = (1 << 17) - 1
    return p


def _rows_at(pools, slots):
    return [p.reshape((-1,) + p.shape[2:])[slots] for p in pools]


@pytest.mark.parametrize("n", [1, 3, 33, 64, 200, 1000])
@pytest.mark.parametrize("H,d_h,r,d,base", [(8, 64, 8, 512, 0.0), (32, 128, 32, 1024, 0.0),
                                            (5, 128, 16, 264, 500000.0)])
def test_append_rope_exact_inputs(n, H, d_h, r, d, base):
    X = S.int_grid_bf16(n, "X", (n, d), -8, 8)
    w = int_weights(n + H, d, d_h, H, r)
    WKR = S.int_grid_bf16(n + H, "WKR", (d, D_ROPE), -8, 8)
    nb = (n + 63) // 64 + 2
    slots = S.permutation(n, "slots", nb * 64)[:n].astype(np.int32)
    pos = _positions(n, n)
    got, st = run_append_rope(H, d_h, r, d, X, w, WKR, slots, pos, nb, base)
    assert st == 0
    ref = oracle_rows(X, w, WKR, pos, base)
    g = _rows_at(got, slots)
    # content columns: bit for bit
    np.testing.assert_array_equal(g[0][:, :d_h], ref[0][:, :d_h], err_msg="s^K")
    for gi, ri, nm in zip(g[1:], ref[1:], ("sV", "zK", "zV")):
        np.testing.assert_array_equal(gi, ri, err_msg=nm)
    # rotated columns: within one bf16 ulp, and almost all identical
    gr, rr = f64(g[0][:, d_h:]), f64(ref[0][:, d_h:])
    assert np.all(np.abs(gr - rr) <= _bf16_ulp(rr)), "k^R beyond one ulp"
    # The rotation's last-bit differences from the plain-double rotation hit ~2e-5 of the rounded
    # values (a CPU model of the arithmetic); allow 1e-4 of them, and at least one.
    assert int((gr != rr).sum()) <= max(1, int(np.ceil(1e-4 * gr.size)))
    # position 0 is the identity rotation: k^R is the plain projection
    np.testing.assert_array_equal(g[0][0, d_h:], oracle_rows(X[:1], w, WKR, np.zeros(1, np.int32), base)[0][0, d_h:])
    # every other slot keeps its previous contents
    untouched = np.setdiff1d(np.arange(nb * 64), slots)
    for p in got:
        assert np.all(p.reshape((-1,) + p.shape[2:])[untouched] == CANARY)


@pytest.mark.parametrize("n,H,d_h,r,d", [(7, 8, 64, 16, 512), (64, 32, 128, 32, 4096), (1000, 32, 128, 16, 4096)])
def test_append_rope_gaussian_within_bound(n, H, d_h, r, d):
    """Gaussian inputs: each fp32 sum lies within K u sum|x w| of the exact one; the rotation mixes two
    columns with weights of magnitude <= 1, so a rotated column lies within 1 ulp(ref) + 2 K u
    (sum|x w_2i| + sum|x w_2i+1|) of the oracle's."""
    X = S.gaussian_bf16(n, "X", (n, d))
    w = weights(n, d, d_h, H, r)
    WKR = S.gaussian_bf16(n, "WKR", (d, D_ROPE), d ** -0.5)
    nb = (n + 63) // 64 + 1
    slots = np.arange(n, dtype=np.int32)
    pos = _positions(n + 1, n)
    got, st = run_append_rope(H, d_h, r, d, X, w, WKR, slots, pos, nb)
    assert st == 0
    ref = oracle_rows(X, w, WKR, pos, 0.0)
    g = _rows_at(got, slots)
    ax = np.abs(f64(X))
    mk = ax @ np.abs(f64(w.WsK))
    mr = ax @ np.abs(f64(WKR))
    mr = np.repeat(mr[:, 0::2] + mr[:, 1::2], 2, axis=1)
    mags = [np.concatenate([mk, mr], 1), ax @ np.abs(f64(w.WsV)),
            np.stack([ax @ np.abs(f64(w.UK[h])) for h in range(H)], 1),
            np.stack([ax @ np.abs(f64(w.UV[h])) for h in range(H)], 1)]
    for gi, ri, mag, nm in zip(g, ref, mags, ("sK", "sV", "zK", "zV")):
        gv, rv = f64(gi), f64(ri)
        assert np.all(np.abs(gv - rv) <= _bf16_ulp(rv) + 2 * d * 2.0 ** -24 * mag), nm
        frac = float((gv != rv).mean())
        print(f"rope append ulp mismatch n={n} H={H} d_h={d_h} r={r} d={d} {nm}: {frac:.2e} of {gv.size}")
        assert frac < 2e-2, nm


def test_append_without_positional_key_ignores_positions():
    """d_rope = 0 keeps the plain layout: a positions pointer is ignored and the rows equal the plain append."""
    H, d_h, r, d, n = 8, 64, 8, 512, 100
    X = S.int_grid_bf16(5, "X", (n, d), -8, 8)
    w = int_weights(5, d, d_h, H, r)
    dims = b.make_dims(H, d_h, r, d)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(2, H, d_h, r, fill=CANARY)))
    slots = np.arange(n, dtype=np.int32)
    b.lrkv_append(dims, dev_bf16(X), dev_bf16(pack_wcat_t(w)), dev_i32(slots), cache,
                  positions=dev_i32(np.full(n, 12345, np.int32)))
    torch.cuda.synchronize()
    ref = oracle.get().append(X, w.WsK, w.WsV, w.UK, w.UV)
    for gi, ri in zip(_rows_at([host_bits(t) for t in cache.tensors()], slots), ref):
        np.testing.assert_array_equal(gi, ri)
