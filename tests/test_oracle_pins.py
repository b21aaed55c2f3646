"""Pins of the fp64 oracle to facts other than itself.

Each ``pin_*`` checks the oracle against something the pages or mathematics fix:
a worked value printed on the pages, a special case that reduces to a library
attention routine (torch SDPA in fp64), an exactly representable integer case,
a symmetry, or a closed form.  ``test_planted_mistakes_are_caught`` rebuilds the
oracle with one deliberate mistake at a time and checks that some pin fails.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import lrkv_synth as S
import oracle
from cases import Weights, empty_pools, f64, random_pools, weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sdpa(q, K, V, scale, causal=False, mask=None):
    """Library attention: q [Hq, Tq, d_h], K/V [Hq, L, d_h] (fp64); mask [Tq, L] bool (True = attend)."""
    m = None if mask is None else torch.from_numpy(mask)
    out = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V),
                                         attn_mask=m, scale=scale, is_causal=causal)
    return out.numpy()


def _lib_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 bits via torch's own fp32 -> bf16 conversion (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------- softmax
def pin_softmax_worked_value(o):
    # Worked value from the MLA lesson, Chapter 5 (golden file cites it).
    for line in open(os.path.join(GOLDEN, "softmax_two_logits.txt")):
        if line.startswith("#") or not line.strip():
            continue
        lg, ex, dec = (s.strip() for s in line.split("|"))
        p = o.softmax([float(v) for v in lg.split()])
        np.testing.assert_array_equal(np.round(p, int(dec)), [float(v) for v in ex.split()])
        # closed form of a two-way softmax: p0 = e^a / (e^a + e^b)
        a, b = (float(v) for v in lg.split())
        assert abs(p[0] - np.exp(a) / (np.exp(a) + np.exp(b))) < 1e-15


def pin_softmax_normalised(o):
    for scale in (1.0, 30.0, 700.0):
        x = S.gaussian(11, f"lg{scale}", 257) * scale
        p = o.softmax(x)
        assert np.all(np.isfinite(p)) and np.all(p >= 0)
        assert abs(p.sum() - 1.0) < 1e-12
        # shift invariance of softmax
        np.testing.assert_allclose(o.softmax(x + 123.25), p, rtol=1e-12, atol=1e-300)


def pin_attend_special_cases(o):
    d_h = 16
    q = S.gaussian(5, "q", d_h)
    V = S.gaussian(5, "V", 9 * d_h).reshape(9, d_h)
    # one token: the output is that token's value row
    K1 = S.gaussian(5, "K1", d_h).reshape(1, d_h)
    np.testing.assert_array_equal(o.attend(q, K1, V[:1]), V[0])
    # identical keys: uniform weights, output is the mean value row
    Keq = np.tile(S.gaussian(5, "Keq", d_h), (9, 1))
    np.testing.assert_allclose(o.attend(q, Keq, V), V.mean(axis=0), rtol=1e-13, atol=1e-15)
    # generic: library attention
    K = S.gaussian(5, "K", 9 * d_h).reshape(9, d_h)
    ref = _sdpa(q[None, None, :], K[None], V[None], 1 / np.sqrt(d_h))[0, 0]
    np.testing.assert_allclose(o.attend(q, K, V), ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------- append (Eqs. 4-5)
def pin_append_integer_exact(o):
    """Integer-grid inputs: every partial sum is exact in fp32, so the cache value is
    the exact integer product, rounded once to bf16 (checked with torch's rounding)."""
    n, d, d_h, H, r = 13, 96, 16, 3, 8
    X = S.int_grid_bf16(1, "X", (n, d), -8, 8)
    w = Weights(*(S.int_grid_bf16(1, nm, sh, -8, 8) for nm, sh in
                  [("a", (d, d_h)), ("b", (d, d_h)), ("c", (H, d, r)), ("e", (H, d, r)),
                   ("f", (H, d_h, r)), ("g", (H, d_h, r))]))
    Xi = f64(X).astype(np.int64)
    sK, sV, zK, zV = o.append(X, w.WsK, w.WsV, w.UK, w.UV)
    exact = lambda Wt: (Xi @ f64(Wt).astype(np.int64)).astype(np.float32)
    np.testing.assert_array_equal(sK, _lib_bf16(exact(w.WsK)))
    np.testing.assert_array_equal(sV, _lib_bf16(exact(w.WsV)))
    for h in range(H):
        np.testing.assert_array_equal(zK[:, h], _lib_bf16(exact(w.UK[h])))
        np.testing.assert_array_equal(zV[:, h], _lib_bf16(exact(w.UV[h])))


def pin_append_gaussian_rounding(o):
    """Gaussian inputs: the cache equals library fp64 GEMM -> fp32 -> bf16 except where the
    fp64 sum order flips a rounding boundary (rare); never more than one bf16 ulp."""
    n, d, d_h, H, r = 64, 512, 64, 4, 16
    X = S.gaussian_bf16(2, "X", (n, d))
    w = weights(2, d, d_h, H, r)
    sK, _, zK, _ = o.append(X, w.WsK, w.WsV, w.UK, w.UV)
    ref_s = _lib_bf16((f64(X) @ f64(w.WsK)).astype(np.float32))
    ref_z = np.stack([_lib_bf16((f64(X) @ f64(w.UK[h])).astype(np.float32)) for h in range(H)], axis=1)
    for got, ref in ((sK, ref_s), (zK, ref_z)):
        diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
        assert diff.max() <= 1
        assert (diff != 0).mean() < 1e-3


# ---------------------------------------------------------------------------- decode / prefill (Eqs. 2-7)
def _ctx(seed, B, L, d):
    return S.gaussian_bf16(seed, "Xctx", (B, L, d))


def pin_r0_is_mqa(o):
    """r = 0: every head shares K_s, V_s, i.e. multi-query attention."""
    B, L, d, d_h, H = 2, 11, 48, 16, 4
    w = weights(3, d, d_h, H, 0)
    X = _ctx(3, B, L, d)
    q = S.gaussian_bf16(3, "q", (B, H, d_h))
    got = o.decode_expanded(X, [L, L - 4], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    for b, Lb in enumerate([L, L - 4]):
        Ks = f64(X[b, :Lb]) @ f64(w.WsK)
        Vs = f64(X[b, :Lb]) @ f64(w.WsV)
        ref = _sdpa(f64(q[b])[:, None, :], np.repeat(Ks[None], H, 0), np.repeat(Vs[None], H, 0),
                    1 / np.sqrt(d_h))[:, 0]
        np.testing.assert_allclose(got[b], ref, rtol=1e-11, atol=1e-13)


def _perm_factor_case(seed, H, d_h, d):
    """W_shared = 0 and B_h = a permutation matrix P_h (r = d_h): W_h = U_h P_h^T,
    whose column i is column pi_h(i) of U_h -- plain multi-head attention."""
    r = d_h
    zeros = np.zeros((d, d_h), np.uint16)
    UK = S.gaussian_bf16(seed, "UK", (H, d, r), 1 / np.sqrt(d))
    UV = S.gaussian_bf16(seed, "UV", (H, d, r), 1 / np.sqrt(d))
    one = np.uint16(0x3F80)
    BK = np.zeros((H, d_h, r), np.uint16)
    BV = np.zeros((H, d_h, r), np.uint16)
    piK, piV = [], []
    for h in range(H):
        pk = S.permutation(seed, f"piK{h}", d_h)
        pv = S.permutation(seed, f"piV{h}", d_h)
        BK[h, np.arange(d_h), pk] = one
        BV[h, np.arange(d_h), pv] = one
        piK.append(pk)
        piV.append(pv)
    return Weights(zeros, zeros.copy(), UK, UV, BK, BV), piK, piV


def pin_mha_special_case(o):
    B, L, d, d_h, H = 2, 9, 40, 8, 3
    w, piK, piV = _perm_factor_case(4, H, d_h, d)
    X = _ctx(4, B, L, d)
    q = S.gaussian_bf16(4, "q", (B, H, d_h))
    got = o.decode_expanded(X, [L, L], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    for b in range(B):
        K = np.stack([f64(X[b]) @ f64(w.UK[h])[:, piK[h]] for h in range(H)])
        V = np.stack([f64(X[b]) @ f64(w.UV[h])[:, piV[h]] for h in range(H)])
        ref = _sdpa(f64(q[b])[:, None, :], K, V, 1 / np.sqrt(d_h))[:, 0]
        np.testing.assert_allclose(got[b], ref, rtol=1e-11, atol=1e-13)
    # causal prefill of the whole sequence against library causal attention
    Tq = L
    qp = S.gaussian_bf16(4, "qp", (B, Tq, H, d_h))
    gotp = o.prefill_expanded(X, [0, 0], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, qp)
    for b in range(B):
        K = np.stack([f64(X[b]) @ f64(w.UK[h])[:, piK[h]] for h in range(H)])
        V = np.stack([f64(X[b]) @ f64(w.UV[h])[:, piV[h]] for h in range(H)])
        ref = _sdpa(np.transpose(f64(qp[b]), (1, 0, 2)), K, V, 1 / np.sqrt(d_h), causal=True)
        np.testing.assert_allclose(gotp[b], np.transpose(ref, (1, 0, 2)), rtol=1e-11, atol=1e-13)


def pin_factored_equals_expanded(o):
    """Eqs. (6)-(7) evaluated in factored form (fp64, numpy) equal the oracle's
    expanded evaluation for the same model (the slides' "two notions of equivalence")."""
    B, L, d, d_h, H, r = 2, 10, 32, 16, 3, 4
    w = weights(6, d, d_h, H, r)
    X = _ctx(6, B, L, d)
    q = S.gaussian_bf16(6, "q", (B, H, d_h))
    got = o.decode_expanded(X, [L, 7], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    for b, Lb in enumerate([L, 7]):
        x = f64(X[b, :Lb])
        Ks, Vs = x @ f64(w.WsK), x @ f64(w.WsV)
        for h in range(H):
            qh = f64(q[b, h])
            RK, RV = x @ f64(w.UK[h]), x @ f64(w.UV[h])
            logits = (qh @ Ks.T + (qh @ f64(w.BK[h])) @ RK.T) / np.sqrt(d_h)
            a = np.exp(logits - logits.max())
            a /= a.sum()
            oh = a @ Vs + (a @ RV) @ f64(w.BV[h]).T
            np.testing.assert_allclose(got[b, h], oh, rtol=1e-11, atol=1e-13)


def _exact_cache_case(o, seed, B, L, d, d_h, H, r, bs=64, extra_pages=3):
    """Small-integer inputs with d small enough that every cache value is an integer of
    magnitude <= 256 and hence exact in bf16: the cache then holds K_s, R_h exactly."""
    X = S.int_grid_bf16(seed, "X", (B, L, d), -1, 1)
    w = Weights(*(S.int_grid_bf16(seed, nm, sh, -1, 1) for nm, sh in
                  [("a", (d, d_h)), ("b", (d, d_h)), ("c", (H, d, r)), ("e", (H, d, r))]),
                BK=S.gaussian_bf16(seed, "BK", (H, d_h, r), 0.5), BV=S.gaussian_bf16(seed, "BV", (H, d_h, r), 0.5))
    pt = S.page_table(seed, [L] * B, bs, spare_blocks=extra_pages)
    pools = empty_pools(pt.num_blocks, H, d_h, r, bs)
    for b in range(B):
        rows = o.append(X[b], w.WsK, w.WsV, w.UK, w.UV)
        oracle.scatter_rows(pools, S.slots_for(pt, b, 0, L), rows)
    return X, w, pt, pools


def pin_cache_path_matches_weight_path(o):
    """E2 (from the paged cache) equals E1 (from X and W_h) when the cache is exact;
    pins the page/slot indexing and the use of B^K for keys and B^V for values."""
    B, L, d, d_h, H, r = 2, 150, 32, 16, 3, 8
    X, w, pt, pools = _exact_cache_case(o, 7, B, L, d, d_h, H, r)
    q = S.gaussian_bf16(7, "q", (B, H, d_h))
    lens = np.array([L, 77], np.int32)
    e1 = o.decode_expanded(X, lens, w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    e2 = o.decode_cache(pools, pt.block_table, lens, w.BK, w.BV, q)
    np.testing.assert_allclose(e2, e1, rtol=1e-12, atol=1e-13)
    Tq = 40
    qs = np.array([L - Tq, 20], np.int32)
    qp = S.gaussian_bf16(7, "qp", (B, Tq, H, d_h))
    p1 = o.prefill_expanded(X, qs, w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, qp)
    p2 = o.prefill_cache(pools, pt.block_table, qs, w.BK, w.BV, qp)
    np.testing.assert_allclose(p2, p1, rtol=1e-12, atol=1e-13)


def pin_head_permutation_equivariance(o):
    B, L, d, d_h, H, r = 1, 12, 24, 8, 4, 4
    w = weights(8, d, d_h, H, r)
    X = _ctx(8, B, L, d)
    q = S.gaussian_bf16(8, "q", (B, H, d_h))
    perm = np.array([2, 0, 3, 1])
    a = o.decode_expanded(X, [L], w.WsK, w.WsV, w.UK, w.UV, w.BK, w.BV, q)
    b = o.decode_expanded(X, [L], w.WsK, w.WsV, w.UK[perm], w.UV[perm], w.BK[perm], w.BV[perm], q[:, perm])
    np.testing.assert_allclose(b, a[:, perm], rtol=1e-13, atol=1e-15)


def pin_page_permutation_invariance(o):
    H, d_h, r, bs = 3, 16, 8, 64
    pt = S.page_table(9, [200, 64, 129], bs)
    pools = random_pools(9, pt.num_blocks, H, d_h, r, bs)
    w = weights(9, 32, d_h, H, r)
    q = S.gaussian_bf16(9, "q", (3, H, d_h))
    a = o.decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    perm = S.permutation(10, "pp", pt.num_blocks)       # new physical location of each page
    pools2 = tuple(np.empty_like(p) for p in pools)
    for p_old, p_new in zip(pools, pools2):
        p_new[perm] = p_old
    bt2 = np.where(pt.block_table >= 0, perm[np.maximum(pt.block_table, 0)], -1).astype(np.int32)
    b = o.decode_cache(pools2, bt2, pt.seq_lens, w.BK, w.BV, q)
    np.testing.assert_array_equal(a, b)


def pin_prefill_causal_edges(o):
    """Query at position 0 sees only token 0: with B^V = 0 its output is s^V of token 0.
    The last query of a chunk sees the whole context, like a decode query."""
    H, d_h, r, bs = 2, 16, 8, 64
    L = 130
    pt = S.page_table(12, [L, L], bs)
    pools = random_pools(12, pt.num_blocks, H, d_h, r, bs)
    w = weights(12, 32, d_h, H, r)
    zeroB = np.zeros_like(w.BV)
    Tq = 130
    qp = S.gaussian_bf16(12, "qp", (2, Tq, H, d_h))
    out = o.prefill_cache(pools, pt.block_table, [0, 0], w.BK, zeroB, qp)
    for b in range(2):
        slot = pt.slot(b, 0)
        sV0 = f64(pools[1].reshape(-1, d_h)[slot])
        for h in range(H):
            np.testing.assert_array_equal(out[b, 0, h], sV0)
    out = o.prefill_cache(pools, pt.block_table, [0, 0], w.BK, w.BV, qp)
    dec = o.decode_cache(pools, pt.block_table, [L, L], w.BK, w.BV, qp[:, -1])
    np.testing.assert_allclose(out[:, -1], dec, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------- absorbed (fused) decode
def _gather_rows(pools, pt, b, L):
    """Token rows 0..L-1 of sequence b from the paged pools: sK, sV [L, d_h]; zK, zV [L, H, r] (fp64)."""
    slots = np.asarray(S.slots_for(pt, b, 0, L), np.int64)
    return tuple(f64(p.reshape((-1,) + p.shape[2:])[slots]) for p in pools)


def pin_fused_is_concatenated_attention(o):
    """With both absorptions in the caller's weights, decode is single-head attention over
    the concatenated features [q | q~] . [s^K | z^K_h] with values [s^V | z^V_h] and the
    scale of the d_h-wide dot product: torch SDPA on exactly those tensors."""
    B, H, d_h, r = 2, 3, 16, 8
    lens = [150, 77]
    pt = S.page_table(21, lens, 64, spare_blocks=2)
    pools = random_pools(21, pt.num_blocks, H, d_h, r)
    q = S.gaussian_bf16(21, "q", (B, H, d_h))
    qt = S.gaussian_bf16(21, "qt", (B, H, r))
    got = o.decode_fused(pools, pt.block_table, lens, q, qt)
    for b in range(B):
        sK, sV, zK, zV = _gather_rows(pools, pt, b, lens[b])
        for h in range(H):
            Kc = np.concatenate([sK, zK[:, h]], axis=1)[None]
            Vc = np.concatenate([sV, zV[:, h]], axis=1)[None]
            qc = np.concatenate([f64(q[b, h]), f64(qt[b, h])])[None, None]
            ref = _sdpa(qc, Kc, Vc, 1.0 / np.sqrt(d_h))[0, 0]
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-14)


def pin_fused_matches_factored_decode(o):
    """On integer q and B^K, q~ = q B^K is exact in bf16, so the absorbed decode must agree
    with the expanded decode: o_s + B^V o_z = softmax(q K_h^T * scale) V_h.  Pins where q~
    enters the logits and that B^V is applied to the aggregated latent, not per token."""
    B, H, d_h, r = 2, 3, 16, 8
    lens = [130, 64]
    pt = S.page_table(22, lens, 64, spare_blocks=1)
    pools = random_pools(22, pt.num_blocks, H, d_h, r)
    q = S.int_grid_bf16(22, "q", (B, H, d_h), -1, 1)
    BK = S.int_grid_bf16(22, "BK", (H, d_h, r), -1, 1)
    BV = S.gaussian_bf16(22, "BV", (H, d_h, r), 0.5)
    qt_exact = np.einsum("bhd,hdr->bhr", f64(q), f64(BK))
    assert np.all(np.abs(qt_exact) <= 256) and np.all(qt_exact == np.round(qt_exact))
    qt = _lib_bf16(qt_exact)
    fused = o.decode_fused(pools, pt.block_table, lens, q, qt)
    o_s, o_z = fused[..., :d_h], fused[..., d_h:]
    recomposed = o_s + np.einsum("hdr,bhr->bhd", f64(BV), o_z)
    ref = o.decode_cache(pools, pt.block_table, lens, BK, BV, q)
    np.testing.assert_allclose(recomposed, ref, rtol=1e-12, atol=1e-13)



def pin_prefill_fused_is_concatenated_causal_attention(o):
    """The absorbed-weights prefill is causal single-head attention over the concatenated
    features: query i of a chunk starting at q_start attends, with [q_i | q~_i], to the keys
    [s^K_j | z^K_{h,j}] of positions j <= q_start + i and aggregates [s^V_j | z^V_{h,j}]:
    torch SDPA with that mask on exactly those tensors.  With a positional key the shared key
    row is [s^K | k^R], the query [q | q^R | q~], the scale 1/sqrt(d_h + d_rope)."""
    B, H, d_h, r, Tq = 2, 3, 16, 8, 40
    qs = [100, 0]
    for d_rope in (0, 16):
        lens = [qs[b] + Tq for b in range(B)]
        pt = S.page_table(23 + d_rope, lens, 64, spare_blocks=2)
        pools = random_pools(23 + d_rope, pt.num_blocks, H, d_h, r, d_rope=d_rope)
        q = S.gaussian_bf16(23, "q", (B, Tq, H, d_h + d_rope))
        qt = S.gaussian_bf16(23, "qt", (B, Tq, H, r))
        got = o.prefill_fused(pools, pt.block_table, qs, q, qt)
        for b in range(B):
            sK, sV, zK, zV = _gather_rows(pools, pt, b, lens[b])
            mask = np.arange(lens[b])[None, :] <= (qs[b] + np.arange(Tq))[:, None]
            for h in range(H):
                Kc = np.concatenate([sK, zK[:, h]], axis=1)[None]
                Vc = np.concatenate([sV, zV[:, h]], axis=1)[None]
                qc = np.concatenate([f64(q[b, :, h]), f64(qt[b, :, h])], axis=1)[None]
                ref = _sdpa(qc, Kc, Vc, 1.0 / np.sqrt(d_h + d_rope), mask=mask)[0]
                np.testing.assert_allclose(got[b, :, h], ref, rtol=1e-12, atol=1e-14)


def pin_prefill_fused_matches_factored_prefill(o):
    """On integer q and B^K, q~ = q B^K is exact in bf16, so every query row of the
    absorbed-weights prefill, recomposed as o_s + B^V o_z, must equal the factored causal
    prefill (which computes q~ and applies B^V itself)."""
    B, H, d_h, r, Tq = 2, 3, 16, 8, 70
    qs = [60, 5]
    lens = [qs[b] + Tq for b in range(B)]
    pt = S.page_table(24, lens, 64, spare_blocks=1)
    pools = random_pools(24, pt.num_blocks, H, d_h, r)
    q = S.int_grid_bf16(24, "q", (B, Tq, H, d_h), -1, 1)
    BK = S.int_grid_bf16(24, "BK", (H, d_h, r), -1, 1)
    BV = S.gaussian_bf16(24, "BV", (H, d_h, r), 0.5)
    qt_exact = np.einsum("bthd,hdr->bthr", f64(q), f64(BK))
    assert np.all(np.abs(qt_exact) <= 256) and np.all(qt_exact == np.round(qt_exact))
    qt = _lib_bf16(qt_exact)
    fused = o.prefill_fused(pools, pt.block_table, qs, q, qt)
    o_s, o_z = fused[..., :d_h], fused[..., d_h:]
    recomposed = o_s + np.einsum("hdr,bthr->bthd", f64(BV), o_z)
    ref = o.prefill_cache(pools, pt.block_table, qs, BK, BV, q)
    np.testing.assert_allclose(recomposed, ref, rtol=1e-12, atol=1e-13)

# ---------------------------------------------------------------------------- decoupled positional key
ROPE_BASE = 10000.0


def _rope_np(v: np.ndarray, pos: np.ndarray, base: float = ROPE_BASE) -> np.ndarray:
    """Rotary encoding written out in numpy: pair (2i, 2i+1) of row t turned by the angle
    pos[t] * base^(-2i / d)."""
    d = v.shape[-1]
    ang = pos[:, None].astype(np.float64) * base ** (-2.0 * np.arange(d // 2) / d)[None, :]
    c, s_ = np.cos(ang), np.sin(ang)
    out = np.empty_like(v, dtype=np.float64)
    out[:, 0::2] = v[:, 0::2] * c - v[:, 1::2] * s_
    out[:, 1::2] = v[:, 0::2] * s_ + v[:, 1::2] * c
    return out


def pin_rope_append_is_rotation(o):
    """With a positional key branch the append writes [x W_s^K | R(pos) x W^KR] into the
    shared key row: on small-integer inputs x W^KR is exact, so the stored positional key
    must equal the closed-form rotation at each row's position, rounded to bf16 by torch;
    the content columns must be those of the plain append."""
    n, d, d_h, H, r, d_rope = 9, 24, 16, 2, 8, 16
    X = S.int_grid_bf16(31, "X", (n, d), -1, 1)
    WsK, WsV, WKR = (S.int_grid_bf16(31, nm, (d, w), -1, 1) for nm, w in [("a", d_h), ("b", d_h), ("c", d_rope)])
    UK, UV = (S.int_grid_bf16(31, nm, (H, d, r), -1, 1) for nm in ["e", "f"])
    pos = np.array([0, 1, 2, 7, 63, 64, 1000, 4097, 32767], np.int32)
    sK, sV, zK, zV = o.append(X, WsK, WsV, UK, UV, WKR=WKR, positions=pos)
    plain = o.append(X, WsK, WsV, UK, UV)
    np.testing.assert_array_equal(sK[:, :d_h], plain[0])
    for a_, b_ in zip((sV, zK, zV), plain[1:]):
        np.testing.assert_array_equal(a_, b_)
    u = f64(X) @ f64(WKR)  # exact integers
    want = _lib_bf16(_rope_np(u, pos).astype(np.float32))
    np.testing.assert_array_equal(sK[:, d_h:], want)


def pin_rope_attention_is_concatenated(o):
    """Decode and causal prefill with the positional branch are textbook attention over the
    concatenated key [K_h | k^R] and query [q | q^R] at the scale of the (d_h + d_rope)-wide
    dot product (the MLA lesson, Ch. 3): torch SDPA on exactly those tensors."""
    B, H, d_h, r, d_rope = 2, 3, 16, 8, 16
    lens = [140, 70]
    pt = S.page_table(32, lens, 64, spare_blocks=1)
    sK, sV, zK, zV = random_pools(32, pt.num_blocks, H, d_h, r)
    kR = S.gaussian_bf16(32, "kR", (pt.num_blocks, 64, d_rope))
    pools = (np.ascontiguousarray(np.concatenate([sK, kR], axis=2)), sV, zK, zV)
    w = weights(32, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(32, "q", (B, H, d_h + d_rope))
    scale = 1.0 / np.sqrt(d_h + d_rope)
    got = o.decode_cache(pools, pt.block_table, lens, w.BK, w.BV, q)
    Tq = 30
    qp = S.gaussian_bf16(32, "qp", (B, Tq, H, d_h + d_rope))
    qs = [lens[0] - Tq, lens[1] - Tq]
    gotp = o.prefill_cache(pools, pt.block_table, qs, w.BK, w.BV, qp)
    for b in range(B):
        rows = _gather_rows(pools, pt, b, lens[b])
        for h in range(H):
            Kc = rows[0][:, :d_h] + rows[2][:, h] @ f64(w.BK[h]).T
            K = np.concatenate([Kc, rows[0][:, d_h:]], axis=1)
            V = rows[1] + rows[3][:, h] @ f64(w.BV[h]).T
            ref = _sdpa(f64(q[b, h])[None, None], K[None], V[None], scale)[0, 0]
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-14)
            # causal: query i at position qs[b] + i sees keys 0 .. qs[b] + i
            mask = np.arange(lens[b])[None, :] <= (qs[b] + np.arange(Tq))[:, None]
            out = F.scaled_dot_product_attention(torch.from_numpy(f64(qp[b, :, h])[None]), torch.from_numpy(K[None]),
                                                 torch.from_numpy(V[None]), attn_mask=torch.from_numpy(mask[None]),
                                                 scale=scale).numpy()[0]
            np.testing.assert_allclose(gotp[b, :, h], out, rtol=1e-12, atol=1e-14)


def pin_rotation_direction_worked_example(o):
    """The rotation the positional key gets is the pages' R(theta) = [[cos, -sin], [sin, cos]]: the
    MLA lesson's worked theta = 90 degree products A.R and R.A (golden file).  The oracle rotates pair i
    of a d_rope-vector by pos * base^(-2i/d_rope); with d_rope = 4, pos = 1 and base = 4/pi^2, pair 1
    turns by exactly pi/2, and the unit inputs e_2, e_3 give the two columns of R."""
    g = {}
    for line in open(os.path.join(GOLDEN, "rotation_90deg.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, vals = (t.strip() for t in line.split("|"))
        g[name] = np.array([float(v) for v in vals.split()]).reshape(2, 2)
    d = 4
    X = _lib_bf16(np.eye(d, dtype=np.float32)[2:4])            # rows e_2, e_3
    WKR = _lib_bf16(np.eye(d, dtype=np.float32))
    rows = o.mla_append(X, np.zeros((d, 8), np.uint16), WKR, np.array([1, 1], np.int32),
                        rope_base=4.0 / np.pi ** 2)
    kr = f64(rows[:, 8:])                                       # [2 inputs, 4]
    R = np.stack([kr[0, 2:4], kr[1, 2:4]], axis=1)              # columns R e_0, R e_1 of the pair
    np.testing.assert_allclose(g["A"] @ R, g["A_R"], atol=1e-6)
    np.testing.assert_allclose(R @ g["A"], g["R_A"], atol=1e-6)


# ---------------------------------------------------------------------------- MLA
def _mla_case(seed, B, H, d_c, d_rope, lens):
    pt = S.page_table(seed, lens, 64, spare_blocks=1)
    kv = S.gaussian_bf16(seed, "mla_kv", (pt.num_blocks, 64, d_c + d_rope))
    return pt, kv


def pin_mla_absorbed_is_mqa(o):
    """Absorbed MLA decode is multi-query attention over the cached rows: keys [c | k^R], values c,
    one query [q~_h | q^R_h] per head, scale 1/sqrt(d_head + d_rope) (the MLA lesson: weight
    absorption; decoupled RoPE; the softmax denominator of the concatenated per-head width).
    Checked against torch SDPA on exactly those tensors, page by page gathered here."""
    B, H, d_c, d_rope, d_head = 2, 3, 64, 16, 32
    lens = [150, 9]
    pt, kv = _mla_case(41, B, H, d_c, d_rope, lens)
    q = S.gaussian_bf16(41, "mla_q", (B, H, d_c + d_rope))
    got = o.mla_decode(kv, pt.block_table, lens, q, d_rope, d_head)
    flat = f64(kv.reshape(-1, d_c + d_rope))
    for b in range(B):
        rows = flat[[pt.slot(b, t) for t in range(lens[b])]]
        ref = _sdpa(f64(q[b])[:, None], np.broadcast_to(rows, (H,) + rows.shape).copy(),
                    np.broadcast_to(rows[:, :d_c], (H, lens[b], d_c)).copy(), 1.0 / np.sqrt(d_head + d_rope))
        np.testing.assert_allclose(got[b], ref[:, 0], rtol=1e-12, atol=1e-14)


def pin_mla_absorbed_equals_expanded(o):
    """Associativity ("Low-Rank Key Value Attention", backup frame "MLA also admits associative
    computation"; the MLA lesson's weight absorption): scoring against the latent with q~ = q^C (W^UK)^T
    and mapping o = a C through W^UV equals reconstructing per-head keys c W^UK and values c W^UV and
    attending to them.  Small-integer q^C and W^UK make q~ exact in bf16."""
    B, H, d_c, d_rope, d_head = 2, 2, 32, 8, 8
    lens = [90, 17]
    pt, kv = _mla_case(42, B, H, d_c, d_rope, lens)
    qC = S.int_grid_bf16(42, "qC", (B, H, d_head), -2, 2)
    qR = S.gaussian_bf16(42, "qR", (B, H, d_rope))
    WUK = S.int_grid_bf16(42, "WUK", (H, d_c, d_head), -2, 2)
    WUV = S.gaussian_bf16(42, "WUV", (H, d_c, d_head), d_c ** -0.5)
    qt = np.einsum("bhe,hce->bhc", f64(qC), f64(WUK))
    assert np.all(np.abs(qt) <= 256)                          # integers, exact in bf16
    q = np.concatenate([_lib_bf16(qt), qR], axis=2)
    o_abs = o.mla_decode(kv, pt.block_table, lens, q, d_rope, d_head)
    got = np.einsum("bhc,hce->bhe", o_abs, f64(WUV))
    flat = kv.reshape(-1, d_c + d_rope)
    Lmax = max(lens)
    rows = np.zeros((B, Lmax, d_c + d_rope), np.uint16)
    for b in range(B):
        rows[b, :lens[b]] = flat[[pt.slot(b, t) for t in range(lens[b])]]
    ref = o.mla_decode_expanded(rows, lens, qC, qR, WUK, WUV)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------- training
def pin_train_is_autograd(o):
    """The training projection K_h = X (W_s + U_h B_h^T) and its gradients: forward against a
    direct fp64 evaluation, backward against torch autograd (fp64) of sum(dK * K) -- the
    derivative of the definition, computed by a library, not by the oracle's formulas."""
    n, d, d_h, H, r = 37, 24, 16, 3, 4
    X = S.gaussian_bf16(51, "X", (n, d))
    Ws = S.gaussian_bf16(51, "Ws", (d, d_h), d ** -0.5)
    U = S.gaussian_bf16(51, "U", (H, d, r), d ** -0.5)
    Bm = S.gaussian_bf16(51, "B", (H, d_h, r), r ** -0.5)
    dK = S.gaussian_bf16(51, "dK", (n, H, d_h))
    tX, tWs, tU, tB = (torch.from_numpy(f64(a)).requires_grad_(True) for a in (X, Ws, U, Bm))
    W = tWs[None] + torch.einsum("hkj,hij->hki", tU, tB)        # [H, d, d_h]
    K = torch.einsum("tk,hki->thi", tX, W)                       # [n, H, d_h]
    np.testing.assert_allclose(o.train_forward(X, Ws, U, Bm), K.detach().numpy(), rtol=1e-12, atol=1e-12)
    (K * torch.from_numpy(f64(dK))).sum().backward()
    got = o.train_backward(X, Ws, U, Bm, dK)
    for g_, ref in zip(got, (tX.grad, tWs.grad, tU.grad, tB.grad)):
        np.testing.assert_allclose(g_, ref.numpy(), rtol=1e-11, atol=1e-11)


PINS = [pin_softmax_worked_value, pin_softmax_normalised, pin_attend_special_cases,
        pin_append_integer_exact, pin_append_gaussian_rounding, pin_r0_is_mqa, pin_mha_special_case,
        pin_factored_equals_expanded, pin_cache_path_matches_weight_path,
        pin_head_permutation_equivariance, pin_page_permutation_invariance, pin_prefill_causal_edges,
        pin_fused_is_concatenated_attention, pin_fused_matches_factored_decode,
        pin_prefill_fused_is_concatenated_causal_attention, pin_prefill_fused_matches_factored_prefill,
        pin_rope_append_is_rotation, pin_rope_attention_is_concatenated, pin_rotation_direction_worked_example,
        pin_mla_absorbed_is_mqa, pin_mla_absorbed_equals_expanded, pin_train_is_autograd]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# Each planted mistake, and what it models:
#  1 residual term U_h B_h^T dropped      2 B^K used for values       3 scale 1/d_h
#  4 causal diagonal excluded             5 shared term dropped       6 B_h read transposed
#  7 absorbed decode drops the residual values z^V
#  8 positional key rotated the wrong way    9 scale of the content width only with a positional key
# 10 MLA scale over the cached row's width  11 MLA values read from the wrong slice of the row
# 12 training: dB_h formed with dK_h B_h in place of X U_h
# 13 absorbed prefill reads q~ of the next head
MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistakes_are_caught(mutant):
    o = oracle.Oracle(mutant)
    failed = []
    for pin in PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant} passed every pin"
