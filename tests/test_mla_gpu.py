"""Multi-head latent attention (absorbed weights) on the GPU against the fp64 oracle.

The cache row is [c_t | k^R_t] (latent d_c = 512 and positional key d_rope = 64, shared by all
heads); head i attends with [q~_i | q^R_i] and returns o_i = sum_t p_t c_t before W^UV_i, scale
1/sqrt(d_head + d_rope) ("Embeddings II: MLA & Architectural Choices": weight absorption,
decoupled RoPE, the softmax denominator).  The kernel splits every sequence over pairs of CTAs
that divide the row's columns and exchange partial logits; the oracle is textbook attention.
"""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import f64
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64
from test_append_gpu import _bf16_ulp

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402

DC, DR, DK = 512, 64, 576
CANARY = 0x7E57


def run_mla(H, kv, pt, q, d_head=128, scale=0.0, seq_lens=None):
    dims = b.make_mla_dims(H, 5120, d_head=d_head, softmax_scale=scale)
    Bn = q.shape[0]
    out = torch.empty((Bn, H, DC), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.mla_decode_workspace_bytes(dims, Bn))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = pt.seq_lens if seq_lens is None else seq_lens
    b.lrkv_mla_decode(dims, dev_bf16(q), dev_bf16(kv), dev_i32(pt.block_table), dev_i32(lens), out, ws, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def mla_case(seed, H, lens, spare=2):
    pt = S.page_table(seed, lens, 64, spare_blocks=spare)
    kv = S.gaussian_bf16(seed, "mla_kv", (pt.num_blocks, 64, DK))
    q = S.gaussian_bf16(seed, "mla_q", (len(lens), H, DK))
    return pt, kv, q


SHAPES = [
    # H, seq_lens
    (128, [256]),
    (128, [8192, 1, 63, 64, 65, 4000]),        # ragged: partial last pages, single-token sequences
    (16, [3000, 129]),
    (1, [700]),
    (100, [2048, 77]),                          # heads not a multiple of 32
    (128, [16384, 9000]),                       # long: many pages per split
    (32, [300] * 90),                           # more sequences than CTA pairs: several splits per pair
]


@pytest.mark.parametrize("H,lens", SHAPES, ids=[f"H{s[0]}_n{len(s[1])}_L{max(s[1])}" for s in SHAPES])
def test_mla_decode_matches_oracle(H, lens):
    pt, kv, q = mla_case(500 + H + len(lens), H, lens)
    out, st = run_mla(H, kv, pt, q)
    assert st == 0
    ref = oracle.get().mla_decode(kv, pt.block_table, pt.seq_lens, q, DR, 128)
    assert_close(host_f64(out), ref, f"MLA decode H={H} lens={lens[:4]}")


def test_mla_decode_explicit_scale_and_bad_length():
    H = 64
    pt, kv, q = mla_case(511, H, [500, 300, 90])
    lens = pt.seq_lens.copy()
    lens[1] = 0
    out, st = run_mla(H, kv, pt, q, scale=0.04, seq_lens=lens)
    assert st & b.DEV_BAD_SEQLEN
    got = host_f64(out)
    assert np.all(got[1] == 0)
    keep = [0, 2]
    ref = oracle.get().mla_decode(kv, pt.block_table[keep], lens[keep], q[keep], DR, 128, scale=0.04)
    assert_close(got[keep], ref, "MLA decode, explicit scale, next to a rejected sequence")


def test_mla_decode_is_deterministic_and_page_order_free():
    """The same inputs give the same bits; permuting the physical pages (table rewritten) does too."""
    H = 128
    pt, kv, q = mla_case(512, H, [5000, 3000])
    out1, _ = run_mla(H, kv, pt, q)
    out2, _ = run_mla(H, kv, pt, q)
    np.testing.assert_array_equal(host_bits(out1), host_bits(out2))
    perm = S.permutation(512, "perm", pt.num_blocks)
    kv2 = np.empty_like(kv)
    kv2[perm] = kv
    pt2 = S.page_table(512, [5000, 3000], 64, spare_blocks=2)
    pt2.block_table[:] = np.where(pt.block_table >= 0, perm[np.maximum(pt.block_table, 0)], pt.block_table)
    out3, _ = run_mla(H, kv2, pt2, q)
    np.testing.assert_array_equal(host_bits(out1), host_bits(out3))


@pytest.mark.parametrize("n", [1, 5, 64, 200])
def test_mla_append_exact_inputs(n):
    """Integer-grid inputs: the latent columns match the oracle bit for bit, the rotated columns to one ulp."""
    d = 1024
    X = S.int_grid_bf16(n, "X", (n, d), -8, 8)
    WDKV = S.int_grid_bf16(n, "WDKV", (d, DC), -8, 8)
    WKR = S.int_grid_bf16(n, "WKR", (d, DR), -8, 8)
    nb = (n + 63) // 64 + 2
    slots = S.permutation(n, "slots", nb * 64)[:n].astype(np.int32)
    pos = S.uniform_int(n, "pos", n, 0, 1 << 17).astype(np.int32)
    kv = torch.from_numpy(np.full((nb, 64, DK), CANARY, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)
    dims = b.make_mla_dims(8, d)
    wt = np.ascontiguousarray(np.concatenate([WDKV.T, WKR.T], axis=0))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_mla_append(dims, dev_bf16(X), dev_bf16(wt), dev_i32(slots), dev_i32(pos), kv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host_bits(kv).reshape(-1, DK)
    ref = oracle.get().mla_append(X, WDKV, WKR, pos)
    np.testing.assert_array_equal(got[slots, :DC], ref[:, :DC])
    gr, rr = f64(got[slots, DC:]), f64(ref[:, DC:])
    assert np.all(np.abs(gr - rr) <= _bf16_ulp(rr))
    # last-bit differences of the rotation: ~2e-5 of the values; allow 1e-4 of them, and at least one
    assert int((gr != rr).sum()) <= max(1, int(np.ceil(1e-4 * gr.size)))
    untouched = np.setdiff1d(np.arange(nb * 64), slots)
    assert np.all(got[untouched] == CANARY)


def test_mla_append_then_decode_end_to_end():
    """Hidden rows appended at their positions, then one decode step: against the oracle's
    append and absorbed decode of the same inputs."""
    H, d = 128, 2048
    lens = [700, 64, 1]
    pt = S.page_table(520, lens, 64, spare_blocks=1)
    WDKV = S.gaussian_bf16(520, "WDKV", (d, DC), d ** -0.5)
    WKR = S.gaussian_bf16(520, "WKR", (d, DR), d ** -0.5)
    wt = dev_bf16(np.ascontiguousarray(np.concatenate([WDKV.T, WKR.T], axis=0)))
    dims = b.make_mla_dims(H, d)
    kv = torch.zeros((pt.num_blocks, 64, DK), dtype=torch.bfloat16, device="cuda")
    ref_kv = np.zeros((pt.num_blocks, 64, DK), np.uint16)
    for bi, L in enumerate(lens):
        X = S.gaussian_bf16(521 + bi, "X", (L, d))
        pos = np.arange(L, dtype=np.int32)
        slots = S.slots_for(pt, bi, 0, L)
        b.lrkv_mla_append(dims, dev_bf16(X), wt, dev_i32(slots), dev_i32(pos), kv)
        ref_kv.reshape(-1, DK)[slots] = oracle.get().mla_append(X, WDKV, WKR, pos)
    q = S.gaussian_bf16(522, "q", (len(lens), H, DK))
    out = torch.empty((len(lens), H, DC), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_mla_decode(dims, dev_bf16(q), kv, dev_i32(pt.block_table), dev_i32(pt.seq_lens), out,
                      b.alloc_workspace(b.mla_decode_workspace_bytes(dims, len(lens))), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.get().mla_decode(ref_kv, pt.block_table, pt.seq_lens, q, DR, 128)
    assert_close(host_f64(out), ref, "MLA append with positions, then decode")
