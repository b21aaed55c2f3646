"""lrkv_decode_fused (both absorptions in the caller's weights) on the GPU against the fp64
oracle: the query arrives as [q | q~] and the result is [o_s | o_z] before the residual
up-projection.  Same shapes and edge cases as the ordinary decode."""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import random_pools
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def run_fused(H, d_h, r, pools, pt, q, qt, status=None, seq_lens=None):
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    Bn = q.shape[0]
    out = torch.empty((Bn, H, d_h + r), dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, Bn))
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = pt.seq_lens if seq_lens is None else seq_lens
    b.lrkv_decode_fused(dims, dev_bf16(q), dev_bf16(qt), cache, dev_i32(pt.block_table), dev_i32(lens), out, ws,
                        status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def fused_case(seed, H, d_h, r, seq_lens, spare=2):
    pt = S.page_table(seed, seq_lens, 64, spare_blocks=spare)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r)
    q = S.gaussian_bf16(seed, "q", (len(seq_lens), H, d_h))
    qt = S.gaussian_bf16(seed, "qt", (len(seq_lens), H, r))
    return pt, pools, q, qt


SHAPES = [
    # H, d_h, r, seq_lens
    (8, 64, 8, [256]),
    (8, 64, 16, [2048, 1, 7, 65, 500]),
    (32, 128, 32, [3000, 129, 64, 1]),
    (128, 128, 16, [700, 64]),
    (20, 128, 16, [333, 1024]),
    (3, 64, 32, [95]),
    (32, 128, 32, [20000, 9000, 31000, 17000]),  # long-context lengths: splits longer than the ring
]


@pytest.mark.parametrize("H,d_h,r,lens", SHAPES, ids=[f"H{s[0]}_dh{s[1]}_r{s[2]}_n{len(s[3])}" for s in SHAPES])
def test_fused_decode_matches_oracle(H, d_h, r, lens):
    pt, pools, q, qt = fused_case(300 + H + r + len(lens), H, d_h, r, lens)
    out, st = run_fused(H, d_h, r, pools, pt, q, qt)
    assert st == 0
    ref = oracle.get().decode_fused(pools, pt.block_table, pt.seq_lens, q, qt)
    assert_close(host_f64(out), ref, f"fused decode H={H} d_h={d_h} r={r}")


def test_fused_decode_bad_length_gives_zero_row_and_status():
    H, d_h, r = 8, 64, 16
    pt, pools, q, qt = fused_case(311, H, d_h, r, [300, 200])
    lens = pt.seq_lens.copy()
    lens[1] = 0
    out, st = run_fused(H, d_h, r, pools, pt, q, qt, seq_lens=lens)
    assert st & 0x2  # LRKV_DEV_BAD_SEQLEN
    got = host_f64(out)
    assert np.all(got[1] == 0)
    ref = oracle.get().decode_fused(pools, pt.block_table, lens[:1], q[:1], qt[:1])
    assert_close(got[:1], ref, "fused decode, valid sequence next to a rejected one")
