"""lrkv_append of a few rows with a weight stream of 64 MiB or more, on the GPU against the oracle.

Eqs. (4)-(5) of "Low-Rank Key Value Attention" at the sizes of a large layer: W_cat^T of the
DeepSeek-V2-scale layer (H=128, d_h=128, r=16, d=16384) is 4352 x 16384 bf16 (142 MB), and a decode
step appends one row per sequence.  Integer-grid inputs (k in [-8, 8]) keep every fp32 partial sum
exact (|sum| <= 64 d < 2^24), so any summation order gives the oracle's value and the content
columns must match bit for bit.  A rotated positional-key column may differ by one bf16 ulp, where
the two sides' double-precision sine and cosine differ in the last bits.

The inputs are drawn by torch's seeded device generator (this much data takes too long for the
host generator) and copied back for the oracle.
"""
import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import empty_pools, f64
from gpu_util import dev_bf16, dev_i32, host_bits
from test_append_gpu import CANARY, _bf16_ulp
from test_append_rope_gpu import _positions
from test_workloads_gpu import _unpack_wcat

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def _int_grid_dev(gen, shape):
    return torch.randint(-8, 9, shape, generator=gen, device="cuda", dtype=torch.int32).to(torch.bfloat16)


@pytest.mark.parametrize("n,H,d_h,r,d,d_rope", [
    (8, 128, 128, 16, 16384, 0),   # the DeepSeek-V2-scale layer, one 8-row block
    (1, 128, 128, 16, 16384, 64),  # one row, with the positional key
    (13, 127, 64, 8, 15560, 0),    # a 16-row block; N = 2160 ends in half a 32-column group; d % 64 != 0
    (40, 127, 64, 8, 15560, 64),   # three row blocks (16, 16, 8), with the positional key
])
def test_append_large_weight_stream_exact(n, H, d_h, r, d, d_rope):
    N = 2 * (d_h + H * r) + d_rope
    assert N * d * 2 >= 64 << 20
    gen = torch.Generator(device="cuda").manual_seed(1000 + n)
    wcat = _int_grid_dev(gen, (N, d))
    X = _int_grid_dev(gen, (n, d))
    nb = (n + 63) // 64 + 2
    slots = S.permutation(n, "slots", nb * 64)[:n].astype(np.int32)
    pos = _positions(n, n)
    dims = b.make_dims(H, d_h, r, d, d_rope=d_rope)
    cache = b.PagedCache(*(dev_bf16(p) for p in empty_pools(nb, H, d_h, r, fill=CANARY, d_rope=d_rope)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.lrkv_append(dims, X, wcat, dev_i32(slots), cache, status=st, positions=dev_i32(pos) if d_rope else None)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = [host_bits(t) for t in cache.tensors()]

    WsK, WsV, UK, UV, WKR = _unpack_wcat(host_bits(wcat), d_h, H, r, d_rope)
    Xh = host_bits(X)
    if d_rope:
        ref = oracle.get().append(Xh, WsK, WsV, UK, UV, WKR=WKR, positions=pos, rope_base=10000.0)
    else:
        ref = oracle.get().append(Xh, WsK, WsV, UK, UV)
    g = [p.reshape((-1,) + p.shape[2:])[slots] for p in got]
    np.testing.assert_array_equal(g[0][:, :d_h], ref[0][:, :d_h], err_msg="s^K")
    for gi, ri, nm in zip(g[1:], ref[1:], ("sV", "zK", "zV")):
        np.testing.assert_array_equal(gi, ri, err_msg=nm)
    if d_rope:
        gr, rr = f64(g[0][:, d_h:]), f64(ref[0][:, d_h:])
        assert np.all(np.abs(gr - rr) <= _bf16_ulp(rr)), "k^R beyond one ulp"
    untouched = np.setdiff1d(np.arange(nb * 64), slots)
    for p in got:
        assert np.all(p.reshape((-1,) + p.shape[2:])[untouched] == CANARY)
