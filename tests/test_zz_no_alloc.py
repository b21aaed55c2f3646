"""lrkv_decode_static_ws: decode for callers that cannot allocate device memory.

Such callers (a serving loop that must not stall the device in cudaMalloc, a host
framework that owns the GPU allocator, a deployment with a memory budget fixed at
start-up) get their decode scratch from a fixed array inside the library instead
of a workspace they pass in.  This file checks, through the C ABI, that two calls
in a row give the same answer as lrkv_decode with a caller workspace, and that a
batch too large for the fixed array is refused with a clear error.  It is named
so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import lrkv_synth as S
import oracle
from cases import random_pools, weights
from gpu_util import assert_close, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu

from compressed_kv_cache_lrkv_gb300 import binding as b  # noqa: E402


def _host_case(seed, H, d_h, r, lens):
    pt = S.page_table(seed, lens, 64, spare_blocks=1)
    pools = random_pools(seed, pt.num_blocks, H, d_h, r)
    w = weights(seed, H * d_h, d_h, H, r)
    q = S.gaussian_bf16(seed, "q", (len(lens), H, d_h))
    return pt, pools, w, q


def _case(seed, H, d_h, r, lens):
    pt, pools, w, q = _host_case(seed, H, d_h, r, lens)
    dims = b.make_dims(H, d_h, r, H * d_h)
    cache = b.PagedCache(*(dev_bf16(p) for p in pools))
    return dims, cache, dev_bf16(q), dev_bf16(w.BK), dev_bf16(w.BV), dev_i32(pt.block_table), dev_i32(pt.seq_lens)


def _with_workspace(dims, cache, q, BK, BV, bt, sl):
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, q.shape[0]))
    b.lrkv_decode(dims, q, BK, BV, cache, bt, sl, out, ws)
    return out


def _static(dims, cache, q, BK, BV, bt, sl):
    """Call the C entry point directly (no binding helper): no workspace argument."""
    lib = b.load()
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = cache.struct()
    rc = lib.lrkv_decode_static_ws(ctypes.byref(dims), q.data_ptr(), BK.data_ptr(), BV.data_ptr(), ctypes.byref(c),
                                   bt.data_ptr(), int(bt.shape[1]), sl.data_ptr(), int(q.shape[0]), out.data_ptr(),
                                   status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.lrkv_last_error()
    return out, status


def test_static_scratch_decode_matches_workspace_decode_twice():
    # two different problems back to back: the second call must not see the first's scratch
    first = _case(41, 32, 128, 32, [9000, 300, 4100])
    second = _case(42, 8, 64, 16, [2048, 1, 77, 1500, 640])
    for args in (first, second):
        ref = _with_workspace(*args)
        got, status = _static(*args)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(host_f64(got), host_f64(ref), "static-scratch decode vs workspace decode")
    # and directly against the fp64 oracle on the first problem, after the second has used the array
    pt, pools, w, q = _host_case(41, 32, 128, 32, [9000, 300, 4100])
    got, status = _static(*first)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.get().decode_cache(pools, pt.block_table, pt.seq_lens, w.BK, w.BV, q)
    assert_close(host_f64(got), ref, "static-scratch decode vs oracle")


def test_static_scratch_rejects_batches_that_do_not_fit():
    H, d_h, r = 128, 128, 32
    dims = b.make_dims(H, d_h, r, H * d_h)
    batch = 4096
    assert b.decode_workspace_bytes(dims, batch) > b.STATIC_WS_BYTES
    lib = b.load()
    c = b.Cache(16, 16, 16, 16, 1)
    rc = lib.lrkv_decode_static_ws(ctypes.byref(dims), 16, 16, 16, ctypes.byref(c), 16, 1, 16, batch, 16, None, None)
    assert rc == 3  # LRKV_ERR_WORKSPACE
    assert b"LRKV_STATIC_WS_BYTES" in lib.lrkv_last_error()
