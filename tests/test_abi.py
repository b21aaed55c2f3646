"""C-ABI surface (no GPU needed): the library builds, loads, exports every entry
point include/lrkv.h declares, and rejects bad host arguments before launching."""
import ctypes
import os
import re

import pytest

from compressed_kv_cache_lrkv_gb300 import binding as b

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lrkv.h")


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(lrkv_[a-z_]+)\s*\(", txt)))


def test_header_declares_expected_calls():
    names = _declared()
    for n in ("lrkv_append", "lrkv_decode", "lrkv_decode_fused", "lrkv_prefill", "lrkv_prefill_fused",
              "lrkv_decode_workspace_bytes",
              "lrkv_status_string", "lrkv_append_layers", "lrkv_decode_layers"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = b.load()
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(b.EXPORTED) | set(_declared())
    assert b.abi_version() == 4


def test_status_strings():
    lib = b.load()
    for code in range(7):
        assert lib.lrkv_status_string(code)
    assert lib.lrkv_status_string(99) == b"unknown status"


def test_cache_block_bytes_matches_accounting():
    from compressed_kv_cache_lrkv_gb300 import accounting as A
    for H, d_h, r in [(8, 64, 8), (8, 64, 16), (128, 128, 16), (32, 128, 32), (32, 128, 16)]:
        assert b.cache_block_bytes(b.make_dims(H, d_h, r, H * d_h)) == A.page_bytes(H, d_h, r)
        assert b.cache_block_bytes(b.make_dims(H, d_h, r, H * d_h, d_rope=64)) == A.page_bytes(H, d_h, r, d_rope=64)


@pytest.mark.parametrize("H,d_h,r,d,bs,why", [
    (8, 96, 8, 512, 64, "d_h"), (8, 64, 12, 512, 64, "r"), (8, 64, 128, 512, 64, "r > d_h"),
    (0, 64, 8, 512, 64, "H"), (129, 64, 8, 512, 64, "H"), (8, 64, 8, 500, 64, "d"), (8, 64, 8, 512, 32, "block"),
])
def test_unsupported_dims_rejected(H, d_h, r, d, bs, why):
    dims = b.make_dims(H, d_h, r, d, bs)
    assert b.cache_block_bytes(dims) == 0, why
    lib = b.load()
    c = b.Cache(16, 16, 16, 16, 1)
    rc = lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, None, ctypes.byref(c), None, None)
    assert rc == 2, lib.lrkv_last_error()


def test_null_and_misaligned_pointers_rejected():
    lib = b.load()
    dims = b.make_dims(8, 64, 8, 512)
    c = b.Cache(16, 16, 16, 16, 1)
    assert lib.lrkv_append(ctypes.byref(dims), None, 16, 1, 16, None, ctypes.byref(c), None, None) == 1
    assert b"X is NULL" in lib.lrkv_last_error()
    assert lib.lrkv_append(ctypes.byref(dims), 24, 16, 1, 16, None, ctypes.byref(c), None, None) == 1
    assert b"aligned" in lib.lrkv_last_error()
    bad = b.Cache(16, 0, 16, 16, 1)
    assert lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, None, ctypes.byref(bad), None, None) == 1
    bad = b.Cache(16, 16, 16, 16, 0)
    assert lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, None, ctypes.byref(bad), None, None) == 1
    assert lib.lrkv_append(ctypes.byref(dims), 16, 16, -1, 16, None, ctypes.byref(c), None, None) == 1
    # zero rows / zero batch are no-ops that succeed without touching the device
    assert lib.lrkv_append(ctypes.byref(dims), None, None, 0, None, None, ctypes.byref(c), None, None) == 0
    assert lib.lrkv_decode(ctypes.byref(dims), 16, 16, 16, ctypes.byref(c), 16, 1, 16, 0, 16, 256, 0, None,
                           None) == 0
    assert lib.lrkv_decode(ctypes.byref(dims), 16, 16, 16, ctypes.byref(c), 16, 0, 16, 1, 16, 256, 0, None,
                           None) == 1
    assert lib.lrkv_prefill(ctypes.byref(dims), 16, 16, 16, ctypes.byref(c), 16, 1, 16, 1, -3, 16, None, 0, None,
                            None) == 1
    # absorbed-weights decode: q~ is required and 16-byte aligned; batch 0 is a no-op
    assert lib.lrkv_decode_fused(ctypes.byref(dims), 16, None, ctypes.byref(c), 16, 1, 16, 1, 16, 256, 0, None,
                                 None) == 1
    assert b"q_tilde" in lib.lrkv_last_error()
    assert lib.lrkv_decode_fused(ctypes.byref(dims), 16, 24, ctypes.byref(c), 16, 1, 16, 1, 16, 256, 0, None,
                                 None) == 1
    assert b"aligned" in lib.lrkv_last_error()
    assert lib.lrkv_decode_fused(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 0, 16, 256, 0, None,
                                 None) == 0
    # token-split decode: partials and the merge need their buffers; a merge of no parts is refused
    assert lib.lrkv_decode_partials(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 1, None, 256, 0, None,
                                    None) == 1
    assert b"partials" in lib.lrkv_last_error()
    assert lib.lrkv_decode_partials(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 0, 16, 256, 0, None,
                                    None) == 0
    assert lib.lrkv_decode_merge(ctypes.byref(dims), 0, 16, 16, 1, 16, None, None) == 1
    assert lib.lrkv_decode_merge(ctypes.byref(dims), 2, None, 16, 1, 16, None, None) == 1
    assert lib.lrkv_decode_merge(ctypes.byref(dims), 2, 16, 24, 1, 16, None, None) == 1
    assert b"aligned" in lib.lrkv_last_error()
    assert lib.lrkv_decode_merge(ctypes.byref(dims), 2, 16, 16, 0, 16, None, None) == 0
    # absorbed-weights prefill: the same rules for q~; batch 0 or Tq 0 is a no-op
    assert lib.lrkv_prefill_fused(ctypes.byref(dims), 16, None, ctypes.byref(c), 16, 1, 16, 1, 4, 16, None,
                                  None) == 1
    assert b"q_tilde" in lib.lrkv_last_error()
    assert lib.lrkv_prefill_fused(ctypes.byref(dims), 16, 24, ctypes.byref(c), 16, 1, 16, 1, 4, 16, None,
                                  None) == 1
    assert b"aligned" in lib.lrkv_last_error()
    assert lib.lrkv_prefill_fused(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 1, -1, 16, None,
                                  None) == 1
    assert lib.lrkv_prefill_fused(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 0, 4, 16, None,
                                  None) == 0
    assert lib.lrkv_prefill_fused(ctypes.byref(dims), 16, 16, ctypes.byref(c), 16, 1, 16, 3, 0, 16, None,
                                  None) == 0


def test_nan_scale_rejected():
    lib = b.load()
    dims = b.make_dims(8, 64, 8, 512, softmax_scale=float("nan"))
    assert b.cache_block_bytes(dims) == 0


@pytest.mark.parametrize("d_rope,base,code", [(32, 0.0, 2), (128, 0.0, 2), (-64, 0.0, 2), (64, float("nan"), 1),
                                              (64, 1.0, 1), (64, -5.0, 1), (64, float("inf"), 1)])
def test_positional_key_dims_rejected(d_rope, base, code):
    """d_rope outside {0, 64} is an unsupported shape; a RoPE base that is NaN, infinite or <= 1 is invalid."""
    lib = b.load()
    dims = b.make_dims(8, 64, 8, 512, d_rope=d_rope, rope_base=base)
    assert b.cache_block_bytes(dims) == 0
    c = b.Cache(16, 16, 16, 16, 1)
    assert lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, 16, ctypes.byref(c), None, None) == code


def test_positional_key_needs_positions():
    lib = b.load()
    dims = b.make_dims(8, 64, 8, 512, d_rope=64)
    c = b.Cache(16, 16, 16, 16, 1)
    assert lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, None, ctypes.byref(c), None, None) == 1
    assert b"positions" in lib.lrkv_last_error()
    # without a positional key the positions pointer is ignored
    plain = b.make_dims(8, 64, 8, 512)
    assert lib.lrkv_append(ctypes.byref(plain), None, None, 0, None, None, ctypes.byref(c), None, None) == 0


@pytest.mark.parametrize("kw,code", [(dict(d_c=256), 2), (dict(d_rope=32), 2), (dict(H=0), 2), (dict(H=129), 2),
                                     (dict(block_size=32), 2), (dict(d=500), 2), (dict(d_head=0), 1),
                                     (dict(softmax_scale=float("nan")), 1), (dict(rope_base=0.5), 1)])
def test_mla_dims_rejected(kw, code):
    """Multi-head latent attention: d_c = 512, d_rope = 64, block 64, 1 <= H <= 128 are the supported shape."""
    lib = b.load()
    base = dict(H=128, d=5120)
    base.update(kw)
    dims = b.make_mla_dims(**base)
    assert b.mla_cache_block_bytes(dims) == 0
    assert lib.lrkv_mla_append(ctypes.byref(dims), 16, 16, 1, 16, 16, 16, 1, None, None) == code
    assert lib.lrkv_mla_decode(ctypes.byref(dims), 16, 16, 1, 16, 1, 16, 1, 16, 256, 1 << 30, None, None) == code


def test_mla_arguments():
    lib = b.load()
    dims = b.make_mla_dims(128, 5120)
    assert b.mla_cache_block_bytes(dims) == 64 * 2 * 576
    # positions are required; zero rows / zero batch are no-ops
    assert lib.lrkv_mla_append(ctypes.byref(dims), 16, 16, 1, 16, None, 16, 1, None, None) == 1
    assert b"positions" in lib.lrkv_last_error()
    assert lib.lrkv_mla_append(ctypes.byref(dims), None, None, 0, None, None, None, 1, None, None) == 0
    assert lib.lrkv_mla_append(ctypes.byref(dims), 24, 16, 1, 16, 16, 16, 1, None, None) == 1
    assert lib.lrkv_mla_decode(ctypes.byref(dims), 16, 16, 1, 16, 1, 16, 0, 16, 256, 0, None, None) == 0
    assert lib.lrkv_mla_decode(ctypes.byref(dims), 16, 16, 0, 16, 1, 16, 1, 16, 256, 0, None, None) == 1
    assert lib.lrkv_mla_decode(ctypes.byref(dims), 16, 16, 1, None, 1, 16, 1, 16, 256, 0, None, None) == 1


def test_header_supported_ranks_match_the_library():
    """The header's supported set of r is the one the library accepts."""
    txt = open(HEADER).read()
    m = re.search(r"r in \{([0-9, ]+)\}", txt)
    assert m, "supported ranks not stated"
    stated = sorted(int(x) for x in m.group(1).split(","))
    accepted = [r for r in range(1, 129) if b.cache_block_bytes(b.make_dims(8, 128, r, 1024)) > 0]
    assert stated == accepted == [8, 16, 32]


@pytest.mark.parametrize("ns,ok", [(0, True), (1, True), (7, True), (65536, True), (-1, False), (65537, False)])
def test_num_splits_range(ns, ok):
    dims = b.make_dims(8, 64, 16, 512, num_splits=ns)
    assert (b.cache_block_bytes(dims) > 0) == ok
    if not ok:
        lib = b.load()
        c = b.Cache(16, 16, 16, 16, 1)
        assert lib.lrkv_append(ctypes.byref(dims), 16, 16, 1, 16, None, ctypes.byref(c), None, None) == 1
        assert b"num_splits" in lib.lrkv_last_error()


def _strides(**kw):
    st = b.LayerStrides()
    for k, v in kw.items():
        setattr(st, k, v)
    return st


def test_layer_batched_calls_validate_strides():
    """Per-layer strides must be multiples of 8 elements and cover one layer's tensor; one layer
    ignores them; checked before anything touches the device."""
    lib = b.load()
    H, d_h, r, d, nb, n = 8, 64, 16, 512, 4, 3
    dims = b.make_dims(H, d_h, r, d)
    c = b.Cache(16, 16, 16, 16, nb)
    rows = nb * 64
    N = 2 * (d_h + H * r)
    good = dict(X=n * d, W_catT=N * d, sK=rows * d_h, sV=rows * d_h, zK=rows * H * r, zV=rows * H * r)
    app = lambda L, st: lib.lrkv_append_layers(ctypes.byref(dims), L, st, 16, 16, n, 16, None, ctypes.byref(c), None,
                                               None)
    assert app(0, ctypes.byref(_strides(**good))) == 1
    assert app(2, None) == 1
    for k in good:
        bad = dict(good)
        bad[k] = good[k] - 8          # layers would overlap
        assert app(2, ctypes.byref(_strides(**bad))) == 1, k
        assert k in lib.lrkv_last_error().decode()
        bad[k] = good[k] + 4          # not 16-byte aligned
        assert app(2, ctypes.byref(_strides(**bad))) == 1, k
    # zero rows: a no-op once the arguments are valid
    assert lib.lrkv_append_layers(ctypes.byref(dims), 3, ctypes.byref(_strides(**good)), None, None, 0, None, None,
                                  ctypes.byref(c), None, None) == 0
    B = 2
    dgood = dict(q=B * H * d_h, BK=H * d_h * r, BV=H * d_h * r, out=B * H * d_h, sK=rows * d_h, sV=rows * d_h,
                 zK=rows * H * r, zV=rows * H * r)
    dec = lambda L, st: lib.lrkv_decode_layers(ctypes.byref(dims), L, st, 16, 16, 16, ctypes.byref(c), 16, 1, 16, B,
                                               16, 256, 1 << 30, None, None)
    for k in dgood:
        bad = dict(dgood)
        bad[k] = dgood[k] - 8
        assert dec(2, ctypes.byref(_strides(**bad))) == 1, k
        assert k in lib.lrkv_last_error().decode()
    assert dec(0, ctypes.byref(_strides(**dgood))) == 1
    assert dec(2, None) == 1
    assert lib.lrkv_decode_layers(ctypes.byref(dims), 2, ctypes.byref(_strides(**dgood)), 16, 16, 16,
                                  ctypes.byref(c), 16, 1, 16, 0, 16, 256, 0, None, None) == 0
