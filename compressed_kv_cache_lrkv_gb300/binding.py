"""Thin ctypes binding of liblrkv.so (include/lrkv.h): argument marshalling only.

Every function here forwards to the C entry point of the same name; tensors
are torch CUDA tensors whose data pointers are passed through.  Nothing is
computed in Python, and there is no fallback: if the library cannot be loaded
(or a call returns an error) an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

LRKV_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace too small", 4: "CUDA error",
                5: "device bounds", 6: "timeout"}
DEV_BAD_BLOCK, DEV_BAD_SEQLEN, DEV_BAD_SLOT, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

EXPORTED = ["lrkv_abi_version", "lrkv_status_string", "lrkv_last_error", "lrkv_cache_block_bytes", "lrkv_append",
            "lrkv_decode_workspace_bytes", "lrkv_decode", "lrkv_decode_fused", "lrkv_decode_static_ws",
            "lrkv_decode_partials", "lrkv_decode_merge",
            "lrkv_append_layers", "lrkv_decode_layers",
            "lrkv_prefill_workspace_bytes", "lrkv_prefill", "lrkv_prefill_fused", "lrkv_mla_cache_block_bytes", "lrkv_mla_append",
            "lrkv_mla_decode_workspace_bytes", "lrkv_mla_decode", "lrkv_train_forward", "lrkv_train_workspace_bytes",
            "lrkv_train_backward"]
STATIC_WS_BYTES = 16 << 20  # LRKV_STATIC_WS_BYTES


class LrkvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("d_h", ctypes.c_int32), ("r", ctypes.c_int32), ("d", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("softmax_scale", ctypes.c_float), ("d_rope", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("num_splits", ctypes.c_int32)]


class LayerStrides(ctypes.Structure):
    """Element strides between consecutive layers' tensors (lrkv_layer_strides)."""
    _fields_ = [(n, ctypes.c_int64) for n in ("X", "W_catT", "q", "BK", "BV", "out", "sK", "sV", "zK", "zV")]


class MlaDims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("d_c", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("d_head", ctypes.c_int32),
                ("d", ctypes.c_int32), ("block_size", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("rope_base", ctypes.c_float)]


class Cache(ctypes.Structure):
    _fields_ = [("sK", ctypes.c_void_p), ("sV", ctypes.c_void_p), ("zK", ctypes.c_void_p), ("zV", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) liblrkv.so and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        path = _build.build()
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    P = ctypes.POINTER
    lib.lrkv_abi_version.restype = ctypes.c_int
    lib.lrkv_status_string.restype = ctypes.c_char_p
    lib.lrkv_status_string.argtypes = [ctypes.c_int]
    lib.lrkv_last_error.restype = ctypes.c_char_p
    lib.lrkv_cache_block_bytes.restype = sz
    lib.lrkv_cache_block_bytes.argtypes = [P(Dims)]
    lib.lrkv_append.restype = ctypes.c_int
    lib.lrkv_append.argtypes = [P(Dims), vp, vp, i32, vp, vp, P(Cache), vp, vp]
    lib.lrkv_decode_workspace_bytes.restype = sz
    lib.lrkv_decode_workspace_bytes.argtypes = [P(Dims), i32]
    lib.lrkv_decode.restype = ctypes.c_int
    lib.lrkv_decode.argtypes = [P(Dims), vp, vp, vp, P(Cache), vp, i32, vp, i32, vp, vp, sz, vp, vp]
    lib.lrkv_decode_fused.restype = ctypes.c_int
    lib.lrkv_decode_fused.argtypes = [P(Dims), vp, vp, P(Cache), vp, i32, vp, i32, vp, vp, sz, vp, vp]
    lib.lrkv_append_layers.restype = ctypes.c_int
    lib.lrkv_append_layers.argtypes = [P(Dims), i32, P(LayerStrides), vp, vp, i32, vp, vp, P(Cache), vp, vp]
    lib.lrkv_decode_layers.restype = ctypes.c_int
    lib.lrkv_decode_layers.argtypes = [P(Dims), i32, P(LayerStrides), vp, vp, vp, P(Cache), vp, i32, vp, i32, vp, vp,
                                       sz, vp, vp]
    lib.lrkv_decode_partials.restype = ctypes.c_int
    lib.lrkv_decode_partials.argtypes = [P(Dims), vp, vp, P(Cache), vp, i32, vp, i32, vp, vp, sz, vp, vp]
    lib.lrkv_decode_merge.restype = ctypes.c_int
    lib.lrkv_decode_merge.argtypes = [P(Dims), i32, vp, vp, i32, vp, vp, vp]
    lib.lrkv_decode_static_ws.restype = ctypes.c_int
    lib.lrkv_decode_static_ws.argtypes = [P(Dims), vp, vp, vp, P(Cache), vp, i32, vp, i32, vp, vp, vp]
    lib.lrkv_prefill_workspace_bytes.restype = sz
    lib.lrkv_prefill_workspace_bytes.argtypes = [P(Dims), i32, i32]
    lib.lrkv_prefill.restype = ctypes.c_int
    lib.lrkv_prefill.argtypes = [P(Dims), vp, vp, vp, P(Cache), vp, i32, vp, i32, i32, vp, vp, sz, vp, vp]
    lib.lrkv_prefill_fused.restype = ctypes.c_int
    lib.lrkv_prefill_fused.argtypes = [P(Dims), vp, vp, P(Cache), vp, i32, vp, i32, i32, vp, vp, vp]
    lib.lrkv_train_forward.restype = ctypes.c_int
    lib.lrkv_train_forward.argtypes = [P(Dims), vp, vp, vp, i32, vp, vp, vp, vp]
    lib.lrkv_train_workspace_bytes.restype = sz
    lib.lrkv_train_workspace_bytes.argtypes = [P(Dims), i32]
    lib.lrkv_train_backward.restype = ctypes.c_int
    lib.lrkv_train_backward.argtypes = [P(Dims), vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp, vp]
    lib.lrkv_mla_cache_block_bytes.restype = sz
    lib.lrkv_mla_cache_block_bytes.argtypes = [P(MlaDims)]
    lib.lrkv_mla_append.restype = ctypes.c_int
    lib.lrkv_mla_append.argtypes = [P(MlaDims), vp, vp, i32, vp, vp, vp, i32, vp, vp]
    lib.lrkv_mla_decode_workspace_bytes.restype = sz
    lib.lrkv_mla_decode_workspace_bytes.argtypes = [P(MlaDims), i32]
    lib.lrkv_mla_decode.restype = ctypes.c_int
    lib.lrkv_mla_decode.argtypes = [P(MlaDims), vp, vp, i32, vp, i32, vp, i32, vp, vp, sz, vp, vp]
    _lib = lib
    return lib


def make_dims(H: int, d_h: int, r: int, d: int, block_size: int = 64, softmax_scale: float = 0.0, d_rope: int = 0,
              rope_base: float = 0.0, num_splits: int = 0) -> Dims:
    return Dims(H, d_h, r, d, block_size, softmax_scale, d_rope, rope_base, num_splits)


def make_mla_dims(H: int, d: int, d_head: int = 128, d_c: int = 512, d_rope: int = 64, block_size: int = 64,
                  softmax_scale: float = 0.0, rope_base: float = 0.0) -> MlaDims:
    return MlaDims(H, d_c, d_rope, d_head, d, block_size, softmax_scale, rope_base)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != LRKV_OK:
        raise LrkvError(rc, where, load().lrkv_last_error().decode())


class PagedCache:
    """One layer's four cache pools (device tensors, bf16 bit patterns as int16/bfloat16)."""

    def __init__(self, sK, sV, zK, zV):
        self.sK, self.sV, self.zK, self.zV = sK, sV, zK, zV
        self.num_blocks = int(sK.shape[0])

    @classmethod
    def empty(cls, num_blocks: int, H: int, d_h: int, r: int, block_size: int = 64, device="cuda", d_rope: int = 0):
        mk = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)
        return cls(mk(num_blocks, block_size, d_h + d_rope), mk(num_blocks, block_size, d_h),
                   mk(num_blocks, block_size, H, r), mk(num_blocks, block_size, H, r))

    def struct(self) -> Cache:
        return Cache(_ptr(self.sK), _ptr(self.sV), _ptr(self.zK), _ptr(self.zV), self.num_blocks)

    def tensors(self):
        return self.sK, self.sV, self.zK, self.zV


def abi_version() -> int:
    return int(load().lrkv_abi_version())


def cache_block_bytes(dims: Dims) -> int:
    return int(load().lrkv_cache_block_bytes(ctypes.byref(dims)))


def decode_workspace_bytes(dims: Dims, batch: int) -> int:
    return int(load().lrkv_decode_workspace_bytes(ctypes.byref(dims), batch))


def prefill_workspace_bytes(dims: Dims, batch: int, Tq: int) -> int:
    return int(load().lrkv_prefill_workspace_bytes(ctypes.byref(dims), batch, Tq))


def lrkv_append(dims: Dims, X, W_catT, slot_mapping, cache: PagedCache, status=None, stream=None, positions=None):
    """Eqs. (4)-(5): write rows of X [n, d] into the cache at slot_mapping [n]; with a
    positional key (dims.d_rope > 0) its columns are rotated at positions [n] (int32)."""
    n = int(X.shape[0])
    c = cache.struct()
    rc = load().lrkv_append(ctypes.byref(dims), _ptr(X), _ptr(W_catT), n, _ptr(slot_mapping), _ptr(positions),
                            ctypes.byref(c), _ptr(status), _stream(stream))
    _check(rc, "lrkv_append")


def lrkv_decode(dims: Dims, q, BK, BV, cache: PagedCache, block_table, seq_lens, out, workspace, status=None,
                stream=None):
    """Factored decode (Eqs. (6)-(7)): q [B, H, d_h] -> out [B, H, d_h]."""
    B = int(q.shape[0])
    c = cache.struct()
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().lrkv_decode(ctypes.byref(dims), _ptr(q), _ptr(BK), _ptr(BV), ctypes.byref(c), _ptr(block_table),
                            int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(out), _ptr(workspace), ws_bytes,
                            _ptr(status), _stream(stream))
    _check(rc, "lrkv_decode")


def lrkv_decode_fused(dims: Dims, q, q_tilde, cache: PagedCache, block_table, seq_lens, out, workspace, status=None,
                      stream=None):
    """Decode with absorbed weights: q [B, H, d_h], q~ [B, H, r] -> out [B, H, d_h + r] = [o_s | o_z]."""
    B = int(q.shape[0])
    c = cache.struct()
    rc = load().lrkv_decode_fused(ctypes.byref(dims), _ptr(q), _ptr(q_tilde), ctypes.byref(c), _ptr(block_table),
                                  int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(out), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()), _ptr(status), _stream(stream))
    _check(rc, "lrkv_decode_fused")


def lrkv_decode_partials(dims: Dims, q, BK, cache: PagedCache, block_table, seq_lens, partials, workspace,
                         status=None, stream=None):
    """Decode partials over this cache's tokens: q [B, H, d_h] -> partials [B, H, d_h + r + 2] fp32
    (acc_s, acc_z, m, l)."""
    B = int(q.shape[0])
    c = cache.struct()
    rc = load().lrkv_decode_partials(ctypes.byref(dims), _ptr(q), _ptr(BK), ctypes.byref(c), _ptr(block_table),
                                     int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(partials), _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()), _ptr(status), _stream(stream))
    _check(rc, "lrkv_decode_partials")


def lrkv_decode_merge(dims: Dims, partials, BV, out, status=None, stream=None):
    """Merge partials [P, B, H, d_h + r + 2] of P parts of the sequences' tokens -> out [B, H, d_h]."""
    P, B = int(partials.shape[0]), int(partials.shape[1])
    rc = load().lrkv_decode_merge(ctypes.byref(dims), P, _ptr(partials), _ptr(BV), B, _ptr(out), _ptr(status),
                                  _stream(stream))
    _check(rc, "lrkv_decode_merge")


def lrkv_decode_static_ws(dims: Dims, q, BK, BV, cache: PagedCache, block_table, seq_lens, out, status=None,
                          stream=None):
    """lrkv_decode with the library's static scratch area instead of a caller
    workspace, for callers that must not allocate device memory (see lrkv.h)."""
    B = int(q.shape[0])
    c = cache.struct()
    rc = load().lrkv_decode_static_ws(ctypes.byref(dims), _ptr(q), _ptr(BK), _ptr(BV), ctypes.byref(c),
                                      _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(out),
                                      _ptr(status), _stream(stream))
    _check(rc, "lrkv_decode_static_ws")


class LayeredCache:
    """Several layers' cache pools as tensors with a leading layer dimension
    ([layers, num_blocks, block_size, ...]); layer l is at l * stride(0) elements."""

    def __init__(self, sK, sV, zK, zV):
        self.sK, self.sV, self.zK, self.zV = sK, sV, zK, zV
        self.num_layers = int(sK.shape[0])
        self.num_blocks = int(sK.shape[1])

    @classmethod
    def empty(cls, num_layers: int, num_blocks: int, H: int, d_h: int, r: int, block_size: int = 64, device="cuda",
              d_rope: int = 0):
        mk = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)
        return cls(mk(num_layers, num_blocks, block_size, d_h + d_rope), mk(num_layers, num_blocks, block_size, d_h),
                   mk(num_layers, num_blocks, block_size, H, r), mk(num_layers, num_blocks, block_size, H, r))

    def struct(self) -> Cache:
        return Cache(_ptr(self.sK), _ptr(self.sV), _ptr(self.zK), _ptr(self.zV), self.num_blocks)

    def tensors(self):
        return self.sK, self.sV, self.zK, self.zV

    def layer(self, l: int) -> PagedCache:
        return PagedCache(self.sK[l], self.sV[l], self.zK[l], self.zV[l])


def _layer_stride(t) -> int:
    return 0 if t is None else int(t.stride(0))


def lrkv_append_layers(dims: Dims, X, W_catT, slot_mapping, cache: LayeredCache, status=None, stream=None,
                       positions=None):
    """lrkv_append of the same slots in every layer: X [L, n, d], W_catT [L, N, d] -> the L layers' pools."""
    L, n = int(X.shape[0]), int(X.shape[1])
    st = LayerStrides(X=_layer_stride(X), W_catT=_layer_stride(W_catT), sK=_layer_stride(cache.sK),
                      sV=_layer_stride(cache.sV), zK=_layer_stride(cache.zK), zV=_layer_stride(cache.zV))
    c = cache.struct()
    rc = load().lrkv_append_layers(ctypes.byref(dims), L, ctypes.byref(st), _ptr(X), _ptr(W_catT), n,
                                   _ptr(slot_mapping), _ptr(positions), ctypes.byref(c), _ptr(status),
                                   _stream(stream))
    _check(rc, "lrkv_append_layers")


def lrkv_decode_layers(dims: Dims, q, BK, BV, cache: LayeredCache, block_table, seq_lens, out, workspace, status=None,
                       stream=None):
    """lrkv_decode of the same batch in every layer: q [L, B, H, d_h], B* [L, H, d_h, r] -> out [L, B, H, d_h];
    workspace of decode_workspace_bytes(dims, L * B) bytes."""
    L, B = int(q.shape[0]), int(q.shape[1])
    st = LayerStrides(q=_layer_stride(q), BK=_layer_stride(BK), BV=_layer_stride(BV), out=_layer_stride(out),
                      sK=_layer_stride(cache.sK), sV=_layer_stride(cache.sV), zK=_layer_stride(cache.zK),
                      zV=_layer_stride(cache.zV))
    c = cache.struct()
    rc = load().lrkv_decode_layers(ctypes.byref(dims), L, ctypes.byref(st), _ptr(q), _ptr(BK), _ptr(BV),
                                   ctypes.byref(c), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B,
                                   _ptr(out), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                   _ptr(status), _stream(stream))
    _check(rc, "lrkv_decode_layers")


def lrkv_prefill(dims: Dims, q, BK, BV, cache: PagedCache, block_table, q_start, out, workspace=None, status=None,
                 stream=None):
    """Causal chunked prefill: q [B, Tq, H, d_h] at positions q_start[b] + i -> out [B, Tq, H, d_h]."""
    B, Tq = int(q.shape[0]), int(q.shape[1])
    c = cache.struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().lrkv_prefill(ctypes.byref(dims), _ptr(q), _ptr(BK), _ptr(BV), ctypes.byref(c), _ptr(block_table),
                             int(block_table.shape[1]), _ptr(q_start), B, Tq, _ptr(out), _ptr(workspace), ws_bytes,
                             _ptr(status), _stream(stream))
    _check(rc, "lrkv_prefill")


def lrkv_prefill_fused(dims: Dims, q, q_tilde, cache: PagedCache, block_table, q_start, out, status=None, stream=None):
    """Causal prefill with absorbed weights: q [B, Tq, H, d_h], q~ [B, Tq, H, r] -> out [B, Tq, H, d_h + r]."""
    B, Tq = int(q.shape[0]), int(q.shape[1])
    c = cache.struct()
    rc = load().lrkv_prefill_fused(ctypes.byref(dims), _ptr(q), _ptr(q_tilde), ctypes.byref(c), _ptr(block_table),
                                   int(block_table.shape[1]), _ptr(q_start), B, Tq, _ptr(out), _ptr(status),
                                   _stream(stream))
    _check(rc, "lrkv_prefill_fused")


def train_workspace_bytes(dims: Dims, n_tok: int) -> int:
    return int(load().lrkv_train_workspace_bytes(ctypes.byref(dims), n_tok))


def lrkv_train_forward(dims: Dims, X, W_T, B, Y, K, status=None, stream=None):
    """Expanded projection: Y = X W_T^T = [S | R] ([n, d_h + H r]) and K = S + R_h B_h^T ([n, H, d_h])."""
    rc = load().lrkv_train_forward(ctypes.byref(dims), _ptr(X), _ptr(W_T), _ptr(B), int(X.shape[0]), _ptr(Y),
                                   _ptr(K), _ptr(status), _stream(stream))
    _check(rc, "lrkv_train_forward")


def lrkv_train_backward(dims: Dims, X, W_T, B, Y, dK, dX, dW_T, dB, workspace, status=None, stream=None):
    """Gradients through K_h = X (W_shared + U_h B_h^T): dX [n, d], dW_T [d_h + H r, d], dB [H, d_h, r]."""
    rc = load().lrkv_train_backward(ctypes.byref(dims), _ptr(X), _ptr(W_T), _ptr(B), _ptr(Y), _ptr(dK),
                                    int(X.shape[0]), _ptr(dX), _ptr(dW_T), _ptr(dB), _ptr(workspace),
                                    int(workspace.numel() * workspace.element_size()), _ptr(status),
                                    _stream(stream))
    _check(rc, "lrkv_train_backward")


def pack_side_t(Ws, U) -> torch.Tensor:
    """W_T [d_h + H r, d] of one projection from W_shared [d, d_h] and U [H, d, r]."""
    H, d, r = U.shape
    return torch.cat([Ws.t(), U.permute(0, 2, 1).reshape(H * r, d)], dim=0).contiguous()


def mla_cache_block_bytes(dims: MlaDims) -> int:
    return int(load().lrkv_mla_cache_block_bytes(ctypes.byref(dims)))


def mla_decode_workspace_bytes(dims: MlaDims, batch: int) -> int:
    return int(load().lrkv_mla_decode_workspace_bytes(ctypes.byref(dims), batch))


def lrkv_mla_append(dims: MlaDims, X, W_T, slot_mapping, positions, kv, status=None, stream=None):
    """MLA cache rows [c | RoPE(k^R)] of X [n, d] into kv [num_blocks, 64, d_c + d_rope] at slot_mapping [n]."""
    rc = load().lrkv_mla_append(ctypes.byref(dims), _ptr(X), _ptr(W_T), int(X.shape[0]), _ptr(slot_mapping),
                                _ptr(positions), _ptr(kv), int(kv.shape[0]), _ptr(status), _stream(stream))
    _check(rc, "lrkv_mla_append")


def lrkv_mla_decode(dims: MlaDims, q, kv, block_table, seq_lens, out, workspace, status=None, stream=None):
    """Absorbed MLA decode: q [B, H, d_c + d_rope] -> out [B, H, d_c]."""
    rc = load().lrkv_mla_decode(ctypes.byref(dims), _ptr(q), _ptr(kv), int(kv.shape[0]), _ptr(block_table),
                                int(block_table.shape[1]), _ptr(seq_lens), int(q.shape[0]), _ptr(out),
                                _ptr(workspace), int(workspace.numel() * workspace.element_size()), _ptr(status),
                                _stream(stream))
    _check(rc, "lrkv_mla_decode")


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned device byte buffer (torch's allocator aligns to 512 B)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def pack_wcat_t(WsK, WsV, UK, UV, WKR=None) -> torch.Tensor:
    """W_cat^T [N, d] from W_shared^{K,V} [d, d_h], U^{K,V} [H, d, r] and the optional positional-key
    projection W^KR [d, d_rope] (column order of lrkv_append)."""
    H, d, r = UK.shape
    parts = [WsK.t()] + ([] if WKR is None else [WKR.t()])
    return torch.cat(parts + [WsV.t(), UK.permute(0, 2, 1).reshape(H * r, d),
                              UV.permute(0, 2, 1).reshape(H * r, d)], dim=0).contiguous()
