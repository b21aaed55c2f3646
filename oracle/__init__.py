"""fp64 CPU oracle for LRKV attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (``compressed_kv_cache_lrkv_gb300``)
never imports it, and it imports nothing from the product path: the two meet
only in the seeded inputs of ``lrkv_synth``.

The arithmetic lives in ``lrkv_oracle.c`` (plain C, fp64, OpenMP over
independent (sequence, head) pairs); this module builds it with gcc and wraps
it with ctypes.  See the C file's header for the equations it follows
("Low-Rank Key Value Attention", Eqs. (2)-(7)).

Pins: every function here is pinned in ``tests/test_oracle_pins.py`` against
facts the pages or mathematics fix (softmax worked value, r=0 -> MQA,
W_shared=0 & B_h=permutation -> MHA through a library attention routine,
L=1 and equal-key special cases, head-permutation equivariance, integer-exact
append, causal-mask special cases, the positional key's rotation against the pages'
worked 90-degree example, absorbed MLA against library multi-query attention and
against its expanded form).  Planted-mistake builds
(``LRKV_ORACLE_MUTANT``) check that those pins catch a dropped term, a wrong
factor, a transposed factor, a wrong scale and an off-by-one causal mask.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lrkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()


def lib_path(mutant: int = 0) -> str:
    name = "liblrkv_oracle.so" if not mutant else f"liblrkv_oracle_m{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, OpenMP, no FP contraction); returns the .so path."""
    out = lib_path(mutant)
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            return out
        os.makedirs(_BUILD, exist_ok=True)
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               f"-DLRKV_ORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u8p_or_null = ctypes.c_void_p
_i32p_or_null = ctypes.c_void_p
_c_int = ctypes.c_int
_c_double = ctypes.c_double


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _want_ptr(want, B, H):
    if want is None:
        return None, None
    w = np.ascontiguousarray(want, dtype=np.uint8).reshape(B, H)
    return w, w.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one build of the oracle library."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self.lib = ctypes.CDLL(build(mutant))
        L = self.lib
        L.oracle_num_threads.restype = _c_int
        L.oracle_round_to_cache.argtypes = [_c_double]
        L.oracle_round_to_cache.restype = ctypes.c_uint16
        L.oracle_softmax.argtypes = [_c_int, _f64p, _f64p]
        L.oracle_attend.argtypes = [_c_int, _c_int, _f64p, _f64p, _f64p, _c_double, _f64p]
        L.oracle_append.argtypes = [_c_int] * 5 + [_u16p] * 5 + [_u16p] * 4
        L.oracle_decode_expanded.argtypes = ([_c_int] * 6 + [_i32p] + [_u16p] * 8 +
                                             [_c_double, _u8p_or_null, _f64p])
        L.oracle_decode_expanded.restype = _c_int
        L.oracle_decode_cache.argtypes = ([_c_int] * 6 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                          [_u16p] * 3 + [_c_double, _u8p_or_null, _f64p])
        L.oracle_decode_cache.restype = _c_int
        L.oracle_decode_fused_rope.argtypes = ([_c_int] * 7 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                               [_u16p, _u16p, _c_double, _u8p_or_null, _f64p])
        L.oracle_decode_fused_rope.restype = _c_int
        L.oracle_decode_cache_rope.argtypes = ([_c_int] * 7 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                               [_u16p] * 3 + [_c_double, _u8p_or_null, _f64p])
        L.oracle_decode_cache_rope.restype = _c_int
        L.oracle_prefill_cache_rope.argtypes = ([_c_int] * 8 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                                [_u16p] * 3 + [_c_double, _u8p_or_null, _f64p])
        L.oracle_prefill_cache_rope.restype = _c_int
        L.oracle_append_rope.argtypes = ([_c_int] * 6 + [_c_double] + [_u16p] * 6 + [_i32p_or_null] +
                                         [_u16p] * 4)
        L.oracle_prefill_expanded.argtypes = ([_c_int] * 7 + [_i32p] + [_u16p] * 8 +
                                              [_c_double, _u8p_or_null, _f64p])
        L.oracle_prefill_expanded.restype = _c_int
        L.oracle_prefill_cache.argtypes = ([_c_int] * 7 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                           [_u16p] * 3 + [_c_double, _u8p_or_null, _f64p])
        L.oracle_prefill_cache.restype = _c_int
        L.oracle_prefill_fused_rope.argtypes = ([_c_int] * 8 + [_u16p] * 4 + [_i32p, _c_int, _i32p] +
                                                [_u16p, _u16p, _c_double, _u8p_or_null, _f64p])
        L.oracle_prefill_fused_rope.restype = _c_int
        L.oracle_mla_decode.argtypes = ([_c_int] * 7 + [_u16p, _i32p, _c_int, _i32p, _u16p] +
                                        [_c_double, _u8p_or_null, _f64p])
        L.oracle_mla_decode.restype = _c_int
        L.oracle_mla_decode_expanded.argtypes = ([_c_int] * 6 + [_i32p] + [_u16p] * 5 + [_c_double, _f64p])
        L.oracle_mla_decode_expanded.restype = _c_int
        L.oracle_train_forward.argtypes = [_c_int] * 5 + [_u16p] * 4 + [_f64p]
        L.oracle_train_backward.argtypes = [_c_int] * 5 + [_u16p] * 5 + [_f64p] * 4

    # -- small pieces ---------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def round_to_cache(self, v: float) -> int:
        return int(self.lib.oracle_round_to_cache(float(v)))

    def softmax(self, logits) -> np.ndarray:
        x = np.ascontiguousarray(logits, dtype=np.float64)
        p = np.empty_like(x)
        self.lib.oracle_softmax(len(x), x, p)
        return p

    def attend(self, q, K, V, scale: float = 0.0) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.float64)
        K = np.ascontiguousarray(K, dtype=np.float64)
        V = np.ascontiguousarray(V, dtype=np.float64)
        d_h = q.shape[0]
        out = np.empty(d_h, dtype=np.float64)
        s = scale if scale != 0.0 else 1.0 / np.sqrt(d_h)
        self.lib.oracle_attend(K.shape[0], d_h, q, K, V, s, out)
        return out

    # -- Eqs. (4)-(5) ---------------------------------------------------------
    def append(self, X, WsK, WsV, UK, UV, WKR=None, positions=None, rope_base=10000.0):
        """Dense cache rows for X [n, d]: (sK [n, d_h + d_rope], sV [n, d_h], zK [n,H,r], zV) as
        bf16 bits.  With WKR [d, d_rope], sK carries the shared positional key rotated at
        positions[t] after its d_h content entries."""
        X = _u16(X)
        n, d = X.shape
        d_h = WsK.shape[1]
        H, _, r = UK.shape
        d_rope = 0 if WKR is None else WKR.shape[1]
        sK = np.empty((n, d_h + d_rope), np.uint16)
        sV = np.empty((n, d_h), np.uint16)
        zK = np.empty((n, H, r), np.uint16)
        zV = np.empty((n, H, r), np.uint16)
        wkr = _u16(WKR) if d_rope else _u16(np.zeros((1, 1), np.uint16))
        pos = _i32(positions) if d_rope else None
        self.lib.oracle_append_rope(n, d, d_h, H, r, d_rope, float(rope_base), X, _u16(WsK), wkr, _u16(WsV),
                                    _u16(UK), _u16(UV), None if pos is None else pos.ctypes.data_as(ctypes.c_void_p),
                                    sK, sV, zK, zV)
        return sK, sV, zK, zV

    # -- decode -----------------------------------------------------------------
    def decode_expanded(self, X, ctx_len, WsK, WsV, UK, UV, BK, BV, q, scale=0.0, want=None):
        """E1 decode.  X [B, Lmax, d]; q [B, H, d_h]; returns out [B, H, d_h] fp64."""
        X = _u16(X)
        B, Lmax, d = X.shape
        H, d_h, r = BK.shape
        out = np.zeros((B, H, d_h), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_decode_expanded(B, H, d_h, r, d, Lmax, _i32(ctx_len), X, _u16(WsK),
                                             _u16(WsV), _u16(UK), _u16(UV), _u16(BK), _u16(BV),
                                             _u16(q), float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_decode_expanded: bad argument")
        return out

    def decode_cache(self, cache, block_table, seq_lens, BK, BV, q, scale=0.0, want=None, bs=64):
        """E2 decode from pools cache=(sK, sV, zK, zV), shaped [nb, bs, d_h + d_rope], [nb, bs, d_h],
        [nb, bs, H, r]; q [B, H, d_h + d_rope] (d_rope > 0: shared positional key after s^K)."""
        sK, sV, zK, zV = (_u16(c) for c in cache)
        H, d_h, r = BK.shape
        d_rope = sK.shape[-1] - d_h
        nb = sK.shape[0]
        bt = _i32(block_table)
        B, max_pages = bt.shape
        out = np.zeros((B, H, d_h), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_decode_cache_rope(B, H, d_h, r, d_rope, bs, nb, sK, sV, zK, zV, bt, max_pages,
                                               _i32(seq_lens), _u16(BK), _u16(BV), _u16(q),
                                               float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_decode_cache: bad block id or length")
        return out

    def decode_fused(self, cache, block_table, seq_lens, q, q_tilde, scale=0.0, want=None, bs=64):
        """Decode with absorbed weights: q [B, H, d_h], q~ [B, H, r] -> [B, H, d_h + r] = [o_s | o_z]."""
        sK, sV, zK, zV = (_u16(c) for c in cache)
        B, H = q.shape[:2]
        d_h = sV.shape[-1]
        d_rope = sK.shape[-1] - d_h
        r = q_tilde.shape[2]
        nb = sK.shape[0]
        bt = _i32(block_table)
        max_pages = bt.shape[1]
        out = np.zeros((B, H, d_h + r), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_decode_fused_rope(B, H, d_h, r, d_rope, bs, nb, sK, sV, zK, zV, bt, max_pages,
                                               _i32(seq_lens), _u16(q), _u16(q_tilde), float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_decode_fused: bad block id or length")
        return out

    # -- MLA (absorbed and expanded) ----------------------------------------------
    def mla_append(self, X, WDKV, WKR, positions, rope_base=10000.0):
        """MLA cache rows [c | k^R] for X [n, d]: c = X W^DKV (d_c), k^R = RoPE(X W^KR, pos) (d_rope),
        each an fp64 sum rounded to fp32 then bf16.  Returns [n, d_c + d_rope] bf16 bits."""
        X = _u16(X)
        n, d = X.shape
        d_c, d_rope = WDKV.shape[1], WKR.shape[1]
        z1 = np.zeros((1, d, 0), np.uint16)
        sK, _, _, _ = self.append(X, WDKV, np.zeros((d, d_c), np.uint16), z1, z1, WKR=WKR, positions=positions,
                                  rope_base=rope_base)
        return sK

    def mla_decode(self, kv, block_table, seq_lens, q, d_rope, d_head, scale=0.0, want=None, bs=64):
        """Absorbed MLA decode: kv [nb, bs, d_c + d_rope] (rows [c | k^R]), q [B, H, d_c + d_rope]
        ([q~ | q^R]) -> o [B, H, d_c] = sum_t p_t c_t; scale 1/sqrt(d_head + d_rope) by default."""
        kv = _u16(kv)
        B, H, dk = q.shape
        d_c = dk - d_rope
        bt = _i32(block_table)
        out = np.zeros((B, H, d_c), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_mla_decode(B, H, d_c, d_rope, d_head, bs, kv.shape[0], kv, bt, bt.shape[1],
                                        _i32(seq_lens), _u16(q), float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_mla_decode: bad block id or length")
        return out

    def mla_decode_expanded(self, rows, ctx_len, qC, qR, WUK, WUV, scale=0.0):
        """MLA decode with per-head keys [c W^UK_h | k^R] and values c W^UV_h formed explicitly:
        rows [B, Lmax, d_c + d_rope], qC [B, H, d_head], qR [B, H, d_rope], WUK, WUV [H, d_c, d_head]
        -> [B, H, d_head]."""
        rows = _u16(rows)
        B, Lmax, dk = rows.shape
        H, d_c, d_head = WUK.shape
        d_rope = dk - d_c
        out = np.zeros((B, H, d_head), np.float64)
        rc = self.lib.oracle_mla_decode_expanded(B, H, d_c, d_rope, d_head, Lmax, _i32(ctx_len), rows, _u16(qC),
                                                 _u16(qR), _u16(WUK), _u16(WUV), float(scale), out)
        if rc != 0:
            raise ValueError("oracle_mla_decode_expanded: bad argument")
        return out

    # -- training: expanded projections ----------------------------------------------
    def train_forward(self, X, Ws, U, B):
        """K_h = X (W_s + U_h B_h^T) for all heads: X [n, d], Ws [d, d_h], U [H, d, r], B [H, d_h, r]
        -> [n, H, d_h] fp64."""
        X = _u16(X)
        n, d = X.shape
        H, d_h, r = B.shape
        K = np.zeros((n, H, d_h), np.float64)
        self.lib.oracle_train_forward(n, d, d_h, H, r, X, _u16(Ws), _u16(U), _u16(B), K)
        return K

    def train_backward(self, X, Ws, U, B, dK):
        """Gradients of sum(dK * K) w.r.t. X, W_s, U, B (the chain rule through K_h = X W_h):
        returns dX [n, d], dWs [d, d_h], dU [H, d, r], dB [H, d_h, r], fp64."""
        X = _u16(X)
        n, d = X.shape
        H, d_h, r = B.shape
        dX = np.zeros((n, d)); dWs = np.zeros((d, d_h)); dU = np.zeros((H, d, r)); dB = np.zeros((H, d_h, r))
        self.lib.oracle_train_backward(n, d, d_h, H, r, X, _u16(Ws), _u16(U), _u16(B), _u16(dK), dX, dWs, dU, dB)
        return dX, dWs, dU, dB

    # -- prefill ----------------------------------------------------------------
    def prefill_expanded(self, X, q_start, WsK, WsV, UK, UV, BK, BV, q, scale=0.0, want=None):
        """E1 causal prefill.  q [B, Tq, H, d_h]; X [B, Lmax, d]; returns [B, Tq, H, d_h]."""
        X = _u16(X)
        B, Lmax, d = X.shape
        _, Tq, H, d_h = q.shape
        r = BK.shape[2]
        out = np.zeros((B, Tq, H, d_h), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_prefill_expanded(B, Tq, H, d_h, r, d, Lmax, _i32(q_start), X,
                                              _u16(WsK), _u16(WsV), _u16(UK), _u16(UV), _u16(BK),
                                              _u16(BV), _u16(q), float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_prefill_expanded: bad argument")
        return out

    def prefill_cache(self, cache, block_table, q_start, BK, BV, q, scale=0.0, want=None, bs=64):
        """E2 causal prefill from the paged pools; q [B, Tq, H, d_h]."""
        sK, sV, zK, zV = (_u16(c) for c in cache)
        _, Tq, H = q.shape[:3]
        d_h, r = BK.shape[1], BK.shape[2]
        d_rope = sK.shape[-1] - d_h
        nb = sK.shape[0]
        bt = _i32(block_table)
        B, max_pages = bt.shape
        out = np.zeros((B, Tq, H, d_h), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_prefill_cache_rope(B, Tq, H, d_h, r, d_rope, bs, nb, sK, sV, zK, zV, bt, max_pages,
                                                _i32(q_start), _u16(BK), _u16(BV), _u16(q), float(scale),
                                                wp, out)
        if rc != 0:
            raise ValueError("oracle_prefill_cache: bad block id or length")
        return out

    def prefill_fused(self, cache, block_table, q_start, q, q_tilde, scale=0.0, want=None, bs=64):
        """E2 causal prefill with absorbed weights: q [B, Tq, H, d_h + d_rope], q~ [B, Tq, H, r]
        -> [B, Tq, H, d_h + r] = [o_s | o_z]."""
        sK, sV, zK, zV = (_u16(c) for c in cache)
        _, Tq, H = q.shape[:3]
        d_h = sV.shape[-1]
        d_rope = sK.shape[-1] - d_h
        r = q_tilde.shape[3]
        nb = sK.shape[0]
        bt = _i32(block_table)
        B, max_pages = bt.shape
        out = np.zeros((B, Tq, H, d_h + r), np.float64)
        w, wp = _want_ptr(want, B, H)
        rc = self.lib.oracle_prefill_fused_rope(B, Tq, H, d_h, r, d_rope, bs, nb, sK, sV, zK, zV, bt, max_pages,
                                                _i32(q_start), _u16(q), _u16(q_tilde), float(scale), wp, out)
        if rc != 0:
            raise ValueError("oracle_prefill_fused: bad block id or length")
        return out


_default = None


def get(mutant: int = 0) -> Oracle:
    """The oracle (built on first use)."""
    global _default
    if mutant:
        return Oracle(mutant)
    if _default is None:
        _default = Oracle(0)
    return _default


def scatter_rows(pools, slots, rows):
    """Place dense cache rows (sK, sV, zK, zV per token) at physical slots of the pools.

    pools: (sK [nb,bs,d_h], sV, zK [nb,bs,H,r], zV); slots: [n] int; rows: 4 arrays [n, ...].
    """
    for pool, row in zip(pools, rows):
        flat = pool.reshape((-1,) + pool.shape[2:])
        flat[np.asarray(slots, dtype=np.int64)] = row
