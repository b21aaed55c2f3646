"""Seeded synthetic inputs for LRKV attention (shared by the oracle side and the CUDA side).

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the fp64 oracle and the CUDA library receive the
exact same bf16 bit patterns from here, so a parity test compares two
implementations on identical inputs.

Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; finaliser constants as published
with Vigna's reference splitmix64.c).  Element ``i`` of stream ``s`` under seed
``k`` is ``mix(base(k, s) + (i + 1) * GOLDEN)``, so any chunk can be produced
independently and in parallel.  Uniforms take the top 53 bits, Gaussians come
from the Box-Muller transform on consecutive pairs, and values are rounded to
bf16 with round-to-nearest-even after an fp64 -> fp32 rounding.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .workloads import WORKLOADS, Workload  # noqa: F401

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place on a uint64 array (wrap-around arithmetic)."""
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _mix_scalar(x: int) -> int:
    return int(_mix(np.array([x & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def _stream_base(seed: int, stream: str) -> np.uint64:
    # FNV-1a over the stream name gives a stable integer id per tensor.
    h = 0xCBF29CE484222325
    for ch in stream.encode():
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return np.uint64(_mix_scalar(_mix_scalar(seed + 0x51ED) ^ h))


def _raw(base: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        idx *= GOLDEN
        idx += base
    return _mix(idx)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _parallel_fill(n: int, fn, out: np.ndarray) -> np.ndarray:
    """Run ``fn(start, stop) -> array`` over chunks and write into ``out``."""
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        if n:
            out[:] = fn(0, n)
        return out

    def work(s):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(s, e)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, starts))
    return out


def uniform(seed: int, stream: str, n: int) -> np.ndarray:
    """n uniforms in the open interval (0, 1), fp64."""
    base = _stream_base(seed, stream)

    def fn(s, e):
        bits = _raw(base, s, e - s) >> np.uint64(11)
        return (bits.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)

    return _parallel_fill(n, fn, np.empty(n, dtype=np.float64))


def _gauss_pairs(base: np.uint64, s: int, e: int, scale: float) -> np.ndarray:
    """Gaussians for pair indices [s, e): 2*(e-s) fp64 values (Box-Muller)."""
    bits = _raw(base, 2 * s, 2 * (e - s)) >> np.uint64(11)
    u = (bits.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1)) * scale
    ang = (2.0 * np.pi) * u2
    out = np.empty(2 * (e - s), dtype=np.float64)
    out[0::2] = rad * np.cos(ang)
    out[1::2] = rad * np.sin(ang)
    return out


def _pairwise(n: int, fn, dtype) -> np.ndarray:
    """Evaluate ``fn(s, e)`` (2*(e-s) values for pair range [s, e)) over all pairs."""
    n2 = (n + 1) // 2
    buf = np.empty(2 * n2, dtype=dtype)
    starts = list(range(0, n2, _CHUNK))

    def work(s):
        e = min(n2, s + _CHUNK)
        buf[2 * s:2 * e] = fn(s, e)

    if len(starts) <= 1:
        if n2:
            work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    return buf[:n]


def gaussian(seed: int, stream: str, n: int, scale: float = 1.0) -> np.ndarray:
    """n draws of scale * N(0, 1) in fp64."""
    base = _stream_base(seed, stream)
    return _pairwise(n, lambda s, e: _gauss_pairs(base, s, e, scale), np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    r = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gaussian_bf16(seed: int, stream: str, shape, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of scale * N(0, 1) (fp64 -> fp32 -> bf16), with the given shape."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if len(shape) else 1
    base = _stream_base(seed, stream)
    fn = lambda s, e: f32_to_bf16_bits(_gauss_pairs(base, s, e, scale).astype(np.float32))
    return _pairwise(n, fn, np.uint16).reshape(shape)


def int_grid_bf16(seed: int, stream: str, shape, lo: int, hi: int, exp2: int = 0) -> np.ndarray:
    """bf16 bits of k * 2**exp2 with k uniform on the integers [lo, hi].

    Products and sums of such values are exact in fp32 as long as partial sums
    stay below 2**24 units, which makes an exactly-rounded GEMM reference
    unambiguous (every summation order gives the same fp32 value).
    """
    n = int(np.prod(shape))
    u = uniform(seed, stream, n)
    k = lo + np.floor(u * (hi - lo + 1)).astype(np.int64)
    k = np.minimum(k, hi)
    v = (k.astype(np.float64) * (2.0 ** exp2)).astype(np.float32)
    return f32_to_bf16_bits(v).reshape(shape)


def uniform_int(seed: int, stream: str, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on the closed interval [lo, hi]."""
    u = uniform(seed, stream, n)
    k = lo + np.floor(u * (hi - lo + 1)).astype(np.int64)
    return np.minimum(k, hi)


def permutation(seed: int, stream: str, n: int) -> np.ndarray:
    """A seeded random permutation of range(n) (argsort of random 64-bit keys)."""
    keys = _raw(_stream_base(seed, stream), 0, n)
    return np.argsort(keys, kind="stable").astype(np.int64)


# ----------------------------------------------------------------------------
# Paged-cache page tables
# ----------------------------------------------------------------------------

@dataclass
class PageTable:
    block_table: np.ndarray  # [B, max_pages] int32, unused entries -1
    seq_lens: np.ndarray     # [B] int32
    num_blocks: int
    block_size: int = 64
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def slot(self, b: int, t: int) -> int:
        """Physical slot (block * block_size + offset) of token t of sequence b."""
        return int(self.block_table[b, t // self.block_size]) * self.block_size + t % self.block_size


def page_table(seed: int, seq_lens, block_size: int = 64, capacity: int | None = None,
               spare_blocks: int = 0) -> PageTable:
    """Block table whose physical pages are a seeded permutation of the pool.

    ``capacity`` (tokens per sequence the table can address) sets max_pages;
    by default it is the longest sequence.  ``spare_blocks`` adds pool pages that
    no sequence uses.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(seq_lens)
    cap = int(capacity if capacity is not None else max(1, int(seq_lens.max())))
    max_pages = (cap + block_size - 1) // block_size
    pages = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    total = sum(pages) + spare_blocks
    perm = permutation(seed, "block_perm", max(total, 1))
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]
    return PageTable(bt, seq_lens.astype(np.int32), max(total, 1), block_size)


def slots_for(pt: PageTable, b: int, t0: int, t1: int) -> np.ndarray:
    """Physical slots of tokens [t0, t1) of sequence b."""
    t = np.arange(t0, t1)
    return (pt.block_table[b, t // pt.block_size].astype(np.int64) * pt.block_size + t % pt.block_size).astype(np.int32)
