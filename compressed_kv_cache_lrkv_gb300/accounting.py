"""Cache, parameter, byte and flop accounting for LRKV attention.

Formulas (source: "Low-Rank Key Value Attention" slide deck):
  * cache elements per token per layer, LRKV: 2(d_h + H r)
    (frame "Can heads share storage while keeping distinct K/V features?", table);
  * cache ratio to MHA, Eq. (9): rho = 2L(d_h + H r) / (2 L H d_h) = 1/H + r/d_h
    (frame "The rank directly sets the theoretical cache budget");
  * K/V parameter counts, Eq. (10): P_LRKV = 2 d d_h + 2 H r (d + d_h), P_MHA = 2 H d d_h
    (frame "Smaller storage trades bandwidth for extra arithmetic").
MHA/GQA/MQA/MLA per-token counts follow "Embeddings II: MLA & Architectural
Choices" (Chapter 1 "Counting the cache, one token at a time"; Chapter 4
"KV Cache Calculator").
"""
from __future__ import annotations

from typing import Iterable

BF16_BYTES = 2


def lrkv_cache_elements(H: int, d_h: int, r: int, d_rope: int = 0) -> int:
    """Elements one token adds to one layer's LRKV cache: s^K, s^V (d_h each) + z^K_h, z^V_h (r each, per head),
    plus the decoupled positional key k^R (d_rope, shared by all heads) when there is one."""
    return 2 * (d_h + H * r) + d_rope


def mha_cache_elements(H: int, d_h: int, layers: int = 1) -> int:
    return 2 * H * d_h * layers


def gqa_cache_elements(n_groups: int, d_h: int, layers: int = 1) -> int:
    return 2 * n_groups * d_h * layers


def mqa_cache_elements(d_h: int, layers: int = 1) -> int:
    return 2 * d_h * layers


def mla_cache_elements(d_c: int, d_h_rope: int, layers: int = 1) -> int:
    return (d_c + d_h_rope) * layers


def cache_ratio(H: int, d_h: int, r: int) -> float:
    """LRKV / MHA cache size, Eq. (9): 1/H + r/d_h."""
    return lrkv_cache_elements(H, d_h, r) / mha_cache_elements(H, d_h)


def kv_params_lrkv(d: int, d_h: int, H: int, r: int) -> int:
    """K/V projection parameters of one LRKV layer, Eq. (10)."""
    return 2 * d * d_h + 2 * H * r * (d + d_h)


def kv_params_mha(d: int, d_h: int, H: int) -> int:
    return 2 * H * d * d_h


def page_bytes(H: int, d_h: int, r: int, block_size: int = 64, d_rope: int = 0) -> int:
    """Bytes of one cache page (all four arrays, bf16)."""
    return block_size * lrkv_cache_elements(H, d_h, r, d_rope) * BF16_BYTES


def decode_algorithmic_bytes(H: int, d_h: int, r: int, seq_lens: Iterable[int], layers: int = 1,
                             d_rope: int = 0) -> int:
    """Bytes one decode step must move: every cached token's compressed row, the
    two factor tensors B^K, B^V, the query [q | q^R] in and the output out (all bf16)."""
    seq_lens = list(int(x) for x in seq_lens)
    B = len(seq_lens)
    per_layer = (sum(seq_lens) * lrkv_cache_elements(H, d_h, r, d_rope) * BF16_BYTES
                 + 2 * H * d_h * r * BF16_BYTES + B * H * (2 * d_h + d_rope) * BF16_BYTES)
    return per_layer * layers


def decode_fused_algorithmic_bytes(H: int, d_h: int, r: int, seq_lens: Iterable[int], layers: int = 1,
                                   d_rope: int = 0) -> int:
    """Bytes of one decode step with both absorptions in the caller's weights: every cached
    token's compressed row, the query [q | q^R | q~] in and [o_s | o_z] out (all bf16)."""
    seq_lens = list(int(x) for x in seq_lens)
    B = len(seq_lens)
    per_layer = (sum(seq_lens) * lrkv_cache_elements(H, d_h, r, d_rope) * BF16_BYTES
                 + B * H * (2 * (d_h + r) + d_rope) * BF16_BYTES)
    return per_layer * layers


def decode_flops(H: int, d_h: int, r: int, seq_lens: Iterable[int], layers: int = 1) -> int:
    """Multiply-adds x 2 of factored decode: per cached token 4H(d_h + r); per sequence
    4 H d_h r for q~ = q B^K and the B^V up-projection."""
    seq_lens = list(int(x) for x in seq_lens)
    return layers * (4 * H * (d_h + r) * sum(seq_lens) + 4 * H * d_h * r * len(seq_lens))


def append_flops(n_tok: int, d: int, H: int, d_h: int, r: int) -> int:
    """2 n d N with N = 2(d_h + H r) output columns."""
    return 2 * n_tok * d * lrkv_cache_elements(H, d_h, r)


def append_algorithmic_bytes(n_tok: int, d: int, H: int, d_h: int, r: int, d_rope: int = 0) -> int:
    """X in, W_cat in, cache rows out (bf16)."""
    N = lrkv_cache_elements(H, d_h, r, d_rope)
    return BF16_BYTES * (n_tok * d + d * N + n_tok * N)


def prefill_flops(B: int, T: int, H: int, d_h: int, r: int, q_start: int = 0, d_rope: int = 0,
                  absorbed: bool = False) -> int:
    """Causal attention flops for queries at positions [q_start, q_start + T): per visible
    (query, key) pair 2 (d_h + d_rope + r) for the logit and 2 (d_h + r) for the value side,
    i.e. 4 (d_h + r) + 2 d_rope, times H B sum_i (q_start + i + 1); plus the q~ absorption and
    the B^V up-projection, 4 B T H d_h r, unless the weights are absorbed by the caller."""
    pairs = T * q_start + T * (T + 1) // 2
    proj = 0 if absorbed else 4 * B * T * H * d_h * r
    return (4 * (d_h + r) + 2 * d_rope) * H * B * pairs + proj


def mla_decode_algorithmic_bytes(H: int, d_c: int, d_rope: int, seq_lens: Iterable[int], layers: int = 1) -> int:
    """Bytes of one absorbed MLA decode step: every cached row [c | k^R], the query [q~ | q^R] in and
    o (width d_c) out, all bf16."""
    seq_lens = list(int(x) for x in seq_lens)
    B = len(seq_lens)
    per_layer = (sum(seq_lens) * (d_c + d_rope) + B * H * (2 * d_c + d_rope)) * BF16_BYTES
    return per_layer * layers


def mla_decode_flops(H: int, d_c: int, d_rope: int, seq_lens: Iterable[int], layers: int = 1) -> int:
    """Multiply-adds x 2 of absorbed MLA decode: per cached token and head (d_c + d_rope) for the
    logit and d_c for the value sum."""
    return layers * 2 * H * (2 * d_c + d_rope) * sum(int(x) for x in seq_lens)


def mla_append_algorithmic_bytes(n_tok: int, d: int, d_c: int, d_rope: int) -> int:
    """X in, [W^DKV | W^KR] in, cache rows out (bf16)."""
    N = d_c + d_rope
    return BF16_BYTES * (n_tok * d + d * N + n_tok * N)


def train_flops(n_tok: int, d: int, H: int, d_h: int, r: int) -> tuple[int, int]:
    """Multiply-adds x 2 of the expanded projection K_h = X (W_shared + U_h B_h^T) through the
    factored route: forward X W_T^T (N = d_h + H r) and the per-head expansion R_h B_h^T; backward
    dR_h = dK_h B_h, dB_h = dK_h^T R_h, dW_T = [G | dR]^T X and dX = [G | dR] W_T.
    Returns (forward, backward)."""
    N = d_h + H * r
    head = 2 * n_tok * H * d_h * r
    fwd = 2 * n_tok * d * N + head
    bwd = 2 * head + 2 * (2 * n_tok * d * N)
    return fwd, bwd
