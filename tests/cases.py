"""Seeded test cases (input layout only; values from lrkv_synth)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import lrkv_synth as S


@dataclass
class Weights:
    WsK: np.ndarray  # [d, d_h]
    WsV: np.ndarray
    UK: np.ndarray   # [H, d, r]
    UV: np.ndarray
    BK: np.ndarray   # [H, d_h, r]
    BV: np.ndarray

    @property
    def dims(self):
        H, d, r = self.UK.shape
        return H, self.WsK.shape[1], r, d


def weights(seed: int, d: int, d_h: int, H: int, r: int, b_scale: float = 1.0, tag: str = "") -> Weights:
    """bf16 weights ~ N(0, 1/fan_in): fan_in(W_shared) = fan_in(U_h) = d, fan_in(B_h) = r."""
    g = lambda name, shape, fan: S.gaussian_bf16(seed, tag + name, shape, 1.0 / np.sqrt(max(fan, 1)))
    return Weights(
        WsK=g("WsK", (d, d_h), d), WsV=g("WsV", (d, d_h), d),
        UK=g("UK", (H, d, r), d), UV=g("UV", (H, d, r), d),
        BK=S.gaussian_bf16(seed, tag + "BK", (H, d_h, r), b_scale / np.sqrt(max(r, 1))),
        BV=S.gaussian_bf16(seed, tag + "BV", (H, d_h, r), b_scale / np.sqrt(max(r, 1))),
    )


def pack_wcat_t(w: Weights, WKR: np.ndarray | None = None) -> np.ndarray:
    """Concatenated projection in the library's layout: W_catT [N, d] (row c = weights of output column c),
    columns ordered [W_shared^K | W^KR | W_shared^V | U_1^K .. U_H^K | U_1^V .. U_H^V] (W^KR [d, d_rope],
    the positional-key projection, only when given)."""
    H, d, r = w.UK.shape
    cols = [w.WsK.T] + ([] if WKR is None else [WKR.T]) + [w.WsV.T,
            np.transpose(w.UK, (0, 2, 1)).reshape(H * r, d),
            np.transpose(w.UV, (0, 2, 1)).reshape(H * r, d)]
    return np.ascontiguousarray(np.concatenate(cols, axis=0))


def empty_pools(num_blocks: int, H: int, d_h: int, r: int, bs: int = 64, fill: int = 0, d_rope: int = 0):
    return (np.full((num_blocks, bs, d_h + d_rope), fill, np.uint16), np.full((num_blocks, bs, d_h), fill, np.uint16),
            np.full((num_blocks, bs, H, r), fill, np.uint16), np.full((num_blocks, bs, H, r), fill, np.uint16))


def random_pools(seed: int, num_blocks: int, H: int, d_h: int, r: int, bs: int = 64, d_rope: int = 0):
    """Cache pools filled with bf16(N(0,1)) -- the distribution of x W with x ~ N(0,1), W ~ N(0, 1/d); a
    rotation keeps that distribution, so the positional key columns (d_rope > 0) are drawn the same way."""
    return (S.gaussian_bf16(seed, "pool_sK", (num_blocks, bs, d_h + d_rope)),
            S.gaussian_bf16(seed, "pool_sV", (num_blocks, bs, d_h)),
            S.gaussian_bf16(seed, "pool_zK", (num_blocks, bs, H, r)),
            S.gaussian_bf16(seed, "pool_zV", (num_blocks, bs, H, r)))


def f64(bits) -> np.ndarray:
    return S.bf16_bits_to_f32(bits).astype(np.float64)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
