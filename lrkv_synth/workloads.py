"""The synthetic workloads (shapes only; no arithmetic of the method).

Shapes follow the pages' models: the 12-layer d=512, 8-head, d_h=64 backbone of
the KVPath experiments page; DeepSeek-V2's 128 heads x 128 of the MLA lesson;
the 6.3B LRKV scale (H=32, d_h=128) of the LRKV slides, which is also the 32 x 128
speed-benchmark shape of the Key-Value Means slides.  In every workload d = H * d_h,
as the LRKV slides assume (frame "LRKV constrains differences between heads").
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    key: str
    description: str
    B: int            # sequences
    L: int            # cached tokens per sequence (upper bound when ragged)
    H: int            # query heads
    d_h: int          # head width
    r: int            # residual rank
    d: int            # hidden size
    layers: int = 1
    L_min: int | None = None   # ragged lengths uniform on [L_min, L]
    chunk: int | None = None   # prefill query chunk
    seed: int = 0
    block_size: int = 64
    d_c: int = 0               # multi-head latent attention: latent width (0: an LRKV workload)
    d_rope: int = 0            # decoupled positional key width

    @property
    def ragged(self) -> bool:
        return self.L_min is not None

    @property
    def N(self) -> int:
        """Append GEMM output width = cache elements per token per layer, 2(d_h + H r)."""
        return 2 * (self.d_h + self.H * self.r)


WORKLOADS = {
    "small": Workload("small", "single layer, batch 1, H=8, d_h=64, d=512, r=8, 256 cached tokens, one decode query",
                      B=1, L=256, H=8, d_h=64, r=8, d=512, seed=0),
    "backbone12": Workload("backbone12", "12-layer backbone d=512, H=8, d_h=64, r=16, batch 16, 2048 cached tokens, one decode step",
                           B=16, L=2048, H=8, d_h=64, r=16, d=512, layers=12, seed=1),
    "dsv2": Workload("dsv2", "DeepSeek-V2-scale layer d=16384, H=128, d_h=128, r=16, batch 8, 8192 cached tokens, decode, 64-token pages",
                     B=8, L=8192, H=128, d_h=128, r=16, d=16384, seed=2),
    "longctx": Workload("longctx", "long-context decode d=4096, H=32, d_h=128, r=32, batch 4, ragged lengths uniform in [16384, 32768]",
                        B=4, L=32768, L_min=16384, H=32, d_h=128, r=32, d=4096, seed=3),
    "mla": Workload("mla", "multi-head latent attention decode at DeepSeek-V2's attention shape (H=128, d_c=512, "
                    "d_h^R=64, d_h=128, d=5120), absorbed weights, batch 8, 16384 cached tokens, 64-token pages",
                    B=8, L=16384, H=128, d_h=128, r=0, d=5120, d_c=512, d_rope=64, seed=5),
    "train": Workload("train", "training-time expanded projection forward + backward (one of K/V) at the 6.3B head "
                      "shape d=4096, H=32, d_h=128, r=16, 8192 tokens (4 x 2048)",
                      B=4, L=2048, H=32, d_h=128, r=16, d=4096, seed=6),
    "prefill": Workload("prefill", "causal chunked prefill + append d=4096, H=32, d_h=128, r=16, batch 2, 4096-token prompts, 512-token chunks",
                        B=2, L=4096, H=32, d_h=128, r=16, d=4096, chunk=512, seed=4),
}
