#!/usr/bin/env python
"""Benchmark of the LRKV hot path on GB300.

Default workload ("longctx"): the long-context decode step.  A step is one
pass of the hot path for one batch: lrkv_append writes the newest token's
compressed row (s^K, s^V, z^K, z^V) of each sequence into the paged cache, then
lrkv_decode attends each sequence's query over its whole cache (q~ absorption,
split-K scan with online softmax, log-sum-exp combine, B^V up-projection).
d=4096, H=32, d_h=128, r=32, batch 4, cached lengths uniform on [16384, 32768]
(seeded), 64-token pages in a permuted pool.  value = algorithmic bytes of the
step (cache rows read, B^K/B^V, q in, out, plus the append's weights, hidden
rows and new cache rows) / device time of the step, in GB/s.

Other workloads (--workload): "dsv2" (H=128, d_h=128, r=16, d=16384, batch 8,
8192 tokens), "backbone12" (12 layers of d=512, H=8, d_h=64, r=16, batch 16,
2048 tokens), "small" (the single-layer parity case) -- decode steps as above;
"prefill": causal chunked prefill plus cache append (d=4096, H=32, d_h=128,
r=16, batch 2, 4096-token prompts in 512-token chunks), value in prompt
tokens/s with the tensor roofline of the prefill kernel; "mla": multi-head latent
attention decode with absorbed weights at DeepSeek-V2's attention shape (H=128,
d_c=512, d_h^R=64, d=5120, batch 8, 16384 cached tokens), GB/s as for decode.  --fused runs a decode
or prefill workload through lrkv_decode_fused / lrkv_prefill_fused (both absorptions in the
caller's weights: q~ given, [o_s | o_z] returned), counting that form's own bytes or flops.
--rope adds the 64-wide decoupled positional key (key rows [s^K | k^R], rotated in the append).

Prints one JSON line.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lrkv|reference] [--workload NAME] [--fused] [--rope]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import lrkv_synth as S  # noqa: E402
from compressed_kv_cache_lrkv_gb300 import accounting as A  # noqa: E402

METRIC_DECODE = "LRKV decode cache-read GB/s (% of GB300 HBM peak) and decode tokens/sec"
METRIC_MLA = "MLA (absorbed) decode cache-read GB/s (% of GB300 HBM peak) and decode tokens/sec"
METRIC_TRAIN = "LRKV expanded projection forward + backward TFLOP/s (bf16 tensor, fp32 accumulate)"
METRIC_PREFILL = "LRKV chunked prefill + append prompt tokens/sec (bf16 tensor TFLOP/s of the prefill kernel)"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
CSRC = os.path.join(ROOT, "compressed_kv_cache_lrkv_gb300", "csrc")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return {k: float(j[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name, sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    try:
        txt = open(os.path.join(ROOT, "profiles", profile_name)).read()
    except OSError:
        return None
    mh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    mt = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    if not mh or not mt or mh.group(1) != source_hash(sources):
        return None
    return int(mt.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        rows = [l for (t, l) in self.lines if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, dist, device="cpu"):
    """Element-wise max of per-rank timings (a barrier-free control-plane reduction)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_seed(rank: int, base: int) -> int:
    """Each rank decodes its own batch (disjoint sequences): weak scaling, no collective."""
    return base + 1000 * rank


def workload_seq_lens(wl):
    if wl.ragged:
        return S.uniform_int(wl.seed, "seq_lens", wl.B, wl.L_min, wl.L).astype(np.int32)
    return np.full(wl.B, wl.L, np.int32)


ROTATION_MAX_COPIES = 64
ROTATION_MAX_BYTES = 32 << 30


def _clone(v):
    """Deep copy of per-step device data: tensors, paged caches, and lists / dicts of them."""
    import torch

    from compressed_kv_cache_lrkv_gb300 import binding as b
    if isinstance(v, torch.Tensor):
        return v.clone()
    if isinstance(v, b.PagedCache):
        return b.PagedCache(*(t.clone() for t in v.tensors()))
    if isinstance(v, b.LayeredCache):
        return b.LayeredCache(*(t.clone() for t in v.tensors()))
    if isinstance(v, list):
        return [_clone(x) for x in v]
    if isinstance(v, dict):
        return {k: _clone(x) for k, x in v.items()}
    return v


def _nbytes(v):
    import torch

    from compressed_kv_cache_lrkv_gb300 import binding as b
    if isinstance(v, torch.Tensor):
        return v.numel() * v.element_size()
    if isinstance(v, (b.PagedCache, b.LayeredCache)):
        return sum(_nbytes(t) for t in v.tensors())
    if isinstance(v, (list, tuple)):
        return sum(_nbytes(x) for x in v)
    if isinstance(v, dict):
        return sum(_nbytes(x) for x in v.values())
    return 0


class Rotating:
    """Independent copies of a harness's per-step device data (caches, weights, activations).

    Successive timed steps use successive copies, round-robin, so no step finds its inputs in
    L2 from the step before: between two uses of a copy, every other copy's data streams
    through.  The number of copies is chosen so that each large class of data (the cache
    pools, the weights, ...) adds up to at least twice the L2 size over all copies; index
    data (block tables, lengths, slots) and the workspace are shared."""

    per_copy = ()  # attribute names that hold per-step device data

    def rotation_classes(self):
        """{label: bytes per copy} of the large data streams whose L2 residency must be broken."""
        raise NotImplementedError

    def copies_needed(self):
        big = [v for v in self.rotation_classes().values() if v >= (1 << 20)]
        need = max([3] + [-(-2 * L2_BYTES // v) for v in big])
        per = max(1, sum(_nbytes(getattr(self, k)) for k in self.per_copy))
        return int(max(1, min(need, ROTATION_MAX_COPIES, max(3, ROTATION_MAX_BYTES // per))))

    def add_copies(self, n):
        base = {k: getattr(self, k) for k in self.per_copy}
        self.sets = [base] + [{k: _clone(v) for k, v in base.items()} for _ in range(n - 1)]
        self.use(0)

    def use(self, k):
        for name, v in self.sets[k].items():
            setattr(self, name, v)

    def rotation_config(self):
        n = len(self.sets)
        per = sum(_nbytes(v) for v in self.sets[0].values())
        return {"copies": n, "bytes_per_copy": int(per),
                "classes_bytes_per_copy": {k: int(v) for k, v in self.rotation_classes().items()},
                "rule": "consecutive steps use different copies round-robin; each large data class totals "
                        ">= 2x L2 over the copies (at least 3 copies)"}

    # end to end through the public API: upload each step's inputs from pinned host buffers into
    # the copy the step uses, run the step's calls, download its result
    def e2e_setup(self):
        t = self.torch
        self.use(0)
        host_in = [x.cpu().pin_memory() for x in self.e2e_inputs()]
        host_out = [t.empty_like(x, device="cpu").pin_memory() for x in self.e2e_outputs()]
        self.e2e_pairs = []
        for k in range(len(self.sets)):
            self.use(k)
            self.e2e_pairs.append((list(zip(host_in, self.e2e_inputs())), list(zip(host_out, self.e2e_outputs()))))
        self.use(0)
        return (sum(_nbytes(h) for h in host_in), sum(_nbytes(h) for h in host_out))

    def e2e_step(self, stream, k=0):
        self.use(k)
        h_in, h_out = self.e2e_pairs[k]
        for h, d in h_in:
            d.copy_(h, non_blocking=True)
        self.step(stream)
        for h, d in h_out:
            h.copy_(d, non_blocking=True)
        stream.synchronize()


# ----------------------------------------------------------------------------- decode
class DecodeHarness(Rotating):
    """Per layer: lrkv_append of each sequence's newest row, then lrkv_decode; several layers
    go through the layer-batched calls (one launch of each kernel for all layers) unless
    per_layer is set."""

    per_copy = ("cache", "q", "BK", "BV", "wcat", "x", "qt", "out")
    profile = "decode_split_longctx.md"
    profiles = {"longctx": "decode_split_longctx.md", "dsv2": "decode_split_dsv2.md",
                "backbone12": "decode_layers_backbone12.md"}  # by workload
    sources = ("decode.cu", "decode_tc.cu", "decode_work.cuh", "lrkv_internal.cuh", "kernels.h")

    def __init__(self, wl, rank, fused=False, d_rope=0, per_layer=False):
        import torch

        from compressed_kv_cache_lrkv_gb300 import binding as b
        self.torch, self.b, self.wl, self.fused, self.d_rope = torch, b, wl, fused, d_rope
        dr = d_rope
        B, H, d_h, r, d, Ly = wl.B, wl.H, wl.d_h, wl.r, wl.d, wl.layers
        # the layer-batched calls have no absorbed-weights form: that one goes layer by layer
        self.layered = Ly > 1 and not per_layer and not fused
        self.seq_lens = workload_seq_lens(wl)
        self.pt = S.page_table(wl.seed, self.seq_lens, 64)
        nb = self.pt.num_blocks
        gen = torch.Generator(device="cuda").manual_seed(replica_seed(rank, 1234))
        rn = lambda *s, scale=1.0: (torch.randn(*s, generator=gen, device="cuda") * scale).to(torch.bfloat16)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        self.dims = b.make_dims(H, d_h, r, d, d_rope=dr)
        # every per-layer tensor carries a leading layer dimension
        self.cache = b.LayeredCache(rn(Ly, nb, 64, d_h + dr), rn(Ly, nb, 64, d_h), rn(Ly, nb, 64, H, r),
                                    rn(Ly, nb, 64, H, r))
        self.q = rn(Ly, B, H, d_h + dr)
        self.BK, self.BV = rn(Ly, H, d_h, r, scale=r ** -0.5), rn(Ly, H, d_h, r, scale=r ** -0.5)
        self.wcat = rn(Ly, 2 * (d_h + H * r) + dr, d, scale=d ** -0.5)
        self.x = rn(Ly, B, d)
        self.qt = rn(Ly, B, H, r) if fused else None
        self.out = torch.empty(Ly, B, H, d_h + (r if fused else 0), dtype=torch.bfloat16, device="cuda")
        self.bt = i32(self.pt.block_table)
        self.sl = i32(self.pt.seq_lens)
        self.slots = i32([self.pt.slot(i, int(L) - 1) for i, L in enumerate(self.seq_lens)])
        self.positions = i32(self.seq_lens - 1) if dr else None  # the newest token's position
        self.ws = b.alloc_workspace(b.decode_workspace_bytes(self.dims, Ly * B))
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.cache_bytes = _nbytes(self.cache)
        acct = A.decode_fused_algorithmic_bytes if fused else A.decode_algorithmic_bytes
        dec = acct(H, d_h, r, self.seq_lens, layers=Ly, d_rope=dr)
        app = Ly * A.append_algorithmic_bytes(B, d, H, d_h, r, d_rope=dr)
        self.kernel_units = dec          # algorithmic bytes of the timed kernel calls
        self.step_units = dec + app      # algorithmic bytes of a step
        per = 3 if fused else 4
        self.launches_per_step = per if self.layered else Ly * per

    def _decode(self, l, stream):
        b = self.b
        if self.fused:
            b.lrkv_decode_fused(self.dims, self.q[l], self.qt[l], self.cache.layer(l), self.bt, self.sl, self.out[l],
                                self.ws, status=self.status, stream=stream)
        else:
            b.lrkv_decode(self.dims, self.q[l], self.BK[l], self.BV[l], self.cache.layer(l), self.bt, self.sl,
                          self.out[l], self.ws, status=self.status, stream=stream)

    def step(self, stream):
        b = self.b
        if self.layered:
            b.lrkv_append_layers(self.dims, self.x, self.wcat, self.slots, self.cache, status=self.status,
                                 stream=stream, positions=self.positions)
            b.lrkv_decode_layers(self.dims, self.q, self.BK, self.BV, self.cache, self.bt, self.sl, self.out,
                                 self.ws, status=self.status, stream=stream)
            return
        for l in range(self.wl.layers):
            b.lrkv_append(self.dims, self.x[l], self.wcat[l], self.slots, self.cache.layer(l), status=self.status,
                          stream=stream, positions=self.positions)
            self._decode(l, stream)

    def kernel(self, stream):
        if self.layered:
            self.b.lrkv_decode_layers(self.dims, self.q, self.BK, self.BV, self.cache, self.bt, self.sl, self.out,
                                      self.ws, status=self.status, stream=stream)
            return
        for l in range(self.wl.layers):
            self._decode(l, stream)

    def rotation_classes(self):
        return {"cache": self.cache_bytes, "weights (W_cat, B^K, B^V)": _nbytes([self.wcat, self.BK, self.BV])}

    def e2e_inputs(self):
        return ([self.x, self.q] + ([self.qt] if self.qt is not None else []) + [self.slots, self.sl] +
                ([self.positions] if self.d_rope else []))

    def e2e_outputs(self):
        return [self.out]

    def report(self, step_s, kernel_s, e2e_s, world, peaks):
        wl = self.wl
        value = self.step_units * world / step_s / 1e9
        achieved = self.kernel_units / kernel_s / 1e9
        return {
            "metric": METRIC_DECODE, "value": value, "unit": "GB/s",
            "tokens_per_s": wl.B * world / step_s, "pct_of_hbm_peak": 100.0 * value / peaks["hbm_gbs"],
            # the decode call alone (cache + factor bytes over its own time), without the step's append
            "decode_pct_of_hbm_peak": 100.0 * achieved / peaks["hbm_gbs"],
            "config": {"workload": f"{wl.key}: {wl.description}", "B": wl.B,
                       "seq_lens": [int(x) for x in self.seq_lens], "layers": wl.layers, "H": wl.H, "d_h": wl.d_h,
                       "r": wl.r, "d": wl.d, "d_rope": self.d_rope, "block_size": 64,
                       "pages_per_layer": int(self.pt.num_blocks),
                       "cache_bytes": int(self.cache_bytes),
                       "l2": (f"inputs larger than L2: cache {self.cache_bytes / 2**20:.0f} MiB vs L2 "
                              f"{L2_BYTES / 2**20:.0f} MiB") if self.cache_bytes > L2_BYTES else
                             "cache fits in L2 (parity-sized workload; not an HBM measurement)",
                       "step": ("all layers at once: lrkv_append_layers (1 row per sequence and layer) + "
                                "lrkv_decode_layers" if self.layered else
                                "per layer: lrkv_append (1 row per sequence" +
                                (", positional key rotated at its position) + " if self.d_rope else ") + ") +
                                ("lrkv_decode_fused (q~ given, [o_s | o_z] returned)" if self.fused else
                                 "lrkv_decode")),
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": {"kernel": "lrkv_decode_fused (split + combine kernels)" if self.fused else
                                   ("lrkv_decode_layers (absorb + split + combine kernels, all layers)"
                                    if self.layered else "lrkv_decode (absorb + split + combine kernels)"),
                         "bound": "hbm",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": recorded_traffic(self.profiles[wl.key], self.sources)
                                    if wl.key in self.profiles and not self.fused and not self.d_rope
                                    and (self.layered or wl.layers == 1) else None,
                         "algorithmic_bytes_per_launch": self.kernel_units // (1 if self.layered else wl.layers),
                         "avg_launch_ms": kernel_s * 1e3 / (1 if self.layered else wl.layers)},
            "e2e_unit_value": lambda s: self.step_units * world / s / 1e9, "e2e_unit": "GB/s",
        }

    def cpu_baseline(self, budget_s):
        """fp64 oracle (E2 decode, all heads) on the first sequence, repeated ~budget_s."""
        import oracle
        wl = self.wl
        o = oracle.get()
        tokens = int(self.seq_lens[0])
        dr = self.d_rope
        pt = S.page_table(wl.seed, [tokens], 64)
        pools = tuple(S.gaussian_bf16(wl.seed, n, shp) for n, shp in
                      [("bl_sK", (pt.num_blocks, 64, wl.d_h + dr)), ("bl_sV", (pt.num_blocks, 64, wl.d_h)),
                       ("bl_zK", (pt.num_blocks, 64, wl.H, wl.r)), ("bl_zV", (pt.num_blocks, 64, wl.H, wl.r))])
        BK = S.gaussian_bf16(wl.seed, "bl_BK", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        BV = S.gaussian_bf16(wl.seed, "bl_BV", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        q = S.gaussian_bf16(wl.seed, "bl_q", (1, wl.H, wl.d_h + dr))
        qt = S.gaussian_bf16(wl.seed, "bl_qt", (1, wl.H, wl.r))
        reps, t0 = 0, time.perf_counter()
        while True:
            if self.fused:
                o.decode_fused(pools, pt.block_table, pt.seq_lens, q, qt)
            else:
                o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        acct = A.decode_fused_algorithmic_bytes if self.fused else A.decode_algorithmic_bytes
        nbytes = acct(wl.H, wl.d_h, wl.r, [tokens], d_rope=dr) * reps
        what = "absorbed-weights decode" if self.fused else "E2 decode"
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                "sample": f"{what} of the workload's first sequence ({tokens} cached tokens, all {wl.H} heads, "
                          f"one layer), {reps} repetitions in {dt:.1f} s; fp64, OpenMP over heads"}


# ----------------------------------------------------------------------------- prefill
class PrefillHarness(Rotating):
    """Per 512-token chunk: lrkv_append of both sequences' rows, then lrkv_prefill (or, with
    absorbed weights, lrkv_prefill_fused)."""

    per_copy = ("cache", "BK", "BV", "wcat", "chunks")

    profile = "prefill_chunked.md"
    sources = ("prefill_tc.cu", "lrkv_internal.cuh", "kernels.h")

    def __init__(self, wl, rank, fused=False, d_rope=0):
        import torch

        from compressed_kv_cache_lrkv_gb300 import binding as b
        self.torch, self.b, self.wl, self.fused, self.d_rope = torch, b, wl, fused, d_rope
        B, H, d_h, r, d, T, C, dr = wl.B, wl.H, wl.d_h, wl.r, wl.d, wl.L, wl.chunk, d_rope
        self.pt = S.page_table(wl.seed, [T] * B, 64)
        nb = self.pt.num_blocks
        gen = torch.Generator(device="cuda").manual_seed(replica_seed(rank, 4321))
        rn = lambda *s, scale=1.0: (torch.randn(*s, generator=gen, device="cuda") * scale).to(torch.bfloat16)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        self.dims = b.make_dims(H, d_h, r, d, d_rope=dr)
        self.cache = b.PagedCache.empty(nb, H, d_h, r, d_rope=dr)
        self.BK, self.BV = rn(H, d_h, r, scale=r ** -0.5), rn(H, d_h, r, scale=r ** -0.5)
        self.wcat = rn(2 * (d_h + H * r) + dr, d, scale=d ** -0.5)
        self.bt = i32(self.pt.block_table)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.chunks = []
        ow = d_h + (r if fused else 0)
        for c0 in range(0, T, C):
            self.chunks.append(dict(
                x=rn(B * C, d),  # both sequences' rows of this chunk
                slots=i32(np.concatenate([S.slots_for(self.pt, bb, c0, c0 + C) for bb in range(B)])),
                pos=i32(np.tile(np.arange(c0, c0 + C), B)) if dr else None,
                q=rn(B, C, H, d_h + dr), qs=i32([c0] * B),
                qt=rn(B, C, H, r) if fused else None,
                out=torch.empty(B, C, H, ow, dtype=torch.bfloat16, device="cuda")))
        self.side = torch.cuda.Stream()
        self.p2 = torch.cuda.Stream()  # every other chunk's prefill
        self.fork, self.join, self.join2 = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        self.appended = [torch.cuda.Event() for _ in self.chunks]
        app = A.append_flops(B * T, d, H, d_h, r) + 2 * B * T * d * dr
        pre = sum(A.prefill_flops(B, C, H, d_h, r, q_start=c0, d_rope=dr, absorbed=fused) for c0 in range(0, T, C))
        self.kernel_units = pre
        self.step_units = app + pre
        self.app_flops = app
        self.launches_per_step = 2 * len(self.chunks)

    def _prefill(self, ch, stream):
        if self.fused:
            self.b.lrkv_prefill_fused(self.dims, ch["q"], ch["qt"], self.cache, self.bt, ch["qs"], ch["out"],
                                      status=self.status, stream=stream)
        else:
            self.b.lrkv_prefill(self.dims, ch["q"], self.BK, self.BV, self.cache, self.bt, ch["qs"], ch["out"],
                                status=self.status, stream=stream)

    def step(self, stream):
        """Chunk c's prefill needs chunk c's rows in the cache; chunk c+1's append only writes
        rows that prefill c never reads (its keys end with chunk c), and no prefill reads
        another's output.  So the appends run in order on a side stream, each prefill waits
        for its own chunk's append, and the prefills alternate between two streams: the side
        stream's GEMMs and the next chunk's CTAs fill the SMs a prefill's last wave leaves idle."""
        b, side = self.b, self.side
        self.fork.record(stream)
        side.wait_event(self.fork)
        self.p2.wait_event(self.fork)
        for ch, ev in zip(self.chunks, self.appended):
            b.lrkv_append(self.dims, ch["x"], self.wcat, ch["slots"], self.cache, status=self.status, stream=side,
                          positions=ch["pos"])
            ev.record(side)
        for i, (ch, ev) in enumerate(zip(self.chunks, self.appended)):
            st = stream if i % 2 == 0 else self.p2
            st.wait_event(ev)
            self._prefill(ch, st)
        self.join.record(side)
        self.join2.record(self.p2)
        stream.wait_event(self.join)
        stream.wait_event(self.join2)

    def kernel(self, stream):
        """The eight chunk prefills alone (cache already filled), alternating between two
        streams as in the step."""
        self.fork.record(stream)
        self.p2.wait_event(self.fork)
        for i, ch in enumerate(self.chunks):
            self._prefill(ch, stream if i % 2 == 0 else self.p2)
        self.join2.record(self.p2)
        stream.wait_event(self.join2)

    def rotation_classes(self):
        return {"activations (X, q, out)": sum(_nbytes([ch["x"], ch["q"], ch["out"]]) for ch in self.chunks),
                "cache": _nbytes(self.cache), "weights (W_cat, B^K, B^V)": _nbytes([self.wcat, self.BK, self.BV])}

    def e2e_inputs(self):
        keys = ("x", "q") + (("qt",) if self.fused else ()) + (("pos",) if self.d_rope else ())
        return [ch[k] for ch in self.chunks for k in keys]

    def e2e_outputs(self):
        return [ch["out"] for ch in self.chunks]

    def report(self, step_s, kernel_s, e2e_s, world, peaks):
        wl = self.wl
        tokens = wl.B * wl.L * world
        achieved = self.kernel_units / kernel_s / 1e12
        return {
            "metric": METRIC_PREFILL, "value": tokens / step_s, "unit": "tokens/s",
            "step_tflops": self.step_units * world / step_s / 1e12,
            "config": {"workload": f"{wl.key}: {wl.description}", "B": wl.B, "prompt": wl.L, "chunk": wl.chunk,
                       "H": wl.H, "d_h": wl.d_h, "r": wl.r, "d": wl.d, "d_rope": self.d_rope,
                       "absorbed_weights": self.fused, "block_size": 64,
                       "l2": "prompt activations (X, q, out) larger than L2",
                       "step": "per 512-token chunk: lrkv_append (1024 rows" +
                               (", positional key rotated at each row's position) + " if self.d_rope else ") + ") +
                               ("lrkv_prefill_fused (q~ given, [o_s | o_z] returned)" if self.fused else
                                "lrkv_prefill") +
                               "; the appends run on a side stream (chunk c+1's append overlaps chunk c's prefill) "
                               "and the prefills alternate between two streams (chunk c+1's CTAs fill chunk c's "
                               "last wave)",
                       "flops_per_step": self.step_units, "append_flops": self.app_flops,
                       "prefill_flops": self.kernel_units,
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": {"kernel": ("lrkv_prefill_fused" if self.fused else "lrkv_prefill") +
                                   " (8 chunk launches on two streams)", "bound": "tensor",
                         "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "traffic": (recorded_traffic(self.profile, self.sources)
                                     if not self.fused and not self.d_rope else None),
                         "algorithmic_flops_per_launch": self.kernel_units / len(self.chunks),
                         "avg_launch_ms": kernel_s * 1e3 / len(self.chunks)},
            "e2e_unit_value": lambda s: tokens / s, "e2e_unit": "tokens/s",
        }

    def cpu_baseline(self, budget_s):
        """fp64 oracle (E2 causal prefill, all heads; absorbed-weights form with --fused) on the
        first chunk of one sequence."""
        import oracle
        wl = self.wl
        o = oracle.get()
        C, dr = wl.chunk, self.d_rope
        pt = S.page_table(wl.seed, [C], 64)
        pools = tuple(S.gaussian_bf16(wl.seed, n, shp) for n, shp in
                      [("bl_sK", (pt.num_blocks, 64, wl.d_h + dr)), ("bl_sV", (pt.num_blocks, 64, wl.d_h)),
                       ("bl_zK", (pt.num_blocks, 64, wl.H, wl.r)), ("bl_zV", (pt.num_blocks, 64, wl.H, wl.r))])
        BK = S.gaussian_bf16(wl.seed, "bl_BK", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        BV = S.gaussian_bf16(wl.seed, "bl_BV", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        q = S.gaussian_bf16(wl.seed, "bl_q", (1, C, wl.H, wl.d_h + dr))
        qt = S.gaussian_bf16(wl.seed, "bl_qt", (1, C, wl.H, wl.r))
        reps, t0 = 0, time.perf_counter()
        while True:
            if self.fused:
                o.prefill_fused(pools, pt.block_table, [0], q, qt)
            else:
                o.prefill_cache(pools, pt.block_table, [0], BK, BV, q)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        what = "absorbed-weights causal prefill" if self.fused else "E2 causal prefill"
        return {"value": C * reps / dt, "unit": "tokens/s", "cores": o.num_threads(), "kind": "oracle",
                "sample": f"{what} of one sequence's first {C}-token chunk (all {wl.H} heads), "
                          f"{reps} repetitions in {dt:.1f} s; fp64, OpenMP over heads"}


# ----------------------------------------------------------------------------- MLA decode
class MlaHarness(Rotating):
    """Multi-head latent attention with absorbed weights, per layer: lrkv_mla_append of each
    sequence's newest row [c | RoPE(k^R)], then lrkv_mla_decode."""

    per_copy = ("kv", "q", "wt", "x", "out")

    profile = "mla_decode.md"
    sources = ("mla_decode.cu", "mla.h", "lrkv_internal.cuh", "kernels.h")

    def __init__(self, wl, rank):
        import torch

        from compressed_kv_cache_lrkv_gb300 import binding as b
        self.torch, self.b, self.wl = torch, b, wl
        B, H, d, dc, dr = wl.B, wl.H, wl.d, wl.d_c, wl.d_rope
        dk = dc + dr
        self.seq_lens = workload_seq_lens(wl)
        self.pt = S.page_table(wl.seed, self.seq_lens, 64)
        nb = self.pt.num_blocks
        gen = torch.Generator(device="cuda").manual_seed(replica_seed(rank, 5678))
        rn = lambda *s, scale=1.0: (torch.randn(*s, generator=gen, device="cuda") * scale).to(torch.bfloat16)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
        self.dims = b.make_mla_dims(H, d, d_head=wl.d_h, d_c=dc, d_rope=dr)
        self.kv = rn(nb, 64, dk)
        self.q = rn(B, H, dk)
        self.wt = rn(dk, d, scale=d ** -0.5)
        self.x = rn(B, d)
        self.out = torch.empty(B, H, dc, dtype=torch.bfloat16, device="cuda")
        self.bt = i32(self.pt.block_table)
        self.sl = i32(self.pt.seq_lens)
        self.slots = i32([self.pt.slot(i, int(L) - 1) for i, L in enumerate(self.seq_lens)])
        self.positions = i32(self.seq_lens - 1)
        self.ws = b.alloc_workspace(b.mla_decode_workspace_bytes(self.dims, B))
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.cache_bytes = self.kv.numel() * self.kv.element_size()
        self.kernel_units = A.mla_decode_algorithmic_bytes(H, dc, dr, self.seq_lens)
        self.step_units = self.kernel_units + A.mla_append_algorithmic_bytes(B, d, dc, dr)
        self.flops = A.mla_decode_flops(H, dc, dr, self.seq_lens)
        self.launches_per_step = 3

    def step(self, stream):
        b = self.b
        b.lrkv_mla_append(self.dims, self.x, self.wt, self.slots, self.positions, self.kv, status=self.status,
                          stream=stream)
        b.lrkv_mla_decode(self.dims, self.q, self.kv, self.bt, self.sl, self.out, self.ws, status=self.status,
                          stream=stream)

    def kernel(self, stream):
        self.b.lrkv_mla_decode(self.dims, self.q, self.kv, self.bt, self.sl, self.out, self.ws, status=self.status,
                               stream=stream)

    def rotation_classes(self):
        return {"cache": self.cache_bytes, "weights ([W^DKV | W^KR])": _nbytes(self.wt)}

    def e2e_inputs(self):
        return [self.x, self.q, self.slots, self.positions, self.sl]

    def e2e_outputs(self):
        return [self.out]

    def report(self, step_s, kernel_s, e2e_s, world, peaks):
        wl = self.wl
        value = self.step_units * world / step_s / 1e9
        achieved = self.kernel_units / kernel_s / 1e9
        return {
            "metric": METRIC_MLA, "value": value, "unit": "GB/s",
            "tokens_per_s": wl.B * world / step_s, "pct_of_hbm_peak": 100.0 * value / peaks["hbm_gbs"],
            "config": {"workload": f"{wl.key}: {wl.description}", "B": wl.B,
                       "seq_lens": [int(x) for x in self.seq_lens], "H": wl.H, "d_c": wl.d_c, "d_rope": wl.d_rope,
                       "d_head": wl.d_h, "d": wl.d, "block_size": 64, "pages": int(self.pt.num_blocks),
                       "cache_bytes": int(self.cache_bytes),
                       "l2": f"inputs larger than L2: cache {self.cache_bytes / 2**20:.0f} MiB vs L2 "
                             f"{L2_BYTES / 2**20:.0f} MiB",
                       "step": "lrkv_mla_append (1 row per sequence, positional key rotated) + lrkv_mla_decode",
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": {"kernel": "lrkv_mla_decode (cluster split + combine kernels)", "bound": "hbm",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": recorded_traffic(self.profile, self.sources),
                         "tensor_tflops": self.flops / kernel_s / 1e12,
                         "tensor_frac": self.flops / kernel_s / 1e12 / peaks["bf16_tflops"],
                         "algorithmic_bytes_per_launch": self.kernel_units,
                         "algorithmic_flops_per_launch": self.flops,
                         "avg_launch_ms": kernel_s * 1e3},
            "e2e_unit_value": lambda s: self.step_units * world / s / 1e9, "e2e_unit": "GB/s",
        }

    def cpu_baseline(self, budget_s):
        """fp64 oracle (absorbed MLA decode, all heads) on a prefix of the first sequence."""
        import oracle
        wl = self.wl
        o = oracle.get()
        dk = wl.d_c + wl.d_rope
        tokens = min(int(self.seq_lens[0]), 2048)
        pt = S.page_table(wl.seed, [tokens], 64)
        kv = S.gaussian_bf16(wl.seed, "bl_kv", (pt.num_blocks, 64, dk))
        q = S.gaussian_bf16(wl.seed, "bl_q", (1, wl.H, dk))
        reps, t0 = 0, time.perf_counter()
        while True:
            o.mla_decode(kv, pt.block_table, pt.seq_lens, q, wl.d_rope, wl.d_h)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        nbytes = A.mla_decode_algorithmic_bytes(wl.H, wl.d_c, wl.d_rope, [tokens]) * reps
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                "sample": f"absorbed MLA decode of the first {tokens} cached tokens of one sequence (all {wl.H} "
                          f"heads), {reps} repetitions in {dt:.1f} s; fp64, OpenMP over heads"}


# ----------------------------------------------------------------------------- training projection
class TrainHarness(Rotating):
    """One projection (keys or values) of a training step: lrkv_train_forward, then
    lrkv_train_backward for a given dK."""

    per_copy = ("X", "Wt", "B", "dK", "Y", "K", "dX", "dWt", "dB")

    profile = "train_projection.md"
    sources = ("train.cu", "train.h", "lrkv_internal.cuh", "kernels.h")

    def __init__(self, wl, rank):
        import torch

        from compressed_kv_cache_lrkv_gb300 import binding as b
        self.torch, self.b, self.wl = torch, b, wl
        n, d, H, d_h, r = wl.B * wl.L, wl.d, wl.H, wl.d_h, wl.r
        self.n = n
        gen = torch.Generator(device="cuda").manual_seed(replica_seed(rank, 9012))
        rn = lambda *s, scale=1.0: (torch.randn(*s, generator=gen, device="cuda") * scale).to(torch.bfloat16)
        self.dims = b.make_dims(H, d_h, r, d)
        N = d_h + H * r
        self.X, self.Wt = rn(n, d), rn(N, d, scale=d ** -0.5)
        self.B, self.dK = rn(H, d_h, r, scale=r ** -0.5), rn(n, H, d_h)
        mk = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
        self.Y, self.K = mk(n, N), mk(n, H, d_h)
        self.dX, self.dWt, self.dB = mk(n, d), mk(N, d), mk(H, d_h, r)
        self.ws = b.alloc_workspace(b.train_workspace_bytes(self.dims, n))
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fwd, bwd = A.train_flops(n, d, H, d_h, r)
        self.kernel_units = bwd
        self.step_units = fwd + bwd
        self.fwd_units = fwd
        self.launches_per_step = 2 + 5

    def step(self, stream):
        b = self.b
        b.lrkv_train_forward(self.dims, self.X, self.Wt, self.B, self.Y, self.K, status=self.status, stream=stream)
        b.lrkv_train_backward(self.dims, self.X, self.Wt, self.B, self.Y, self.dK, self.dX, self.dWt, self.dB,
                              self.ws, status=self.status, stream=stream)

    def kernel(self, stream):
        self.b.lrkv_train_backward(self.dims, self.X, self.Wt, self.B, self.Y, self.dK, self.dX, self.dWt, self.dB,
                                   self.ws, status=self.status, stream=stream)

    def rotation_classes(self):
        return {"activations (X, dK, Y, K, dX)": _nbytes([self.X, self.dK, self.Y, self.K, self.dX]),
                "weights (W_T, B, dW_T, dB)": _nbytes([self.Wt, self.B, self.dWt, self.dB])}

    def e2e_inputs(self):
        return [self.X, self.dK]

    def e2e_outputs(self):
        return [self.dB]

    def report(self, step_s, kernel_s, e2e_s, world, peaks):
        wl = self.wl
        achieved = self.kernel_units / kernel_s / 1e12
        return {
            "metric": METRIC_TRAIN, "value": self.step_units * world / step_s / 1e12, "unit": "TFLOP/s",
            "tokens_per_s": self.n * world / step_s,
            "config": {"workload": f"{wl.key}: {wl.description}", "tokens": self.n, "H": wl.H, "d_h": wl.d_h,
                       "r": wl.r, "d": wl.d, "flops_per_step": self.step_units, "forward_flops": self.fwd_units,
                       "backward_flops": self.kernel_units,
                       "l2": "activations (X, dK, Y, K, dX: 224 MiB) larger than L2",
                       "step": "lrkv_train_forward (Y, K) + lrkv_train_backward (dX, dW_T, dB)",
                       "parallelism": f"replicas x{world} (independent micro-batches)"},
            "roofline": {"kernel": "lrkv_train_backward (head sum + 4 tcgen05 GEMM launches + dB reduce)",
                         "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"],
                         "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                         "traffic": recorded_traffic(self.profile, self.sources),
                         "algorithmic_flops_per_launch": self.kernel_units, "avg_launch_ms": kernel_s * 1e3},
            "e2e_unit_value": lambda s: self.step_units * world / s / 1e12, "e2e_unit": "TFLOP/s",
        }

    def cpu_baseline(self, budget_s):
        """fp64 oracle (forward + backward) on a 64-token sample of the workload's shape."""
        import oracle
        wl = self.wl
        o = oracle.get()
        n = 64
        X = S.gaussian_bf16(wl.seed, "bl_X", (n, wl.d))
        Ws = S.gaussian_bf16(wl.seed, "bl_Ws", (wl.d, wl.d_h), wl.d ** -0.5)
        U = S.gaussian_bf16(wl.seed, "bl_U", (wl.H, wl.d, wl.r), wl.d ** -0.5)
        Bm = S.gaussian_bf16(wl.seed, "bl_B", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        dK = S.gaussian_bf16(wl.seed, "bl_dK", (n, wl.H, wl.d_h))
        reps, t0 = 0, time.perf_counter()
        while True:
            o.train_forward(X, Ws, U, Bm)
            o.train_backward(X, Ws, U, Bm, dK)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
        f, bw = A.train_flops(n, wl.d, wl.H, wl.d_h, wl.r)
        return {"value": (f + bw) * reps / dt / 1e12, "unit": "TFLOP/s", "cores": o.num_threads(), "kind": "oracle",
                "sample": f"expanded projection forward + backward of {n} tokens at the workload's shape, "
                          f"{reps} repetitions in {dt:.1f} s; fp64 (algorithmic flop count of the factored route)"}


HARNESS = {"longctx": DecodeHarness, "dsv2": DecodeHarness, "backbone12": DecodeHarness, "small": DecodeHarness,
           "prefill": PrefillHarness, "mla": MlaHarness, "train": TrainHarness}


# ----------------------------------------------------------------------------- arms
def run_gpu(args, world, rank, local):
    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl = S.WORKLOADS[args.workload]
    if (args.fused or args.rope) and HARNESS[args.workload] not in (DecodeHarness, PrefillHarness):
        raise SystemExit("--fused and --rope apply to the decode and prefill workloads")
    if args.per_layer and HARNESS[args.workload] is not DecodeHarness:
        raise SystemExit("--per-layer applies to the decode workloads")
    if HARNESS[args.workload] is DecodeHarness:
        hz = DecodeHarness(wl, rank, fused=args.fused, d_rope=64 if args.rope else 0, per_layer=args.per_layer)
    elif HARNESS[args.workload] is PrefillHarness:
        hz = PrefillHarness(wl, rank, fused=args.fused, d_rope=64 if args.rope else 0)
    else:
        hz = HARNESS[args.workload](wl, rank)
    stream = torch.cuda.current_stream()

    # The timed steps are CUDA graphs of the public calls, so host launch overhead stays out
    # of the device-timed region; a second set of graphs holds only the dominant call
    # (lrkv_decode / lrkv_prefill / ...) for the roofline.  The per-step data comes in
    # independent copies used round-robin (Rotating), so no timed step or call reads inputs
    # that the previous one left in L2.  One graph per copy holds one step; one "cycle" graph
    # holds one step on every copy in turn, so that K steps are K / copies cycle replays (plus
    # single-step replays for the remainder) and the gap between two graph launches is paid
    # once per cycle, not once per step.
    n_copies = args.copies or hz.copies_needed()
    hz.add_copies(n_copies)
    for k in range(n_copies):
        hz.use(k)
        hz.step(stream)
    for _ in range(2):
        hz.use(0)
        hz.step(stream)
    torch.cuda.synchronize()
    g_step = [torch.cuda.CUDAGraph() for _ in range(n_copies)]
    g_ker = [torch.cuda.CUDAGraph() for _ in range(n_copies)]
    g_step_cycle, g_ker_cycle = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for k in range(n_copies):
            hz.use(k)
            with torch.cuda.graph(g_step[k], stream=cap):
                hz.step(cap)
            with torch.cuda.graph(g_ker[k], stream=cap):
                hz.kernel(cap)
        with torch.cuda.graph(g_step_cycle, stream=cap):
            for k in range(n_copies):
                hz.use(k)
                hz.step(cap)
        with torch.cuda.graph(g_ker_cycle, stream=cap):
            for k in range(n_copies):
                hz.use(k)
                hz.kernel(cap)
        # the same number of steps on copy 0 alone, back to back (for the L2-warm figures)
        hz.use(0)
        g_step_warm, g_ker_warm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step_warm, stream=cap):
            for k in range(n_copies):
                hz.step(cap)
        with torch.cuda.graph(g_ker_warm, stream=cap):
            for k in range(n_copies):
                hz.kernel(cap)
    hz.use(0)
    stream.wait_stream(cap)
    torch.cuda.synchronize()

    def timed_steps(cycle, singles, steps):
        """Seconds per step over exactly `steps` steps on the copies in turn: steps // copies
        replays of the cycle graph, then single-step graphs for the remainder (CUDA events)."""
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps // n_copies):
            cycle.replay()
        for k in range(steps % n_copies):
            singles[k].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) * 1e-3 / steps

    sampler = ClockSampler(local)
    sampler.start()
    for i in range(max(args.warmup, 3)):
        g_step[i % n_copies].replay()
    for g in (g_step_cycle, g_ker_cycle, g_step_warm, g_ker_warm):
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    step_s = timed_steps(g_step_cycle, g_step, args.steps)
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # per-step spread, from a separate shorter loop so the timed region above has no extra events
    nd = max(1, min(args.steps, 200))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nd + 1)]
    evs[0].record(stream)
    for i in range(nd):
        g_step[(args.steps + i) % n_copies].replay()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(nd))
    kernel_s = timed_steps(g_ker_cycle, g_ker, args.steps)
    # the same graphs on one copy back to back: whatever of its inputs stays in L2 between
    # replays is served from there (reported beside the rotated numbers, not as them)
    kernel_warm_s = timed_steps(g_ker_warm, [g_ker[0]] * n_copies, args.steps)
    step_warm_s = timed_steps(g_step_warm, [g_step[0]] * n_copies, args.steps)
    if int(hz.status.item()) != 0:
        raise RuntimeError(f"device status {int(hz.status.item()):#x}")

    # end to end through the public API with pinned host buffers, copies in the timed region
    h2d, d2h = hz.e2e_setup()
    e2e_steps = max(1, min(args.steps, 200))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        hz.e2e_step(stream, i % n_copies)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    hz.use(0)
    sampler.stop()

    if dist:
        step_s, kernel_s, e2e_s, kernel_warm_s, step_warm_s = max_over_ranks(
            [step_s, kernel_s, e2e_s, kernel_warm_s, step_warm_s], dist, device="cuda")
    if rank != 0:
        dist.destroy_process_group()
        return
    peaks, peak_kind = measured_peaks()
    rep = hz.report(step_s, kernel_s, e2e_s, world, peaks)
    e2e_fn, e2e_unit = rep.pop("e2e_unit_value"), rep.pop("e2e_unit")
    rep["roofline"]["peak_kind"] = peak_kind
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = hz.cpu_baseline(budget_s=15.0)
    line = {"metric": rep.pop("metric"), "value": rep.pop("value"), "unit": rep.pop("unit"), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    line.update(rep)
    line["cpu_baseline"] = cpu
    line["e2e"] = {"value": e2e_fn(e2e_s), "unit": e2e_unit, "ms_per_step": e2e_s * 1e3,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}
    line["step_ms_spread"] = {"median": statistics.median(per_step_ms), "min": per_step_ms[0],
                              "max": per_step_ms[-1], "reps": nd}
    line["gpu_launches"] = hz.launches_per_step * args.steps
    line["timing"] = ("each step is one pass of the public calls on its own copy of the inputs, the copies used "
                      "round-robin (see config.l2_rotation); one CUDA graph holds one step on every copy in turn and "
                      "is replayed steps // copies times, single-step graphs take the remainder; CUDA events on the "
                      "stream")
    line["config"]["l2"] = "rotated input copies (no step reads inputs the previous step left in L2): " + \
        line["config"].get("l2", "")
    line["config"]["l2_rotation"] = hz.rotation_config()
    rf = line["roofline"]
    rf["avg_launch_ms_l2_warm"] = rf["avg_launch_ms"] * kernel_warm_s / kernel_s
    rf["frac_l2_warm"] = rf["frac"] * kernel_s / kernel_warm_s
    line["l2_warm"] = {"ms_per_step": step_warm_s * 1e3, "value": line["value"] * step_s / step_warm_s,
                       "note": "one input copy replayed back to back (inputs may stay in L2 between steps); "
                               "context only, not the reported value"}
    line["clocks"] = sampler.summary(t_wall0 - 0.3, t_wall1 + 0.3)
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def run_reference(args, world, rank):
    """--impl reference: the fp64 oracle on the host cores; each step is a bounded sample
    of the workload (decode: E2 decode of a prefix of the first sequence, all heads; the
    MLA, prefill and training workloads: see their functions below)."""
    if rank != 0:
        return
    import oracle

    wl = S.WORKLOADS[args.workload]
    if (args.fused or args.rope) and HARNESS[args.workload] not in (DecodeHarness, PrefillHarness):
        raise SystemExit("--fused and --rope apply to the decode and prefill workloads")
    o = oracle.get()
    per_step_budget = max(0.01, 90.0 / max(args.steps + args.warmup, 1))
    if args.workload == "prefill":
        return run_reference_prefill(args, wl, o, per_step_budget)
    if args.workload == "train":
        return run_reference_train(args, wl, o, per_step_budget)
    seq_lens = workload_seq_lens(wl)

    if wl.d_c:
        return run_reference_mla(args, wl, seq_lens, o, per_step_budget)

    dr = 64 if args.rope else 0

    def inputs(tokens):
        pt = S.page_table(wl.seed, [tokens], 64)
        pools = tuple(S.gaussian_bf16(wl.seed, n, shp) for n, shp in
                      [("rf_sK", (pt.num_blocks, 64, wl.d_h + dr)), ("rf_sV", (pt.num_blocks, 64, wl.d_h)),
                       ("rf_zK", (pt.num_blocks, 64, wl.H, wl.r)), ("rf_zV", (pt.num_blocks, 64, wl.H, wl.r))])
        BK = S.gaussian_bf16(wl.seed, "rf_BK", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        BV = S.gaussian_bf16(wl.seed, "rf_BV", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        q = S.gaussian_bf16(wl.seed, "rf_q", (1, wl.H, wl.d_h + dr))
        qt = S.gaussian_bf16(wl.seed, "rf_qt", (1, wl.H, wl.r))
        return pt, pools, BK, BV, q, qt

    def step(pt, pools, BK, BV, q, qt):
        if args.fused:
            o.decode_fused(pools, pt.block_table, pt.seq_lens, q, qt)
        else:
            o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)

    probe = 256
    a_in = inputs(probe)
    t0 = time.perf_counter()
    step(*a_in)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    tokens = max(64, int(min(int(seq_lens[0]), rate * per_step_budget)) // 64 * 64)
    a_in = inputs(tokens)
    for _ in range(args.warmup):
        step(*a_in)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(*a_in)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    acct = A.decode_fused_algorithmic_bytes if args.fused else A.decode_algorithmic_bytes
    val = acct(wl.H, wl.d_h, wl.r, [tokens], d_rope=dr) / dt / 1e9
    what = "absorbed-weights decode" if args.fused else "E2 decode"
    print(json.dumps({
        "impl": "reference", "metric": METRIC_DECODE, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.key}: {wl.description}", "sample_tokens_per_step": tokens, "H": wl.H,
                   "d_h": wl.d_h, "r": wl.r, "d_rope": dr, "absorbed_weights": bool(args.fused)},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"{what} of the first {tokens} tokens of one sequence, all heads, per step"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def run_reference_mla(args, wl, seq_lens, o, per_step_budget):
    """--impl reference on the MLA workload: the oracle's absorbed MLA decode of a prefix of the
    first sequence, all heads, each step."""
    dk = wl.d_c + wl.d_rope

    def inputs(tokens):
        pt = S.page_table(wl.seed, [tokens], 64)
        return (pt, S.gaussian_bf16(wl.seed, "rf_kv", (pt.num_blocks, 64, dk)),
                S.gaussian_bf16(wl.seed, "rf_q", (1, wl.H, dk)))

    probe = 256
    pt, kv, q = inputs(probe)
    t0 = time.perf_counter()
    o.mla_decode(kv, pt.block_table, pt.seq_lens, q, wl.d_rope, wl.d_h)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    tokens = max(64, int(min(int(seq_lens[0]), rate * per_step_budget)) // 64 * 64)
    pt, kv, q = inputs(tokens)
    for _ in range(args.warmup):
        o.mla_decode(kv, pt.block_table, pt.seq_lens, q, wl.d_rope, wl.d_h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.mla_decode(kv, pt.block_table, pt.seq_lens, q, wl.d_rope, wl.d_h)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    val = A.mla_decode_algorithmic_bytes(wl.H, wl.d_c, wl.d_rope, [tokens]) / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC_MLA, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.key}: {wl.description}", "sample_tokens_per_step": tokens, "H": wl.H,
                   "d_c": wl.d_c, "d_rope": wl.d_rope},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"absorbed MLA decode of the first {tokens} tokens of one sequence, all heads, "
                                   f"per step"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def _timed_steps(args, fn):
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    return (time.perf_counter() - t0) / max(args.steps, 1)


def run_reference_prefill(args, wl, o, per_step_budget):
    """--impl reference on the prefill workload: each step, the oracle appends one sequence's
    first Tq prompt rows (the cache rows from X and the weights) and runs the E2 causal prefill of
    those Tq queries over them, all heads; Tq (a multiple of 64, at most one chunk) sized from a
    probe so that a step takes about its share of the run's budget.  With --rope the append
    also rotates the positional key at each row's position; with --fused the prefill takes q~
    and returns [o_s | o_z] (the oracle's absorbed-weights prefill)."""
    d, H, d_h, r = wl.d, wl.H, wl.d_h, wl.r
    dr = 64 if args.rope else 0

    def inputs(tq):
        X = S.gaussian_bf16(wl.seed, "rp_X", (tq, d))
        W = [S.gaussian_bf16(wl.seed, "rp_WsK", (d, d_h), d ** -0.5),
             S.gaussian_bf16(wl.seed, "rp_WsV", (d, d_h), d ** -0.5),
             S.gaussian_bf16(wl.seed, "rp_UK", (H, d, r), d ** -0.5),
             S.gaussian_bf16(wl.seed, "rp_UV", (H, d, r), d ** -0.5)]
        WKR = S.gaussian_bf16(wl.seed, "rp_WKR", (d, dr), d ** -0.5) if dr else None
        BK = S.gaussian_bf16(wl.seed, "rp_BK", (H, d_h, r), r ** -0.5)
        BV = S.gaussian_bf16(wl.seed, "rp_BV", (H, d_h, r), r ** -0.5)
        q = S.gaussian_bf16(wl.seed, "rp_q", (1, tq, H, d_h + dr))
        qt = S.gaussian_bf16(wl.seed, "rp_qt", (1, tq, H, r))
        pt = S.page_table(wl.seed, [tq], 64)
        return X, W, WKR, BK, BV, q, qt, pt

    def step(tq, X, W, WKR, BK, BV, q, qt, pt):
        # (sK, sV, zK, zV) rows, bf16 bits, token order
        rows = o.append(X, *W, WKR=WKR, positions=np.arange(tq, dtype=np.int32) if dr else None)
        nb = pt.num_blocks
        pools = [np.zeros((nb * 64,) + a.shape[1:], np.uint16) for a in rows]
        slots = S.slots_for(pt, 0, 0, tq)
        for pool, a in zip(pools, rows):
            pool[slots] = a
        pools = tuple(pool.reshape((nb, 64) + pool.shape[1:]) for pool in pools)
        if args.fused:
            o.prefill_fused(pools, pt.block_table, [0], q, qt)
        else:
            o.prefill_cache(pools, pt.block_table, [0], BK, BV, q)

    probe = 64
    args_p = inputs(probe)
    t0 = time.perf_counter()
    step(probe, *args_p)
    dt0 = max(time.perf_counter() - t0, 1e-6)
    tq = probe
    while tq * 2 <= wl.chunk and dt0 * (tq * 2 / probe) ** 2 <= per_step_budget:
        tq *= 2
    a_in = inputs(tq)
    dt = _timed_steps(args, lambda: step(tq, *a_in))
    val = tq / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC_PREFILL, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.key}: {wl.description}", "sample_prompt_tokens_per_step": tq, "H": H,
                   "d_h": d_h, "r": r, "d": d, "d_rope": dr, "absorbed_weights": bool(args.fused)},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"append of one sequence's first {tq} prompt rows and the "
                                   f"{'absorbed-weights' if args.fused else 'E2'} causal prefill "
                                   f"of those {tq} queries (all {H} heads), per step"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def run_reference_train(args, wl, o, per_step_budget):
    """--impl reference on the training workload: each step, the oracle's expanded projection
    forward and backward on n tokens at the workload's shape (d, H, d_h, r), n (a multiple of 8)
    sized from a probe to the step's share of the budget; TFLOP/s of the algorithmic flops."""
    d, H, d_h, r = wl.d, wl.H, wl.d_h, wl.r

    def inputs(n):
        return (S.gaussian_bf16(wl.seed, "rt_X", (n, d)),
                S.gaussian_bf16(wl.seed, "rt_Ws", (d, d_h), d ** -0.5),
                S.gaussian_bf16(wl.seed, "rt_U", (H, d, r), d ** -0.5),
                S.gaussian_bf16(wl.seed, "rt_B", (H, d_h, r), r ** -0.5),
                S.gaussian_bf16(wl.seed, "rt_dK", (n, H, d_h)))

    def step(X, Ws, U, Bm, dK):
        o.train_forward(X, Ws, U, Bm)
        o.train_backward(X, Ws, U, Bm, dK)

    probe = 8
    t0 = time.perf_counter()
    step(*inputs(probe))
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    n = max(8, min(wl.B * wl.L, int(rate * per_step_budget)) // 8 * 8)
    a_in = inputs(n)
    dt = _timed_steps(args, lambda: step(*a_in))
    f, bw = A.train_flops(n, d, H, d_h, r)
    val = (f + bw) / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC_TRAIN, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.key}: {wl.description}", "sample_tokens_per_step": n, "H": H, "d_h": d_h,
                   "r": r, "d": d, "flops_per_step": f + bw},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": f"expanded projection forward + backward of {n} tokens at the workload's shape, "
                                   f"per step (algorithmic flop count of the factored route)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lrkv", choices=["lrkv", "reference"])
    ap.add_argument("--workload", default="longctx", choices=sorted(HARNESS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-layer", action="store_true",
                    help="multi-layer decode workloads: one lrkv_append + lrkv_decode per layer instead of the "
                         "layer-batched calls")
    ap.add_argument("--copies", type=int, default=0,
                    help="independent input copies replayed round-robin (0: enough to break L2 residency)")
    ap.add_argument("--fused", action="store_true",
                    help="decode or prefill with absorbed weights (lrkv_decode_fused / lrkv_prefill_fused: "
                         "q~ given, [o_s | o_z] returned)")
    ap.add_argument("--rope", action="store_true",
                    help="decode or prefill with a 64-wide decoupled positional key shared by all heads "
                         "(d_rope = 64)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
