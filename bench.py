#!/usr/bin/env python
"""Benchmark of the LRKV decode step on the long-context workload.

A step is one pass of the hot path for one batch: lrkv_append writes the newest
token's compressed row (s^K, s^V, z^K, z^V) of each sequence into the paged
cache, then lrkv_decode attends each sequence's query over its whole cache
(q~ absorption, split-K scan with online softmax, log-sum-exp combine and the
B^V up-projection).  Workload: d=4096, H=32, d_h=128, r=32, batch 4, cached
lengths uniform on [16384, 32768] (seeded), 64-token pages in a permuted pool.

Prints one JSON line.  value = algorithmic bytes of the step (cache rows read,
B^K/B^V, q in, out, plus the append's weights, hidden rows and new cache rows)
divided by the device time of the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lrkv|reference]
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

METRIC = "LRKV decode cache-read GB/s (% of GB300 HBM peak) and decode tokens/sec"
WORKLOAD = "longctx"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def workload_dims():
    wl = S.WORKLOADS[WORKLOAD]
    seq_lens = S.uniform_int(wl.seed, "seq_lens", wl.B, wl.L_min, wl.L).astype(np.int32)
    return wl, seq_lens


def step_bytes(wl, seq_lens):
    dec = A.decode_algorithmic_bytes(wl.H, wl.d_h, wl.r, seq_lens)
    app = A.append_algorithmic_bytes(wl.B, wl.d, wl.H, wl.d_h, wl.r)
    return dec, app


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode.cu", "lrkv_internal.cuh", "kernels.h"):
        with open(os.path.join(ROOT, "compressed_kv_cache_lrkv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current decode kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_split_longctx.md")
    try:
        txt = open(p).read()
    except OSError:
        return None
    mh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    mt = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    if not mh or not mt or mh.group(1) != kernel_source_hash():
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
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
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
        if not rows:
            return None
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
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_baseline_sample(wl, seq_lens, budget_s: float):
    """Time the fp64 oracle (E2 decode, all heads) on the workload's first sequence,
    repeated until about budget_s seconds have passed; returns the baseline dict."""
    import oracle

    o = oracle.get()
    tokens = int(seq_lens[0])
    pt = S.page_table(wl.seed, [tokens], 64)
    pools = tuple(S.gaussian_bf16(wl.seed, n, shp) for n, shp in
                  [("bl_sK", (pt.num_blocks, 64, wl.d_h)), ("bl_sV", (pt.num_blocks, 64, wl.d_h)),
                   ("bl_zK", (pt.num_blocks, 64, wl.H, wl.r)), ("bl_zV", (pt.num_blocks, 64, wl.H, wl.r))])
    BK = S.gaussian_bf16(wl.seed, "bl_BK", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
    BV = S.gaussian_bf16(wl.seed, "bl_BV", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
    q = S.gaussian_bf16(wl.seed, "bl_q", (1, wl.H, wl.d_h))
    reps = 0
    t0 = time.perf_counter()
    while True:
        o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    nbytes = A.decode_algorithmic_bytes(wl.H, wl.d_h, wl.r, [tokens]) * reps
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"E2 decode of the workload's first sequence ({tokens} cached tokens, all {wl.H} heads), "
                      f"{reps} repetitions in {dt:.1f} s; fp64, OpenMP over heads"}


def run_reference(args, world, rank):
    """--impl reference: the fp64 oracle on the host cores, bounded sample per step."""
    wl, seq_lens = workload_dims()
    if rank != 0:
        print(json.dumps({"impl": "reference", "rank": rank, "skipped": True}), file=sys.stderr)
        return
    import oracle

    o = oracle.get()
    total_steps = args.steps + args.warmup
    per_step_budget = max(0.01, 90.0 / max(total_steps, 1))
    # calibrate tokens per step
    probe = 256
    pt = S.page_table(wl.seed, [probe], 64)

    def inputs(tokens):
        pt = S.page_table(wl.seed, [tokens], 64)
        pools = tuple(S.gaussian_bf16(wl.seed, n, shp) for n, shp in
                      [("rf_sK", (pt.num_blocks, 64, wl.d_h)), ("rf_sV", (pt.num_blocks, 64, wl.d_h)),
                       ("rf_zK", (pt.num_blocks, 64, wl.H, wl.r)), ("rf_zV", (pt.num_blocks, 64, wl.H, wl.r))])
        BK = S.gaussian_bf16(wl.seed, "rf_BK", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        BV = S.gaussian_bf16(wl.seed, "rf_BV", (wl.H, wl.d_h, wl.r), wl.r ** -0.5)
        q = S.gaussian_bf16(wl.seed, "rf_q", (1, wl.H, wl.d_h))
        return pt, pools, BK, BV, q

    pt, pools, BK, BV, q = inputs(probe)
    t0 = time.perf_counter()
    o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    tokens = int(max(64, min(int(seq_lens[0]), rate * per_step_budget)) // 64 * 64) or 64
    pt, pools, BK, BV, q = inputs(tokens)
    for _ in range(args.warmup):
        o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.decode_cache(pools, pt.block_table, pt.seq_lens, BK, BV, q)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    nbytes = A.decode_algorithmic_bytes(wl.H, wl.d_h, wl.r, [tokens])
    val = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": S.WORKLOADS[WORKLOAD].description, "B": 1, "tokens_per_step": tokens,
                       "H": wl.H, "d_h": wl.d_h, "r": wl.r},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                             "sample": f"E2 decode, one sequence, first {tokens} tokens, all heads, per step"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_gpu(args, world, rank, local):
    import torch

    from compressed_kv_cache_lrkv_gb300 import binding as b

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl, seq_lens = workload_dims()
    B, H, d_h, r, d = wl.B, wl.H, wl.d_h, wl.r, wl.d
    pt = S.page_table(wl.seed, seq_lens, 64)
    nb = pt.num_blocks
    gen = torch.Generator(device="cuda").manual_seed(1234 + rank)
    randn = lambda *s, scale=1.0: (torch.randn(*s, generator=gen, device="cuda") * scale).to(torch.bfloat16)
    cache = b.PagedCache(randn(nb, 64, d_h), randn(nb, 64, d_h), randn(nb, 64, H, r), randn(nb, 64, H, r))
    q = randn(B, H, d_h)
    BK = randn(H, d_h, r, scale=r ** -0.5)
    BV = randn(H, d_h, r, scale=r ** -0.5)
    wcat = randn(2 * (d_h + H * r), d, scale=d ** -0.5)
    x_new = randn(B, d)
    dev_i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    bt = dev_i32(pt.block_table)
    sl = dev_i32(pt.seq_lens)
    slots = dev_i32([pt.slot(i, int(L) - 1) for i, L in enumerate(seq_lens)])
    dims = b.make_dims(H, d_h, r, d)
    out = torch.empty(B, H, d_h, dtype=torch.bfloat16, device="cuda")
    ws = b.alloc_workspace(b.decode_workspace_bytes(dims, B))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    cache_bytes = sum(t.numel() * t.element_size() for t in cache.tensors())

    def step():
        b.lrkv_append(dims, x_new, wcat, slots, cache, status=status, stream=stream)
        b.lrkv_decode(dims, q, BK, BV, cache, bt, sl, out, ws, status=status, stream=stream)

    # The timed step is a CUDA graph of the two public calls, so host launch overhead
    # stays out of the device-timed region; a second graph holds lrkv_decode alone.
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    g_step, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(g_step, stream=cap_stream):
            b.lrkv_append(dims, x_new, wcat, slots, cache, status=status, stream=cap_stream)
            b.lrkv_decode(dims, q, BK, BV, cache, bt, sl, out, ws, status=status, stream=cap_stream)
        with torch.cuda.graph(g_dec, stream=cap_stream):
            b.lrkv_decode(dims, q, BK, BV, cache, bt, sl, out, ws, status=status, stream=cap_stream)
    stream.wait_stream(cap_stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(args.warmup, 3)):
        g_step.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        g_step.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    # lrkv_decode alone (absorb + split + combine kernels), same workload, same stream
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for k in range(args.steps):
        g_dec.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dec_avg_ms = d0.elapsed_time(d1) / args.steps
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x}")

    # end to end through the public API with host buffers (pinned), copies in the timed region
    x_h = x_new.cpu().pin_memory()
    q_h = q.cpu().pin_memory()
    slots_h = slots.cpu().pin_memory()
    sl_h = sl.cpu().pin_memory()
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (x_h, q_h, slots_h, sl_h))
    d2h = out_h.numel() * out_h.element_size()
    e2e_steps = max(1, min(args.steps, 500))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x_new.copy_(x_h, non_blocking=True)
        q.copy_(q_h, non_blocking=True)
        slots.copy_(slots_h, non_blocking=True)
        sl.copy_(sl_h, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    sampler.stop()

    step_ms = total_ms / args.steps
    if dist:
        t = torch.tensor([step_ms, e2e_s], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms, e2e_s = float(t[0]), float(t[1])
    if rank != 0:
        dist.destroy_process_group()
        return
    dec_bytes, app_bytes = step_bytes(wl, seq_lens)
    bytes_step = (dec_bytes + app_bytes) * world
    value = bytes_step / (step_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic()
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_sample(wl, seq_lens, budget_s=15.0)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {wl.description}", "B": B, "seq_lens": [int(x) for x in seq_lens],
                   "H": H, "d_h": d_h, "r": r, "d": d, "block_size": 64, "pages": int(nb),
                   "cache_bytes": int(cache_bytes),
                   "l2": f"inputs larger than L2: cache {cache_bytes / 2**20:.0f} MiB vs L2 {L2_BYTES / 2**20:.0f} MiB",
                   "step": "lrkv_append (1 row per sequence) + lrkv_decode",
                   "parallelism": f"replicas x{world} (independent batches)"},
        "tokens_per_s": B * world / (step_ms * 1e-3),
        "pct_of_hbm_peak": 100.0 * value / peak,
        "roofline": {"kernel": "lrkv_decode (absorb + split + combine kernels)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": dec_bytes,
                     "avg_launch_ms": dec_avg_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": bytes_step / e2e_s / 1e9, "unit": "GB/s", "ms_per_step": e2e_s * 1e3,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 4 * args.steps,
        "timing": "each step is one replay of a CUDA graph holding lrkv_append + lrkv_decode",
        "clocks": sampler.summary(t_wall0 - 0.3, t_wall1 + 0.3),
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lrkv", choices=["lrkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
