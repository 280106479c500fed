#!/usr/bin/env python3
"""Benchmark of the paged GQA attention path on GB300.

Headline (one JSON line on stdout): a decode step of the decode-attention
workload -- batch 64, Qwen3-0.6B attention shapes (16 query heads, 8 KV heads,
head_dim 128, bf16), 256-token blocks, context lengths uniform in
[512, 4096], physical blocks a random permutation of a pool 1.25x the blocks
used.  One step = the new token's slot, its KV write and the decode attention,
through the C ABI call that fuses them (pkv_decode_append: split-K decode +
combine launches); the same step through the three separate calls is reported
beside it.  value = KV bytes the attention reads per step / step time, in GB/s.

The same line carries:
  roofline      the decode attention call's achieved HBM GB/s (KV bytes per
                call / CUDA-event time of the call) against the measured copy
                bandwidth, plus DRAM traffic per launch from the committed ncu
                summary when the kernel source is unchanged since it was taken
  e2e           the same metric with host buffers: pinned-host -> device copies
                of the step's inputs and the device -> host copy of its output
                inside the timed region
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  secondary     prefill TFLOP/s (32 prompts with prefix-cache hits), long-
                context decode GB/s (batch 8, 16k-40k), and the full 28-layer
                decode step + sampler (batch 256) in tokens/s
  clocks        SM clocks and throttle reasons sampled during the timed region

``--impl reference`` times the CPU oracle instead (the only other arm: the
pages ship no code to run), on the same metric and workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

# The CPU baseline runs the oracle on the host's own cores: its BLAS threads are pinned to the
# cores this process may run on (unless the caller sets them), before NumPy loads OpenBLAS, so
# the count reported is the count that ran.
try:
    _HOST_CORES = sorted(os.sched_getaffinity(0))
except AttributeError:          # not Linux
    _HOST_CORES = list(range(os.cpu_count() or 1))
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(len(_HOST_CORES)))
os.environ.setdefault("OMP_NUM_THREADS", os.environ["OPENBLAS_NUM_THREADS"])

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn HBM GB/s (% of peak); prefill TFLOP/s; decode tok/s at batch"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
DECODE_SRC = os.path.join(ROOT, "paged_kv_attention_29_gb300", "csrc", "decode.cu")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file, src_path):
    """DRAM bytes per launch from a committed ncu summary, if the source is unchanged."""
    try:
        with open(os.path.join(PROFILE_DIR, kernel_file)) as f:
            rec = json.load(f)
        if rec.get("source_sha256_16") == source_hash(src_path):
            return rec.get("traffic_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0, interval_ms=50):
        self.proc = None
        self.t0 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t0 = time.time()
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]), reasons=parts[4:9]))
            except ValueError:
                continue
        return rows

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names[1:], r["reasons"][1:]):
                if v.lower() in ("active", "1", "true"):
                    reasons.add(n)
        loaded = [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(value, dist, device="cuda"):
    """The slowest rank's time: every rank's timed region ends at the barrier after it."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank, ms_slowest, world_size):
    """Whole-job throughput in GB/s: every rank processed its own replica of the workload."""
    return bytes_per_rank * world_size / (ms_slowest * 1e-3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference arm)
# ---------------------------------------------------------------------------

def oracle_decode_sample(wl, k_cache, v_cache, q, k_new, v_new, rows):
    """The oracle's decode step (scatter + attention) for the given sequences,
    on a compact pool that holds only their blocks.  Returns KV bytes covered."""
    from oracle import paged_attention as pa
    ids = sorted({int(x) for r in rows for x in wl.block_tables[r] if x >= 0})
    remap = {b: i for i, b in enumerate(ids)}
    kc = k_cache[ids]
    vc = v_cache[ids]
    bt = np.full((len(rows), wl.block_tables.shape[1]), -1, dtype=np.int64)
    for i, r in enumerate(rows):
        for j, x in enumerate(wl.block_tables[r]):
            if x >= 0:
                bt[i, j] = remap[int(x)]
    lens = wl.kv_lens[rows]
    slots = pa.slot_mapping(np.ones(len(rows), np.int64), lens, bt, wl.block_size)
    kc, vc = pa.store_kvcache(kc, vc, k_new[rows], v_new[rows], slots, wl.block_size)
    pa.decode(q[rows], kc, vc, bt, lens, wl.block_size, wl.softmax_scale)
    return int(lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * 2


def cpu_inputs(wl, device_vals=None):
    """Float32 CPU copies of the workload's values (exact for bf16)."""
    if device_vals is None:
        device_vals = W.paged_values(wl, device="cpu")
    f = lambda t: t.detach().to("cpu").float().numpy()  # noqa: E731
    return (f(device_vals.k_cache), f(device_vals.v_cache), f(device_vals.q), f(device_vals.k_new),
            f(device_vals.v_new))


def time_oracle(wl, arrays, budget_s, min_rows=1):
    """Run oracle decode steps on growing prefixes of the batch until ~budget_s."""
    kc, vc, q, kn, vn = arrays
    t0 = time.perf_counter()
    bytes_done = 0
    rows_done = 0
    r = 0
    while True:
        rows = [r % wl.batch]
        bytes_done += oracle_decode_sample(wl, kc, vc, q, kn, vn, rows)
        rows_done += 1
        r += 1
        if time.perf_counter() - t0 >= budget_s and rows_done >= min_rows:
            break
    dt = time.perf_counter() - t0
    return bytes_done / dt / 1e9, rows_done, dt


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = W.decode_b64()
    arrays = cpu_inputs(wl)
    # calibrate one sequence, then size each step so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle_decode_sample(wl, *arrays, rows=[0])
    t_one = max(time.perf_counter() - t0, 1e-3)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(min(wl.batch, max(1, per_step // t_one)))
    kc, vc, q, kn, vn = arrays
    for i in range(args.warmup):
        oracle_decode_sample(wl, kc, vc, q, kn, vn, [(i * n_rows + j) % wl.batch for j in range(n_rows)])
    tot_bytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        tot_bytes += oracle_decode_sample(wl, kc, vc, q, kn, vn, [(i * n_rows + j) % wl.batch for j in range(n_rows)])
    dt = time.perf_counter() - t0
    value = tot_bytes / dt / 1e9
    threads = os.environ["OPENBLAS_NUM_THREADS"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config_dict(wl),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": int(threads), "kind": "oracle",
                         "sample": f"{n_rows} of {wl.batch} sequences per step (KV scatter + fp64 gather-then-dense "
                                   f"attention), compact pool of their blocks",
                         "host_cpus": os.cpu_count(), "affinity": _HOST_CORES},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def decode_config_dict(wl):
    return {"workload": "decode attention, one layer: batch 64, Hq 16, Hkv 8, d 128, bf16, block 256, "
                        "context U[512,4096], pool 1.25x blocks used, random block permutation",
            "batch": wl.batch, "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "kv_bytes_per_step": wl.kv_bytes_read, "seed": wl.seed,
            "l2": f"inputs larger than L2 (KV {wl.kv_bytes_read / 1e9:.2f} GB per step vs 0.13 GB L2)"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class DecodeStep:
    """Device-resident decode workload and its step (slot map + scatter + decode)."""

    def __init__(self, pkv, torch, wl, layers=1, seed_offset=0):
        self.pkv, self.torch, self.wl = pkv, torch, wl
        dev = "cuda"
        self.layers = []
        for layer in range(layers):
            v = W.paged_values(wl, device=dev, layer=layer + seed_offset)
            self.layers.append(v)
        self.block_tables = torch.from_numpy(wl.block_tables).to(dev)
        self.ctx = torch.from_numpy(wl.kv_lens).to(dev)
        self.slots = torch.empty(wl.batch, dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.layers[0].q)
        self.ws = pkv.decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim)
        self.max_ctx = int(wl.kv_lens.max())
        self.ev = None
        self.calls = [None] * layers          # prepared pkv_decode_append per layer, made on first use

    def layer(self, i, q=None, k_new=None, v_new=None, events=None):
        """One decode step of one layer: the new token's slot, its K/V write and the
        attention, fused in pkv_decode_append (split-K decode + combine launches)."""
        v = self.layers[i]
        pkv, wl = self.pkv, self.wl
        if q is not None or k_new is not None or v_new is not None:
            if events is not None:
                events[0].record()
            pkv.pkv_decode_append(q if q is not None else v.q, k_new if k_new is not None else v.k_new,
                                  v_new if v_new is not None else v.v_new, v.k_cache, v.v_cache,
                                  self.block_tables, self.ctx, self.max_ctx, wl.softmax_scale, out=self.out,
                                  slot_mapping=self.slots, workspace=self.ws)
        else:
            if self.calls[i] is None:
                self.calls[i] = pkv.DecodeAppendCall(v.q, v.k_new, v.v_new, v.k_cache, v.v_cache,
                                                     self.block_tables, self.ctx, self.max_ctx, wl.softmax_scale,
                                                     out=self.out, slot_mapping=self.slots, workspace=self.ws)
            if events is not None:
                events[0].record()
            self.calls[i]()
        if events is not None:
            events[1].record()
        return self.out

    def layer_unfused(self, i, events=None):
        """The same step through the separate calls: slot mapping, scatter, decode."""
        v = self.layers[i]
        pkv, wl = self.pkv, self.wl
        pkv.pkv_slot_mapping(self.block_tables, wl.num_blocks, wl.block_size, self.slots, context_lens=self.ctx)
        pkv.pkv_store_kvcache(v.k_new, v.v_new, self.slots, v.k_cache, v.v_cache)
        if events is not None:
            events[0].record()
        pkv.pkv_decode(v.q, v.k_cache, v.v_cache, self.block_tables, self.ctx, self.max_ctx, wl.softmax_scale,
                       out=self.out, workspace=self.ws)
        if events is not None:
            events[1].record()
        return self.out

    LAUNCHES_PER_LAYER = 2   # fused split-K decode (slot + KV write + attention), combine


HEADLINE_MIN_S = 0.5    # the K-step timed region is repeated until this much GPU time is covered


def bench_headline(args, pkv, torch, dist, ws, rank, peaks):
    wl = W.decode_b64()
    step = DecodeStep(pkv, torch, wl)
    cpu_arrays = None
    if rank == 0 and not args.no_cpu_baseline:
        v = step.layers[0]
        f = lambda t: t.detach().to("cpu").float().numpy()  # noqa: E731
        cpu_arrays = (f(v.k_cache), f(v.v_cache), f(v.q), f(v.k_new), f(v.v_new))  # before any kernel runs
    for _ in range(args.warmup):
        step.layer(0)
    torch.cuda.synchronize()
    K = args.steps
    # One timed region is K steps back to back on the launching stream, events at its two ends
    # only (an event between calls would sit between one call's combine and the next call's
    # split-K grid and stop the programmatic launch of the latter from overlapping the former).
    # A short region is repeated until HEADLINE_MIN_S of GPU time is covered, so the clocks are
    # sampled over a steady stretch; the headline is the median repeat, the spread is reported.
    t0 = time.perf_counter()
    for _ in range(K):
        step.layer(0)
    torch.cuda.synchronize()
    repeats = int(min(2000, max(1, math.ceil(HEADLINE_MIN_S / max(time.perf_counter() - t0, 1e-6)))))
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(repeats)]
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    time.sleep(0.2)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for start, end in pairs:
        start.record()
        for _ in range(K):
            step.layer(0)
        end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clock_rows = clocks.stop()
    region_ms = sorted(a.elapsed_time(b) for a, b in pairs)
    elapsed_ms = statistics.median(region_ms)
    elapsed_ms = max_over_ranks(elapsed_ms, dist)
    ms_per_step = elapsed_ms / K
    value = weak_scaling_value(wl.kv_bytes_read, ms_per_step, ws)
    hbm, _, _, peak_kind = peaks
    # a step is one pkv_decode_append call, so the call's average duration is the timed region / K
    call_mean = statistics.median(region_ms) / K
    achieved = wl.kv_bytes_read / (call_mean * 1e-3) / 1e9
    # the conservative figure: the same call bracketed by its own pair of events, one call at a
    # time (no overlap with the previous call's tail through programmatic launch)
    K_iso = max(50, K)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_iso)]
    for k in range(K_iso):
        step.layer(0, events=evs[k])
    torch.cuda.synchronize()
    call_iso = float(np.median([a.elapsed_time(b) for a, b in evs]))
    iso_gbs = wl.kv_bytes_read / (call_iso * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": profiled_traffic("decode_splitk_b64_traffic.json", DECODE_SRC),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "kernel": "pkv_decode_append call (split-K decode with the fused KV write + combine): average "
                          "duration over the timed region (CUDA events on the launching stream)",
                "algorithmic_bytes_per_launch": wl.kv_bytes_read,
                "call_ms_with_own_events": call_iso,
                "per_call": {"achieved": iso_gbs, "frac": iso_gbs / hbm,
                             "how": f"median of {K_iso} calls, each between its own pair of events (conservative)"},
                "repeats": {"regions": repeats, "steps_per_region": K,
                            "region_ms": {"min": region_ms[0], "median": statistics.median(region_ms),
                                          "max": region_ms[-1]},
                            "gbs": {"min": wl.kv_bytes_read * K / (region_ms[-1] * 1e-3) / 1e9,
                                    "median": wl.kv_bytes_read * K / (statistics.median(region_ms) * 1e-3) / 1e9,
                                    "max": wl.kv_bytes_read * K / (region_ms[0] * 1e-3) / 1e9}}}
    # the same step through the three separate calls (4 launches), for comparison
    K2 = max(10, K // 4)
    su, eu = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        step.layer_unfused(0)
    torch.cuda.synchronize()
    su.record()
    for _ in range(K2):
        step.layer_unfused(0)
    eu.record()
    torch.cuda.synchronize()
    unfused_ms = su.elapsed_time(eu) / K2
    e2e = bench_e2e(args, pkv, torch, step, dist, ws)
    res = dict(value=value, ms_per_step=ms_per_step, roofline=roofline, e2e=e2e,
               clocks=ClockSampler.summary(clock_rows), gpu_launches=K * DecodeStep.LAUNCHES_PER_LAYER,
               config=decode_config_dict(wl), call_ms=call_mean,
               unfused=dict(ms_per_step=unfused_ms, gbs=wl.kv_bytes_read / (unfused_ms * 1e-3) / 1e9,
                            launches_per_step=4, calls="pkv_slot_mapping + pkv_store_kvcache + pkv_decode"))
    return res, cpu_arrays, wl


def bench_e2e(args, pkv, torch, step, dist, ws):
    """Same step through the public API with host buffers and copies in the timed region.

    As a serving loop runs it: each step's inputs (q, the new K/V rows, block
    tables, context lengths) go up from one packed pinned buffer in a single
    copy on an upload stream, the decode runs on the compute stream, and its
    output comes back to pinned memory on a download stream; two buffer slots
    let step i+1's upload and step i's download overlap step i's compute.
    Every step's copies are inside the timed region, which ends when the last
    download has landed."""
    wl = step.wl
    v = step.layers[0]
    parts = [v.q, v.k_new, v.v_new, torch.from_numpy(wl.block_tables), torch.from_numpy(wl.kv_lens)]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    out_bytes = v.q.numel() * v.q.element_size()

    def views(buf):
        res = []
        for t, o in zip(parts, offs):
            n = t.numel() * t.element_size()
            res.append(buf[o:o + n].view(t.dtype).view(tuple(t.shape)))
        return res

    slots = []
    for _ in range(2):
        h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        for dst, src in zip(views(h_in), parts):
            dst.copy_(src.cpu())
        d_in = torch.empty(total, dtype=torch.uint8, device="cuda")
        slots.append({"h_in": h_in, "d_in": d_in, "d": views(d_in), "d_out": torch.empty_like(v.q),
                      "h_out": torch.empty(tuple(v.q.shape), dtype=v.q.dtype).pin_memory(),
                      "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event()})
    comp = torch.cuda.current_stream()
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    for sl in slots:
        sl["d_in"].copy_(sl["h_in"])
        q, kn, vn, bt, ctx = sl["d"]
        sl["call"] = pkv.DecodeAppendCall(q, kn, vn, v.k_cache, v.v_cache, bt, ctx, step.max_ctx, wl.softmax_scale,
                                          out=sl["d_out"], slot_mapping=step.slots, workspace=step.ws, stream=comp)
    torch.cuda.synchronize()
    h2d, d2h = total, out_bytes
    K = max(10, args.steps // 4)

    def one(i):
        sl = slots[i % 2]
        if i >= 2:
            up_s.wait_event(sl["done"])                 # step i-2's decode no longer reads this slot
        with torch.cuda.stream(up_s):
            sl["d_in"].copy_(sl["h_in"], non_blocking=True)
        sl["up"].record(up_s)
        comp.wait_event(sl["up"])
        if i >= 2:
            comp.wait_event(sl["down"])                 # step i-2's output has been read back
        sl["call"]()
        sl["done"].record(comp)
        down_s.wait_event(sl["done"])
        with torch.cuda.stream(down_s):
            sl["h_out"].copy_(sl["d_out"], non_blocking=True)
        sl["down"].record(down_s)

    def run(n):
        for i in range(n):
            one(i)
        for sl in slots:
            comp.wait_event(sl["down"])

    run(max(3, args.warmup))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(comp)
    up_s.wait_event(s)
    run(K)
    e.record(comp)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / K
    ms = max_over_ranks(ms, dist)
    ok = all(torch.equal(sl["h_out"], sl["d_out"].cpu()) for sl in slots)
    return {"value": weak_scaling_value(wl.kv_bytes_read, ms, ws), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": K, "copies_checked": ok,
            "pipeline": "1 packed upload + 1 download per step on their own streams, 2 buffer slots"}


class L2Flush:
    """Evict L2 between timed calls: write a buffer twice the size of L2, then read another one.

    The read pass pushes the written lines' write-backs to DRAM before the timed
    region starts, so the next call finds clean, unrelated lines in L2 and pays
    neither for its own inputs being cached nor for the flush's dirty data."""

    def __init__(self, torch, dev="cuda"):
        n = 2 * L2_BYTES // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.add_(1)
        self.r.amax()


def flush_l2(torch, flush):
    flush()


def bench_prefill(args, pkv, torch, peaks):
    wl = W.prefill_prefix()
    dev = "cuda"
    v = W.paged_values(wl, device=dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cu_q = torch.from_numpy(wl.cu_seqlens_q).to(dev)
    cu_k = torch.from_numpy(wl.cu_seqlens_k).to(dev)
    slots = torch.empty(wl.total_q, dtype=torch.int32, device=dev)
    out = torch.empty_like(v.q)
    flush = L2Flush(torch, dev)
    pairs = 0
    for ql, kl in zip(wl.q_lens.astype(np.int64), wl.kv_lens.astype(np.int64)):
        pairs += ql * (kl - ql) + ql * (ql + 1) // 2      # unmasked (query, key) pairs per head
    flops = 4 * wl.head_dim * wl.num_heads * pairs

    def step(evs=None):
        pkv.pkv_slot_mapping(bt, wl.num_blocks, wl.block_size, slots, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
        pkv.pkv_store_kvcache(v.k_new, v.v_new, slots, v.k_cache, v.v_cache)
        if evs:
            evs[0].record()
        pkv.pkv_prefill_varlen(v.q, v.k_cache, v.v_cache, cu_q, cu_k, bt, int(wl.q_lens.max()),
                               int(wl.kv_lens.max()), wl.softmax_scale, out=out)
        if evs:
            evs[1].record()

    for _ in range(max(3, args.warmup // 10)):
        step()
    K = max(10, min(200, args.steps // 10))
    step_ms, call_ms = [], []
    for _ in range(K):
        flush_l2(torch, flush)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        step((a, b))
        e.record()
        torch.cuda.synchronize()
        step_ms.append(s.elapsed_time(e))
        call_ms.append(a.elapsed_time(b))
    # the same attention on a plan made once for the batch (as every layer after the first of a
    # model's prefill step runs): pkv_prefill_plan before the loop, pkv_prefill_varlen_planned timed
    ws = pkv.pkv_prefill_plan(cu_q, cu_k, wl.total_q, int(wl.q_lens.max()), int(wl.kv_lens.max()), wl.num_heads,
                              wl.num_kv_heads, wl.head_dim, wl.block_size, bt.shape[1])
    planned_ms = []
    for i in range(K + 3):
        pkv.pkv_slot_mapping(bt, wl.num_blocks, wl.block_size, slots, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
        pkv.pkv_store_kvcache(v.k_new, v.v_new, slots, v.k_cache, v.v_cache)
        flush_l2(torch, flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pkv.pkv_prefill_varlen_planned(v.q, v.k_cache, v.v_cache, cu_q, cu_k, bt, int(wl.q_lens.max()),
                                       int(wl.kv_lens.max()), wl.softmax_scale, ws, out=out)
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            planned_ms.append(a.elapsed_time(b))
    _, bf16, bf16_sus, kind = peaks
    call = float(np.median(call_ms))
    tflops = flops / (call * 1e-3) / 1e12
    pcall = float(np.median(planned_ms))
    ptflops = flops / (pcall * 1e-3) / 1e12
    return {"workload": "varlen prefill with prefix-cache hits: 32 prompts U[100,1024], 0-2 shared 256-token blocks "
                        "per group of 4, Hq 16, Hkv 8, d 128, bf16",
            "tflops": tflops, "unit": "TFLOP/s", "algorithmic_flops": int(flops), "call_ms_median": call,
            "step_ms_median": float(np.median(step_ms)), "frac_of_bf16_peak": tflops / bf16,
            "peak": bf16, "peak_source": kind, "steps": K, "l2": "flushed between steps (256 MB write, then 256 MB clean read)",
            "total_q": wl.total_q,
            "planned": {"tflops": ptflops, "call_ms_median": pcall, "frac_of_bf16_peak": ptflops / bf16,
                        "steps": K, "how": "pkv_prefill_plan once for the batch, then pkv_prefill_varlen_planned per "
                                           "call (each layer after the first of a prefill step); L2 flushed before "
                                           "each call"}}


def bench_rope_store(args, pkv, torch, peaks):
    """RoPE fused into the KV write over the prefill workload's tokens, against the plain scatter.

    Headline figure: back-to-back calls cycling over ROPE_SETS independent copies of the inputs,
    outputs and pools (together far larger than L2), so each call's writes are pushed to DRAM by
    the calls after it, inside the timed region.  A single call after an L2 flush is reported
    beside it: its writes can still sit in L2 when its end event fires."""
    ROPE_SETS, ROUNDS = 8, 3
    wl = W.prefill_prefix()
    dev = "cuda"
    n = wl.total_q
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cu_q = torch.from_numpy(wl.cu_seqlens_q).to(dev)
    cu_k = torch.from_numpy(wl.cu_seqlens_k).to(dev)
    pos = torch.from_numpy(np.concatenate([np.arange(kl - ql, kl) for ql, kl in zip(wl.q_lens, wl.kv_lens)])
                           .astype(np.int32)).to(dev)
    sets = []
    for i in range(ROPE_SETS):
        v = W.paged_values(wl, device=dev, layer=i)
        slots = torch.empty(n, dtype=torch.int32, device=dev)
        pkv.pkv_slot_mapping(bt, wl.num_blocks, wl.block_size, slots, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
        sets.append((v, slots, torch.empty_like(v.q), pos.clone()))
    flush = L2Flush(torch, dev)
    q_row, kv_row = wl.num_heads * wl.head_dim * 2, wl.num_kv_heads * wl.head_dim * 2
    rope_bytes = n * (2 * q_row + 4 * kv_row + 8)        # q in/out, k in/out, v in/out, position, slot
    store_bytes = n * (4 * kv_row + 4)

    def rope(i):
        v, slots, q_out, p = sets[i % ROPE_SETS]
        pkv.pkv_rope_store_kvcache(v.q, v.k_new, v.v_new, p, slots, v.k_cache, v.v_cache, 1e6, q_out=q_out)

    def store(i):
        v, slots, _, _ = sets[i % ROPE_SETS]
        pkv.pkv_store_kvcache(v.k_new, v.v_new, slots, v.k_cache, v.v_cache)

    def back_to_back(fn):
        for i in range(2 * ROPE_SETS):
            fn(i)
        flush_l2(torch, flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        calls = ROUNDS * ROPE_SETS
        a.record()
        for i in range(calls):
            fn(i)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / calls

    def single(fn):
        ms = []
        for k in range(max(10, min(100, args.steps // 30))):
            flush_l2(torch, flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(k)
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return float(np.median(ms))

    rope_ms, store_ms = back_to_back(rope), back_to_back(store)
    rope_single, store_single = single(rope), single(store)
    gbs = rope_bytes / (rope_ms * 1e-3) / 1e9
    return {"workload": f"rotary embedding + KV write of the prefill workload's {n} tokens (Hq 16, Hkv 8, d 128, "
                        "base 1e6)", "gbs": gbs, "unit": "GB/s", "call_ms": rope_ms,
            "frac_of_hbm": gbs / peaks[0], "algorithmic_bytes": int(rope_bytes),
            "how": f"{ROUNDS * ROPE_SETS} calls back to back over {ROPE_SETS} independent input/output/pool sets "
                   "(writes reach DRAM inside the timed region), after an L2 flush",
            "plain_store_ms": store_ms, "plain_store_gbs": store_bytes / (store_ms * 1e-3) / 1e9,
            "single_call_after_flush": {"rope_ms_median": rope_single,
                                        "rope_gbs": rope_bytes / (rope_single * 1e-3) / 1e9,
                                        "store_ms_median": store_single,
                                        "store_gbs": store_bytes / (store_single * 1e-3) / 1e9,
                                        "note": "writes may still be in L2 when the end event fires"}}


def bench_long_decode(args, pkv, torch, peaks):
    wl = W.long_decode()
    st = DecodeStep(pkv, torch, wl)
    for _ in range(3):
        st.layer(0)
    K = max(10, min(200, args.steps // 10))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        st.layer(0)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    gbs = wl.kv_bytes_read / (ms * 1e-3) / 1e9
    res = {"workload": "long-context decode: batch 8, context U[16384,40960], pool 1400 blocks",
           "gbs": gbs, "unit": "GB/s", "call_ms": ms, "frac_of_hbm": gbs / peaks[0], "kv_bytes": wl.kv_bytes_read}
    del st
    torch.cuda.empty_cache()
    return res


def bench_decode_sweep(args, pkv, torch, peaks):
    """The fused decode step across batch sizes and context lengths (every sequence of a batch
    at the same length), each call timed cold: L2 flushed before it, events around it alone."""
    flush = L2Flush(torch)
    rows = []
    for L in (512, 4096, 32768):
        for B in (1, 4, 16, 64, 256):
            if B * L * 4096 > 16e9:
                continue
            wl = W.build_workload(f"sweep-b{B}-l{L}", np.ones(B, np.int32), np.full(B, L, np.int32),
                                  seed=3000 + B + L)
            st = DecodeStep(pkv, torch, wl)
            for _ in range(3):
                st.layer(0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(20):
                flush()
                a.record()
                st.layer(0)
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            ms = float(np.median(ts))
            rows.append({"batch": B, "context": L, "call_us": ms * 1e3, "gbs": wl.kv_bytes_read / (ms * 1e-3) / 1e9,
                         "frac_of_hbm": wl.kv_bytes_read / (ms * 1e-3) / 1e9 / peaks[0],
                         "tok_per_s_per_layer": B / (ms * 1e-3)})
            del st
            torch.cuda.empty_cache()
    return {"workload": "pkv_decode_append, batch x context grid, each sequence at the same length, "
                        "L2 flushed before every call (median of 20)", "rows": rows}


def bench_sample(args, pkv, torch, peaks):
    """The sampler alone on the full decode step's logits ([256, 151936] fp32), L2 flushed before
    each call (the logits, 156 MB, are larger than L2 anyway)."""
    s_in = W.sampler_inputs(batch=256, device="cuda")
    ids = torch.empty(256, dtype=torch.int64, device="cuda")
    flush = L2Flush(torch)
    for k in range(3):
        pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed + k, 0, out_ids=ids)
    ms = []
    for k in range(max(10, min(100, args.steps // 30))):
        flush_l2(torch, flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed + k, 0, out_ids=ids)
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    call = float(np.median(ms))
    nbytes = 256 * W.VOCAB_QWEN3 * 4
    gbs = nbytes / (call * 1e-3) / 1e9
    return {"workload": "temperature sampler on [256, 151936] fp32 logits N(0, 3^2), T in [0.5, 1]",
            "gbs": gbs, "unit": "GB/s", "call_ms_median": call, "frac_of_hbm": gbs / peaks[0],
            "algorithmic_bytes": nbytes, "l2": "flushed before every call"}


def bench_full_step(args, pkv, torch, peaks):
    wl = W.full_step()
    st = DecodeStep(pkv, torch, wl, layers=wl.num_layers)
    s_in = W.sampler_inputs(batch=wl.batch, device="cuda")
    ids = torch.empty(wl.batch, dtype=torch.int64, device="cuda")

    def step(k, evs=None):
        for layer in range(wl.num_layers):
            st.layer(layer)
        if evs:
            evs[0].record()
        pkv.pkv_sample(s_in.logits, s_in.temperatures, s_in.seed + k, 0, out_ids=ids)
        if evs:
            evs[1].record()

    for k in range(3):
        step(k)
    K = max(5, min(30, args.steps // 100))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    samp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    s.record()
    for k in range(K):
        step(k, samp[k])
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / K
    sample_ms = float(np.mean([a.elapsed_time(b) for a, b in samp]))
    graph_ms = bench_full_step_graph(pkv, torch, st, s_in, K)
    kv = wl.kv_bytes_read * wl.num_layers
    logits_bytes = wl.batch * W.VOCAB_QWEN3 * 4
    res = {"workload": "full decode step: 28 layers x (slot map + scatter + decode), batch 256, context "
                       "U[128,2048], per-layer pools, then the sampler on [256, 151936] fp32 logits",
           "tok_per_s": wl.batch / (ms * 1e-3), "step_ms": ms, "kv_gbs": (kv + logits_bytes) / (ms * 1e-3) / 1e9,
           "sampler_ms": sample_ms, "sampler_gbs": logits_bytes / (sample_ms * 1e-3) / 1e9,
           "kv_bytes_per_step": kv, "steps": K,
           "gpu_launches_per_step": wl.num_layers * DecodeStep.LAUNCHES_PER_LAYER + 1,
           "graph": {"step_ms": graph_ms, "tok_per_s": wl.batch / (graph_ms * 1e-3),
                     "how": "the step (28 x pkv_decode_append + pkv_sample_dev + noise-offset update) "
                            "captured once in a CUDA graph and replayed"}}
    del st
    torch.cuda.empty_cache()
    return res


def bench_full_step_graph(pkv, torch, st, s_in, K):
    """The full decode step captured in a CUDA graph, replayed K times."""
    wl = st.wl
    ids = torch.empty(wl.batch, dtype=torch.int64, device="cuda")
    seed_offset = torch.tensor([s_in.seed, 0], dtype=torch.int64, device="cuda")

    def step():
        for layer in range(wl.num_layers):
            st.layer(layer)
        pkv.pkv_sample_dev(s_in.logits, s_in.temperatures, seed_offset, out_ids=ids)
        seed_offset[1:].add_(wl.batch)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(K):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / K


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-secondary", action="store_true", help="headline only")
    ap.add_argument("--parts", default="prefill,long,full,rope,sample",
                    help="secondary workloads to run: any of prefill,long,full,rope,sample,sweep (sweep is opt-in)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        return run_reference(args)

    import torch
    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)
    import paged_kv_attention_29_gb300 as pkv
    pkv.load()
    peaks = load_peaks()

    head, cpu_arrays, wl = bench_headline(args, pkv, torch, dist, ws, rank, peaks)
    secondary = {"unfused_decode_step": head["unfused"]}
    parts = set() if args.no_secondary else {x.strip() for x in args.parts.split(",") if x.strip()}
    if rank == 0:
        # each part runs inside an NVTX range of its own name, so a profiler can select one
        # (ncu --nvtx --nvtx-include "full_step/")
        for key, part, fn in (("prefill", "prefill", bench_prefill), ("long", "long_decode", bench_long_decode),
                              ("full", "full_step", bench_full_step), ("rope", "rope_store", bench_rope_store),
                              ("sample", "sample", bench_sample), ("sweep", "decode_sweep", bench_decode_sweep)):
            if key in parts:
                torch.cuda.nvtx.range_push(part)
                try:
                    secondary[part] = fn(args, pkv, torch, peaks)
                finally:
                    torch.cuda.nvtx.range_pop()
    code, info = pkv.pkv_get_device_error(clear=True)
    if code:
        raise RuntimeError(f"device error {code} ({pkv.DEVERR.get(code)}), info {info}")

    cpu_baseline = None
    if rank == 0 and cpu_arrays is not None:
        gbs, rows, dt = time_oracle(wl, cpu_arrays, args.cpu_budget)
        threads = os.environ["OPENBLAS_NUM_THREADS"]
        cpu_baseline = {"value": gbs, "unit": "GB/s", "cores": int(threads), "kind": "oracle",
                        "sample": f"{rows} sequences of the batch-64 decode workload, one at a time "
                                  f"(KV scatter + fp64 gather-then-dense attention), {dt:.1f} s",
                        "host_cpus": os.cpu_count(), "affinity": _HOST_CORES,
                        "threads": f"OPENBLAS_NUM_THREADS={threads}, OMP_NUM_THREADS={os.environ['OMP_NUM_THREADS']}"}
    if dist is not None:
        dist.barrier()
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1))",
                "config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu_baseline,
                "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                "secondary": secondary}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
