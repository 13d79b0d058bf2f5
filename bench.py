#!/usr/bin/env python3
"""Benchmark of the routed-MoE layer served from the shared GPU expert cache.

Headline (``value``): Qwen3.6-35B-A3B-shaped decode — 40 MoE layers, hidden
2048, per-expert SwiGLU intermediate 512, 256 experts, top-8, one shared
expert, bf16 weights ~N(0, 0.02) and bf16 activations, batch 1, AR(1) router
logits (logit_t = 0.8 logit_{t-1} + 0.6 N(0,1)), cache of 5,120 slots (50% of
the 10,240 layer-experts) backed by a 64.4 GB pinned host pool, misses filled
by cudaMemcpyAsync on the copy streams.  One step = one decode token through
all 40 layers (router, cache control, fills, expert FFN, combine).  W warm-up
steps start from a cold cache; the K timed steps continue the same trace.

The same JSON line carries the other legs of the metric, each measured the
same way (one pair of CUDA events around the timed steps, per-launch
profiling off; per-launch statistics come from a separate pass):
  decode_c2_device  the headline workload with device-driven fills;
  decode_c3_b1/b8   DeepSeek-V4-Flash-shaped FP4 decode at batch 1 and 8;
  prefill_c4        a 4096-token prompt through the 43 FP4 layers;
  elastic_c5        Qwen3.6-shaped decode with the cache resized 60% -> 25%
                    -> 80% of the layer-experts at steps 512 and 1280.
All inputs are seeded and synthetic.  Prints one JSON line.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl native|reference] [--legs ...]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import configs  # noqa: E402

METRIC = "MoE decode tok/s + prefill tok/s; HBM GB/s (tensor %) vs peak; cache hit rate"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ALL_LEGS = ("c2_device", "c3", "c4", "c4_w4a4", "c5")
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : bf16 tensor rate


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0}, "fallback"


def blas_threads() -> int | None:
    """Threads numpy's BLAS uses (None when it cannot be asked)."""
    try:
        import threadpoolctl

        info = threadpoolctl.threadpool_info()
        n = [d.get("num_threads") for d in info if d.get("user_api") == "blas"]
        return int(n[0]) if n else None
    except Exception:
        for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
            if os.environ.get(v, "").isdigit():
                return int(os.environ[v])
        return None


# ------------------------------------------------------------ multi-rank --
def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (every rank gets it); x itself without a
    process group.  The timed region of each rank is reduced this way, so a
    whole-job rate divides the units all ranks processed by the slowest rank's
    time."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.dev = device_index
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.seek(0)
        lines = self.f.read().splitlines()
        self.f.close()
        sm, mx, power, reasons = [], 0.0, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ oracle leg --
def oracle_tokens(w, lg, n_tokens, layers=None, pool_np=None):
    """Run the CPU oracle (router, cache simulator, expert FFN, combine) over
    n_tokens decode tokens; returns (layer calls done, seconds)."""
    from oracle import ffn, lru, records, router

    layers = list(range(w.L)) if layers is None else layers
    sim = lru.CacheSim(w.L, w.E, w.C)
    S = synth.record_bytes(w.H, w.I, w.wdtype)

    def rec(key):
        if pool_np is not None and key < w.LE:
            return pool_np[key]
        return synth.records_array(w.seed, key, 1, w.H, w.I, w.wdtype)[0]

    # inputs the oracle reads: records (host pool bytes), x, logits
    xs = {(s, l): synth.bf16_bits_to_f32(synth.activations_bf16(w.seed, s, l, w.B, w.H)).astype(np.float64)
          for s in range(n_tokens) for l in layers}
    needed = {}
    for s in range(n_tokens):
        for l in layers:
            ids, _ = router.topk_softmax(lg[s, l].astype(np.float64), w.k)
            for e in set(ids.reshape(-1).tolist()):
                needed[l * w.E + e] = None
            if w.shared:
                needed[w.LE + l] = None
    raw = {key: rec(key) for key in needed}
    assert all(r.size == S for r in raw.values())
    t0 = time.perf_counter()
    calls = 0
    for s in range(n_tokens):
        for l in layers:
            ids, wts = router.topk_softmax(lg[s, l].astype(np.float64), w.k)
            sim.access(l, ids)
            sh = records.parse(raw[w.LE + l], w.H, w.I, w.wdtype) if w.shared else None
            ffn.moe_layer(xs[(s, l)], ids, wts, lambda e, l=l: records.parse(raw[l * w.E + e], w.H, w.I, w.wdtype), sh)
            calls += 1
    return calls, time.perf_counter() - t0


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, on the host cores, on a
    bounded sample per step (4 layer calls of one token)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step_layers = 4
    T = args.warmup + args.steps
    lg = synth.ar1_logits(w.seed, max(T, 1), w.L, w.B, w.E)
    done = 0
    for s in range(args.warmup):  # warm-up steps, untimed
        oracle_tokens(w, lg[s:s + 1], 1, layers=[(s * per_step_layers + i) % w.L for i in range(per_step_layers)])
    secs = 0.0
    for s in range(args.warmup, T):
        c, dt = oracle_tokens(w, lg[s:s + 1], 1, layers=[(s * per_step_layers + i) % w.L for i in range(per_step_layers)])
        done += c
        secs += dt
    tokens = done / w.L * w.B
    value = tokens / secs if secs > 0 else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s (decode)", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(w),
        "cpu_baseline": {"value": value, "unit": "tok/s (decode)", "cores": os.cpu_count(),
                         "blas_threads": blas_threads(), "kind": "oracle",
                         "sample": f"{per_step_layers} layer calls of one token per step, float64 numpy"},
        "e2e": {"value": value, "unit": "tok/s (decode)", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ native legs --
def decode_config(w):
    return {"workload": w.name, "layers": w.L, "experts": w.E, "top_k": w.k, "hidden": w.H, "intermediate": w.I,
            "shared_expert": w.shared, "batch": w.B, "cache_slots": w.C,
            "weights": synth.WD_NAMES[w.wdtype] + (" (e2m1 + e4m3 per 16)" if w.wdtype == synth.WD_FP4 else ""),
            "record_bytes": synth.record_bytes(w.H, w.I, w.wdtype),
            "host_pool_GB": round(w.LE * synth.record_bytes(w.H, w.I, w.wdtype) / 1e9, 2),
            "trace": "AR(1) logits rho=0.8 sd=0.6 per (layer, sequence, expert), cold cache at warm-up start",
            "l2": "per-step expert stream >> 129 MB L2 (no reuse across layers); no flush"}


def touch_pool(dev, pool, chunk=1 << 30):
    """Copy the whole pinned pool to the device once, 1 GiB at a time, before
    anything is timed, so that no timed pass pays the first DMA access to a
    host page (on a C2C-attached host that first access is several times
    slower than the next ones).  Returns the GB/s of this first sweep."""
    import torch

    flat = pool.view(-1)
    dst = torch.empty(min(chunk, flat.numel()), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for a in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - a)
        dst[:n].copy_(flat[a:a + n], non_blocking=True)
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    del dst
    return flat.numel() / secs / 1e9


def measure_link(dev, pool, S, n=96):
    """B_P: sustained host->device bandwidth of back-to-back cudaMemcpyAsync of
    expert records spread evenly over the whole pinned pool, GB/s (the link
    rate varies across the pool's pages, so one record is not representative)."""
    import torch

    dst = torch.empty(S, dtype=torch.uint8, device=dev)
    rows = [(r * pool.shape[0]) // n for r in range(n)]
    dst.copy_(pool[rows[0]], non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for r in rows:
        dst.copy_(pool[r], non_blocking=True)
    b.record()
    b.synchronize()
    return n * S / (a.elapsed_time(b) / 1e3) / 1e9


class DecodeInputs:
    """Pinned pool, shared experts, logits and activations of a decode workload."""

    def __init__(self, w, T, dev, pool=None, x_from_synth=True):
        import torch

        from expert_cache_serving_gb300 import runner

        t0 = time.perf_counter()
        self.w, self.T, self.dev = w, T, dev
        self.pool = runner.build_pool(w) if pool is None else pool
        self.shared = runner.build_shared(w, dev)
        self.S = synth.record_bytes(w.H, w.I, w.wdtype)
        self.lg_host = synth.ar1_logits(w.seed, T, w.L, w.B, w.E)
        if x_from_synth:
            self.x_host = torch.stack([torch.stack([runner.activations(w, s, l) for l in range(w.L)])
                                       for s in range(T)])
        else:  # long traces: seeded N(0,1) activations drawn on the host by torch
            g = torch.Generator().manual_seed(w.seed)
            self.x_host = torch.randn((T, w.L, w.B, w.H), generator=g).to(runner.x_dtype(w))
        self.lg_dev = torch.from_numpy(self.lg_host).to(dev)
        self.x_dev = self.x_host.to(dev)
        self.y_dev = torch.empty_like(self.x_dev[0])
        self.setup_s = time.perf_counter() - t0


def decode_pass(inp, W, K, fill_mode, profile=0, host_io=False, resize=None, max_slots=0):
    """One fresh cache; W untimed warm-up steps from cold, then K steps timed
    with one pair of CUDA events on the launching stream (per-launch events
    only when profile > 0).  host_io: every timed step copies its activations
    and logits from pinned host memory and its outputs back (end to end).
    resize: {step: slots}, applied at the safe point before that step; the
    phases between resizes are timed separately.  Returns a dict."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w, dev = inp.w, inp.dev
    stream = torch.cuda.current_stream()
    cache = runner.Cache(w, inp.pool, inp.shared, max_slots=max_slots)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE if fill_mode == "device" else mc.MOE_FILL_COPY)
    y = inp.y_dev

    def step(s, x, lg):
        for l in range(w.L):
            st = cache.forward(l, x[l], lg[l], y[l], w.B, stream=stream)
            if st != mc.MOE_OK:
                raise mc.MoeError(st, "moe_layer_forward")

    for s in range(W):
        step(s, inp.x_dev[s], inp.lg_dev[s])
    torch.cuda.synchronize()
    mc.check(mc.moe_cache_sync(cache.handle, stream), "moe_cache_sync")
    mc.moe_cache_reset_stats(cache.handle)
    mc.moe_cache_set_profiling(cache.handle, profile)
    h2d = d2h = 0
    if host_io:
        x_pin = inp.x_host.pin_memory()
        lg_pin = torch.from_numpy(inp.lg_host).pin_memory()
        y_pin = torch.empty_like(x_pin[:1]).pin_memory()
        xs = torch.empty_like(inp.x_dev[0])
        ls = torch.empty_like(inp.lg_dev[0])
        h2d = xs.numel() * xs.element_size() + ls.numel() * ls.element_size()
        d2h = y.numel() * y.element_size()
    bounds = sorted(set([W] + [s for s in (resize or {}) if W < s < W + K] + [W + K]))
    phases = []
    clk = ClockSampler(dev.index or 0).start()
    for a, b in zip(bounds, bounds[1:]):
        resize_ms = None
        if resize and a in resize and a > W:
            t0 = time.perf_counter()
            torch.cuda.synchronize()
            mc.check(mc.moe_cache_sync(cache.handle, stream), "moe_cache_sync")
            mc.moe_cache_resize(cache.handle, resize[a], stream)
            torch.cuda.synchronize()
            resize_ms = (time.perf_counter() - t0) * 1e3
            st_r = mc.moe_cache_stats(cache.handle)  # counters since the previous phase's reset: this resize only
            resize_counts = {"moves": st_r["resize_moves"], "evictions": st_r["resize_evictions"]}
        else:
            resize_counts = None
        mc.moe_cache_reset_stats(cache.handle)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(a, b):
            if host_io:
                xs.copy_(x_pin[s], non_blocking=True)
                ls.copy_(lg_pin[s], non_blocking=True)
                step(s, xs, ls)
                y_pin[0].copy_(y, non_blocking=True)
            else:
                step(s, inp.x_dev[s], inp.lg_dev[s])
        e1.record(stream)
        torch.cuda.synchronize()
        mc.check(mc.moe_cache_sync(cache.handle, stream), "moe_cache_sync")
        ms = e0.elapsed_time(e1)
        st = mc.moe_cache_stats(cache.handle)
        phases.append({"steps": [a, b], "ms": ms, "stats": st, "resize_ms": resize_ms, "resize": resize_counts,
                       "slots": mc.moe_cache_state(cache.handle, 0)[2]})
    clocks = clk.stop()
    mc.moe_cache_set_profiling(cache.handle, 0)
    pt = mc.moe_cache_phase_times(cache.handle) if profile >= 2 else None
    cache.close()
    ms = sum(p["ms"] for p in phases)
    tot = {}
    for p in phases:
        for k_, v in p["stats"].items():
            tot[k_] = tot.get(k_, 0) + v
    return {"ms": ms, "stats": tot, "phases": phases, "clocks": clocks, "h2d": h2d, "d2h": d2h, "phase_us": pt}


def replay_pass(inp, W, K, fill_mode="device"):
    """The layer kernel's steady state on calls without fills: after W warm-up
    steps, step W-1 (whose experts are all resident now) is replayed K times,
    timed with one pair of CUDA events (launches back to back, nothing
    between them).  Returns (ms per launch, records per launch)."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = inp.w
    stream = torch.cuda.current_stream()
    cache = runner.Cache(w, inp.pool, inp.shared)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE if fill_mode == "device" else mc.MOE_FILL_COPY)
    y = inp.y_dev

    def step(s):
        for l in range(w.L):
            st = cache.forward(l, inp.x_dev[s][l], inp.lg_dev[s][l], y[l], w.B, stream=stream)
            if st != mc.MOE_OK:
                raise mc.MoeError(st, "moe_layer_forward")

    for s in range(W):
        step(s)
    step(W - 1)
    torch.cuda.synchronize()
    mc.check(mc.moe_cache_sync(cache.handle, stream), "moe_cache_sync")
    mc.moe_cache_reset_stats(cache.handle)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step(W - 1)
    e1.record(stream)
    torch.cuda.synchronize()
    mc.check(mc.moe_cache_sync(cache.handle, stream), "moe_cache_sync")
    st = mc.moe_cache_stats(cache.handle)
    cache.close()
    assert st["misses"] == 0, "the replayed step must hit everywhere"
    launches = st["layer_launches"]
    return e0.elapsed_time(e1) / launches, st["records_streamed"] / launches


def hit_rate(st):
    return st["hits"] / (st["hits"] + st["misses"]) if st["hits"] + st["misses"] else None


def read_ceiling(nbytes, peak):
    """HBM read rate of a kernel that does nothing but read the same bytes per
    launch (moe_measure_read_rate: the layer kernel's 16-byte evict-first
    loads on every SM, buffers rotated so that no launch finds its bytes in
    L2): the practical ceiling for one layer call of that size."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc

    nbytes = int(nbytes) // 16 * 16
    n_bufs = max(2, min(16, (2 << 30) // max(nbytes, 1)))
    buf = torch.empty(n_bufs * nbytes, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    reps = 3 * n_bufs
    gbps = mc.moe_measure_read_rate(buf, nbytes, n_bufs, reps, torch.cuda.current_stream())
    del buf
    return {"GBps": gbps, "frac_of_peak": gbps / peak, "bytes_per_launch": nbytes, "launches": reps,
            "kernel": "reads only (moe_measure_read_rate), one 512-thread CTA per SM, rotating buffers"}


def kernel_roofline(inp, W, K, peak, prof_stats=None):
    """Layer-kernel HBM roofline: algorithmic bytes per launch (records
    streamed x record bytes) over the average launch time of calls without
    fills, from a replay of one warmed step (launches back to back, one event
    pair); the per-launch CUDA-event times of a profiled pass are added for
    reference (events between launches keep them from overlapping)."""
    ms, recs = replay_pass(inp, W, K)
    achieved = recs * inp.S / (ms / 1e3) / 1e9
    out = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
           "traffic": None, "algorithmic_bytes_per_launch": recs * inp.S, "avg_launch_us": ms * 1e3,
           "launches": K * inp.w.L,
           "kernel": "layer_kernel, calls without fills: one warmed step replayed K times, device-fill mode"}
    ceil = read_ceiling(recs * inp.S, peak)
    out["read_ceiling"] = ceil
    out["frac_of_read_ceiling"] = achieved / ceil["GBps"] if ceil["GBps"] else None
    if prof_stats is not None:
        n = prof_stats["hit_only_timed"]
        out["profiled_hit_only_avg_us"] = prof_stats["hit_only_ms"] * 1e3 / n if n else None
        out["profiled_all_launches_avg_us"] = prof_stats["layer_ms"] * 1e3 / max(1, prof_stats["layer_timed"])
    return out


def decode_leg(inp, W, K, peak, b_p, fill_mode="copy", profile=True):
    """Timed pass (profiling off) plus a profiled pass for the kernel roofline."""
    w = inp.w
    decode_pass(inp, W, K, fill_mode)  # untimed first pass (see run_native)
    main = decode_pass(inp, W, K, fill_mode)
    st = main["stats"]
    value = w.B * K / (main["ms"] / 1e3)
    hbm_s = st["records_streamed"] * inp.S / (peak * 1e9)
    link_s = st["bytes_filled"] / (b_p * 1e9)
    roof = w.B * K / max(hbm_s, link_s) if max(hbm_s, link_s) > 0 else None
    out = {"value": value, "unit": "tok/s (decode)", "ms_per_step": main["ms"] / K, "steps": K, "warmup": W,
           "fill_mode": fill_mode, "hit_rate": hit_rate(st),
           "hit_rate_note": f"over the {K} timed steps after {W} warm-up steps from a cold cache",
           "routed_pair_hit_rate": st["routed_pair_hits"] / st["routed_pairs"] if st["routed_pairs"] else None,
           "fill_GB_per_token": st["bytes_filled"] / 1e9 / (w.B * K),
           "link": {"B_P_GBps": b_p, "roofline_tok_s": roof, "frac": value / roof if roof else None,
                    "note": "bound = max(expert bytes / HBM peak, fill bytes / B_P) over the timed steps"},
           "deferred_calls": st["deferred_calls"], "gpu_launches": st["layer_launches"] + st["finish_launches"],
           "host_us_per_call": {"wait_for_miss_list": st["host_wait_us"] / max(1, st["calls"]),
                                "issue_fills": st["host_issue_us"] / max(1, st["calls"])},
           "clocks": main["clocks"]}
    if profile:
        prof = decode_pass(inp, W, K, "device", profile=1)
        out["roofline"] = kernel_roofline(inp, W, K, peak, prof["stats"])
    return out, main


def prefill_leg(w, pool, dev, W, K, peaks, peak_kind, w4a4=False, hbm_peak=FALLBACK_HBM_GBS):
    """Config 4: one T-token prompt through every layer of the FP4 model per
    step, layer l+1's experts streamed host->device while layer l runs.
    w4a4: activations quantised to FP4 and block-scaled FP4 x FP4 GEMMs."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    T, L = w.B, w.L
    xs = np.stack([synth.activations_bf16(w.seed, 0, l, T, w.H) for l in range(L)])
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    del xs
    logits = torch.from_numpy(synth.iid_logits(w.seed, L, T, w.E)).to(dev)
    y = torch.empty_like(x)
    cache = runner.Cache(w, pool, None, C=w.C, max_tokens=1)
    if w4a4:
        mc.moe_cache_set_prefill_precision(cache.handle, mc.MOE_PREFILL_W4A4)
    stream = torch.cuda.current_stream()

    def step():
        st = mc.moe_prefill_stream(cache.handle, 0, L, x, logits, T, y, stream)
        if st != mc.MOE_OK:
            raise mc.MoeError(st, "moe_prefill_stream")

    def timed(n, profile):
        mc.moe_cache_reset_stats(cache.handle)
        mc.moe_cache_set_profiling(cache.handle, profile)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        mc.moe_cache_set_profiling(cache.handle, 0)
        return e0.elapsed_time(e1), mc.moe_cache_stats(cache.handle)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(dev.index or 0).start()
    ms, _ = timed(K, 0)
    clocks = clk.stop()
    pms, st = timed(1, 1)
    cache.close()
    S = synth.record_bytes(w.H, w.I, w.wdtype)
    value = T * K / (ms / 1e3)
    gemm_tflops = st["prefill_gemm_flop"] / (st["prefill_gemm_ms"] / 1e3) / 1e12 if st["prefill_gemm_ms"] else None
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)))
    copy_bytes = L * w.E * S
    roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_tf, "unit": "TFLOP/s",
            "frac": gemm_tflops / peak_tf if gemm_tflops else None, "traffic": None,
            "kernel": "grouped tcgen05 GEMMs (gate/up + down), weights resident in the layer buffer",
            "peak_kind": peak_kind + " bf16 sustained (f16 dense rate is the same)",
            "gemm_ms_per_step": st["prefill_gemm_ms"], "flop_per_step": st["prefill_gemm_flop"]}
    dtype = "f16 operands (FP4 weights expanded exactly), fp32 accumulation"
    if w4a4:
        # per layer: every expert's weights once, the quantised activations and
        # SwiGLU output once each way, the float32 down-GEMM rows written once
        pairs = T * w.k + (T if w.shared else 0)
        gemm_bytes = L * (w.E * S + pairs * (w.H + 2 * w.I) * 9 / 16 + pairs * w.H * 4)
        fp4_peak = peak_tf * FP4_OVER_BF16
        t = st["prefill_gemm_ms"] / 1e3 if st["prefill_gemm_ms"] else None
        gbps = gemm_bytes / t / 1e9 if t else None
        roof = {"bound": "hbm", "achieved": gbps, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbps / hbm_peak if gbps else None, "traffic": None,
                "algorithmic_bytes_per_step": gemm_bytes,
                "kernel": "block-scaled FP4 x FP4 tcgen05 GEMMs (kind::mxf4nvf4), weights resident in the layer buffer",
                "peak_kind": peak_kind + " hbm_gbs (copy)",
                "tensor": {"achieved_tflops": gemm_tflops, "peak_tflops": fp4_peak,
                           "frac": gemm_tflops / fp4_peak if gemm_tflops else None,
                           "peak_kind": peak_kind + " bf16 sustained x 6 (nominal FP4 : bf16 dense ratio)"},
                "gemm_ms_per_step": st["prefill_gemm_ms"], "flop_per_step": st["prefill_gemm_flop"],
                "note": "at ~96 rows per expert every weight byte feeds ~340 flop, below the FP4 ridge (~1,500 flop per byte): "
                        "the GEMMs are bound by streaming the weights from HBM"}
        dtype = "e2m1 x e2m1 with e4m3 block scales (activations quantised), fp32 accumulation"
    return {
        "value": value, "unit": "tok/s (prefill)", "ms_per_step": ms / K, "steps": K, "warmup": W,
        "dtype": dtype,
        "config": {"workload": w.name, "layers": L, "experts": w.E, "top_k": w.k, "hidden": w.H,
                   "intermediate": w.I, "prompt_tokens": T, "cache_slots": w.C, "record_bytes": S,
                   "step": "one prompt through all layers", "logits": "i.i.d. N(0,1) per (token, layer, expert)",
                   "l2": "each layer streams 3.6 GB of experts >> 129 MB L2; no flush"},
        "roofline": roof,
        "link": {"copy_ms_per_step": st["prefill_copy_ms"], "compute_ms_per_step": st["prefill_compute_ms"],
                 "profiled_step_ms": pms,
                 "exposed_copy_ms_per_step": max(0.0, ms / K - st["prefill_compute_ms"]),
                 "bound_ms_per_step": max(st["prefill_copy_ms"], st["prefill_compute_ms"]),
                 "frac_of_bound": max(st["prefill_copy_ms"], st["prefill_compute_ms"]) / (ms / K),
                 "stream_GBps": copy_bytes / (st["prefill_copy_ms"] / 1e3) / 1e9 if st["prefill_copy_ms"] else None,
                 "note": "copy/compute split from a separate profiled step"},
        "clocks": clocks,
    }


def elastic_leg(w, dev, batches, fill_mode="copy"):
    """Config 5: the cache budget resized 60% -> 25% -> 80% at fixed safe-point
    steps; hit rate and tok/s per phase, the moves, and the host pool's
    address and checksum before and after."""
    import torch

    out = {"fill_mode": fill_mode, "schedule": [[s, c] for s, c in w.resize], "initial_slots": w.C, "batches": {}}
    pool = None
    for B in batches:
        wb = w.with_(B=B)
        inp = DecodeInputs(wb, wb.steps, dev, pool=pool, x_from_synth=False)
        if pool is None:
            touch_pool(dev, inp.pool)
        pool = inp.pool
        ptr = pool.data_ptr()
        digest = hashlib.blake2b(pool[::997].numpy().tobytes(), digest_size=16).hexdigest()
        res = decode_pass(inp, 0, wb.steps, fill_mode, resize=dict(wb.resize), max_slots=wb.LE)
        phases = []
        for p in res["phases"]:
            st = p["stats"]
            n = p["steps"][1] - p["steps"][0]
            phases.append({"steps": p["steps"], "slots": p["slots"], "tok_s": B * n / (p["ms"] / 1e3),
                           "hit_rate": hit_rate(st), "misses": st["misses"], "evictions": st["evictions"],
                           "resize_moves": (p["resize"] or {}).get("moves", 0),
                           "resize_evictions": (p["resize"] or {}).get("evictions", 0),
                           "resize_ms": p["resize_ms"]})
        after = hashlib.blake2b(pool[::997].numpy().tobytes(), digest_size=16).hexdigest()
        out["batches"][str(B)] = {"phases": phases, "tok_s": B * wb.steps / (res["ms"] / 1e3),
                                  "pool_unchanged": after == digest and pool.data_ptr() == ptr,
                                  "clocks": res["clocks"]}
        del inp, res
    out["note"] = ("whole 2048-step trace from a cold cache; resize time (a synchronising safe point) is "
                   "reported per phase and excluded from the phase's tok/s")
    torch.cuda.empty_cache()
    return out


def run_native(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    W, K = args.warmup, args.steps
    legs = set(ALL_LEGS if args.legs == "all" else [x for x in args.legs.split(",") if x])
    t_all = time.perf_counter()

    # ---- headline: config 2, copy-mode fills ---------------------------------------
    w = {"c2": configs.C2, "small": configs.SMALL_BF16,
         "small-fp4": configs.SMALL_FP4.with_(name="small-fp4-L2-E16-k6", C=16, steps=W + K)}[args.workload]
    inp = DecodeInputs(w, W + K, dev)
    first_touch = touch_pool(dev, inp.pool)
    b_p = measure_link(dev, inp.pool, inp.S)
    # one untimed pass first: the first cache created in a process runs its
    # first steps slower (first use of freshly mapped slot memory, host page
    # translations), which is setup, not per-step work
    prime = decode_pass(inp, W, K, "copy")
    if dist:
        dist.barrier()
    head = decode_pass(inp, W, K, "copy")
    ms = max_over_ranks(head["ms"], dist, dev)
    value = w.B * K * world / (ms / 1e3)
    if dist:
        dist.barrier()
    e2e = decode_pass(inp, W, K, "copy", host_io=True)
    e2e_ms = max_over_ranks(e2e["ms"], dist, dev)
    st = head["stats"]
    prof = decode_pass(inp, W, K, "device", profile=2 if args.profile >= 2 else 1)
    hbm_s = st["records_streamed"] * inp.S / (hbm_peak * 1e9)
    link_s = st["bytes_filled"] / (b_p * 1e9)
    roof_tok_s = w.B * K / max(hbm_s, link_s)
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s (decode)", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(decode_config(w), fill_mode="copy"),
        "hit_rate": hit_rate(st),
        "hit_rate_note": f"distinct (call, expert) accesses over the {K} timed steps, after {W} warm-up steps "
                         f"from a cold cache",
        "routed_pair_hit_rate": st["routed_pair_hits"] / st["routed_pairs"] if st["routed_pairs"] else None,
        "fill_GB_per_token": st["bytes_filled"] / 1e9 / (w.B * K),
        "roofline": dict(kernel_roofline(inp, W, K, hbm_peak, prof["stats"]), peak_kind=peak_kind + " hbm_gbs (copy)"),
        "link": {"B_P_GBps": b_p, "pool_first_touch_GBps": first_touch, "fill_bytes": st["bytes_filled"],
                 "roofline_tok_s": roof_tok_s,
                 "frac": value / world / roof_tok_s,
                 "note": "tok/s bound = max(expert bytes / HBM peak, fill bytes / B_P) over the timed steps"},
        "e2e": {"value": w.B * K * world / (e2e_ms / 1e3), "unit": "tok/s (decode)",
                "h2d_bytes_per_step": e2e["h2d"] * w.L, "d2h_bytes_per_step": e2e["d2h"] * w.L, "steps": K,
                "note": "same trace steps and cache history as value; per step the activations and logits of "
                        "every layer are copied from pinned host memory and the outputs back"},
        "first_pass_tok_s": w.B * K / (prime["ms"] / 1e3),
        "gpu_launches": st["layer_launches"] + st["finish_launches"],
        "pdl_launches": st["pdl_launches"],
        "deferred_calls": st["deferred_calls"],
        "host_us_per_call": {"wait_for_miss_list": st["host_wait_us"] / max(1, st["calls"]),
                             "issue_fills": st["host_issue_us"] / max(1, st["calls"])},
        "phase_us": prof["phase_us"],
        "clocks": head["clocks"],
        "legs": {},
    }
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = args.cpu_tokens
        calls, secs = oracle_tokens(w, inp.lg_host, n_tok, pool_np=inp.pool.numpy())
        line["cpu_baseline"] = {"value": calls / w.L * w.B / secs, "unit": "tok/s (decode)",
                                "cores": os.cpu_count(), "blas_threads": blas_threads(), "kind": "oracle",
                                "sample": f"first {n_tok} tokens x {w.L} layers of the trace, float64 numpy, "
                                          f"{secs:.1f} s"}
    if "c2_device" in legs:
        dev_leg, _ = decode_leg(inp, W, K, hbm_peak, b_p, fill_mode="device", profile=False)
        line["legs"]["decode_c2_device"] = dev_leg
    del inp
    torch.cuda.empty_cache()

    # ---- configs 3 and 4: the FP4 model -------------------------------------------
    if "c3" in legs or "c4" in legs or "c4_w4a4" in legs:
        from expert_cache_serving_gb300 import runner

        pool3 = runner.build_pool(configs.C3)
        S3 = synth.record_bytes(configs.C3.H, configs.C3.I, configs.C3.wdtype)
        touch_pool(dev, pool3)
        b_p3 = measure_link(dev, pool3, S3)
        if "c3" in legs:
            for B in (1, 8):
                w3 = configs.C3.with_(B=B, name=configs.C3.name if B == 1 else configs.C3_B8.name)
                inp3 = DecodeInputs(w3, W + K, dev, pool=pool3)
                leg, _ = decode_leg(inp3, W, K, hbm_peak, b_p3)
                leg["config"] = decode_config(w3)
                line["legs"][f"decode_c3_b{B}"] = leg
                del inp3
                torch.cuda.empty_cache()
        if "c4" in legs:
            w4 = configs.C4
            leg = prefill_leg(w4, pool3, dev, args.prefill_warmup, args.prefill_steps, peaks, peak_kind)
            leg["config"]["weights"] = "the config-3 model's pool (seed 3); prompt activations and logits seed 4"
            leg["link"]["B_P_GBps"] = b_p3
            line["legs"]["prefill_c4"] = leg
        if "c4_w4a4" in legs:
            leg = prefill_leg(configs.C4, pool3, dev, args.prefill_warmup, args.prefill_steps, peaks, peak_kind,
                              w4a4=True, hbm_peak=hbm_peak)
            leg["config"]["weights"] = "the config-3 model's pool (seed 3); prompt activations and logits seed 4"
            leg["link"]["B_P_GBps"] = b_p3
            line["legs"]["prefill_c4_w4a4"] = leg
        del pool3
        torch.cuda.empty_cache()

    # ---- config 5: elastic resize --------------------------------------------------
    if "c5" in legs:
        bs = [int(b) for b in args.elastic_batches.split(",") if b]
        line["legs"]["elastic_c5"] = elastic_leg(configs.C5, dev, bs)

    line["wall_s"] = round(time.perf_counter() - t_all, 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_prefill_only(args):
    """The prefill leg alone, printed as its own line (profiler captures)."""
    import torch

    from expert_cache_serving_gb300 import runner

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks, peak_kind = load_peaks()
    full = args.workload.startswith("c4")
    w = configs.C4 if full else configs.C4.with_(name="small-fp4-prefill-256", L=2, E=16, C=32, B=256)
    pool = runner.build_pool(configs.C3 if full else w)
    touch_pool(dev, pool)
    leg = prefill_leg(w, pool, dev, args.warmup, args.steps, peaks, peak_kind, w4a4=args.workload.endswith("w4a4"),
                      hbm_peak=float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)))
    line = dict(leg, metric=METRIC, n_gpus=1, higher_is_better=True, scaling="weak", vs_baseline=None,
                data="synthetic")
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="c2",
                    choices=["c2", "small", "small-fp4", "c4", "small-prefill", "c4-w4a4", "small-prefill-w4a4"],
                    help="c2: the full benchmark (default); small / small-fp4: a 3-layer bf16 or 2-layer FP4 "
                         "(config-3 shapes) decode headline for profiler captures; c4 / small-prefill: only the prefill leg, at full size or on 2 layers of "
                         "16 experts with 256 tokens (profiler captures); -w4a4: the same with FP4 x FP4 GEMMs")
    ap.add_argument("--legs", default="all",
                    help="comma list of extra legs: c2_device, c3, c4, c4_w4a4, c5 ('all' default, '' for none)")
    ap.add_argument("--prefill-steps", type=int, default=3)
    ap.add_argument("--prefill-warmup", type=int, default=2)
    ap.add_argument("--elastic-batches", default="1,4")
    ap.add_argument("--cpu-tokens", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", type=int, default=1, help="2: also record phase timestamps in the profiled pass")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, configs.C2)
    if args.workload.startswith("c4") or args.workload.startswith("small-prefill"):
        return run_prefill_only(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
