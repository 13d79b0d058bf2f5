#!/usr/bin/env python3
"""Decode benchmark of the routed-MoE layer served from the shared GPU expert cache.

Workload (default): Qwen3.6-35B-A3B-shaped decode — 40 MoE layers, hidden
2048, per-expert SwiGLU intermediate 512, 256 experts, top-8, one shared
expert, bf16 weights ~N(0, 0.02) and bf16 activations, batch 1, AR(1) router
logits (logit_t = 0.8 logit_{t-1} + 0.6 N(0,1)), cache of 5,120 slots (50% of
the 10,240 layer-experts) backed by a 64.4 GB pinned host pool.  All inputs
are seeded and synthetic.

One step = one decode token through all 40 layers (router, cache control,
fills, expert FFN, combine).  W warm-up steps start from a cold cache; the K
timed steps continue the same trace.  Prints one JSON line.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl native|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

# the oracle leg runs on one host thread: pin BLAS before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import configs  # noqa: E402

METRIC = "MoE decode tok/s + prefill tok/s; HBM GB/s (tensor %) vs peak; cache hit rate"
FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


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
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, path, device_index=0):
        self.path = path
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


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
    """The reference arm: the CPU oracle as it stands, on host cores, on a
    bounded sample per step (4 layer calls of one token)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step_layers = 4
    T = args.warmup + args.steps
    lg = synth.ar1_logits(w.seed, max(T, 1), w.L, w.B, w.E)
    done = 0
    # warm-up steps untimed
    for s in range(args.warmup):
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
        "config": {"workload": w.name, "layers": w.L, "experts": w.E, "top_k": w.k, "hidden": w.H,
                   "intermediate": w.I, "batch": w.B, "cache_slots": w.C},
        "cpu_baseline": {"value": value, "unit": "tok/s (decode)", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step_layers} layer calls of one token per step, float64 numpy"},
        "e2e": {"value": value, "unit": "tok/s (decode)", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ native leg --
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


def run_native(args, w):
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

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
    out_dir = os.path.join(ROOT, "gpurun_out")
    os.makedirs(out_dir, exist_ok=True)

    W, K = args.warmup, args.steps
    K_e2e = K if args.e2e_steps is None else args.e2e_steps
    T = W + K + K_e2e
    t_setup = time.perf_counter()
    pool = runner.build_pool(w)
    shared = runner.build_shared(w, dev)
    S = synth.record_bytes(w.H, w.I, w.wdtype)
    lg_host = synth.ar1_logits(w.seed, T, w.L, w.B, w.E)
    x_host = torch.stack([torch.stack([runner.activations(w, s, l) for l in range(w.L)]) for s in range(T)])
    lg_dev = torch.from_numpy(lg_host).to(dev)
    x_dev = x_host.to(dev)
    y_dev = torch.empty_like(x_dev)
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE if args.fill_mode == "device" else mc.MOE_FILL_COPY)
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream()

    def step(s, x, lg, y):
        for l in range(w.L):
            st = cache.forward(l, x[s, l], lg[s, l], y[s, l], w.B, stream=stream)
            if st != mc.MOE_OK:
                raise mc.MoeError(st, "moe_layer_forward")

    for s in range(W):
        step(s, x_dev, lg_dev, y_dev)
    torch.cuda.synchronize()
    mc.moe_cache_reset_stats(cache.handle)
    mc.moe_cache_set_profiling(cache.handle, args.profile)
    clk = ClockSampler(os.path.join(out_dir, f"clocks_rank{rank}.csv"), local)
    clk.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for s in range(W, W + K):
        step(s, x_dev, lg_dev, y_dev)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = ev0.elapsed_time(ev1)
    mc.moe_cache_set_profiling(cache.handle, False)
    stats = mc.moe_cache_stats(cache.handle)
    phases = mc.moe_cache_phase_times(cache.handle) if args.profile >= 2 else None
    ms = max_over_ranks(ms, dist, dev)
    tokens = w.B * K * world
    value = tokens / (ms / 1e3)

    # end to end through the C ABI with host buffers: per step copy the
    # step's activations and logits from pinned host memory, run the layers,
    # copy the outputs back
    x_pin = x_host.pin_memory()
    lg_pin = torch.from_numpy(lg_host).pin_memory()
    y_pin = torch.empty_like(x_pin).pin_memory()
    xs_dev = torch.empty((1,) + tuple(x_dev.shape[1:]), dtype=x_dev.dtype, device=dev)
    ls_dev = torch.empty((1,) + tuple(lg_dev.shape[1:]), dtype=lg_dev.dtype, device=dev)
    ys_dev = torch.empty_like(xs_dev)
    h2d = xs_dev.numel() * xs_dev.element_size() + ls_dev.numel() * ls_dev.element_size()
    d2h = ys_dev.numel() * ys_dev.element_size()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(W + K, T):
        xs_dev.copy_(x_pin[s:s + 1], non_blocking=True)
        ls_dev.copy_(lg_pin[s:s + 1], non_blocking=True)
        step(0, xs_dev, ls_dev, ys_dev)
        y_pin[s:s + 1].copy_(ys_dev, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = w.B * K_e2e * world / (e2e_ms / 1e3) if K_e2e else None

    # ablation: the same timed steps with the other fill mechanism (copy
    # engine + stream flags vs the kernel pulling misses over the host link)
    ablation = None
    if not args.no_ablation:
        other = "device" if args.fill_mode == "copy" else "copy"
        cache.close()
        cache_b = runner.Cache(w, pool, shared)
        mc.moe_cache_set_fill_mode(cache_b.handle, mc.MOE_FILL_DEVICE if other == "device" else mc.MOE_FILL_COPY)

        def step_b(s):
            for l in range(w.L):
                st = cache_b.forward(l, x_dev[s, l], lg_dev[s, l], y_dev[s, l], w.B, stream=stream)
                if st != mc.MOE_OK:
                    raise mc.MoeError(st, "moe_layer_forward")

        for s in range(W):
            step_b(s)
        torch.cuda.synchronize()
        mc.moe_cache_reset_stats(cache_b.handle)
        mc.moe_cache_set_profiling(cache_b.handle, 1)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for s in range(W, W + K):
            step_b(s)
        a1.record(stream)
        torch.cuda.synchronize()
        ms_b = a0.elapsed_time(a1)
        mc.moe_cache_set_profiling(cache_b.handle, False)
        sb = mc.moe_cache_stats(cache_b.handle)
        ablation = {"fill_mode": other, "value": w.B * K * world / (ms_b / 1e3), "unit": "tok/s (decode)",
                    "ms_per_step": ms_b / K,
                    "hit_only_avg_launch_us": sb["hit_only_ms"] * 1e3 / max(1, sb["hit_only_timed"]),
                    "all_launches_avg_us": sb["layer_ms"] * 1e3 / max(1, sb["layer_timed"]),
                    "hit_rate": sb["hits"] / max(1, sb["hits"] + sb["misses"]),
                    "note": "same trace steps and pool, measured after the main leg in the same process"}
        cache = cache_b

    # roofline of the dominant kernel (the layer kernel): algorithmic bytes =
    # every expert record it streams once (S bytes each).  Calls with fills
    # also wait for the host link inside the kernel, so the HBM figure is
    # taken over the launches of calls without fills; the link-inclusive
    # bound covers every call.
    hit_bytes = stats["hit_only_records"] * S
    # DRAM traffic of the layer kernel from the committed ncu capture
    # (profiles/decode_layer_kernel_small_full.md: same expert shape, 8
    # resident records read 50.508 MB + wrote 0.321 MB), scaled per record to
    # this run's records per hit-only launch; valid for this expert shape only
    recs_per_launch = stats["hit_only_records"] / max(1, stats["hit_only_timed"])
    traffic = (50.508288e6 + 0.320512e6) / 8 * recs_per_launch if S == 6291456 else None
    hit_s = stats["hit_only_ms"] / 1e3
    achieved = hit_bytes / hit_s / 1e9 if hit_s > 0 else None
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    b_p = measure_link(dev, pool, S)
    hbm_s = stats["records_streamed"] * S / (peak * 1e9)
    link_s = stats["bytes_filled"] / (b_p * 1e9)
    roof_tok_s = w.B * K / max(hbm_s, link_s) if max(hbm_s, link_s) > 0 else None
    hits, misses = stats["hits"], stats["misses"]
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s (decode)", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": w.L, "experts": w.E, "top_k": w.k, "hidden": w.H,
                   "intermediate": w.I, "shared_expert": w.shared, "batch": w.B, "cache_slots": w.C,
                   "record_bytes": S, "host_pool_GB": round(w.LE * S / 1e9, 2), "fill_mode": args.fill_mode,
                   "trace": "AR(1) logits rho=0.8 sd=0.6, cold cache at warm-up start",
                   "l2": "per-step expert stream >> 129 MB L2 (no reuse across layers); no flush"},
        "hit_rate": hits / (hits + misses) if hits + misses else None,
        "routed_pair_hit_rate": stats["routed_pair_hits"] / stats["routed_pairs"] if stats["routed_pairs"] else None,
        "fill_GB_per_token": stats["bytes_filled"] / 1e9 / (w.B * K),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None, "traffic": traffic,
                     "algorithmic_bytes_per_launch": recs_per_launch * S,
                     "kernel": "layer_kernel (calls without fills)", "peak_kind": peak_kind + " hbm_gbs (copy)",
                     "launches": stats["hit_only_timed"],
                     "avg_launch_us": stats["hit_only_ms"] * 1e3 / max(1, stats["hit_only_timed"]),
                     "all_launches_avg_us": stats["layer_ms"] * 1e3 / max(1, stats["layer_timed"])},
        "link": {"B_P_GBps": b_p, "fill_bytes": stats["bytes_filled"],
                 "roofline_tok_s": roof_tok_s,
                 "frac": value / roof_tok_s if roof_tok_s else None,
                 "note": "tok/s bound = max(expert bytes / HBM peak, fill bytes / B_P) over the timed steps"},
        "e2e": {"value": e2e_value, "unit": "tok/s (decode)", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": K_e2e},
        "ablation": ablation,
        "gpu_launches": stats["layer_launches"],
        "phase_us": phases,
        "host_us_per_call": {"wait_for_miss_list": stats["host_wait_us"] / max(1, stats["calls"]),
                             "issue_fills": stats["host_issue_us"] / max(1, stats["calls"])},
        "clocks": clocks,
        "setup_s": round(setup_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = args.cpu_tokens
        calls, secs = oracle_tokens(w, lg_host, n_tok, pool_np=pool.numpy())
        cpu_v = calls / w.L * w.B / secs
        line["cpu_baseline"] = {"value": cpu_v, "unit": "tok/s (decode)", "cores": 1, "kind": "oracle",
                                "sample": f"first {n_tok} tokens x {w.L} layers of the trace, float64 numpy, "
                                          f"{secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    cache.close()
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------ prefill leg --
def run_prefill(args, w):
    """Config 4: one T-token prompt through every layer of the config-3 model
    per step, layer l+1's experts streamed host->device while layer l runs."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks, peak_kind = load_peaks()
    T, L = w.B, w.L
    t0 = time.perf_counter()
    pool = runner.build_pool(w)
    xs = np.stack([synth.activations_bf16(w.seed, 0, l, T, w.H) for l in range(L)])
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    del xs
    logits = torch.from_numpy(synth.iid_logits(w.seed, L, T, w.E)).to(dev)
    y = torch.empty_like(x)
    cache = runner.Cache(w, pool, None, C=w.C, max_tokens=1)
    setup_s = time.perf_counter() - t0
    stream = torch.cuda.current_stream()

    def step():
        st = mc.moe_prefill_stream(cache.handle, 0, L, x, logits, T, y, stream)
        if st != mc.MOE_OK:
            raise mc.MoeError(st, "moe_prefill_stream")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    mc.moe_cache_reset_stats(cache.handle)
    mc.moe_cache_set_profiling(cache.handle, 1)
    clk = ClockSampler(os.path.join(ROOT, "gpurun_out", "clocks_prefill.csv"))
    os.makedirs(os.path.join(ROOT, "gpurun_out"), exist_ok=True)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    st = mc.moe_cache_stats(cache.handle)
    S = synth.record_bytes(w.H, w.I, w.wdtype)
    b_p = measure_link(dev, pool, S)
    value = T * args.steps / (ms / 1e3)
    gemm_tflops = st["prefill_gemm_flop"] / (st["prefill_gemm_ms"] / 1e3) / 1e12 if st["prefill_gemm_ms"] else None
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
    copy_bytes = L * w.E * S * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s (prefill)", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (FP4 weights dequantised exactly)", "data": "synthetic",
        "config": {"workload": w.name, "layers": L, "experts": w.E, "top_k": w.k, "hidden": w.H,
                   "intermediate": w.I, "prompt_tokens": T, "cache_slots": w.C, "record_bytes": S,
                   "host_pool_GB": round(w.LE * S / 1e9, 1), "step": "one prompt through all layers",
                   "l2": "each layer streams 3.6 GB of experts >> 129 MB L2; no flush"},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": gemm_tflops / peak_tf if gemm_tflops else None, "traffic": None,
                     "kernel": "grouped tcgen05 GEMMs (gate/up + down)", "peak_kind": peak_kind + " bf16 sustained",
                     "gemm_ms_per_step": st["prefill_gemm_ms"] / args.steps},
        "link": {"B_P_GBps": b_p, "copy_ms_per_step": st["prefill_copy_ms"] / args.steps,
                 "compute_ms_per_step": st["prefill_compute_ms"] / args.steps,
                 "exposed_copy_ms_per_step": ms / args.steps - st["prefill_compute_ms"] / args.steps,
                 "bound_ms_per_step": max(st["prefill_copy_ms"], st["prefill_compute_ms"]) / args.steps,
                 "frac_of_bound": max(st["prefill_copy_ms"], st["prefill_compute_ms"]) / ms,
                 "stream_GBps": copy_bytes / (st["prefill_copy_ms"] / 1e3) / 1e9 if st["prefill_copy_ms"] else None},
        "gpu_launches": None, "clocks": clocks, "setup_s": round(setup_s, 1),
    }
    print(json.dumps(line), flush=True)
    cache.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="c2", choices=["c2", "c4", "small", "small-prefill"],
                    help="c2: Qwen3.6-shaped decode (default); c4: 4096-token FP4 prefill over 43 layers; "
                         "small / small-prefill: 3-layer bf16 decode / 2-layer FP4 prefill for profiler captures")
    ap.add_argument("--cpu-tokens", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", type=int, default=1, help="1: CUDA events per launch; 2: also phase timestamps")
    ap.add_argument("--no-ablation", action="store_true", help="skip the timed pass with the other fill mode")
    ap.add_argument("--fill-mode", default="copy", choices=["copy", "device"],
                    help="copy: host-issued cudaMemcpyAsync fills (default); device: the kernel pulls misses itself")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "c4":
        return run_prefill(args, configs.C4)
    if args.workload == "small-prefill":
        return run_prefill(args, configs.C4.with_(name="small-fp4-prefill-256", L=2, E=16, C=32, B=256))
    w = configs.C2 if args.workload == "c2" else configs.SMALL_BF16
    if args.impl == "reference":
        return run_reference(args, w)
    return run_native(args, w)


if __name__ == "__main__":
    sys.exit(main())
