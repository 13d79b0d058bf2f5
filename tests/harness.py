"""Test harness: runs a decode workload through the C ABI on the GPU and the
same calls through the CPU oracle, and collects what each side produced."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import synth
from oracle import ffn, lru, permute, records, router
from synth.configs import Workload


@dataclass
class CallOut:
    step: int
    layer: int
    status: int = 0
    ids: np.ndarray | None = None
    w: np.ndarray | None = None
    slots: np.ndarray | None = None
    perm: np.ndarray | None = None
    offsets: np.ndarray | None = None
    y: np.ndarray | None = None  # float64


@dataclass
class RunOut:
    calls: list = field(default_factory=list)
    events: list = field(default_factory=list)


def decode_calls(w: Workload, steps: int | None = None):
    return [(s, l) for s in range(steps if steps is not None else w.steps) for l in range(w.L)]


def trace_logits(w: Workload, steps: int | None = None) -> np.ndarray:
    """float32 [T, L, B, E] AR(1) logits of the workload."""
    return synth.ar1_logits(w.seed, steps if steps is not None else w.steps, w.L, w.B, w.E)


def x_f64(w: Workload, step: int, layer: int) -> np.ndarray:
    if w.wdtype == synth.WD_FP32:
        return synth.activations_f32(w.seed, step, layer, w.B, w.H).astype(np.float64)
    return synth.bf16_bits_to_f32(synth.activations_bf16(w.seed, step, layer, w.B, w.H)).astype(np.float64)


class ExpertBank:
    """Parsed float64 expert matrices, regenerated on demand from the seeded generator."""

    def __init__(self, w: Workload):
        self.w = w
        self.cache = {}

    def get(self, key: int):
        if key not in self.cache:
            rec = synth.records_array(self.w.seed, key, 1, self.w.H, self.w.I, self.w.wdtype, self.w.sigma)[0]
            self.cache[key] = records.parse(rec, self.w.H, self.w.I, self.w.wdtype)
        return self.cache[key]


def run_oracle(w: Workload, calls, logits=None, router_w=None, C=None, y_for=None, resize=None) -> RunOut:
    """Oracle side.  y_for: set of call indices whose layer output to compute (None = all).
    resize: {call index: new C} applied before that call."""
    sim = lru.CacheSim(w.L, w.E, w.C if C is None else C)
    bank = ExpertBank(w)
    out = RunOut()
    for ci, (s, l) in enumerate(calls):
        if resize and ci in resize:
            out.events += [e.as_tuple() for e in sim.resize(resize[ci])]
        x = x_f64(w, s, l)
        if w.router:
            lg = router.logits_from_router(x, router_w[l])
            assert router.topk_margin(lg, w.k) > 1e-4, f"seeded input has a near-tie at call {ci}"
        else:
            lg = logits[s, l].astype(np.float64)
        ids, wts = router.topk_softmax(lg, w.k)
        co = CallOut(s, l)
        try:
            ev, slots = sim.access(l, ids)
        except lru.CapacityError:
            co.status = 3
            out.calls.append(co)
            continue
        out.events += [e.as_tuple() for e in ev]
        co.ids, co.w, co.slots = ids, wts, slots
        co.perm, co.offsets = permute.permutation(ids, w.E)
        if y_for is None or ci in y_for:
            shared = bank.get(w.LE + l) if w.shared else None
            co.y = ffn.moe_layer(x, ids, wts, lambda e, l=l: bank.get(l * w.E + e), shared)
        out.calls.append(co)
    return out


def run_gpu(w: Workload, calls, logits=None, router_w=None, C=None, max_slots=0, resize=None, keep_y=True,
            pool=None, shared=None, inject=None, fill_mode=0, y_for=None, light=False, wait_ns=None):
    """GPU side through the C ABI; returns (RunOut, final cache state, stats).
    inject: {call index: number of fills that succeed before the injected failure}.
    y_for: call indices whose output to keep (None = all, when keep_y).
    light: only ids and slots are read back per call (full-size runs).
    wait_ns: (gate/up, W_down) fill wait limits of the layer kernel (None: the library's).
    Ends with moe_cache_sync, which must report no error."""
    import torch

    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    dev = torch.device("cuda")
    pool = runner.build_pool(w) if pool is None else pool
    shared = runner.build_shared(w) if shared is None else shared
    cache = runner.Cache(w, pool, shared, C=C, max_slots=max_slots)
    mc.moe_cache_set_trace(cache.handle, True)
    mc.moe_cache_set_fill_mode(cache.handle, fill_mode)
    if wait_ns is not None:
        mc.moe_cache_set_wait_limit_ns(cache.handle, *wait_ns)
    B, k, E, H = w.B, w.k, w.E, w.H
    xdt = runner.x_dtype(w)
    ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    wts = torch.empty((B, k), dtype=torch.float32, device=dev)
    slots = torch.empty((B, k), dtype=torch.int32, device=dev)
    perm = torch.empty((B * k,), dtype=torch.int32, device=dev)
    offs = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    lg_dev = torch.from_numpy(np.ascontiguousarray(logits)).to(dev) if logits is not None else None
    wr_dev = torch.from_numpy(router_w).to(dev) if router_w is not None else None
    y = torch.empty((B, H), dtype=xdt, device=dev)
    out = RunOut()
    stream = torch.cuda.current_stream()
    for ci, (s, l) in enumerate(calls):
        if resize and ci in resize:
            torch.cuda.synchronize()
            mc.moe_cache_resize(cache.handle, resize[ci], stream)
        if inject and ci in inject:
            mc.moe_cache_inject_fill_failure(cache.handle, inject[ci])
        x = runner.activations(w, s, l).to(dev)
        aux = {"ids": ids, "slots": slots} if light else \
            {"ids": ids, "weights": wts, "slots": slots, "perm": perm, "offsets": offs}
        lg = lg_dev[s, l] if lg_dev is not None else None
        st = cache.forward(l, x, lg, y, B, router_w=(wr_dev[l] if wr_dev is not None else None), stream=stream,
                           aux=aux)
        co = CallOut(s, l, status=st)
        if st == mc.MOE_OK:
            co.ids = ids.cpu().numpy().copy()
            co.slots = slots.cpu().numpy().copy()
            if not light:
                co.w = wts.cpu().numpy().astype(np.float64)
                co.perm = perm.cpu().numpy().copy()
                co.offsets = offs.cpu().numpy().copy()
            if keep_y and (y_for is None or ci in y_for):
                co.y = y.float().cpu().numpy().astype(np.float64)
        out.calls.append(co)
    torch.cuda.synchronize()
    st = mc.moe_cache_sync(cache.handle, stream)
    assert st == mc.MOE_OK, mc.moe_last_error()
    out.events = mc.moe_cache_trace(cache.handle)
    state = mc.moe_cache_state(cache.handle, cache.w.LE if max_slots == 0 else max_slots)
    stats = mc.moe_cache_stats(cache.handle)
    cache.close()
    return out, state, stats


def assert_layer_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    """max|y_gpu - y_ref| <= 1e-2 * max|y_ref| (bf16 compute against the float64 oracle)."""
    ref_max = float(np.max(np.abs(y_ref)))
    err = float(np.max(np.abs(y_gpu - y_ref)))
    assert err <= 1e-2 * ref_max, f"{what}: max err {err:.3e} > 1e-2 * {ref_max:.3e}"
    return err / ref_max if ref_max else 0.0
