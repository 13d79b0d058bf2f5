"""GPU parity of moe_prefill_stream (full-layer double buffering, grouped
tcgen05 GEMMs) against the CPU oracle, through the C ABI.

Layer outputs within max|err| <= 1e-2 * max|ref|; the cache keeps working for
decode afterwards (the two buffers' slots are emptied, every other slot is
untouched), checked event for event against the oracle simulator.
"""
import numpy as np
import pytest

import synth
from oracle import ffn, lru, router
from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def prefill_inputs(w, T, n_layers):
    xs = np.stack([synth.activations_bf16(w.seed + 100, 0, l, T, w.H) for l in range(n_layers)])
    lg = synth.iid_logits(w.seed, n_layers, T, w.E)
    return xs, lg


def oracle_prefill(w, xs, lg, layers, bank):
    out = []
    for li, l in enumerate(layers):
        x = synth.bf16_bits_to_f32(xs[li]).astype(np.float64)
        ids, wts = router.topk_softmax(lg[li].astype(np.float64), w.k)
        shared = bank.get(w.LE + l) if w.shared else None
        out.append(ffn.moe_layer(x, ids, wts, lambda e, l=l: bank.get(l * w.E + e), shared))
    return out


def run_prefill(w, T, layers, C, pool=None, shared=None, profile=False):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    dev = torch.device("cuda")
    pool = runner.build_pool(w) if pool is None else pool
    shared = runner.build_shared(w) if shared is None else shared
    cache = runner.Cache(w, pool, shared, C=C)
    if profile:
        mc.moe_cache_set_profiling(cache.handle, 1)
    xs, lg = prefill_inputs(w, T, len(layers))
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(lg).to(dev)
    y = torch.empty_like(x)
    st = mc.moe_prefill_stream(cache.handle, layers[0], layers[-1] + 1, x, logits, T, y,
                               torch.cuda.current_stream())
    assert st == mc.MOE_OK, mc.moe_last_error()
    torch.cuda.synchronize()
    return cache, xs, lg, y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T", [200, 333])
def test_prefill_bf16_shared_parity(T):
    w = configs.SMALL_BF16.with_(C=70)
    layers = [0, 1, 2]
    cache, xs, lg, y = run_prefill(w, T, layers, C=70)
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"prefill layer {layers[li]}")
    cache.close()


def test_prefill_fp4_full_shape_parity():
    w = configs.SMALL_FP4.with_(C=32)
    layers = [0, 1]
    cache, xs, lg, y = run_prefill(w, 160, layers, C=32)
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"prefill layer {layers[li]}")
    cache.close()


def test_prefill_needs_two_full_layer_buffers():
    from expert_cache_serving_gb300 import moecache as mc

    w = configs.SMALL_BF16
    with pytest.raises(AssertionError):
        run_prefill(w, 16, [0], C=2 * w.E - 1)
    assert "two full-layer buffers" in mc.moe_last_error()


def test_decode_after_prefill_keeps_lru_consistent():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=1, C=80, steps=6)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    dev = torch.device("cuda")
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_trace(cache.handle, True)
    y = torch.empty((w.B, w.H), dtype=torch.bfloat16, device=dev)
    sim = lru.CacheSim(w.L, w.E, w.C)
    events = []

    def decode(ci_range):
        for ci in ci_range:
            s, l = calls[ci]
            assert cache.forward(l, runner.activations(w, s, l).to(dev), torch.from_numpy(lg[s, l]).to(dev), y, 1) == 0
            ids, _ = router.topk_softmax(lg[s, l].astype(np.float64), w.k)
            ev, _ = sim.access(l, ids)
            events.extend(e.as_tuple() for e in ev)

    decode(range(0, 8))
    xs, plg = prefill_inputs(w, 64, 2)
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    yp = torch.empty_like(x)
    assert mc.moe_prefill_stream(cache.handle, 0, 2, x, torch.from_numpy(plg).to(dev), 64, yp,
                                 torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    for s in range(w.C - 2 * w.E, w.C):  # the two buffers' slots are emptied
        key = int(sim.owner[s])
        if key >= 0:
            sim.map[key] = -1
        sim.owner[s] = -1
        sim.stamp[s] = 0
    decode(range(8, len(calls)))
    torch.cuda.synchronize()
    assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == events
    cache.close()
