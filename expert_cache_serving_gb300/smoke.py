"""Small decode and prefill runs on cuda:0 checked against the CPU oracle.

Runs the tiny fp32 workload (2 layers, 16 experts, top-2, 12 cache slots)
for a few steps and a small bf16 workload with a shared expert through the C
ABI, and compares routing, slots, the cache event log and the layer outputs
with the oracle; then one 64-token FP4 prefill layer (H 512, I 256, 24
experts, top-4) through the tcgen05 grouped GEMMs.  Raises on any mismatch.
"""
from __future__ import annotations

import numpy as np


def run() -> None:
    import torch

    import synth
    from oracle import ffn, lru, records, router
    from synth import configs

    from . import moecache as mc
    from . import runner

    assert torch.cuda.is_available(), "smoke needs cuda:0"
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    for w, steps in ((configs.C1, 6), (configs.SMALL_BF16.with_(L=2, E=16, C=12), 4)):
        pool, shared = runner.build_pool(w), runner.build_shared(w)
        cache = runner.Cache(w, pool, shared)
        mc.moe_cache_set_trace(cache.handle, True)
        wr = synth.router_weights(w.seed, w.L, w.E, w.H) if w.router else None
        wr_dev = torch.from_numpy(wr).to(dev) if wr is not None else None
        lg = None if w.router else synth.ar1_logits(w.seed, steps, w.L, w.B, w.E)
        sim = lru.CacheSim(w.L, w.E, w.C)
        want_events = []
        ids_d = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
        y = torch.empty((w.B, w.H), dtype=runner.x_dtype(w), device=dev)
        for s in range(steps):
            for l in range(w.L):
                x = runner.activations(w, s, l)
                x64 = x.float().numpy().astype(np.float64)
                logits_host = router.logits_from_router(x64, wr[l]) if w.router else lg[s, l].astype(np.float64)
                st = cache.forward(l, x.to(dev), None if w.router else torch.from_numpy(lg[s, l]).to(dev), y, w.B,
                                   router_w=wr_dev[l] if wr_dev is not None else None, aux={"ids": ids_d})
                mc.check(st, "moe_layer_forward")
                ids, wts = router.topk_softmax(logits_host, w.k)
                ev, _ = sim.access(l, ids)
                want_events += [e.as_tuple() for e in ev]
                assert (ids_d.cpu().numpy() == ids).all(), "routing mismatch"

                def expert(e, l=l):
                    rec = synth.records_array(w.seed, l * w.E + e, 1, w.H, w.I, w.wdtype)[0]
                    return records.parse(rec, w.H, w.I, w.wdtype)

                sh = None
                if w.shared:
                    sh = records.parse(synth.records_array(w.seed, w.LE + l, 1, w.H, w.I, w.wdtype)[0], w.H, w.I,
                                       w.wdtype)
                ref = ffn.moe_layer(x64, ids, wts, expert, sh)
                got = y.float().cpu().numpy().astype(np.float64)
                err = np.max(np.abs(got - ref))
                assert err <= 1e-2 * np.max(np.abs(ref)), f"layer output error {err}"
        torch.cuda.synchronize()
        mc.check(mc.moe_cache_sync(cache.handle, torch.cuda.current_stream()), "moe_cache_sync")
        assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == want_events, "cache event log mismatch"
        cache.close()

    # one FP4 prefill layer (tensor-core grouped GEMMs reading FP4 codes)
    w = configs.SMALL_FP4_NARROW.with_(C=48)
    T = 64
    pool = runner.build_pool(w)
    cache = runner.Cache(w, pool, None, C=w.C, max_tokens=1)
    xs = synth.activations_bf16(w.seed + 100, 0, 0, T, w.H)
    lg = synth.iid_logits(w.seed, 1, T, w.E)
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.empty_like(x)
    mc.check(mc.moe_prefill_stream(cache.handle, 0, 1, x, torch.from_numpy(lg).to(dev), T, y,
                                   torch.cuda.current_stream()), "moe_prefill_stream")
    torch.cuda.synchronize()
    ids, wts = router.topk_softmax(lg[0].astype(np.float64), w.k)

    def expert0(e):
        return records.parse(synth.records_array(w.seed, e, 1, w.H, w.I, w.wdtype)[0], w.H, w.I, w.wdtype)

    ref = ffn.moe_layer(synth.bf16_bits_to_f32(xs).astype(np.float64), ids, wts, expert0, None)
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.max(np.abs(got - ref))
    assert err <= 1e-2 * np.max(np.abs(ref)), f"prefill output error {err}"
    cache.close()
    print("smoke: ok")
