"""Parity at the full sizes of the five configurations, in the launch
configuration bench.py times (the fused layer kernel, copy-mode fills).

Every call's selected experts and slots and the whole hit/miss/eviction log
must match the oracle bit for bit; layer outputs are compared on a seeded
sample of calls (the oracle computes them one by one); with the elastic
schedule the outputs must also equal, bit for bit, those of a run at full
residency.  Pools are built on the GPU and freed after each test.
"""
import gc
import os

import numpy as np
import pytest

import synth
from synth import configs
from tests import harness as H

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def sample_calls(n_calls, n, seed):
    rng = np.random.default_rng(seed)
    return set(int(i) for i in rng.choice(n_calls, size=n, replace=False))


def check_light(gpu, ref):
    assert len(gpu.calls) == len(ref.calls)
    for ci, (g, r) in enumerate(zip(gpu.calls, ref.calls)):
        assert g.status == r.status, f"call {ci}"
        if r.status:
            continue
        assert (g.ids == r.ids).all(), f"call {ci}: ids"
        assert (g.slots == r.slots).all(), f"call {ci}: slots"
        if r.y is not None:
            H.assert_layer_close(g.y, r.y, f"call {ci}")
    assert [tuple(e) for e in gpu.events] == [tuple(e) for e in ref.events]


def free(*objs):
    for o in objs:
        del o
    gc.collect()
    torch.cuda.empty_cache()


def test_qwen36_shape_decode_full():
    w = configs.C2
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ys = sample_calls(len(calls), 24, 0)
    ref = H.run_oracle(w, calls, logits=lg, y_for=ys)
    gpu, _, stats = H.run_gpu(w, calls, logits=lg, light=True, y_for=ys)
    check_light(gpu, ref)
    assert 0.5 < stats["hits"] / (stats["hits"] + stats["misses"]) < 0.95
    free(gpu, ref)


@pytest.mark.parametrize("B,n_y", [(1, 6), (8, 2)])
def test_dsv4_shape_fp4_decode_full(B, n_y):
    w = configs.C3.with_(B=B)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ys = sample_calls(len(calls), n_y, B)
    ref = H.run_oracle(w, calls, logits=lg, y_for=ys)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg, light=True, y_for=ys)
    check_light(gpu, ref)
    free(gpu, ref)


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_elastic_schedule_full(B):
    w = configs.C5.with_(B=B)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    # resize before steps 512 and 1280: call index = step * L
    resize = {step * w.L: C for step, C in w.resize}
    ys = sample_calls(len(calls), 6, 10 + B) | {511 * w.L + 3, 512 * w.L + 3, 1280 * w.L + 7}
    ref = H.run_oracle(w, calls, logits=lg, resize=resize, y_for=ys)
    from expert_cache_serving_gb300 import runner

    pool, shared = runner.build_pool(w), runner.build_shared(w)
    before = pool[::997].clone()
    gpu, state, stats = H.run_gpu(w, calls, logits=lg, max_slots=w.LE, resize=resize, light=True, y_for=ys,
                                  pool=pool, shared=shared)
    check_light(gpu, ref)
    assert stats["resize_calls"] == 2
    # outputs equal a run at full residency, bit for bit
    full, _, _ = H.run_gpu(w, [calls[ci] for ci in sorted(ys)], logits=lg, C=w.LE, light=True, pool=pool,
                           shared=shared)
    for ci, f in zip(sorted(ys), full.calls):
        assert (gpu.calls[ci].y == f.y).all()
    # the host pool is never written
    assert torch.equal(pool[::997], before)
    free(gpu, ref, full, pool, shared)


# ---- prefill at full size: the oracle on a seeded sample of tokens -------------

def _expert_outputs(args):
    """Oracle worker (spawned process): o = expert(x) of one (layer, expert) for
    the sampled tokens routed to it."""
    import numpy as np

    import synth
    from oracle import ffn, nvfp4, records

    seed, key, H, I, wdtype, x, w4a4 = args
    rec = synth.records_array(seed, key, 1, H, I, wdtype)[0]
    if w4a4:
        return key, nvfp4.expert(x.astype(np.float32), *records.parse(rec, H, I, wdtype))
    return key, ffn.expert(x, *records.parse(rec, H, I, wdtype))


def sampled_prefill_reference(w, xs, lg, layers, tokens, workers=16, w4a4=False):
    """y [len(layers), len(tokens), H] from the oracle: routing and combine here,
    the expert FFNs of the distinct (layer, expert) pairs in a spawned pool."""
    import multiprocessing as mp

    from oracle import router

    jobs, plan = [], []
    for li, l in enumerate(layers):
        x = synth.bf16_bits_to_f32(xs[li][tokens]).astype(np.float64)
        ids, wts = router.topk_softmax(lg[li][tokens].astype(np.float64), w.k)
        plan.append((x, ids, wts))
        for e in sorted(set(ids.reshape(-1).tolist())):
            jobs.append((w.seed, l * w.E + e, w.H, w.I, w.wdtype, x, w4a4))
        if w.shared:
            jobs.append((w.seed, w.LE + l, w.H, w.I, w.wdtype, x, w4a4))
    with mp.get_context("spawn").Pool(min(workers, os.cpu_count() or 1)) as pool:
        outs = dict(pool.map(_expert_outputs, jobs, chunksize=1))
    ys = []
    for li, l in enumerate(layers):
        x, ids, wts = plan[li]
        y = np.zeros_like(x)
        for t in range(len(tokens)):
            for j in range(w.k):
                y[t] += wts[t, j] * outs[l * w.E + int(ids[t, j])][t]
            if w.shared:
                y[t] += outs[w.LE + l][t]
        ys.append(y)
    return ys


@pytest.mark.parametrize("w,w4a4", [(configs.C4, False), (configs.C2.with_(name="qwen3.6-shape-prefill-4096", B=4096),
                                                         False), (configs.C4, True)],
                         ids=["dsv4-fp4-4096x43", "qwen36-bf16-4096x40", "dsv4-fp4xfp4-4096x43"])
def test_prefill_full_size_sampled(w, w4a4):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    T, L = w.B, w.L
    layers = [0, 1, L // 2, L - 1]
    rng = np.random.default_rng(w.seed)
    tokens = np.sort(rng.choice(T, size=64, replace=False))
    xs = np.stack([synth.activations_bf16(w.seed, 0, l, T, w.H) for l in range(L)])
    lg = synth.iid_logits(w.seed, L, T, w.E)
    ref = sampled_prefill_reference(w, xs[layers], lg[layers], layers, tokens, w4a4=w4a4)
    dev = torch.device("cuda")
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared, C=w.C, max_tokens=1)
    if w4a4:
        mc.moe_cache_set_prefill_precision(cache.handle, mc.MOE_PREFILL_W4A4)
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    del xs
    y = torch.empty_like(x)
    st = mc.moe_prefill_stream(cache.handle, 0, L, x, torch.from_numpy(lg).to(dev), T, y, torch.cuda.current_stream())
    assert st == mc.MOE_OK, mc.moe_last_error()
    torch.cuda.synchronize()
    assert mc.moe_cache_sync(cache.handle, torch.cuda.current_stream()) == mc.MOE_OK
    for li, l in enumerate(layers):
        got = y[l][torch.from_numpy(tokens).to(dev)].float().cpu().numpy().astype(np.float64)
        H.assert_layer_close(got, ref[li], f"layer {l}")
    cache.close()
    free(x, y, pool, shared)
