"""GPU parity of moe_prefill_stream (full-layer double buffering, grouped
tcgen05 GEMMs) against the CPU oracle, through the C ABI.

Routing (ids, weights), the grouping permutation and offsets and the slot
each expert is read from are compared bit for bit (weights to float32
rounding), including ties, signed zeros, NaN, -inf and +inf logits; layer
outputs within max|err| <= 1e-2 * max|ref|.  The cache state after prefill
(the buffers' contents seed decode, resident experts are read in place) and
the decode calls that follow are checked event for event against the oracle
simulator.
"""
import numpy as np
import pytest

import synth
from oracle import ffn, lru, permute, router
from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def prefill_inputs(w, T, n_layers, edge=False):
    xs = np.stack([synth.activations_bf16(w.seed + 100, 0, l, T, w.H) for l in range(n_layers)])
    lg = synth.iid_logits(w.seed, n_layers, T, w.E)
    if edge:  # the routing edge cases in the first tokens of every layer
        lg[:, 0, :] = 0.5                                   # all equal
        lg[:, 1, :] = -1.0
        lg[:, 1, [1, 3, 5, 9]] = [-0.0, 0.0, -0.0, 0.0]     # zeros of both signs tie at the top
        lg[:, 2, :4] = np.nan                               # NaN and -inf below the real logits
        lg[:, 2, 4:8] = -np.inf
        lg[:, 3, :] = -np.inf                               # no real logit at all
        lg[:, 3, 2::5] = np.nan
        lg[:, 4, 7] = np.inf                                # +inf entries share the weight
        lg[:, 4, 11] = np.inf
        lg[:, 5, ::3] = 2.0                                 # many copies of the maximum
    return xs, lg


def oracle_prefill(w, xs, lg, layers, bank, tokens=None):
    out = []
    for li, l in enumerate(layers):
        t_sel = np.arange(xs.shape[1]) if tokens is None else np.asarray(tokens)
        x = synth.bf16_bits_to_f32(xs[li][t_sel]).astype(np.float64)
        ids, wts = router.topk_softmax(lg[li][t_sel].astype(np.float64), w.k)
        shared = bank.get(w.LE + l) if w.shared else None
        out.append(ffn.moe_layer(x, ids, wts, lambda e, l=l: bank.get(l * w.E + e), shared))
    return out


def run_prefill(w, T, layers, C, pool=None, shared=None, edge=False, aux=False, cache=None):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    dev = torch.device("cuda")
    if cache is None:
        pool = runner.build_pool(w) if pool is None else pool
        shared = runner.build_shared(w) if shared is None else shared
        cache = runner.Cache(w, pool, shared, C=C)
    xs, lg = prefill_inputs(w, T, len(layers), edge)
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(lg).to(dev)
    y = torch.empty_like(x)
    n = len(layers)
    a = None
    if aux:
        a = {"ids": torch.empty((n, T, w.k), dtype=torch.int32, device=dev),
             "weights": torch.empty((n, T, w.k), dtype=torch.float32, device=dev),
             "perm": torch.empty((n, T * w.k), dtype=torch.int32, device=dev),
             "offsets": torch.empty((n, w.E + 1), dtype=torch.int32, device=dev),
             "slots": torch.empty((n, w.E), dtype=torch.int32, device=dev)}
    st = mc.moe_prefill_stream(cache.handle, layers[0], layers[-1] + 1, x, logits, T, y,
                               torch.cuda.current_stream(), aux=a)
    assert st == mc.MOE_OK, mc.moe_last_error()
    torch.cuda.synchronize()
    assert mc.moe_cache_sync(cache.handle, torch.cuda.current_stream()) == mc.MOE_OK
    got = {k: v.cpu().numpy() for k, v in a.items()} if aux else None
    return cache, xs, lg, y.float().cpu().numpy().astype(np.float64), got


@pytest.mark.parametrize("T", [200, 333])
def test_prefill_bf16_shared_parity(T):
    w = configs.SMALL_BF16.with_(C=70)
    layers = [0, 1, 2]
    cache, xs, lg, y, _ = run_prefill(w, T, layers, C=70)
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"prefill layer {layers[li]}")
    cache.close()


def test_prefill_fp4_full_shape_parity():
    w = configs.SMALL_FP4.with_(C=32)
    layers = [0, 1]
    cache, xs, lg, y, _ = run_prefill(w, 160, layers, C=32)
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"prefill layer {layers[li]}")
    cache.close()


def test_prefill_fp4_experts_spanning_several_row_tiles():
    # 512 tokens, top-6 of 8 experts: ~384 rows per expert, three or four
    # 128-row tiles each, the last one ragged
    w = configs.SMALL_FP4.with_(name="fp4-multi-tile", E=8, C=16)
    T = 512
    cache, xs, lg, y, got = run_prefill(w, T, [0], C=16, aux=True)
    ids, _ = router.topk_softmax(lg[0].astype(np.float64), w.k)
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    assert counts.min() > 128 and counts.max() > 256
    sample = list(range(0, T, 7)) + [T - 1]
    ref = oracle_prefill(w, xs, lg, [0], H.ExpertBank(w), tokens=sample)
    H.assert_layer_close(y[0][sample], ref[0], "prefill layer 0")
    cache.close()


def test_prefill_routing_grouping_and_slots_bit_exact():
    w = configs.SMALL_BF16.with_(C=80)
    layers = [0, 1]
    T = 64
    cache, xs, lg, y, got = run_prefill(w, T, layers, C=80, edge=True, aux=True)
    sim = lru.CacheSim(w.L, w.E, w.C)
    _, table = sim.prefill(layers[0], layers[-1] + 1)
    for li in range(len(layers)):
        ids, wts = router.topk_softmax(lg[li].astype(np.float64), w.k)
        assert (got["ids"][li] == ids).all(), f"layer {li}: ids"
        assert np.allclose(got["weights"][li], wts, rtol=0, atol=2e-6), f"layer {li}: weights"
        perm, offsets = permute.permutation(ids, w.E)
        assert (got["perm"][li] == perm).all(), f"layer {li}: perm"
        assert (got["offsets"][li] == offsets).all(), f"layer {li}: offsets"
        assert (got["slots"][li] == table[li]).all(), f"layer {li}: slots"
    # the crafted rows select what the rule says
    ids0, w0 = router.topk_softmax(lg[0].astype(np.float64), w.k)
    assert ids0[0].tolist() == list(range(w.k))
    assert ids0[1].tolist()[:4] == [1, 3, 5, 9]
    assert np.allclose(w0[3], 1.0 / w.k) and ids0[4].tolist()[:2] == [7, 11]
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"prefill layer {layers[li]}")
    cache.close()


@pytest.mark.parametrize("w,C", [(configs.SMALL_BF16.with_(B=1, steps=4), 20),
                                 (configs.SMALL_FP4_NARROW.with_(B=1, steps=4), 7)], ids=["bf16", "fp4"])
def test_prefill_on_demand_when_two_buffers_do_not_fit(w, C):
    # C < 2E: each layer's routed experts are loaded in chunks of at most C,
    # each chunk like one decode call, then evaluated
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = w.with_(C=C)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    calls = H.decode_calls(w, 2)
    lg = H.trace_logits(w, 2)
    dev = torch.device("cuda")
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_trace(cache.handle, True)
    y = torch.empty((w.B, w.H), dtype=torch.bfloat16, device=dev)
    sim = lru.CacheSim(w.L, w.E, w.C)
    events = []
    for s, l in calls:  # some decode first, so some experts are resident
        assert cache.forward(l, runner.activations(w, s, l).to(dev), torch.from_numpy(lg[s, l]).to(dev), y, 1) == 0
        ev, _ = sim.access(l, router.topk_softmax(lg[s, l].astype(np.float64), w.k)[0])
        events += [e.as_tuple() for e in ev]
    layers = [0, 1]
    _, xs, plg, yp, got = run_prefill(w, 48, layers, C=w.C, aux=True, cache=cache)
    for li, l in enumerate(layers):
        ids, _ = router.topk_softmax(plg[li].astype(np.float64), w.k)
        ev, slot_of = sim.prefill_on_demand(l, ids)
        events += [e.as_tuple() for e in ev]
        want = np.full(w.E, -1)
        for e, s in slot_of.items():
            want[e] = s
        assert (got["slots"][li] == want).all(), f"layer {l}: slots"
    ref = oracle_prefill(w, xs, plg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(yp[li], ref[li], f"prefill layer {layers[li]}")
    assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == events
    owner, stamp, n, g = mc.moe_cache_state(cache.handle, w.C)
    assert (owner == sim.owner).all() and g == sim.g
    occ = owner >= 0
    assert (stamp[occ] == sim.stamp[occ]).all()
    cache.close()


def test_prefill_seeds_decode_and_reads_resident_experts_in_place():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=1, C=80, steps=8)
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

    decode(range(0, 9))
    mc.moe_cache_reset_stats(cache.handle)
    _, xs, plg, yp, got = run_prefill(w, 64, [0, 1], C=w.C, aux=True, cache=cache)
    ev, table = sim.prefill(0, 2)
    events.extend(e.as_tuple() for e in ev)
    assert (got["slots"] == table).all()
    stats = mc.moe_cache_stats(cache.handle)
    assert stats["prefill_records_in_place"] > 0
    assert stats["prefill_records_streamed"] + stats["prefill_records_in_place"] == 2 * w.E
    ref = oracle_prefill(w, xs, plg, [0, 1], H.ExpertBank(w))
    for li in range(2):
        H.assert_layer_close(yp[li], ref[li], f"prefill layer {li}")
    owner, stamp, n, g = mc.moe_cache_state(cache.handle, w.C)
    assert (owner == sim.owner).all() and g == sim.g
    occ = owner >= 0
    assert (stamp[occ] == sim.stamp[occ]).all()
    decode(range(9, len(calls)))
    torch.cuda.synchronize()
    assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == events
    cache.close()


def test_long_prompt_runs_in_chunks():
    from expert_cache_serving_gb300 import moecache as mc

    w = configs.SMALL_BF16.with_(L=3, E=16, k=4, C=40)
    T = 8192 + 300
    layers = [0, 1]
    cache, xs, lg, y, _ = run_prefill(w, T, layers, C=w.C)
    sample = [0, 1, 4000, 8190, 8191, 8192, 8193, T - 1]
    ref = oracle_prefill(w, xs, lg, layers, H.ExpertBank(w), tokens=sample)
    for li in range(2):
        H.assert_layer_close(y[li][sample], ref[li], f"prefill layer {li}")
    sim = lru.CacheSim(w.L, w.E, w.C)
    sim.prefill(0, 2, chunks=2)
    owner, stamp, n, g = mc.moe_cache_state(cache.handle, w.C)
    assert (owner == sim.owner).all() and g == sim.g
    cache.close()
