"""GPU parity of the decode path against the CPU oracle (through the C ABI).

Integer results (selected experts, slots, the hit/miss/eviction log, the
grouping permutation and offsets) must match bit for bit; routing weights to
float32 rounding; layer outputs within max|err| <= 1e-2 * max|ref| of the
float64 oracle.  Outputs must also be bitwise identical across cache
capacities, resizes and hit/miss patterns (a GPU self-invariant).
"""
import numpy as np
import pytest

import synth
from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def compare(gpu, ref, check_y=True):
    assert len(gpu.calls) == len(ref.calls)
    worst = 0.0
    for ci, (g, r) in enumerate(zip(gpu.calls, ref.calls)):
        assert g.status == r.status, f"call {ci}: status {g.status} vs {r.status}"
        if r.status != 0:
            continue
        assert (g.ids == r.ids).all(), f"call {ci}: ids"
        assert np.allclose(g.w, r.w, rtol=0, atol=2e-6), f"call {ci}: weights"
        assert (g.slots == r.slots).all(), f"call {ci}: slots"
        assert (g.perm == r.perm).all(), f"call {ci}: perm"
        assert (g.offsets == r.offsets).all(), f"call {ci}: offsets"
        if check_y and r.y is not None:
            worst = max(worst, H.assert_layer_close(g.y, r.y, f"call {ci} (step {g.step}, layer {g.layer})"))
    assert [tuple(e) for e in gpu.events] == [tuple(e) for e in ref.events]
    return worst


def test_tiny_fp32_router_full_parity():
    w = configs.C1
    calls = H.decode_calls(w)
    wr = synth.router_weights(w.seed, w.L, w.E, w.H)
    ref = H.run_oracle(w, calls, router_w=wr)
    gpu, state, stats = H.run_gpu(w, calls, router_w=wr)
    compare(gpu, ref)
    assert stats["hits"] + stats["misses"] == sum(1 for e in ref.events if e[3] in (0, 1))
    assert stats["evictions"] > 0


@pytest.mark.parametrize("B", [1, 3])
def test_small_bf16_shared_parity(B):
    w = configs.SMALL_BF16.with_(B=B, C=40 if B == 1 else 80)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, state, stats = H.run_gpu(w, calls, logits=lg)
    compare(gpu, ref)
    assert stats["misses"] > 0 and stats["hits"] > 0


def test_small_fp4_parity_full_shape():
    w = configs.SMALL_FP4
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    sample = {0, 1, 9, len(calls) - 1}
    ref = H.run_oracle(w, calls, logits=lg, y_for=sample)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    compare(gpu, ref)


@pytest.mark.parametrize("B,C", [(1, 11), (8, 30)])
def test_small_fp4_narrow_parity(B, C):
    w = configs.SMALL_FP4_NARROW.with_(B=B, C=C)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    compare(gpu, ref)


def test_max_batch_and_k():
    # B = 16 tokens, k = 16 of 64 experts: up to 64 distinct experts per call
    w = configs.SMALL_BF16.with_(name="edge-b16-k16", L=2, E=64, k=16, H=256, I=128, shared=True, B=16, C=100,
                                 steps=6)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    compare(gpu, ref)


def test_wide_router_k1():
    w = configs.SMALL_BF16.with_(name="edge-e1024-k1", L=2, E=1024, k=1, H=256, I=64, shared=False, B=2, C=5,
                                 steps=20)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    compare(gpu, ref)


def test_outputs_bitwise_identical_across_capacities():
    w = configs.SMALL_BF16.with_(B=2, steps=10)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    from expert_cache_serving_gb300 import runner

    pool, shared = runner.build_pool(w), runner.build_shared(w)
    outs = []
    for C in (17, 40, w.LE):  # heavy eviction, some eviction, full residency (never evicts)
        gpu, _, stats = H.run_gpu(w, calls, logits=lg, C=C, pool=pool, shared=shared)
        outs.append(gpu)
        if C == w.LE:
            assert stats["evictions"] == 0
    for a, b in zip(outs, outs[1:]):
        for ca, cb in zip(a.calls, b.calls):
            assert (ca.y == cb.y).all()
            assert (ca.ids == cb.ids).all()


def test_capacity_error_leaves_cache_unchanged_and_resize_recovers():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=1, C=5, steps=3)  # k = 8 distinct experts per call > 5 slots
    lg = H.trace_logits(w)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared, max_slots=64)
    dev = torch.device("cuda")
    x = runner.activations(w, 0, 0).to(dev)
    y = torch.empty((1, w.H), dtype=torch.bfloat16, device=dev)
    st = cache.forward(0, x, torch.from_numpy(lg[0, 0]).to(dev), y, 1)
    assert st == mc.MOE_ERR_CAPACITY
    owner, stamp, n, g = mc.moe_cache_state(cache.handle, 64)
    assert n == 5 and (owner == -1).all() and g == 0
    mc.moe_cache_resize(cache.handle, 20)
    st = cache.forward(0, x, torch.from_numpy(lg[0, 0]).to(dev), y, 1)
    assert st == mc.MOE_OK
    ref = H.run_oracle(w, [(0, 0)], logits=lg, C=20)
    H.assert_layer_close(y.float().cpu().numpy().astype(np.float64), ref.calls[0].y)
    cache.close()


def test_fill_failure_rolls_back_recency_and_empties_victims():
    from oracle import lru

    w = configs.SMALL_BF16.with_(B=1, C=20, steps=8)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    fail_at, ok_fills = 10, 1
    gpu, state, _ = H.run_gpu(w, calls, logits=lg, inject={fail_at: ok_fills})
    assert gpu.calls[fail_at].status == 5  # MOE_ERR_CUDA
    # oracle model of the rollback: recency and counter as before the call,
    # every victim slot of the failed call empty
    from oracle import router
    sim = lru.CacheSim(w.L, w.E, w.C)
    events = []
    for ci, (s, l) in enumerate(calls):
        ids, _ = router.topk_softmax(lg[s, l].astype(np.float64), w.k)
        if ci == fail_at:
            snap_stamp, g, ncalls = sim.stamp.copy(), sim.g, sim.calls
            ev, _ = sim.access(l, ids)
            sim.stamp[:] = snap_stamp
            sim.g, sim.calls = g, ncalls
            for e in ev:
                if e.kind == lru.MISS:
                    sim.map[l * w.E + e.expert] = -1
                    sim.owner[e.slot] = -1
                    sim.stamp[e.slot] = 0
            continue
        ev, _ = sim.access(l, ids)
        events += [e.as_tuple() for e in ev]
    assert [tuple(e) for e in gpu.events] == events
    owner, stamp, n, g = state
    assert (owner[:w.C] == sim.owner).all()
    occupied = owner[:w.C] >= 0
    assert (stamp[:w.C][occupied] == sim.stamp[occupied]).all()
    assert g == sim.g


def test_resize_schedule_parity_and_output_identity():
    w = configs.SMALL_BF16.with_(B=2, C=40, steps=16)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    resize = {12: 17, 24: 70, 36: 9, 40: 33}
    ref = H.run_oracle(w, calls, logits=lg, resize=resize, y_for=set())
    from expert_cache_serving_gb300 import runner

    pool, shared = runner.build_pool(w), runner.build_shared(w)
    gpu, state, stats = H.run_gpu(w, calls, logits=lg, max_slots=w.LE, resize=resize, pool=pool, shared=shared)
    compare(gpu, ref, check_y=False)
    assert stats["resize_calls"] == 4 and stats["resize_moves"] > 0
    plain, _, _ = H.run_gpu(w, calls, logits=lg, C=w.LE, pool=pool, shared=shared)
    n_same = 0
    for a, b in zip(gpu.calls, plain.calls):
        if a.status == 0:  # calls after the shrink to 9 slots may exceed the capacity
            assert (a.y == b.y).all()
            n_same += 1
    assert n_same > len(calls) // 2
    # the host pool is never written
    fresh = runner.build_pool(w)
    assert torch.equal(pool, fresh)


# ---- device-driven fills (the layer kernel pulls misses from the pool) ------

@pytest.mark.parametrize("B", [1, 3])
def test_device_fill_bf16_parity(B):
    w = configs.SMALL_BF16.with_(B=B, C=40 if B == 1 else 80)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, stats = H.run_gpu(w, calls, logits=lg, fill_mode=1)
    compare(gpu, ref)
    assert stats["misses"] > 0


@pytest.mark.parametrize("B,C", [(1, 11), (8, 30)])
def test_device_fill_fp4_parity(B, C):
    w = configs.SMALL_FP4_NARROW.with_(B=B, C=C)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg, fill_mode=1)
    compare(gpu, ref)


def test_fill_modes_bitwise_identical_and_slots_hold_records():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_FP4.with_(steps=6)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    a, sa, _ = H.run_gpu(w, calls, logits=lg, pool=pool, shared=shared, fill_mode=0)
    b, sb, _ = H.run_gpu(w, calls, logits=lg, pool=pool, shared=shared, fill_mode=1)
    for ca, cb in zip(a.calls, b.calls):
        assert (ca.y == cb.y).all()
    assert [tuple(e) for e in a.events] == [tuple(e) for e in b.events]
    # after a device-driven run every occupied slot holds its expert's record byte for byte
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_fill_mode(cache.handle, 1)
    dev = torch.device("cuda")
    y = torch.empty((w.B, w.H), dtype=torch.bfloat16, device=dev)
    for (s, l) in calls:
        assert cache.forward(l, runner.activations(w, s, l).to(dev), torch.from_numpy(lg[s, l]).to(dev), y, w.B) == 0
    torch.cuda.synchronize()
    owner, _, n, _ = mc.moe_cache_state(cache.handle, w.C)
    S = synth.record_bytes(w.H, w.I, w.wdtype)
    class SlotView:  # zero-copy device view of one slot
        def __init__(self, ptr):
            self.__cuda_array_interface__ = {"shape": (S,), "typestr": "|u1", "data": (ptr, False), "version": 3}

    for slot, key in enumerate(owner):
        if key < 0:
            continue
        got = torch.as_tensor(SlotView(mc.moe_cache_slot_ptr(cache.handle, slot)), device=dev)
        assert torch.equal(got.cpu(), pool[key]), f"slot {slot} does not hold record {key}"
    cache.close()


def test_device_fill_with_resize():
    w = configs.SMALL_BF16.with_(B=2, C=40, steps=12)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    resize = {10: 19, 20: 60}
    ref = H.run_oracle(w, calls, logits=lg, resize=resize, y_for=set())
    gpu, _, _ = H.run_gpu(w, calls, logits=lg, max_slots=w.LE, resize=resize, fill_mode=1)
    compare(gpu, ref, check_y=False)
