"""Late fills, busy resizes and the status of calls, on the GPU (through the C ABI).

No test here faults, traps or hangs the GPU.  A late fill is made by giving
the layer kernel's bounded fill waits a zero limit: whenever a copy has not
landed at the first look, the kernel hands the rest of the call to the
completion kernel that runs after the call's copies.  The outputs must still
match the oracle and be bitwise identical to a run where the kernel waited,
the hand-overs must show in the statistics, and moe_cache_sync must report
no error (a late fill is not one).
"""
import numpy as np
import pytest

from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

from tests.test_gpu_decode import compare  # noqa: E402


@pytest.mark.parametrize("wait_ns,stage", [((0, 5_000_000_000), "gate/up"), ((5_000_000_000, 0), "W_down"),
                                           ((0, 0), "both")])
def test_late_fills_finish_on_the_completion_kernel(wait_ns, stage):
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=2, C=40, steps=10)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    ref = H.run_oracle(w, calls, logits=lg)
    waited, _, s_wait = H.run_gpu(w, calls, logits=lg, pool=pool, shared=shared,
                                  wait_ns=(5_000_000_000, 5_000_000_000))
    late, state, s_late = H.run_gpu(w, calls, logits=lg, pool=pool, shared=shared, wait_ns=wait_ns)
    compare(late, ref)
    for a, b in zip(waited.calls, late.calls):
        assert (a.y == b.y).all(), f"{stage}: outputs differ from a run that waited for its fills"
    assert s_wait["deferred_calls"] == 0
    if stage != "W_down":
        # every call with fills hands over: its first gate/up half cannot have
        # landed when the kernel first looks (the host issues it after the miss list)
        assert s_late["deferred_calls"] > 0
        assert s_late["deferred_calls"] <= sum(1 for c in ref.calls if c.status == 0)


def test_fp4_late_fills_at_batch_8():
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_FP4_NARROW.with_(B=8, C=30, steps=6)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    pool = runner.build_pool(w)
    ref = H.run_oracle(w, calls, logits=lg)
    late, _, stats = H.run_gpu(w, calls, logits=lg, pool=pool, wait_ns=(0, 0))
    compare(late, ref)
    assert stats["deferred_calls"] > 0
    dev_fill, _, _ = H.run_gpu(w, calls, logits=lg, pool=pool, fill_mode=1)
    for a, b in zip(late.calls, dev_fill.calls):
        assert (a.y == b.y).all()


def test_next_call_after_a_hand_over_is_clean():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=1, C=40, steps=4)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared)
    dev = torch.device("cuda")
    y = torch.empty((1, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    for ci, (s, l) in enumerate(calls):
        # alternate: hand over at once, then wait normally
        mc.moe_cache_set_wait_limit_ns(cache.handle, *((0, 0) if ci % 2 == 0 else (2_000_000, 2_000_000)))
        st = cache.forward(l, runner.activations(w, s, l).to(dev), torch.from_numpy(lg[s, l]).to(dev), y, 1)
        assert st == mc.MOE_OK
        assert mc.moe_cache_sync(cache.handle, stream) == mc.MOE_OK
        H.assert_layer_close(y.float().cpu().numpy().astype(np.float64), ref.calls[ci].y, f"call {ci}")
    stats = mc.moe_cache_stats(cache.handle)
    assert stats["deferred_calls"] > 0
    cache.close()


def test_resize_is_busy_while_a_forward_runs():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=1, C=40, steps=2)
    lg = H.trace_logits(w)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared, max_slots=64)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE)  # the call returns without waiting
    dev = torch.device("cuda")
    x = runner.activations(w, 0, 0).to(dev)
    logits = torch.from_numpy(lg[0, 0]).to(dev)
    y = torch.empty((1, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # keeps the stream busy for ~0.1 s (a bounded spin)
    assert cache.forward(0, x, logits, y, 1, stream=stream) == mc.MOE_OK
    with pytest.raises(mc.MoeError) as ei:
        mc.moe_cache_resize(cache.handle, 20, stream)
    assert ei.value.status == mc.MOE_ERR_BUSY
    assert mc.moe_cache_sync(cache.handle, stream) == mc.MOE_OK
    mc.moe_cache_resize(cache.handle, 20, stream)  # now idle
    owner, _, n, _ = mc.moe_cache_state(cache.handle, 64)
    assert n == 20 and (owner >= 0).sum() == w.k
    ref = H.run_oracle(w, [(0, 0)], logits=lg)
    H.assert_layer_close(y.float().cpu().numpy().astype(np.float64), ref.calls[0].y)
    cache.close()


def test_device_fill_calls_run_ahead_and_sync_reads_their_summaries():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=2, C=40, steps=12)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg, y_for=set())
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_trace(cache.handle, True)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE)
    dev = torch.device("cuda")
    xs = [runner.activations(w, s, l).to(dev) for (s, l) in calls]
    lgs = torch.from_numpy(lg).to(dev)
    ys = torch.empty((len(calls), w.B, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)  # the host enqueues every call before the GPU starts them
    for ci, (s, l) in enumerate(calls):
        assert cache.forward(l, xs[ci], lgs[s, l], ys[ci], w.B, stream=stream) == mc.MOE_OK
    assert mc.moe_cache_sync(cache.handle, stream) == mc.MOE_OK
    assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == [tuple(e) for e in ref.events]
    stats = mc.moe_cache_stats(cache.handle)
    assert stats["calls"] == len(calls) and stats["host_wait_us"] == 0.0
    cache.close()
