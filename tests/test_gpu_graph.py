"""Whole decode steps captured into a CUDA graph and replayed (graph mode,
device-driven fills), through the C ABI.

The control step runs on the device, so a step of L layer calls needs no host
decision and can be a graph ("CUDA Graph와 공존하는 LRU 캐시" in the FreeToken
write-up).  Each replay must be a new call sequence: the hit/miss/evict log
equals the oracle simulator's, event for event, and the outputs equal those
of the same steps launched one call at a time, bit for bit.
"""
import numpy as np
import pytest

from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.mark.parametrize("B", [1, 3])
def test_captured_steps_replay_as_new_calls(B):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=B, C=40 if B == 1 else 80, steps=14)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    eager, _, _ = H.run_gpu(w, calls, logits=lg, fill_mode=mc.MOE_FILL_DEVICE)

    dev = torch.device("cuda")
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_trace(cache.handle, True)
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE)
    mc.moe_cache_set_graph_mode(cache.handle, 1)
    xdt = runner.x_dtype(w)
    x_all = torch.stack([torch.stack([runner.activations(w, s, l) for l in range(w.L)])
                         for s in range(w.steps)]).to(dev)
    lg_all = torch.from_numpy(np.ascontiguousarray(lg)).to(dev)
    x_in = torch.empty((w.L, B, w.H), dtype=xdt, device=dev)
    lg_in = torch.empty((w.L, B, w.E), dtype=torch.float32, device=dev)
    y_out = torch.empty((w.L, B, w.H), dtype=xdt, device=dev)

    def step_calls(stream):
        for l in range(w.L):
            st = cache.forward(l, x_in[l], lg_in[l], y_out[l], B, stream=stream)
            assert st == mc.MOE_OK, mc.moe_last_error()

    ys = []
    # step 0 launched directly (graph mode, not captured), then captured once
    x_in.copy_(x_all[0])
    lg_in.copy_(lg_all[0])
    step_calls(torch.cuda.current_stream())
    ys.append(y_out.clone())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_calls(torch.cuda.current_stream())
    for s in range(1, w.steps):
        x_in.copy_(x_all[s])
        lg_in.copy_(lg_all[s])
        g.replay()
        ys.append(y_out.clone())
    torch.cuda.synchronize()
    assert mc.moe_cache_sync(cache.handle, torch.cuda.current_stream()) == mc.MOE_OK, mc.moe_last_error()
    events = mc.moe_cache_trace(cache.handle)
    stats = mc.moe_cache_stats(cache.handle)
    assert stats["summaries_lost"] == 0
    assert stats["layer_launches"] == len(calls)
    assert [tuple(e) for e in events] == [tuple(e) for e in ref.events]
    for ci, (s, l) in enumerate(calls):
        got = ys[s][l].float().cpu().numpy().astype(np.float64)
        assert np.array_equal(got, eager.calls[ci].y), f"step {s} layer {l}: output differs from the launched run"
    del g
    mc.moe_cache_set_graph_mode(cache.handle, 0)
    cache.close()


def test_graph_mode_needs_device_fills():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16
    cache = runner.Cache(w, runner.build_pool(w), runner.build_shared(w))
    assert mc.lib.moe_cache_set_graph_mode(cache.handle, 1) == mc.MOE_ERR_INVALID_ARG
    mc.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_DEVICE)
    mc.moe_cache_set_graph_mode(cache.handle, 1)
    assert mc.lib.moe_cache_set_fill_mode(cache.handle, mc.MOE_FILL_COPY) == mc.MOE_ERR_INVALID_ARG
    mc.moe_cache_set_graph_mode(cache.handle, 0)
    cache.close()
