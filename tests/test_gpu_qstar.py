"""The fill count q* of the bandwidth split, derived by the layer kernel's
control step, against the oracle (oracle.qstar, pinned by the Fig. 2 worked
example) for every call of a decode trace, at the pages' Table 1 bandwidth
ratios and at ratios that put m * B_P / B_H exactly on a half.  This build has
no host execution branch, so every miss is still filled: the cache's
hit/miss/eviction log must not depend on the bandwidths."""
import numpy as np
import pytest

from oracle import lru, qstar, router
from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.mark.parametrize("bp,bh", [(1.0, 4.0), (52.7, 77.3), (11.8, 47.5), (1.0, 2.0), (3.0, 4.0), (5.0, 2.0),
                                   (0.0, 0.0)])
def test_control_step_derives_qstar(bp, bh):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16.with_(B=2, C=40, steps=8)
    calls = H.decode_calls(w)
    lg = H.trace_logits(w)
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared)
    mc.moe_cache_set_trace(cache.handle, True)
    mc.moe_cache_set_split_bandwidths(cache.handle, bp, bh)
    dev = torch.device("cuda")
    y = torch.empty((w.B, w.H), dtype=torch.bfloat16, device=dev)
    q = torch.empty(1, dtype=torch.int32, device=dev)
    sim = lru.CacheSim(w.L, w.E, w.C)
    events, total = [], 0
    for s, l in calls:
        st = cache.forward(l, runner.activations(w, s, l).to(dev), torch.from_numpy(lg[s, l]).to(dev), y, w.B,
                           aux={"qstar": q})
        assert st == mc.MOE_OK
        ids, _ = router.topk_softmax(lg[s, l].astype(np.float64), w.k)
        ev, _ = sim.access(l, ids)
        events += [e.as_tuple() for e in ev]
        m = sum(1 for e in ev if e.kind == lru.MISS)
        want = qstar.qstar(m, bp, bh) if bp > 0 and bh > 0 else m
        assert int(q.item()) == want, f"call ({s}, {l}): m={m}"
        total += want
    torch.cuda.synchronize()
    assert [tuple(e) for e in mc.moe_cache_trace(cache.handle)] == events
    assert mc.moe_cache_stats(cache.handle)["qstar_fills"] == total
    cache.close()
