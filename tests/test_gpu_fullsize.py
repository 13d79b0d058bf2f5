"""Parity at the full sizes of the five configurations, in the launch
configuration bench.py times (the fused layer kernel, copy-mode fills).

Every call's selected experts and slots and the whole hit/miss/eviction log
must match the oracle bit for bit; layer outputs are compared on a seeded
sample of calls (the oracle computes them one by one); with the elastic
schedule the outputs must also equal, bit for bit, those of a run at full
residency.  Pools are built on the GPU and freed after each test.
"""
import gc

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
