"""Routing edge cases on the GPU against the oracle (through the C ABI).

The router's rule: top-k by logit, descending, ties to the lower expert id,
a NaN logit counts as -inf, -0 equals +0; weights = softmax over the k taken
logits.  Crafted logits put every tie case at the top of the ranking (all
logits equal; zeros of both signs; many copies of the maximum; NaN and -inf
next to real values; a single real logit above a sea of -inf, where the rest
of the top-k are taken by index with weight 0).  Selected ids, weights, slots,
the event log and the layer outputs must match the oracle.
"""
import numpy as np
import pytest

from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def edge_logits(w):
    lg = H.trace_logits(w).copy()  # [steps, L, B, E]
    # step 0: token 0 all equal; token 1: zeros of both signs tie at the top
    lg[0, :, 0, :] = 0.5
    lg[0, :, 1, :] = -1.0
    for e, v in ((1, -0.0), (3, 0.0), (5, -0.0), (9, 0.0)):
        lg[0, :, 1, e] = v
    # step 1: NaN and -inf below every real logit; copies of the maximum
    lg[1, :, 0, :4] = np.nan
    lg[1, :, 0, 4:8] = -np.inf
    lg[1, :, 1, ::3] = 2.0
    # step 2: one real logit, every other one -inf or NaN
    lg[2, :, 0, :] = -np.inf
    lg[2, :, 0, 2::5] = np.nan
    lg[2, :, 0, 17] = 0.25
    lg[2, :, 1, :] = np.float32(-3.0)
    lg[2, :, 1, 30] = np.float32(-2.0)
    return lg


def test_router_ties_nan_and_signed_zero():
    w = configs.SMALL_BF16.with_(B=2, C=40, steps=3)
    calls = H.decode_calls(w)
    lg = edge_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    assert len(gpu.calls) == len(ref.calls)
    for ci, (g, r) in enumerate(zip(gpu.calls, ref.calls)):
        assert g.status == r.status == 0, f"call {ci}"
        assert (g.ids == r.ids).all(), f"call {ci}: ids {g.ids.tolist()} vs {r.ids.tolist()}"
        assert np.allclose(g.w, r.w, rtol=0, atol=2e-6), f"call {ci}: weights"
        assert (g.slots == r.slots).all(), f"call {ci}: slots"
        H.assert_layer_close(g.y, r.y, f"call {ci}")
    assert [tuple(e) for e in gpu.events] == [tuple(e) for e in ref.events]
    # the crafted cases select what the rule says
    first = ref.calls[0]
    assert first.ids[0].tolist() == list(range(w.k))
    assert first.ids[1].tolist()[:4] == [1, 3, 5, 9]


@pytest.mark.parametrize("E,k", [(256, 8), (100, 6), (64, 8)])
def test_router_edges_wide_expert_counts(E, k):
    """The same crafted cases with 64..256 experts (several logits per lane)."""
    w = configs.SMALL_BF16.with_(name=f"edge-e{E}-k{k}", L=2, E=E, k=k, H=256, I=64, B=3, C=100, steps=5)
    calls = H.decode_calls(w)
    lg = edge_logits(w)
    ref = H.run_oracle(w, calls, logits=lg)
    gpu, _, _ = H.run_gpu(w, calls, logits=lg)
    for ci, (g, r) in enumerate(zip(gpu.calls, ref.calls)):
        assert g.status == r.status == 0, f"call {ci}"
        assert (g.ids == r.ids).all(), f"call {ci}: ids {g.ids.tolist()} vs {r.ids.tolist()}"
        assert np.allclose(g.w, r.w, rtol=0, atol=2e-6), f"call {ci}: weights"
        H.assert_layer_close(g.y, r.y, f"call {ci}")
    assert [tuple(e) for e in gpu.events] == [tuple(e) for e in ref.events]
