"""The no-allocation entry point (moe_layer_forward_resident_noalloc) against
the CPU oracle and against moe_layer_forward, through the C ABI.

It serves callers that cannot allocate device memory: its scratch is a fixed
array inside the library.  Two calls in a row must match the oracle and the
cached entry point's outputs within the layer tolerance (max|err| <= 1e-2 *
max|ref|), for fp32, bf16 (with a shared expert) and FP4 weights, with the
router's tie, signed-zero, NaN and infinity cases; sizes beyond the scratch
must be rejected.  This file is collected last so a failure here does not
hide the other tests' results; it passes both alone and after them.
"""
import numpy as np
import pytest

from synth import configs
from tests import harness as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def edge_rows(lg):
    """Put the router's edge cases into the first tokens of every call."""
    lg = lg.copy()
    E = lg.shape[-1]
    lg[:, :, 0, :] = 0.5                      # all equal
    if lg.shape[2] > 1:
        lg[:, :, 1, :] = -np.inf              # no real logit at all (uniform weights)
        lg[:, :, 1, 2::5] = np.nan
    if lg.shape[2] > 2:
        lg[:, :, 2, :] = -1.0
        lg[:, :, 2, [1, 3]] = [-0.0, 0.0]     # zeros of both signs tie at the top
        lg[:, :, 2, E - 1] = np.inf           # +inf takes the whole weight
    return lg


@pytest.mark.parametrize("w", [configs.SMALL_BF16.with_(B=3, steps=2),
                               configs.SMALL_FP4_NARROW.with_(B=3, C=40, steps=2),
                               configs.C1.with_(router=False, B=3, C=32, steps=2)],
                         ids=["bf16-shared", "fp4", "fp32"])
def test_noalloc_matches_oracle_and_cached_forward_two_calls(w):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    dev = torch.device("cuda")
    pool, shared = runner.build_pool(w), runner.build_shared(w)
    cache = runner.Cache(w, pool, shared)
    lg = edge_rows(H.trace_logits(w))
    calls = [(0, 0), (1, w.L - 1)]  # two calls in a row, different layers
    ref = H.run_oracle(w, calls, logits=lg)
    xdt = runner.x_dtype(w)
    y_ref = torch.empty((w.B, w.H), dtype=xdt, device=dev)
    y_new = torch.empty((w.B, w.H), dtype=xdt, device=dev)
    for ci, (s, l) in enumerate(calls):
        x = runner.activations(w, s, l).to(dev)
        logits = torch.from_numpy(lg[s, l]).to(dev)
        assert cache.forward(l, x, logits, y_ref, w.B) == mc.MOE_OK
        bank = pool[l * w.E:(l + 1) * w.E].to(dev)
        sh = shared[l] if shared is not None else None
        st = mc.moe_layer_forward_resident_noalloc(cache.desc, bank, sh, x, logits, w.B, y_new,
                                                   torch.cuda.current_stream())
        assert st == mc.MOE_OK, mc.moe_last_error()
        torch.cuda.synchronize()
        got = y_new.float().cpu().numpy().astype(np.float64)
        H.assert_layer_close(got, ref.calls[ci].y, f"call ({s}, {l}) against the oracle")
        H.assert_layer_close(got, y_ref.float().cpu().numpy().astype(np.float64), f"call ({s}, {l}) against "
                                                                                   f"moe_layer_forward")
    cache.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from expert_cache_serving_gb300 import moecache as mc

    dev = torch.device("cuda")
    # (16 * 16 + 16) * 8192 * 4 bytes of intermediate: more than the 4 MiB scratch
    desc = mc.moe_model_desc(1, 64, 16, 256, 8192, mc.MOE_BF16, 1, 16)
    t = torch.zeros(16, dtype=torch.uint8, device=dev)
    st = mc.moe_layer_forward_resident_noalloc(desc, t, t, t, t, 16, t, None)
    assert st == mc.MOE_ERR_INVALID_ARG
    assert "4 MiB" in mc.moe_last_error()
