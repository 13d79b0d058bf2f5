"""GPU parity of the FP4 x FP4 prefill (activations quantised to the weights'
e2m1 + e4m3-per-16 format, block-scaled tcgen05 GEMMs) against the oracle,
through the C ABI.

The quantiser (moe_quantize_fp4) is compared bit for bit on float32 and bf16
rows, including blocks that are zero, tiny (scale rounding to 0 or into the
e4m3 subnormals), huge (saturating scales), values on rounding ties and
negative values that round to zero.  Layer outputs are compared within
max|err| <= 1e-2 * max|ref|: the SwiGLU output is quantised from float32
sums whose order differs from the oracle's, so a code next to a rounding
boundary may differ by one step; the bound covers that.
"""
import numpy as np
import pytest

import synth
from oracle import nvfp4, router
from synth import configs
from tests import harness as H
from tests.test_gpu_prefill import prefill_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def _edge_rows(K, rng):
    rows = []
    rows.append(np.zeros(K, np.float32))                                  # all-zero blocks
    rows.append(np.full(K, 1e-30, np.float32))                            # scale rounds to 0
    rows.append((rng.standard_normal(K) * 2e-3).astype(np.float32))       # e4m3 subnormal scales
    rows.append((rng.standard_normal(K) * 1e4).astype(np.float32))        # saturating scales
    ties = np.tile(np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.2, -0.75, -5, 4, 2, 1, 0.5],
                            np.float32), K // 16)
    rows.append(ties)                                                     # amax 6 -> scale 1: exact ties
    rows.append((ties * np.float32(0.0625)).astype(np.float32))           # the same ties at scale 2^-4
    v = rng.standard_normal(K).astype(np.float32)
    v[::16] = 0
    rows.append(v)
    return np.stack(rows)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_quantizer_bit_exact(dtype):
    from expert_cache_serving_gb300 import moecache as mc

    rng = np.random.default_rng(21)
    R, K = 400, 512
    x = (rng.standard_normal((R, K)) * np.exp(rng.uniform(-6, 6, (R, 1)))).astype(np.float32)
    x = np.concatenate([x, _edge_rows(K, rng)])
    if dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        x = xt.float().numpy()
        xd = xt.cuda()
        kind = mc.MOE_BF16
    else:
        xd = torch.from_numpy(x).cuda()
        kind = mc.MOE_FP32
    rows = x.shape[0]
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    mc.moe_quantize_fp4(xd, kind, rows, K, codes, scales, torch.cuda.current_stream())
    torch.cuda.synchronize()
    rc, rs = nvfp4.quantize(x)
    gs, gc = scales.cpu().numpy(), codes.cpu().numpy()
    bad_s = np.argwhere(gs != rs)
    assert bad_s.size == 0, f"scales differ at {bad_s[:5].tolist()}: gpu {gs[tuple(bad_s[0])]} oracle {rs[tuple(bad_s[0])]}"
    bad_c = np.argwhere(gc != rc)
    assert bad_c.size == 0, f"codes differ at {bad_c[:5].tolist()}"


def test_quantizer_rejects_bad_arguments():
    from expert_cache_serving_gb300 import moecache as mc

    x = torch.zeros((4, 24), dtype=torch.float32, device="cuda")
    c = torch.empty((4, 16), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    st = mc.lib.moe_quantize_fp4(x.data_ptr(), mc.MOE_FP32, 4, 24, c.data_ptr(), s.data_ptr(), None)
    assert st == mc.MOE_ERR_INVALID_ARG
    st = mc.lib.moe_quantize_fp4(x.data_ptr(), 7, 4, 16, c.data_ptr(), s.data_ptr(), None)
    assert st == mc.MOE_ERR_INVALID_ARG


def oracle_w4a4(w, xs, lg, layers, bank, tokens=None):
    out = []
    for li, l in enumerate(layers):
        t_sel = np.arange(xs.shape[1]) if tokens is None else np.asarray(tokens)
        x = synth.bf16_bits_to_f32(xs[li][t_sel]).astype(np.float32)
        ids, wts = router.topk_softmax(lg[li][t_sel].astype(np.float64), w.k)
        shared = bank.get(w.LE + l) if w.shared else None
        out.append(nvfp4.moe_layer(x, ids, wts, lambda e, l=l: bank.get(l * w.E + e), shared))
    return out


def run_w4a4(w, T, layers, C, pool=None, shared=None):
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    dev = torch.device("cuda")
    pool = runner.build_pool(w) if pool is None else pool
    shared = runner.build_shared(w) if shared is None else shared
    cache = runner.Cache(w, pool, shared, C=C)
    mc.moe_cache_set_prefill_precision(cache.handle, mc.MOE_PREFILL_W4A4)
    xs, lg = prefill_inputs(w, T, len(layers))
    x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(lg).to(dev)
    y = torch.empty_like(x)
    st = mc.moe_prefill_stream(cache.handle, layers[0], layers[-1] + 1, x, logits, T, y, torch.cuda.current_stream())
    assert st == mc.MOE_OK, mc.moe_last_error()
    torch.cuda.synchronize()
    assert mc.moe_cache_sync(cache.handle, torch.cuda.current_stream()) == mc.MOE_OK
    return cache, xs, lg, y.float().cpu().numpy().astype(np.float64)


def test_w4a4_full_shape_parity():
    w = configs.SMALL_FP4.with_(C=32)
    layers = [0, 1]
    cache, xs, lg, y = run_w4a4(w, 160, layers, C=32)
    ref = oracle_w4a4(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"W4A4 prefill layer {layers[li]}")
    cache.close()


def test_w4a4_experts_spanning_several_row_tiles():
    w = configs.SMALL_FP4.with_(name="fp4-multi-tile", E=8, C=16)
    T = 512
    cache, xs, lg, y = run_w4a4(w, T, [0], C=16)
    ids, _ = router.topk_softmax(lg[0].astype(np.float64), w.k)
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    assert counts.min() > 128 and counts.max() > 256
    sample = list(range(0, T, 7)) + [T - 1]
    ref = oracle_w4a4(w, xs, lg, [0], H.ExpertBank(w), tokens=sample)
    H.assert_layer_close(y[0][sample], ref[0], "W4A4 prefill layer 0")
    cache.close()


def test_w4a4_narrow_shape_with_shared_expert():
    w = configs.SMALL_FP4_NARROW.with_(name="fp4-narrow-shared", shared=True, C=48)
    layers = [0, 1]
    cache, xs, lg, y = run_w4a4(w, 97, layers, C=48)
    ref = oracle_w4a4(w, xs, lg, layers, H.ExpertBank(w))
    for li in range(len(layers)):
        H.assert_layer_close(y[li], ref[li], f"W4A4 prefill layer {layers[li]}")
    cache.close()


def test_w4a4_needs_an_fp4_model():
    from expert_cache_serving_gb300 import moecache as mc
    from expert_cache_serving_gb300 import runner

    w = configs.SMALL_BF16
    cache = runner.Cache(w, runner.build_pool(w), runner.build_shared(w))
    st = mc.lib.moe_cache_set_prefill_precision(cache.handle, mc.MOE_PREFILL_W4A4)
    assert st == mc.MOE_ERR_INVALID_ARG
    cache.close()
