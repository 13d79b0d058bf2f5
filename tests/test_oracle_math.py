"""Pins for the oracle's router, permutation, FP4 decoding, records, SwiGLU
expert, layer combine and q* (oracle.*).  Each check rests on something other
than the oracle's own formula: the formats' published constants, closed-form
identities, library routines, brute-force loops, or the pages' worked numbers
(tests/golden/)."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import synth
from oracle import ffn, fp4, permute, qstar, records, router

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


# ---------------------------------------------------------------- router ----

def test_router_selection_property_with_ties():
    rng = np.random.default_rng(0)
    for _ in range(200):
        E = int(rng.integers(2, 12))
        k = int(rng.integers(1, E + 1))
        logits = rng.integers(-2, 3, size=(3, E)).astype(np.float64)  # many ties
        ids, w = router.topk_softmax(logits, k)
        for t in range(3):
            sel = list(ids[t])
            assert len(set(sel)) == k
            rest = [e for e in range(E) if e not in sel]
            for a in sel:
                for b in rest:
                    assert logits[t, a] > logits[t, b] or (logits[t, a] == logits[t, b] and a < b)
            # selection order: non-increasing logit, equal logits by ascending id
            for a, b in zip(sel, sel[1:]):
                assert logits[t, a] > logits[t, b] or (logits[t, a] == logits[t, b] and a < b)


def test_router_weights_closed_forms():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((5, 16))
    ids, w = router.topk_softmax(logits, 4)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    for t in range(5):
        for a, b in itertools.combinations(range(4), 2):
            assert math.isclose(w[t, a] / w[t, b], math.exp(logits[t, ids[t, a]] - logits[t, ids[t, b]]),
                                rel_tol=1e-12)
    # renormalised full softmax over the selected experts (library softmax)
    p = scipy.special.softmax(logits, axis=1)
    for t in range(5):
        sel = p[t, ids[t]]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-12)


def test_router_k_equals_E_is_full_softmax():
    logits = np.random.default_rng(2).standard_normal((4, 6))
    ids, w = router.topk_softmax(logits, 6)
    full = scipy.special.softmax(logits, axis=1)
    for t in range(4):
        assert np.allclose(w[t], full[t, ids[t]], rtol=1e-12)


def test_router_degenerate_cases():
    ids, w = router.topk_softmax(np.zeros((2, 8)), 3)
    assert (ids == [[0, 1, 2], [0, 1, 2]]).all()
    assert np.allclose(w, 1.0 / 3)
    row = np.array([[np.nan, 1.0, np.nan, -5.0]])
    ids, _ = router.topk_softmax(row, 2)
    assert list(ids[0]) == [1, 3]


def test_router_non_finite_rows_take_the_equal_logit_limit():
    # every selected logit -inf (or NaN): the limit of a softmax over equal
    # logits, i.e. uniform weights over the k lowest ids (library softmax on
    # equal finite logits gives the same)
    for row in (np.full((1, 6), -np.inf), np.full((1, 6), np.nan)):
        ids, w = router.topk_softmax(row, 3)
        assert list(ids[0]) == [0, 1, 2]
        assert np.allclose(w[0], scipy.special.softmax(np.zeros(3)), rtol=0, atol=1e-15)
    # +inf entries share the weight: the limit of softmax([M, M, 0]) as M grows
    row = np.array([[0.0, np.inf, -1.0, np.inf]])
    ids, w = router.topk_softmax(row, 3)
    assert list(ids[0]) == [1, 3, 0]
    assert np.allclose(w[0], scipy.special.softmax(np.array([800.0, 800.0, 0.0])), rtol=0, atol=1e-15)
    # a single real logit above -inf: all the weight on it
    row = np.array([[-np.inf, -np.inf, 0.25, np.nan]])
    ids, w = router.topk_softmax(row, 3)
    assert list(ids[0]) == [2, 0, 1] and list(w[0]) == [1.0, 0.0, 0.0]


def test_router_logits_brute_force():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 5))
    wr = rng.standard_normal((3, 5))
    got = router.logits_from_router(x, wr)
    for t in range(2):
        for e in range(3):
            assert math.isclose(got[t, e], sum(x[t, h] * wr[e, h] for h in range(5)), rel_tol=1e-12, abs_tol=1e-12)
    assert router.topk_margin(np.array([[3.0, 1.0, 2.0]]), 1) == 1.0


# ----------------------------------------------------------- permutation ----

def test_permutation_matches_bucket_sort():
    rng = np.random.default_rng(4)
    for _ in range(50):
        E = int(rng.integers(1, 9))
        ids = rng.integers(0, E, size=(int(rng.integers(1, 6)), int(rng.integers(1, 4))))
        perm, off = permute.permutation(ids, E)
        buckets = [[] for _ in range(E)]
        for p, e in enumerate(ids.reshape(-1)):
            buckets[e].append(p)
        assert list(perm) == [p for b in buckets for p in b]
        assert list(np.diff(off)) == [len(b) for b in buckets]
        assert off[0] == 0 and off[-1] == ids.size


# ------------------------------------------------------------------- fp4 ----

def test_e2m1_table_matches_spec_values():
    # OCP MX v1.0, FP4 (E2M1): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = mags[c & 7] * (-1.0 if c >= 8 else 1.0)
        assert fp4.e2m1_value(c) == want
        assert fp4.E2M1[c] == want


def test_e4m3_exhaustive_against_integer_construction():
    # e4m3 = sign * (8 + m) * 2^(e - 10) for e >= 1, sign * m * 2^-9 for e = 0;
    # exponent 15 with mantissa 7 is NaN.
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e, m = (b >> 3) & 15, b & 7
        v = fp4.e4m3_value(b)
        if e == 15 and m == 7:
            assert math.isnan(v)
            continue
        want = s * (m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10))
        assert v == want
    # published landmarks
    assert fp4.e4m3_value(0x7E) == 448.0
    assert fp4.e4m3_value(0x08) == 2.0 ** -6
    assert fp4.e4m3_value(0x01) == 2.0 ** -9
    assert fp4.e4m3_value(0x38) == 1.0
    assert fp4.e4m3_value(0xC0) == -2.0


def test_fp4_products_exact_in_float32_and_bf16():
    # every e2m1 * e4m3 product must be exactly representable in float32 and in bf16
    for c in range(16):
        for b in range(256):
            if b in (0x7F, 0xFF):
                continue
            p = fp4.E2M1[c] * fp4.E4M3[b]
            assert float(np.float32(p)) == p
            assert float(synth.bf16_bits_to_f32(synth.to_bf16_bits(np.float32([p])))[0]) == p


def test_dequant_nibble_order_and_scale_axis():
    codes = np.array([[0x21, 0xF7] + [0] * 6], dtype=np.uint8)  # 16 elements
    scales = np.array([[0x40]], dtype=np.uint8)  # e4m3 0x40 = 2.0
    w = fp4.dequant_rows(codes, scales)
    assert list(w[0, :4]) == [1.0, 2.0, 12.0, -12.0]  # 0.5*2, 1*2, 6*2, -6*2
    codes = np.full((1, 16), 0x22, dtype=np.uint8)  # 32 elements of 1.0
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)  # block 0 scale 1, block 1 scale 2
    w = fp4.dequant_rows(codes, scales)
    assert (w[0, :16] == 1.0).all() and (w[0, 16:] == 2.0).all()


def test_fp4_record_within_quantisation_bound():
    # dequantised weights stay within the e2m1 rounding bound of the values the
    # generator quantised: half the local e2m1 gap times the block scale, or
    # the saturation excess above 6 * scale.
    H, I = 64, 32
    rec = synth.expert_record(5, 9, H, I, synth.WD_FP4)
    g, u, d = records.parse(rec, H, I, records.FP4)
    v = synth.element_values(5, 9, 0, 3 * H * I, 0.02).astype(np.float64)
    for t, (m, R, K) in enumerate([(g, I, H), (u, I, H), (d, H, I)]):
        orig = v[t * H * I:(t + 1) * H * I].reshape(R, K)
        blocks = orig.reshape(R, K // 16, 16)
        scale = np.array([[fp4.E4M3[synth._rne_encode(np.float32(np.abs(b).max() / 6), synth.E4M3_ENC)]
                           for b in row] for row in blocks])
        err = np.abs(m.reshape(R, K // 16, 16) - blocks)
        bound = np.maximum(1.0 * scale[:, :, None], np.abs(blocks) - 6 * scale[:, :, None]) + 1e-12
        assert (err <= bound).all()


# --------------------------------------------------------------- records ----

def test_record_sizes_match_pages_pool_size():
    gd = read_golden("pool_bytes.txt")
    S = records.record_size(int(gd["H"]), int(gd["I"]), records.BF16)
    pool = gd["L"] * gd["E"] * S
    assert abs(pool / 1e9 - gd["pool_GB"]) < 0.05
    t = pool / 1e9 / gd["B_P_GBps"]
    assert gd["chunk_s_lo"] - 0.01 <= t <= gd["chunk_s_hi"] + 0.01


def test_record_parse_bf16_and_fp32_layout():
    H, I = 32, 16
    v = synth.element_values(2, 3, 0, 3 * H * I, 0.02)
    g, u, d = records.parse(synth.expert_record(2, 3, H, I, synth.WD_FP32), H, I, records.FP32)
    assert (g == v[:H * I].reshape(I, H)).all() and (d == v[2 * H * I:].reshape(H, I)).all()
    g, u, d = records.parse(synth.expert_record(2, 3, H, I, synth.WD_BF16), H, I, records.BF16)
    assert np.allclose(u, v[H * I:2 * H * I].reshape(I, H), rtol=2 ** -8, atol=0)


# ------------------------------------------------------------------- ffn ----

def brute_expert(x, wg, wu, wd):
    n, H = len(x), len(x[0])
    I = len(wg)
    out = []
    for t in range(n):
        h = []
        for i in range(I):
            a = sum(x[t][c] * wg[i][c] for c in range(H))
            b = sum(x[t][c] * wu[i][c] for c in range(H))
            h.append(a / (1 + math.exp(-a)) * b)
        out.append([sum(h[i] * wd[r][i] for i in range(I)) for r in range(H)])
    return np.array(out)


def test_expert_brute_force():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 6))
    wg, wu, wd = rng.standard_normal((4, 6)), rng.standard_normal((4, 6)), rng.standard_normal((6, 4))
    assert np.allclose(ffn.expert(x, wg, wu, wd), brute_expert(x.tolist(), wg.tolist(), wu.tolist(), wd.tolist()),
                       rtol=1e-12, atol=1e-12)


def test_silu_identities():
    z = np.linspace(-30, 30, 601)
    assert np.allclose(ffn.silu(z) - ffn.silu(-z), z, rtol=0, atol=1e-12)  # z*s(z) + z*s(-z) = z
    assert ffn.silu(np.array([0.0]))[0] == 0.0
    assert math.isclose(ffn.silu(np.array([40.0]))[0], 40.0, rel_tol=1e-15)
    assert math.isclose(ffn.silu(np.array([1.0]))[0], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)


def test_expert_zero_gate_and_linearity():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 8))
    wg, wu, wd = rng.standard_normal((5, 8)), rng.standard_normal((5, 8)), rng.standard_normal((8, 5))
    assert (ffn.expert(x, np.zeros_like(wg), wu, wd) == 0).all()
    assert np.allclose(ffn.expert(x, wg, 3 * wu, wd), 3 * ffn.expert(x, wg, wu, wd), rtol=1e-12)
    assert np.allclose(ffn.expert(x, wg, wu, -2 * wd), -2 * ffn.expert(x, wg, wu, wd), rtol=1e-12)


def _toy_experts(E, H, I, seed=7):
    rng = np.random.default_rng(seed)
    ws = [(rng.standard_normal((I, H)) * 0.3, rng.standard_normal((I, H)) * 0.3, rng.standard_normal((H, I)) * 0.3)
          for _ in range(E)]
    return ws


def test_layer_equals_dense_gate_masked_evaluation():
    E, H, I, k, B = 6, 8, 5, 2, 4
    ws = _toy_experts(E, H, I)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((B, H))
    logits = rng.standard_normal((B, E))
    ids, w = router.topk_softmax(logits, k)
    y = ffn.moe_layer(x, ids, w, lambda e: ws[e])
    p = scipy.special.softmax(logits, axis=1)
    gates = np.zeros((B, E))
    for t in range(B):
        top = np.argsort(-logits[t], kind="stable")[:k]
        gates[t, top] = p[t, top] / p[t, top].sum()
    assert np.allclose(y, ffn.dense_layer(x, gates, lambda e: ws[e], E), rtol=1e-10, atol=1e-12)
    # k = E: plain softmax-weighted sum of every expert
    ids, w = router.topk_softmax(logits, E)
    assert np.allclose(ffn.moe_layer(x, ids, w, lambda e: ws[e]), ffn.dense_layer(x, p, lambda e: ws[e], E),
                       rtol=1e-10, atol=1e-12)


def test_layer_shared_expert_is_additive():
    E, H, I = 4, 6, 3
    ws = _toy_experts(E, H, I)
    sh = _toy_experts(1, H, I, seed=9)[0]
    x = np.random.default_rng(10).standard_normal((3, H))
    ids, w = router.topk_softmax(np.random.default_rng(11).standard_normal((3, E)), 2)
    diff = ffn.moe_layer(x, ids, w, lambda e: ws[e], sh) - ffn.moe_layer(x, ids, w, lambda e: ws[e])
    assert np.allclose(diff, ffn.expert(x, *sh), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- qstar ----

def test_qstar_worked_example():
    gd = read_golden("qstar_fig2.txt")
    m = int(gd["m"])
    assert int(gd["routed"]) - int(gd["hits"]) == m
    q = qstar.qstar(m, gd["B_P"], gd["B_H"])
    assert q == int(gd["qstar"])
    assert m - q == int(gd["cpu"])


def test_qstar_limits_and_balance():
    assert qstar.qstar(0, 1, 4) == 0
    assert qstar.qstar(7, 10, 10) == 7          # B_H -> B_P: pure on-demand fill
    assert qstar.qstar(7, 10, 10.0001) == 7
    assert qstar.qstar(3, 1, 1000) == 1          # at least one fill keeps warming the cache
    m, S, bp, bh = 6, 1.0, 2.0, 6.0              # q* = 2 exactly
    q = qstar.qstar(m, bp, bh)
    tf, tc = qstar.branch_times(m, q, S, bp, bh)
    assert q == 2 and math.isclose(tf, tc, rel_tol=1e-12)
