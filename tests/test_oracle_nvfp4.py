"""Pins of the FP4 x FP4 oracle (oracle/nvfp4.py) against independent facts:
brute-force nearest-value searches, printed format constants, exact round
trips of representable blocks, the quantisation error bound and a pure-Python
brute-force layer on tiny inputs."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp4, nvfp4


def _nearest_even(v: float, values: list[float]) -> int:
    """Brute force: the code whose value is nearest to v (exact rational
    distances), ties to the even code."""
    best, best_d = None, None
    for c, val in enumerate(values):
        d = abs(Fraction(val) - Fraction(v))
        if best is None or d < best_d or (d == best_d and c % 2 == 0 and best % 2 == 1):
            best, best_d = c, d
    return best


E4M3_VALUES = [fp4.e4m3_value(b) for b in range(127)]
E2M1_VALUES = [fp4.e2m1_value(c) for c in range(8)]


def _probe_values(values, rng, n_random):
    """Every table value, every midpoint, the float32 neighbours of both, random
    magnitudes over the table's range and beyond."""
    out = []
    for a, b in zip(values, values[1:]):
        for m in (a, (a + b) / 2):
            f = np.float32(m)
            out += [f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(np.inf))]
    top = values[-1]
    out += list(rng.uniform(0, top * 1.2, n_random).astype(np.float32))
    out += list((np.exp(rng.uniform(math.log(1e-6), math.log(top * 4), n_random))).astype(np.float32))
    out += [np.float32(top * 1.01), np.float32(top * 10), np.float32(1e30)]
    return np.array(out, dtype=np.float32)


def test_e4m3_rne_matches_brute_force_nearest_even():
    rng = np.random.default_rng(11)
    v = _probe_values(E4M3_VALUES, rng, 3000)
    got = nvfp4.e4m3_rne(v)
    for x, g in zip(v, got):
        assert int(g) == _nearest_even(float(x), E4M3_VALUES), (float(x), int(g))
    neg = nvfp4.e4m3_rne(-v)
    assert np.array_equal(neg, np.where(got != 0, got | 0x80, 0).astype(np.uint8))


def test_e2m1_rne_matches_brute_force_nearest_even():
    rng = np.random.default_rng(12)
    v = _probe_values(E2M1_VALUES, rng, 3000)
    got = nvfp4.e2m1_rne(v)
    for x, g in zip(v, got):
        assert int(g) == _nearest_even(float(x), E2M1_VALUES), (float(x), int(g))
    neg = nvfp4.e2m1_rne(-v)
    assert np.array_equal(neg, np.where(got != 0, got | 0x8, 0).astype(np.uint8))


def test_format_constants():
    # OCP e4m3: 1.0 = 0x38, largest finite 448 = 0x7E, smallest subnormal 2^-9 = 0x01
    assert nvfp4.e4m3_rne(np.float32(1.0)) == 0x38
    assert nvfp4.e4m3_rne(np.float32(448.0)) == 0x7E
    assert nvfp4.e4m3_rne(np.float32(1e6)) == 0x7E  # saturating
    assert nvfp4.e4m3_rne(np.float32(2.0 ** -9)) == 0x01
    assert nvfp4.e4m3_rne(np.float32(2.0 ** -10)) == 0x00  # tie between 0 and 2^-9 -> even
    assert nvfp4.e4m3_rne(np.float32(3 * 2.0 ** -10)) == 0x02  # tie between 0x01 and 0x02 -> even
    # e2m1 grid 0, 0.5, 1, 1.5, 2, 3, 4, 6: ties to the even code
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 7.0: 7, 100.0: 7,
             -0.2: 0, -0.3: 0x9, -6.5: 0xF, 0.0: 0}
    for v, c in cases.items():
        assert nvfp4.e2m1_rne(np.float32(v)) == c, v
    assert nvfp4.e2m1_rne(np.float32(-0.0)) == 0


def test_quantize_round_trips_representable_blocks():
    """A block whose largest magnitude is code 7 (6 x scale) is reproduced exactly:
    amax / 6 is the scale itself and every element divides to a grid value."""
    rng = np.random.default_rng(13)
    R, K = 64, 128
    scale = rng.integers(0x08, 0x70, size=(R, K // 16)).astype(np.uint8)  # normal e4m3, 6*s exact
    elem = rng.integers(0, 8, size=(R, K)).astype(np.uint8)
    elem[:, ::16] = 7  # the block maximum
    sign = rng.integers(0, 2, size=(R, K)).astype(np.uint8) * 8
    elem = np.where(elem != 0, elem | sign, 0).astype(np.uint8)
    codes = (elem[:, 0::2] | (elem[:, 1::2] << 4)).astype(np.uint8)
    v = fp4.dequant_rows(codes, scale).astype(np.float32)
    qc, qs = nvfp4.quantize(v)
    assert np.array_equal(qs, scale)
    assert np.array_equal(qc, codes)


def test_quantize_nibble_order_and_zero_blocks():
    v = np.zeros((1, 32), dtype=np.float32)
    v[0, :16] = [6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, 0]
    codes, scales = nvfp4.quantize(v)
    assert scales[0, 0] == 0x38 and scales[0, 1] == 0  # scale 1.0; the all-zero block gets scale 0
    assert codes[0, 0] == (7 | (6 << 4))  # element 0 in the low nibble
    assert codes[0, 3] == (1 | (0 << 4))
    assert codes[0, 4] == (0xF | (0xE << 4))
    assert np.all(codes[0, 8:] == 0)


def test_quantize_error_bound():
    """|q(v) - v| <= half the local grid spacing x scale inside the grid, and the
    saturation distance above it; the scale is within e4m3 rounding of amax/6."""
    rng = np.random.default_rng(14)
    v = (rng.standard_normal((256, 256)) * np.exp(rng.uniform(-4, 4, (256, 1)))).astype(np.float32)
    codes, scales = nvfp4.quantize(v)
    s = fp4.E4M3[scales]
    amax = np.abs(v.reshape(256, 16, 16)).max(-1).astype(np.float64)
    assert np.all(np.abs(s - amax / 6) <= s * 2.0 ** -4 + 2.0 ** -10)
    q = np.abs(v.astype(np.float64)) / np.repeat(s, 16, axis=1)
    gap = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    bound = np.maximum(0.5 * gap, q - 6.0) * np.repeat(s, 16, axis=1)
    err = np.abs(nvfp4.dequant(codes, scales) - v.astype(np.float64))
    assert np.all(err <= bound * (1 + 1e-12) + 1e-300)


def _bf_quant(vals: list[float]) -> list[float]:
    """Pure-Python fake quantisation of one row (float32 steps via numpy scalars)."""
    out = []
    for b in range(0, len(vals), 16):
        blk = [np.float32(x) for x in vals[b:b + 16]]
        amax = max(abs(x) for x in blk)
        sc = E4M3_VALUES[_nearest_even(float(np.float32(amax) / np.float32(6.0)), E4M3_VALUES)]
        for x in blk:
            if sc == 0:
                out.append(0.0)
                continue
            q = float(np.float32(x) / np.float32(sc))
            mag = E2M1_VALUES[_nearest_even(abs(q), E2M1_VALUES)]
            out.append(math.copysign(mag, q) * sc)
    return out


def test_layer_brute_force_tiny():
    rng = np.random.default_rng(15)
    T, H, I, E, k = 5, 32, 32, 3, 2
    mats = []
    for _ in range(E + 1):
        trip = []
        for rows, cols in ((I, H), (I, H), (H, I)):
            c = rng.integers(0, 256, size=(rows, cols // 2)).astype(np.uint8)
            s = rng.integers(0x20, 0x40, size=(rows, cols // 16)).astype(np.uint8)
            trip.append(fp4.dequant_rows(c, s))
        mats.append(trip)
    x = rng.standard_normal((T, H)).astype(np.float32)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)])
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    got = nvfp4.moe_layer(x, ids, w, lambda e: mats[e], shared=mats[E])

    def bf_expert(xt, trip):
        wg, wu, wd = trip
        xq = _bf_quant(list(xt))
        g = [sum(xq[c] * wg[r, c] for c in range(H)) for r in range(I)]
        u = [sum(xq[c] * wu[r, c] for c in range(H)) for r in range(I)]
        h = [float(np.float32(g[r] / (1.0 + math.exp(-g[r])) * u[r])) for r in range(I)]
        hq = _bf_quant(h)
        return [sum(hq[c] * wd[r, c] for c in range(I)) for r in range(H)]

    for t in range(T):
        ref = [0.0] * H
        for j in range(k):
            o = bf_expert(x[t], mats[ids[t, j]])
            ref = [a + float(w[t, j]) * b for a, b in zip(ref, o)]
        o = bf_expert(x[t], mats[E])
        ref = [a + b for a, b in zip(ref, o)]
        np.testing.assert_allclose(got[t], ref, rtol=1e-9, atol=1e-9 * max(abs(r) for r in ref))


def test_layer_zero_input_and_weight_linearity():
    rng = np.random.default_rng(16)
    H, I = 64, 32
    trip = [fp4.dequant_rows(rng.integers(0, 256, size=(r, c // 2)).astype(np.uint8),
                             rng.integers(0x20, 0x40, size=(r, c // 16)).astype(np.uint8))
            for r, c in ((I, H), (I, H), (H, I))]
    x = np.zeros((2, H), dtype=np.float32)
    assert np.all(nvfp4.expert(x, *trip) == 0)
    x = rng.standard_normal((3, H)).astype(np.float32)
    ids = np.zeros((3, 2), dtype=np.int64)
    ids[:, 1] = 1
    w = np.array([[0.25, 0.75], [1.0, 0.0], [0.5, 0.5]], dtype=np.float32)
    y = nvfp4.moe_layer(x, ids, w, lambda e: trip)
    np.testing.assert_allclose(y, nvfp4.expert(x, *trip), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("K", [8, 24])
def test_quantize_rejects_partial_blocks(K):
    with pytest.raises(ValueError):
        nvfp4.quantize(np.zeros((1, K), dtype=np.float32))
