"""FP4 x FP4 prefill arithmetic: activations quantised to the weights' format (oracle).

TEST INFRASTRUCTURE ONLY: plain NumPy, imported by tests, smoke() and the
bench's CPU baseline, never by the GPU path.

The pages deploy DeepSeek-V4-Flash experts in MXFP4 and GLM-5.2 / Qwen3.6 in
NVFP4 (FreeToken write-up, experimental setup); on Blackwell tensor cores a
block-scaled FP4 x FP4 product needs both operands in that format, so the
activations of the prefill GEMMs are quantised too.  The pages say nothing
about activation quantisation; the readings taken here:

* format: the weights' own (fp4.py): e2m1 codes, one e4m3 scale per block of
  16 consecutive elements along the contraction dimension, no per-tensor
  scale; element 2c in the low nibble of byte c;
* quantiser: scale = e4m3(amax / 6) and code = e2m1(v / scale), both rounded
  to nearest with ties to the even code and saturated to the largest finite
  value (448 for e4m3, 6 for e2m1); amax / 6 and v / scale are float32
  divisions, so both sides of a parity test take every rounding decision on
  the same float32 numbers; a block whose scale rounds to 0 gets codes 0; a
  value that rounds to magnitude 0 gets code 0 (never the negative zero 0x8);
* what is quantised: the layer input x (bf16, so exact in float32) before the
  gate/up contraction, and the SwiGLU output h, rounded to float32, before the
  down contraction; the contractions themselves are exact sums of products of
  the dequantised values (float64 here).
"""
from __future__ import annotations

import numpy as np

from . import ffn, fp4

E4M3_POS = fp4.E4M3[:127]   # codes 0x00..0x7E: every finite non-negative e4m3 value, ascending
E2M1_POS = fp4.E2M1[:8]     # codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6
E4M3_MAX, E2M1_MAX = 448.0, 6.0


def _round_to_table(mag: np.ndarray, table: np.ndarray, top: float) -> np.ndarray:
    """Index of the nearest entry of an ascending table of magnitudes; ties to
    the even index; magnitudes at or above `top` saturate to the last entry."""
    a = np.asarray(mag, dtype=np.float64)
    last = len(table) - 1
    lo = np.clip(np.searchsorted(table, a, side="right") - 1, 0, last)
    hi = np.minimum(lo + 1, last)
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    pick_hi = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)))
    idx = np.where(pick_hi, hi, lo)
    return np.where(a >= top, last, idx).astype(np.int64)


def e4m3_rne(v) -> np.ndarray:
    """float32 values -> e4m3 bytes (round to nearest even, saturating)."""
    v = np.asarray(v, dtype=np.float32)
    code = _round_to_table(np.abs(v), E4M3_POS, E4M3_MAX)
    neg = np.signbit(v) & (code != 0)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def e2m1_rne(v) -> np.ndarray:
    """float32 values -> e2m1 codes 0..15 (round to nearest even, saturating at 6;
    magnitude 0 always gets code 0)."""
    v = np.asarray(v, dtype=np.float32)
    code = _round_to_table(np.abs(v), E2M1_POS, E2M1_MAX)
    neg = np.signbit(v) & (code != 0)
    return (code | np.where(neg, 0x8, 0)).astype(np.uint8)


def quantize(v) -> tuple[np.ndarray, np.ndarray]:
    """v float32 [..., K] (K a multiple of 16) -> (codes u8 [..., K/2], scales u8 [..., K/16])."""
    v = np.asarray(v, dtype=np.float32)
    K = v.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    blocks = v.reshape(v.shape[:-1] + (K // 16, 16))
    amax = np.max(np.abs(blocks), axis=-1)
    scales = e4m3_rne(amax / np.float32(6.0))
    s = fp4.E4M3[scales].astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, blocks / np.where(s > 0, s, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    elem = e2m1_rne(q).reshape(v.shape)
    codes = (elem[..., 0::2] | (elem[..., 1::2] << 4)).astype(np.uint8)
    return codes, scales


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse of quantize's encoding for any leading shape -> float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    lead = codes.shape[:-1]
    return fp4.dequant_rows(codes.reshape(-1, codes.shape[-1]), scales.reshape(-1, scales.shape[-1])).reshape(
        lead + (2 * codes.shape[-1],))


def fake_quant(v) -> np.ndarray:
    """dequant(quantize(v)): the value the FP4 x FP4 GEMM sees for v (float64)."""
    return dequant(*quantize(v))


def expert(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """FP4 x FP4 SwiGLU expert on x [n, H] (float32 values) -> [n, H] float64.

    The weights are the dequantised FP4 matrices (float64, exact)."""
    xq = fake_quant(np.asarray(x, dtype=np.float32))
    h = (ffn.silu(xq @ w_gate.T) * (xq @ w_up.T)).astype(np.float32)
    return fake_quant(h) @ w_down.T


def moe_layer(x: np.ndarray, ids: np.ndarray, w: np.ndarray, get_expert, shared=None) -> np.ndarray:
    """y [T, H] = sum_j w[t, j] * expert_{ids[t, j]}(x_t) (+ shared(x_t)), rank order, float64.

    get_expert(e) -> (W_gate, W_up, W_down) dequantised; shared is None or such a triple."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    y = np.zeros((T, H), dtype=np.float64)
    by_expert: dict[int, list[tuple[int, int]]] = {}
    for t in range(T):
        for j in range(ids.shape[1]):
            by_expert.setdefault(int(ids[t, j]), []).append((t, j))
    contrib = np.zeros((T, ids.shape[1], H), dtype=np.float64)
    for e, pairs in by_expert.items():
        rows = np.array([t for t, _ in pairs])
        o = expert(x[rows], *get_expert(e))
        for (t, j), oi in zip(pairs, o):
            contrib[t, j] = oi
    for j in range(ids.shape[1]):
        y += w[:, j:j + 1].astype(np.float64) * contrib[:, j]
    if shared is not None:
        y += expert(x, *shared)
    return y
