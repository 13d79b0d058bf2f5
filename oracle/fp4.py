"""FP4 expert weights: e2m1 element codes with one e4m3 scale per 16 elements (oracle).

The pages deploy DeepSeek-V4-Flash experts in MXFP4 and GLM-5.2 / Qwen3.6 in
NVFP4 (FreeToken write-up, experimental setup).  The format decoded here is an
e2m1 element code times an e4m3 scale shared by a block of 16 consecutive
elements of a row (OCP Microscaling Formats v1.0 element encodings).

Readings where the pages are silent: element 2c of a row sits in the low
nibble of code byte c; scale blocks run along the row (the input dimension of
the matrix); there is no further per-tensor scale.

Every decoded weight is exactly representable in float32 (at most 2 + 4
significant bits, exponent within range), so dequantisation is exact.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        mag = 0.5 * man  # subnormal: 2^(1-1) * (m / 2)
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + 0.5 * man)
    return sign * mag


def e4m3_value(byte: int) -> float:
    """Value of an e4m3 byte: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.

    Exponent 15 with mantissa 7 is NaN (no infinities)."""
    sign = -1.0 if byte & 0x80 else 1.0
    exp = (byte >> 3) & 0xF
    man = byte & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        mag = 2.0 ** -6 * (man / 8.0)
    else:
        mag = 2.0 ** (exp - 7) * (1.0 + man / 8.0)
    return sign * mag


E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3 = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def dequant_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes u8 [R, K/2], scales u8 [R, K/16] -> float64 weights [R, K]."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    R, half = codes.shape
    K = 2 * half
    elem = np.empty((R, K), dtype=np.uint8)
    elem[:, 0::2] = codes & 0x0F
    elem[:, 1::2] = codes >> 4
    scale_per_elem = np.repeat(E4M3[scales], 16, axis=1)
    return E2M1[elem] * scale_per_elem
