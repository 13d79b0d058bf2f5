"""Expert records: the bytes one cache slot (or host-pool row) holds (oracle).

FreeToken write-up, "expert banks and the FTW format" section: expert weights
are stored in banks whose leading dimension is the flat id ``l*E + e``; the
rows with the same id make up one expert, and a cache slot holds every tensor
of one (layer, expert) pair ("FreeToken's design" section).  The record here
holds the three SwiGLU matrices of one expert (the Luce Spark post: a swap
copies three weight tensors).

Layout (row-major, [out][in]):
* fp32 / bf16: ``W_gate[I][H] | W_up[I][H] | W_down[H][I]``.
* FP4: ``gate codes[I][H/2] | up codes[I][H/2] | gate scales[I][H/16] |
  up scales[I][H/16] | down codes[H][I/2] | down scales[H][I/16]``.
"""
from __future__ import annotations

import numpy as np

from . import fp4

FP32, BF16, FP4 = 0, 1, 2


def record_size(H: int, I: int, wdtype: int) -> int:
    if wdtype == FP32:
        return 4 * 3 * H * I
    if wdtype == BF16:
        return 2 * 3 * H * I
    if wdtype == FP4:
        return 3 * H * I // 2 + 3 * H * I // 16
    raise ValueError(wdtype)


def _bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def parse(record: np.ndarray, H: int, I: int, wdtype: int):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) as float64 from one record's bytes."""
    rec = np.ascontiguousarray(record, dtype=np.uint8).reshape(-1)
    if rec.size != record_size(H, I, wdtype):
        raise ValueError("record size mismatch")
    HI = H * I
    if wdtype == FP32:
        v = rec.view(np.float32).astype(np.float64)
    elif wdtype == BF16:
        v = _bf16_to_f64(rec.view(np.uint16))
    else:
        q, e = HI // 2, HI // 16  # code and scale bytes of one matrix
        gc, uc = rec[0:q], rec[q:2 * q]
        gs, us = rec[2 * q:2 * q + e], rec[2 * q + e:2 * q + 2 * e]
        dc, ds = rec[2 * q + 2 * e:3 * q + 2 * e], rec[3 * q + 2 * e:]
        g = fp4.dequant_rows(gc.reshape(I, H // 2), gs.reshape(I, H // 16))
        u = fp4.dequant_rows(uc.reshape(I, H // 2), us.reshape(I, H // 16))
        d = fp4.dequant_rows(dc.reshape(H, I // 2), ds.reshape(H, I // 16))
        return g, u, d
    return v[:HI].reshape(I, H), v[HI:2 * HI].reshape(I, H), v[2 * HI:].reshape(H, I)
