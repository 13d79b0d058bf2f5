"""Workload driver over the C ABI: builds the pinned host expert pool and the
device-resident shared experts for a workload, creates the cache and runs
decode steps.  Used by the GPU tests, smoke() and bench.py; it only moves
inputs and calls the library (every step of the layer runs in CUDA)."""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth.configs import Workload

from . import moecache as mc


def model_desc(w: Workload, max_tokens: int | None = None) -> mc.moe_model_desc:
    return mc.moe_model_desc(w.L, w.E, w.k, w.H, w.I, w.wdtype, int(w.shared), max_tokens or w.B)


def build_pool(w: Workload, threads: int | None = None) -> torch.Tensor:
    """Host tensor u8 [L*E, S] over exact-size pinned memory holding every routed
    expert record, generated on the GPU (the seeded generator's CUDA twin)."""
    return torch.from_numpy(synth.pinned_pool(w.seed, w.LE, w.H, w.I, w.wdtype, w.sigma))


def build_shared(w: Workload, device="cuda") -> torch.Tensor | None:
    """Device tensor u8 [L, S] of the per-layer shared experts (keys L*E + l), or None."""
    if not w.shared:
        return None
    recs = synth.records_array(w.seed, w.LE, w.L, w.H, w.I, w.wdtype, w.sigma)
    return torch.from_numpy(recs).to(device)


def x_dtype(w: Workload):
    return torch.float32 if w.wdtype == synth.WD_FP32 else torch.bfloat16


def activations(w: Workload, step: int, layer: int, B: int | None = None) -> torch.Tensor:
    """Host tensor [B, H] (fp32 for fp32 models, bf16 otherwise) of N(0,1) activations."""
    B = B or w.B
    if w.wdtype == synth.WD_FP32:
        return torch.from_numpy(synth.activations_f32(w.seed, step, layer, B, w.H))
    bits = synth.activations_bf16(w.seed, step, layer, B, w.H)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


class Cache:
    """Owns one moecache cache plus the pool it reads."""

    def __init__(self, w: Workload, pool: torch.Tensor, shared: torch.Tensor | None, C: int | None = None,
                 max_slots: int = 0, max_tokens: int | None = None):
        self.w = w
        self.pool = pool
        self.shared = shared
        self.desc = model_desc(w, max_tokens)
        self.handle = mc.moe_cache_create(self.desc, pool, shared, w.C if C is None else C, max_slots)

    def forward(self, layer, x, logits, y, B, router_w=None, stream=None, aux=None) -> int:
        if stream is None:
            stream = torch.cuda.current_stream()
        return mc.moe_layer_forward(self.handle, layer, x, logits, router_w, B, y, stream, aux)

    def close(self):
        if self.handle:
            mc.moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
