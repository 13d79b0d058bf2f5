"""Workload shapes: the five seeded configurations and the small parity cases.

A workload names its model shape (L, E, k, H, I, weight format, shared
expert), its cache capacity, its routing trace (decode steps and tokens per
step, AR(1) logits) and its seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

from . import WD_BF16, WD_FP32, WD_FP4


@dataclass(frozen=True)
class Workload:
    name: str
    L: int
    E: int
    k: int
    H: int
    I: int
    wdtype: int
    shared: bool
    C: int
    steps: int
    B: int
    seed: int
    router: bool = False          # logits = x W_r^T (else AR(1) trace logits)
    sigma: float = 0.02
    resize: tuple = field(default_factory=tuple)  # ((step, new_C), ...) applied before the step

    @property
    def LE(self) -> int:
        return self.L * self.E

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Tiny MoE: 2 layers, hidden 256, intermediate 128, 16 experts, top-2, fp32,
# router logits x W_r^T, 64 decode tokens at batch 1, 12 cache slots.
C1 = Workload("tiny-fp32-L2-E16-k2", L=2, E=16, k=2, H=256, I=128, wdtype=WD_FP32, shared=False, C=12,
              steps=64, B=1, seed=1, router=True)
# Qwen3.6-35B-A3B-shaped decode: 40 layers, hidden 2048, intermediate 512,
# 256 experts, top-8, one shared expert, bf16, 256 tokens at batch 1, cache of
# 50% of the 10,240 layer-experts.
C2 = Workload("qwen3.6-35b-a3b-shape-bf16-decode", L=40, E=256, k=8, H=2048, I=512, wdtype=WD_BF16, shared=True,
              C=5120, steps=256, B=1, seed=2)
# DeepSeek-V4-Flash-shaped decode: 43 layers, hidden 4096, intermediate 2048,
# 256 experts, top-6, FP4 e2m1 + e4m3/16, 512 tokens at batch 1 or 8, cache of
# 30% of the 11,008 layer-experts.
C3 = Workload("dsv4-flash-shape-fp4-decode", L=43, E=256, k=6, H=4096, I=2048, wdtype=WD_FP4, shared=False,
              C=3302, steps=512, B=1, seed=3)
C3_B8 = C3.with_(name="dsv4-flash-shape-fp4-decode-b8", B=8)
# Prefill through the config-3 model: one 4096-token prompt.
C4 = C3.with_(name="dsv4-flash-shape-fp4-prefill-4096", steps=1, B=4096, seed=4)
# Elastic cache: config-2 shapes, 2048 tokens, slots 60% -> 25% -> 80% of the
# 10,240 layer-experts before steps 512 and 1280.
C5 = C2.with_(name="qwen3.6-shape-elastic", steps=2048, B=1, seed=5, C=6144, resize=((512, 2560), (1280, 8192)))

# Small parity cases: full hidden/intermediate sizes (so every kernel spans
# many tiles and a ragged per-CTA row split) with few layers and experts.
SMALL_BF16 = C2.with_(name="small-bf16", L=3, E=32, C=40, steps=24)
SMALL_FP4 = C3.with_(name="small-fp4", L=2, E=16, C=14, steps=12)
SMALL_FP4_NARROW = C3.with_(name="small-fp4-narrow", L=2, E=24, k=4, H=512, I=256, C=11, steps=40)
