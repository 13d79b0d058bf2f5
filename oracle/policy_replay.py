"""Miss rate versus cache capacity of the four placement policies on the
seeded synthetic routing traces (the Fig. 4b analogue of the FreeToken
write-up's expert-locality paragraph).  CPU only; prints a markdown table.

    python -m oracle.policy_replay [--prompt 256] [--decode 512]

Traces: the AR(1) router logits of the Qwen3.6-shaped (40 layers, 256
experts, top-8) and DeepSeek-V4-Flash-shaped (43 layers, 256 experts, top-6)
configurations at batch 1; the first `prompt` tokens are what the policies
may learn from, the next `decode` tokens are replayed and counted.
"""
from __future__ import annotations

import argparse
import os
import sys

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402
from oracle import policies  # noqa: E402
from synth import configs  # noqa: E402


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--prompt", type=int, default=256)
    ap.add_argument("--decode", type=int, default=512)
    args = ap.parse_args()
    fracs = [0.1, 0.2, 0.3, 0.37, 0.5, 0.6, 0.8, 1.0]
    print("| trace | capacity | " + " | ".join(policies.POLICIES) + " |")
    print("|---|---|" + "---|" * len(policies.POLICIES))
    for w in (configs.C2, configs.C3):
        T = args.prompt + args.decode
        lg = synth.ar1_logits(w.seed, T, w.L, 1, w.E)
        ids = policies.routed_ids(lg, w.k)
        for f in fracs:
            C = max(w.k, int(f * w.LE))
            rates = []
            for pol in policies.POLICIES:
                m, a = policies.replay(ids, args.prompt, w.E, C, pol)
                rates.append(f"{100.0 * m / a:.1f}%")
            print(f"| {w.name} | {f:.0%} ({C} slots) | " + " | ".join(rates) + " |")


if __name__ == "__main__":
    main()
