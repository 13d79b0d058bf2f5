"""CPU oracle for the routed-MoE layer served from a shared GPU expert cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the layer computes, written from the FreeToken write-ups
("FreeToken: 프론티어급 MoE 모델을 게이밍 데스크톱 수준에서 서빙하기 위한 Edge-Serving
에 대한 연구", discuss.pytorch.kr, and the qqtang-code.github.io reading of the
same paper).  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import it.  The CUDA library never calls it and shares no
code with it; the only common source of inputs is the ``synth`` package.

Modules
-------
``router``   top-k softmax routing (decode co-design section: "the router and
             cache lookup run on the GPU").
``lru``      the shared all-layer LRU expert cache as a stamp-based simulator:
             hits refresh recency, fills admit the selected expert, evictions
             take the expert not requested for the longest time, victims are
             found in one pass (CUDA-Graph LRU cache section), plus resizing at
             a safe point (elastic memory management section).
``permute``  stable grouping of (token, rank) pairs by expert.
``fp4``      e2m1 / e4m3 decoding of FP4 expert records.
``records``  parsing of one expert record into its three matrices.
``ffn``      the SwiGLU expert and the weighted combine (exact merge of
             partial sums, Fig. 2 caption).
``qstar``    the bandwidth-adaptive fill count q* (decode co-design section,
             equations for T_fill, T_cpu and q*).

Every floating-point result is computed in float64.  Pinning: see
``tests/test_oracle_*.py``; every function here has at least one pin that does
not restate its own formula.
"""
from . import fp4, ffn, lru, permute, qstar, records, router  # noqa: F401
