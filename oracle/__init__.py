"""Oracle for the paged-expert MoE layer.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, CPU restatement of what
the paged-expert MoE layer computes, written from the article "Running an MoE
Model Larger Than Your VRAM: SGLang Paged Experts, the PCIe Math, and the
4-Request Cliff" and the post on the llama.cpp MoE expert cache ("Locality of
reference helped ..."). Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it. The CUDA library never
calls it, links it or shares code with it; the only thing both sides use is the
seeded input generator package ``workloads``, which holds none of the method's
arithmetic.

Precision: float64 for all floating-point arithmetic (inputs are bf16 / fp32 /
fp8 / int4 and upcast exactly), integers exact.

Modules
  router     softmax over E, top-k selection, renormalisation
  formats    exact decoding of an expert's bytes (bf16, block-FP8 e4m3, GPTQ int4)
  moe        SwiGLU expert MLP and the top_k-weighted combine (the unpaged layer)
  permute    token->expert histogram, exclusive scan and stable grouping
  lru        brute-force per-layer K-slot LRU / wave simulator
  preflight  the article's sizing arithmetic (slot cost, batch cap, miss bounds)

Every function names the passage it follows. Points where the pages are silent
are stated in the docstrings of the functions that take a reading.
"""

from . import router, formats, moe, permute, lru, preflight  # noqa: F401
