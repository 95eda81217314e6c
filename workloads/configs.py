"""The workload shapes: a tiny layer and Qwen3-30B-A3B-shaped MoE layers.

Qwen3-30B-A3B MoE shape ("Running an MoE Model Larger Than Your VRAM", section
"What does Paged Experts actually do?"): 48 layers, 128 experts, 8 per token,
hidden 2048, MoE intermediate 768.
"""

from dataclasses import dataclass, field


@dataclass(frozen=True)
class LayerShape:
    E: int
    top_k: int
    H: int
    I: int


QWEN3_30B_A3B = LayerShape(E=128, top_k=8, H=2048, I=768)
TINY = LayerShape(E=8, top_k=2, H=128, I=64)

BF16, FP8_BLOCK128, INT4_GPTQ_G128 = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    fmt: int
    K: int
    layers: int = 1
    batches: tuple = ()
    steps: int = 0
    prefill_tokens: int = 0
    reuse_p: float = 0.8
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)


CONFIGS = {
    "tiny": Workload("tiny bf16 layer E=8 top_k=2 H=128 I=64 K=8, 4 tokens", TINY, BF16, K=8,
                     batches=(4,), steps=1),
    "decode_bf16": Workload("Qwen3-30B-A3B MoE layer bf16 decode B=1/2/4 x 256 steps, K=40, p=0.8 reuse",
                            QWEN3_30B_A3B, BF16, K=40, batches=(1, 2, 4), steps=256),
    "prefill_bf16": Workload("Qwen3-30B-A3B MoE layer bf16 prefill 2048 tokens, K=92 cold, uniform routing",
                             QWEN3_30B_A3B, BF16, K=92, prefill_tokens=2048),
    "fp8": Workload("Qwen3-30B-A3B MoE layer block-FP8, K=40, decode B=1 x 256 (p=0.8) + prefill 512",
                    QWEN3_30B_A3B, FP8_BLOCK128, K=40, batches=(1,), steps=256, prefill_tokens=512),
    "stack_int4": Workload("48-layer Qwen3-30B-A3B MoE stack, GPTQ int4 g128, K=26, decode B=1 vs 4, 256 steps",
                           QWEN3_30B_A3B, INT4_GPTQ_G128, K=26, layers=48, batches=(1, 4), steps=256),
}
