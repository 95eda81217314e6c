"""The article's sizing arithmetic, restated as separate closed forms.

Source: "Running an MoE Model Larger Than Your VRAM", sections "Why is it fast
when experts keep crossing PCIe?", "What does a resident slot cost in context
length?" and "A preflight script before you turn it on". The quantities:

  slot cost               = expert size x MoE layers   (a slot exists in every layer)
  KV tokens one slot buys = slot bytes / KV bytes per token
  single-wave batch cap   = K // top_k
  all-miss traffic        = layers x top_k x expert size per token
  highest miss rate a measured speed allows
                          = link bandwidth / (tokens per second x all-miss traffic)
  miss rate under uniform random routing = 1 - K / E
  verdict: reuse is implied when the allowed maximum is below 0.8 x the random
  rate; otherwise the numbers are inconclusive.
  bf16 KV bytes per token for Qwen3-30B-A3B = 2 (K and V) x 48 layers x 4 KV heads
  x 128 head dim x 2 bytes.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from dataclasses import dataclass


def kv_bytes_per_token(layers=48, kv_heads=4, head_dim=128, elem_bytes=2):
    return 2 * layers * kv_heads * head_dim * elem_bytes


def slot_cost_mb(expert_mb, layers):
    return expert_mb * layers


def batch_cap(K, top_k):
    return K // top_k


def all_miss_gb_per_token(expert_mb, layers, top_k):
    return expert_mb * layers * top_k / 1000.0


def max_miss_allowed(link_gbps, tok_s, all_miss_gb):
    return link_gbps / (tok_s * all_miss_gb)


def random_routing_miss(K, E):
    return 1.0 - K / E


@dataclass
class Sizing:
    slot_mb: float
    kv_tokens_per_slot: float
    batch_cap: int
    random_miss: float
    max_miss: float
    reuse_implied: bool


def size_deployment(E, top_k, layers, expert_mb, K, link_gbps, tok_s, kv_bytes):
    slot = slot_cost_mb(expert_mb, layers)
    mx = max_miss_allowed(link_gbps, tok_s, all_miss_gb_per_token(expert_mb, layers, top_k))
    rnd = random_routing_miss(K, E)
    return Sizing(slot_mb=slot, kv_tokens_per_slot=slot * 1e6 / kv_bytes,
                  batch_cap=batch_cap(K, top_k), random_miss=rnd, max_miss=mx,
                  reuse_implied=mx < 0.8 * rnd)


def activations_per_token(layers, top_k):
    """Expert activations of one decode token: one per (layer, rank)."""
    return layers * top_k
