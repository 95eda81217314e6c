"""Shared helpers of the GPU parity tests: seeded layers, caches and the comparisons.

Inputs come from ``workloads``; expected values come from ``oracle`` only.
"""

import numpy as np

from oracle import formats as ofmt
from oracle import moe as omoe
from oracle import router as orouter
from workloads import generators as gen

REL_FROB_BF16 = 1e-2      # bf16 / int4 layer outputs: relative Frobenius error
MAX_ABS_BF16 = 3e-2       # ... and max-abs error relative to max |reference|
REL_FROB_FP8 = 3e-2       # block-FP8 layer outputs


def rel_frob(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_layer_close(y_gpu, y_ref, fmt):
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    rf = rel_frob(y_gpu, y_ref)
    if fmt == 1:
        assert rf <= REL_FROB_FP8, f"rel-Frobenius {rf:.3e} > {REL_FROB_FP8}"
    else:
        ma = float(np.abs(y_gpu - y_ref).max() / max(np.abs(y_ref).max(), 1e-300))
        assert rf <= REL_FROB_BF16, f"rel-Frobenius {rf:.3e} > {REL_FROB_BF16}"
        assert ma <= MAX_ABS_BF16, f"max-abs {ma:.3e} x max|ref| > {MAX_ABS_BF16}"
    return rf


def bf16_to_f64(t):
    """torch bf16 tensor (any device) -> float64 numpy."""
    import torch
    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)


class SyntheticLayer:
    """One layer's experts (bytes from the generator) and its oracle view."""

    def __init__(self, fmt, E, H, I, seed=0, layer=0, fast_int4=False):
        self.fmt, self.E, self.H, self.I = fmt, E, H, I
        self.store = gen.layer_store(fmt, H, I, E, seed, layer, fast=fast_int4)
        self.experts = omoe.ExpertSource(lambda e: self.store[e], fmt, H, I, cache=48)

    def oracle_y(self, x_bits, ids, w):
        x = gen.bf16_bits_to_float(x_bits).astype(np.float64)
        y, _ = omoe.moe_layer(x, ids, w, self.experts)
        return y


def make_cache(layers, top_k, K, max_tokens=8, mode=0, device=0):
    import paged_expert_moe_gb300 as pm
    L0 = layers[0]
    c = pm.ExpertCache(L0.E, top_k, L0.H, L0.I, K, num_layers=len(layers), fmt=L0.fmt, max_tokens=max_tokens,
                       pagein_mode=mode, device=device)
    for l, L in enumerate(layers):
        c.load_layer(l, L.store)
    return c


def step_inputs(rng, sets, E, H):
    """(x bf16 bits [T,H], logits [T,E]) for one step whose routed sets are `sets`."""
    logits = gen.logits_for_sets(rng, sets, E)
    x = gen.activations_bf16(rng, len(sets), H)
    return x, logits


def oracle_route(logits, top_k):
    return orouter.router_topk(logits, top_k)


def to_device_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def decode_bytes(buf, fmt, H, I):
    return ofmt.decode_expert(buf, fmt, H, I)
