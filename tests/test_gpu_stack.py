"""GPU parity of the multi-layer stack (GPTQ-int4 experts, residual stream, prefetch of the
next layer's page-in while the current layer computes), through the C ABI.

The oracle is the unpaged stack h_{l+1} = h_l + moe_l(h_l) in float64 with the same
per-layer routing; the per-layer slot tables, misses and waves are checked against one
LRU simulator per layer; the prefetching stack call is bit for bit equal to per-layer
forward calls without prefetch.
"""

import numpy as np
import pytest

from oracle import lru as olru
from oracle import moe as omoe
from oracle import router as orouter
from tests import _harness as hz
from workloads import generators as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_expert_moe_gb300 as pm
    pm.load()
    return pm


def _stack_inputs(L, E, k, H, B, steps, seed):
    rng = np.random.default_rng(seed)
    traces = [gen.reuse_routing_trace(rng, E, k, B, steps) for _ in range(L)]
    logits = np.stack([np.stack([gen.logits_for_sets(rng, traces[l][s], E) for l in range(L)])
                       for s in range(steps)])  # [steps, L, B, E]
    xs = [gen.activations_bf16(rng, B, H) for _ in range(steps)]
    return traces, logits, xs


@pytest.mark.parametrize("B,mode", [(4, 0), (1, 0), (4, 1), (1, 1), (2, 1)])
def test_int4_stack_against_oracle_and_without_prefetch(pm, B, mode):
    """SM-pull mode with B * top_k <= K (B = 1, 2 at K = 26) runs all layers in one
    persistent launch; B = 4 there (several waves) and copy-engine mode run per layer."""
    L, E, k, H, I, K, steps = 4, 128, 8, 2048, 768, 26, 5
    layers = [hz.SyntheticLayer(2, E, H, I, seed=600, layer=l, fast_int4=True) for l in range(L)]
    traces, logits, xs = _stack_inputs(L, E, k, H, B, steps, seed=601 + B)
    stack = hz.make_cache(layers, k, K, max_tokens=B, mode=mode)
    plain = hz.make_cache(layers, k, K, max_tokens=B, mode=mode)
    sims = [olru.LayerLRU(E, K) for _ in range(L)]
    for s in range(steps):
        lg = torch.from_numpy(logits[s].reshape(L * B, E)).cuda()
        ids, w = pm.moe_router_topk(lg, k)
        x = hz.to_device_bf16(xs[s])
        y = stack.moe_paged_stack_forward(x, ids, w)
        # the same layers, one forward call each, no prefetch
        h = x
        for l in range(L):
            h = plain.moe_paged_forward(l, h, ids[l * B:(l + 1) * B], w[l * B:(l + 1) * B], residual=h)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), h.view(torch.int16)), f"step {s}"
        # oracle: unpaged float64 stack with the same routing
        oracle_layers = []
        for l in range(L):
            ids_o, w_o = orouter.router_topk(logits[s, l], k)
            oracle_layers.append((ids_o, w_o, layers[l].experts))
            sims[l].step(ids_o.ravel().tolist())
        ref, n_act = omoe.moe_stack(gen.bf16_bits_to_float(xs[s]).astype(np.float64), oracle_layers, residual=True)
        assert n_act == L * B * k
        hz.assert_layer_close(hz.bf16_to_f64(y), ref, 2)
    for l in range(L):
        st = stack.expert_cache_stats(l)
        assert (st["misses"], st["hits"], st["waves"]) == (sims[l].misses, sims[l].hits, sims[l].waves), l
        exp_in, last = stack.expert_cache_slot_table(l)
        assert exp_in.tolist() == sims[l].expert_in and last.tolist() == sims[l].last_use
    if B == 4:
        assert sum(sims[l].waves for l in range(L)) > L * steps  # B=4 exceeds K // top_k = 3
    stack.close()
    plain.close()


@pytest.mark.parametrize("fmt", [0, 1, 3, 4])
def test_one_launch_stack_equals_per_layer_calls(pm, fmt):
    """bf16, block-FP8, MXFP4 and NVFP4 experts: the persistent stack launch (every layer
    one wave: B * top_k = 8 <= K = 12) equals one forward call per layer with residual =
    input, bit for bit, step after step, and the tables agree."""
    L, E, k, H, I, K, B, steps = 3, 32, 4, 512, 256, 12, 2, 4
    layers = [hz.SyntheticLayer(fmt, E, H, I, seed=620 + fmt, layer=l) for l in range(L)]
    traces, logits, xs = _stack_inputs(L, E, k, H, B, steps, seed=630 + fmt)
    mode = pm.PMOE_PAGEIN_SM_PULL
    stack = hz.make_cache(layers, k, K, max_tokens=B, mode=mode)
    plain = hz.make_cache(layers, k, K, max_tokens=B, mode=mode)
    for s in range(steps):
        lg = torch.from_numpy(logits[s].reshape(L * B, E)).cuda()
        ids, w = pm.moe_router_topk(lg, k)
        x = hz.to_device_bf16(xs[s])
        y = stack.moe_paged_stack_forward(x, ids, w)
        h = x
        for l in range(L):
            h = plain.moe_paged_forward(l, h, ids[l * B:(l + 1) * B], w[l * B:(l + 1) * B], residual=h)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), h.view(torch.int16)), f"step {s}"
    for l in range(L):
        assert stack.expert_cache_stats(l) == plain.expert_cache_stats(l)
        assert stack.expert_cache_slot_table(l)[0].tolist() == plain.expert_cache_slot_table(l)[0].tolist()
    stack.close()
    plain.close()
