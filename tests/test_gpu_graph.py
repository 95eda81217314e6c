"""CUDA-graph capture of single-wave decode steps (SM-pull page-in, no host round trip).

The article's "What happens with more than one request?" section notes that the
single-wave decode step is the case a CUDA graph can capture. A step captured once and
replayed with new inputs must give the same bits, slot tables and counters as the
same steps run without a graph; a copy-engine cache refuses capture (its page-in reads
the plan on the host).
"""

import numpy as np
import pytest

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


@pytest.mark.parametrize("B", [1, 4])
def test_captured_decode_step_matches_uncaptured(pm, B):
    """The headline configuration (E=128, K=40, SM-pull page-in inside the decode kernel,
    the step replayed as one graph): every replayed step equals the uncaptured run bit
    for bit and the oracle within the bf16 tolerances."""
    from oracle import router as orouter
    E, k, H, I, K, steps = 128, 8, 2048, 768, 40, 12
    L = hz.SyntheticLayer(0, E, H, I, seed=700)
    rng = np.random.default_rng(700 + B)
    trace = gen.reuse_routing_trace(rng, E, k, B, steps)
    inputs = [hz.step_inputs(rng, sets, E, H) for sets in trace]
    ref = hz.make_cache([L], k, K, max_tokens=B, mode=pm.PMOE_PAGEIN_SM_PULL)
    ys_ref = []
    for x_bits, logits in inputs:
        ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
        ys_ref.append(ref.moe_paged_forward(0, hz.to_device_bf16(x_bits), ids, w).clone())
    torch.cuda.synchronize()

    cache = hz.make_cache([L], k, K, max_tokens=B, mode=pm.PMOE_PAGEIN_SM_PULL)
    x_s = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
    l_s = torch.zeros((B, E), dtype=torch.float32, device="cuda")
    ids_s = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    w_s = torch.zeros((B, k), dtype=torch.float32, device="cuda")
    y_s = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pm.moe_router_topk(l_s, k, ids_out=ids_s, w_out=w_s)
        cache.moe_paged_forward(0, x_s, ids_s, w_s, y=y_s)
    for i, (x_bits, logits) in enumerate(inputs):
        x_s.copy_(hz.to_device_bf16(x_bits))
        l_s.copy_(torch.from_numpy(logits).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_s.view(torch.int16), ys_ref[i].view(torch.int16)), f"step {i}"
        ids_o, w_o = orouter.router_topk(logits, k)
        assert np.array_equal(ids_s.cpu().numpy(), ids_o), f"step {i}: routing"
        hz.assert_layer_close(hz.bf16_to_f64(y_s), L.oracle_y(x_bits, ids_o, w_o), 0)
    assert cache.expert_cache_stats(0) == ref.expert_cache_stats(0)
    assert cache.expert_cache_slot_table(0)[0].tolist() == ref.expert_cache_slot_table(0)[0].tolist()
    cache.close()
    ref.close()


def test_captured_int4_stack_matches_uncaptured(pm):
    Lyr, E, k, H, I, K, B, steps = 4, 128, 8, 2048, 768, 26, 1, 6
    layers = [hz.SyntheticLayer(2, E, H, I, seed=710, layer=l, fast_int4=True) for l in range(Lyr)]
    rng = np.random.default_rng(711)
    traces = [gen.reuse_routing_trace(rng, E, k, B, steps) for _ in range(Lyr)]
    logits = [np.concatenate([gen.logits_for_sets(rng, traces[l][s], E) for l in range(Lyr)]) for s in range(steps)]
    xs = [gen.activations_bf16(rng, B, H) for _ in range(steps)]
    ref = hz.make_cache(layers, k, K, max_tokens=B, mode=pm.PMOE_PAGEIN_SM_PULL)
    ys_ref = []
    for s in range(steps):
        ids, w = pm.moe_router_topk(torch.from_numpy(logits[s]).cuda(), k)
        ys_ref.append(ref.moe_paged_stack_forward(hz.to_device_bf16(xs[s]), ids, w).clone())
    torch.cuda.synchronize()
    cache = hz.make_cache(layers, k, K, max_tokens=B, mode=pm.PMOE_PAGEIN_SM_PULL)
    x_s = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
    l_s = torch.zeros((Lyr * B, E), dtype=torch.float32, device="cuda")
    ids_s = torch.zeros((Lyr * B, k), dtype=torch.int32, device="cuda")
    w_s = torch.zeros((Lyr * B, k), dtype=torch.float32, device="cuda")
    y_s = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
    work = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pm.moe_router_topk(l_s, k, ids_out=ids_s, w_out=w_s)
        cache.moe_paged_stack_forward(x_s, ids_s, w_s, y=y_s, work=work)
    for s in range(steps):
        x_s.copy_(hz.to_device_bf16(xs[s]))
        l_s.copy_(torch.from_numpy(logits[s]).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_s.view(torch.int16), ys_ref[s].view(torch.int16)), f"step {s}"
    for l in range(Lyr):
        assert cache.expert_cache_stats(l) == ref.expert_cache_stats(l)
    cache.close()
    ref.close()


def test_copy_engine_cache_refuses_capture(pm):
    L = hz.SyntheticLayer(0, 8, 128, 64, seed=720)
    cache = hz.make_cache([L], 2, 4, max_tokens=2)
    x = torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    w = torch.full((2, 2), 0.5, dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    g = torch.cuda.CUDAGraph()
    with pytest.raises(pm.PmoeError) as ei:
        with torch.cuda.graph(g):
            cache.moe_paged_forward(0, x, ids, w, y=y)
    assert ei.value.status == pm.PMOE_EUNSUPPORTED
    cache.close()
