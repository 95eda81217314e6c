"""GPU parity of expert_cache_prefetch, through the C ABI.

A prefetch is one residency step for a predicted expert set, followed by its page-in,
with nothing computed. Expected values come from the oracle only:
- the LRU simulator treats the prefetch as an ordinary step, so slot tables, misses
  and waves must match it bit for bit;
- the forward that follows must return exactly what it returns without any prefetch
  (paging never changes the result: article "Running an MoE Model Larger Than Your
  VRAM", section "Can paging change the model's outputs?"), and match the oracle
  within the stated tolerances.
"""

import numpy as np
import pytest

from oracle import lru as olru
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


def _ids_tensor(flat):
    return torch.tensor(flat, dtype=torch.int32).cuda()


def _check_table(cache, sim, layer=0):
    exp_in, last = cache.expert_cache_slot_table(layer)
    assert exp_in.tolist() == sim.expert_in
    assert last.tolist() == sim.last_use


def _forward(pm, cache, x_bits, logits, k):
    x = hz.to_device_bf16(x_bits)
    ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
    return cache.moe_paged_forward(0, x, ids, w)


@pytest.mark.parametrize("mode", [0, 1])
def test_prefetch_steps_match_simulator_and_leave_outputs_unchanged(pm, mode):
    """E=16, top_k=2, H=128, I=64, K=3, 2 tokens per step. Before every forward, a
    prefetch of a predicted set: the exact next set, four distinct random experts (more
    than K: two waves), or four draws with repeats; the simulator sees each prefetch as
    a step."""
    E, k, H, I, K, B, n = 16, 2, 128, 64, 3, 2, 40
    L = hz.SyntheticLayer(0, E, H, I, seed=11)
    rng = np.random.default_rng(11)
    trace = gen.reuse_routing_trace(rng, E, k, B, n)
    steps = [hz.step_inputs(rng, sets, E, H) for sets in trace]
    pred_rng = np.random.default_rng(12)

    plain = hz.make_cache([L], k, K, max_tokens=B, mode=mode)
    ref = [_forward(pm, plain, *st, k) for st in steps]
    torch.cuda.synchronize()
    plain.close()

    cache = hz.make_cache([L], k, K, max_tokens=B, mode=mode)
    sim = olru.LayerLRU(E, K)
    outs = []
    for s, (sets, st) in enumerate(zip(trace, steps)):
        real = [e for t in sets for e in t]
        kind = s % 3
        if kind == 0:
            pred = list(real)
        elif kind == 1:
            pred = [int(e) for e in pred_rng.choice(E, size=B * k, replace=False)]
        else:
            pred = [int(e) for e in pred_rng.choice(E, size=B * k, replace=True)]
        cache.expert_cache_prefetch(0, _ids_tensor(pred))
        sim.step(pred)
        before = cache.expert_cache_stats(0)["misses"]
        outs.append(_forward(pm, cache, *st, k))
        out = sim.step(real)
        torch.cuda.synchronize()
        if kind == 0 and len(set(real)) <= K:
            assert out["n_misses"] == 0
            assert cache.expert_cache_stats(0)["misses"] == before
        if s % 8 == 0:
            _check_table(cache, sim)
    torch.cuda.synchronize()
    _check_table(cache, sim)
    stt = cache.expert_cache_stats(0)
    assert (stt["misses"], stt["hits"], stt["waves"]) == (sim.misses, sim.hits, sim.waves)
    for a, b in zip(outs, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    exp_in, _ = cache.expert_cache_slot_table(0)
    for slot, e in enumerate(exp_in.tolist()):
        if e >= 0:
            assert np.array_equal(cache.expert_cache_read_slot(0, slot), L.store[e]), (slot, e)
    cache.close()
    for i in (0, n // 2, n - 1):
        x_bits, logits = steps[i]
        ids, w = orouter.router_topk(logits, k)
        hz.assert_layer_close(hz.bf16_to_f64(outs[i]), L.oracle_y(x_bits, ids, w), 0)


def test_prefetch_of_a_qwen_layer_removes_the_forward_misses(pm):
    """Qwen3-30B-A3B-shaped bf16 layer, K=40, B=1, SM-pull: prefetching each step's own
    experts makes every forward miss-free; the outputs are bit for bit those of the
    run without prefetch."""
    E, k, H, I, K, n = 128, 8, 2048, 768, 40, 12
    L = hz.SyntheticLayer(0, E, H, I, seed=5)
    rng = np.random.default_rng(5)
    trace = gen.reuse_routing_trace(rng, E, k, 1, n)
    steps = [hz.step_inputs(rng, sets, E, H) for sets in trace]
    plain = hz.make_cache([L], k, K, max_tokens=1, mode=1)
    ref = [_forward(pm, plain, *st, k) for st in steps]
    torch.cuda.synchronize()
    plain_misses = plain.expert_cache_stats(0)["misses"]
    plain.close()
    cache = hz.make_cache([L], k, K, max_tokens=1, mode=1)
    outs = []
    for sets, st in zip(trace, steps):
        cache.expert_cache_prefetch(0, _ids_tensor([e for t in sets for e in t]))
        before = cache.expert_cache_stats(0)["misses"]
        outs.append(_forward(pm, cache, *st, k))
        torch.cuda.synchronize()
        assert cache.expert_cache_stats(0)["misses"] == before
    assert cache.expert_cache_stats(0)["misses"] == plain_misses  # the same misses, taken by the prefetches
    for a, b in zip(outs, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    cache.close()
    x_bits, logits = steps[-1]
    ids, w = orouter.router_topk(logits, k)
    hz.assert_layer_close(hz.bf16_to_f64(outs[-1]), L.oracle_y(x_bits, ids, w), 0)


def test_prefetch_argument_errors(pm):
    L = hz.SyntheticLayer(0, 8, 128, 64, seed=1)
    cache = hz.make_cache([L], 2, 4, max_tokens=2)
    ids = _ids_tensor([0, 1])
    with pytest.raises(RuntimeError):
        cache.expert_cache_prefetch(1, ids)  # no such layer
    with pytest.raises(RuntimeError):
        cache.expert_cache_prefetch(0, _ids_tensor([0, 1, 2, 3, 4]))  # more ids than max_tokens * top_k
    cache.expert_cache_prefetch(0, ids[:0])  # an empty prediction is a step with nothing routed
    torch.cuda.synchronize()
    cache.close()
