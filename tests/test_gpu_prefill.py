"""GPU parity of the prefill path (tcgen05 grouped GEMMs) through the C ABI.

Small layers span several M tiles, ragged pair counts (including an expert with more
than 256 pairs, which is split over two N tiles) and several waves; the full-size
Qwen3-30B-A3B prefill (2048 tokens, K=92, cold) is checked on sampled tokens against
the oracle and bit for bit against K=128.
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


def _skewed_sets(rng, T, E, k, hot=0):
    """Every token routes to expert `hot` plus k-1 uniform others."""
    sets = []
    for _ in range(T):
        others = rng.choice(np.setdiff1d(np.arange(E), [hot]), size=k - 1, replace=False)
        sets.append([hot] + list(others))
    return sets


def _forward(cache, x_bits, logits, k):
    x = hz.to_device_bf16(x_bits)
    import paged_expert_moe_gb300 as pm
    ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
    y = cache.moe_paged_forward(0, x, ids, w)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("T,skew,fmt", [(300, True, 0), (9, False, 0), (64, False, 0), (1000, False, 0),
                                        (300, True, 1), (64, False, 1), (128, True, 1), (1000, False, 1),
                                        (300, True, 2), (64, False, 2), (300, True, 3), (64, False, 3),
                                        (300, True, 4), (64, False, 4)])
def test_prefill_small_layer_parity_and_bitwise_k_invariance(pm, T, skew, fmt):
    """bf16, block-FP8, GPTQ-int4 and MXFP4 prefill tiles. Block-FP8 with few pairs per
    expert (T=64, and T=128 skewed, where hot experts take several 64-pair tiles) runs
    e4m3 MMAs on two-plane activations; with more (T=300, 1000) its weights are
    dequantised to bf16 in shared memory, like int4, MXFP4 and NVFP4 (whose fp32 tensor
    scale multiplies the accumulators)."""
    E, k, H, I = 16, 4, 256, 384
    L = hz.SyntheticLayer(fmt, E, H, I, seed=200 + T)
    rng = np.random.default_rng(200 + T)
    sets = _skewed_sets(rng, T, E, k) if skew else gen.uniform_routing_sets(rng, T, E, k)
    x_bits, logits = hz.step_inputs(rng, sets, E, H)
    ys = {}
    for K in (16, 5, 1):
        cache = hz.make_cache([L], k, K, max_tokens=T)
        ys[K] = _forward(cache, x_bits, logits, k)
        st = cache.expert_cache_stats(0)
        sim = olru.LayerLRU(E, K)
        out = sim.step(np.asarray(sets).ravel().tolist())
        assert (st["misses"], st["waves"]) == (out["n_misses"], len(out["waves"]))
        cache.close()
    ids, w = orouter.router_topk(logits, k)
    hz.assert_layer_close(hz.bf16_to_f64(ys[16]), L.oracle_y(x_bits, ids, w), fmt)
    for K in (5, 1):
        assert torch.equal(ys[K].view(torch.int16), ys[16].view(torch.int16)), f"K={K} differs"


def test_prefill_qwen3_layer_cold_k92(pm):
    """2048 tokens, uniform routing, K=92, cold: 128 misses, 2 waves; sampled tokens against
    the oracle and all outputs bit for bit against K=128."""
    E, k, H, I, T = 128, 8, 2048, 768, 2048
    L = hz.SyntheticLayer(0, E, H, I, seed=300)
    rng = np.random.default_rng(300)
    sets = gen.uniform_routing_sets(rng, T, E, k)
    x_bits, logits = hz.step_inputs(rng, sets, E, H)
    cache = hz.make_cache([L], k, 92, max_tokens=T)
    y92 = _forward(cache, x_bits, logits, k)
    st = cache.expert_cache_stats(0)
    assert st["misses"] == 128 and st["waves"] == 2
    exp_in, _ = cache.expert_cache_slot_table(0)
    assert exp_in.tolist() == [92 + i if i < 36 else i for i in range(92)]
    cache.close()
    cache = hz.make_cache([L], k, 128, max_tokens=T)
    y128 = _forward(cache, x_bits, logits, k)
    cache.close()
    assert torch.equal(y92.view(torch.int16), y128.view(torch.int16))
    sample = np.random.default_rng(301).choice(T, size=24, replace=False)
    ids, w = orouter.router_topk(logits[sample], k)
    ref = L.oracle_y(x_bits[sample], ids, w)
    hz.assert_layer_close(hz.bf16_to_f64(y92)[sample], ref, 0)


def test_gemv_and_tensor_core_paths_agree_at_the_boundary(pm):
    """T=8 runs the decode kernels, T=9 the tensor-core kernels: both match the oracle."""
    E, k, H, I = 32, 8, 512, 256
    L = hz.SyntheticLayer(0, E, H, I, seed=400)
    rng = np.random.default_rng(400)
    for T in (8, 9):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        x_bits, logits = hz.step_inputs(rng, sets, E, H)
        cache = hz.make_cache([L], k, 24, max_tokens=16)
        y = _forward(cache, x_bits, logits, k)
        cache.close()
        ids, w = orouter.router_topk(logits, k)
        hz.assert_layer_close(hz.bf16_to_f64(y), L.oracle_y(x_bits, ids, w), 0)


@pytest.mark.parametrize("fmt", [1, 3, 4])
def test_prefill_quantised_512_tokens_k40(pm, fmt):
    """Block-FP8 (rel-Frobenius 3e-2) and MXFP4 (the bf16 tolerances: E2M1 times an E8M0
    scale is exact in bf16) Qwen3-30B-A3B layers, 512-token prefill, K=40 (several waves):
    sampled tokens against the oracle and all outputs bit for bit against K=128."""
    E, k, H, I, T = 128, 8, 2048, 768, 512
    L = hz.SyntheticLayer(fmt, E, H, I, seed=500)
    rng = np.random.default_rng(500)
    sets = gen.uniform_routing_sets(rng, T, E, k)
    x_bits, logits = hz.step_inputs(rng, sets, E, H)
    cache = hz.make_cache([L], k, 40, max_tokens=T)
    y40 = _forward(cache, x_bits, logits, k)
    st = cache.expert_cache_stats(0)
    sim = olru.LayerLRU(E, 40)
    out = sim.step(np.asarray(sets).ravel().tolist())
    assert (st["misses"], st["waves"]) == (out["n_misses"], len(out["waves"]))
    cache.close()
    cache = hz.make_cache([L], k, 128, max_tokens=T)
    y128 = _forward(cache, x_bits, logits, k)
    cache.close()
    assert torch.equal(y40.view(torch.int16), y128.view(torch.int16))
    sample = np.random.default_rng(501).choice(T, size=16, replace=False)
    ids, w = orouter.router_topk(logits[sample], k)
    hz.assert_layer_close(hz.bf16_to_f64(y40)[sample], L.oracle_y(x_bits[sample], ids, w), fmt)


@pytest.mark.parametrize("T,fmt", [(300, 0), (300, 1), (64, 1), (300, 4)])
def test_prefill_sm_pull_mode_is_bitwise_identical_to_copy_engine(pm, T, fmt):
    """SM-pull page-in (plan kept on the device, a pull kernel per wave, GEMMs launched for
    an upper bound of waves that skip the ones the plan does not have) against copy-engine
    page-in, in one cache per mode carried over several steps: the same misses and waves
    as the LRU simulator and the same output bits. bf16, block-FP8 on both of its tile
    paths, NVFP4; K = 5 (several waves a step) and K = 16 (all resident after the first)."""
    E, k, H, I = 16, 4, 256, 384
    L = hz.SyntheticLayer(fmt, E, H, I, seed=400 + T + fmt)
    rng = np.random.default_rng(400 + T + fmt)
    steps = []
    for _ in range(3):
        sets = _skewed_sets(rng, T, E, k, hot=int(rng.integers(E)))
        steps.append((sets,) + hz.step_inputs(rng, sets, E, H))
    for K in (5, 16):
        ys = {}
        for mode in (0, 1):
            cache = hz.make_cache([L], k, K, max_tokens=T, mode=mode)
            sim = olru.LayerLRU(E, K)
            ys[mode] = []
            for sets, x_bits, logits in steps:
                before = cache.expert_cache_stats(0)
                ys[mode].append(_forward(cache, x_bits, logits, k))
                st = cache.expert_cache_stats(0)
                out = sim.step(np.asarray(sets).ravel().tolist())
                assert st["misses"] - before["misses"] == out["n_misses"]
                assert st["waves"] - before["waves"] == len(out["waves"])
            cache.close()
        for i, (a, b) in enumerate(zip(ys[0], ys[1])):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"K={K} step {i}"
    ids, w = orouter.router_topk(steps[-1][2], k)
    hz.assert_layer_close(hz.bf16_to_f64(ys[1][-1]), L.oracle_y(steps[-1][1], ids, w), fmt)
