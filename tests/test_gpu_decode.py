"""GPU parity of the router, the residency step and the decode layer, through the C ABI.

Expected values come from the oracle only: router ids bit-exact and weights within a
derived fp32 bound; slot tables, misses and waves bit-exact against the LRU
simulator; layer outputs within the stated float tolerances and bitwise identical
for every K.
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


def _router_rtol(k):
    # fp32: expf within 2 ulp, k-1 additions and one division each within half an ulp
    return (k + 3) * 2.0 ** -23


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (1, 128, 8), (7, 128, 8), (2048, 128, 8), (33, 33, 5),
                                   (5, 1024, 32), (3, 1, 1), (16, 64, 64 // 2)])
def test_router_matches_oracle(pm, T, E, k):
    rng = np.random.default_rng(100 + T + E + k)
    sets = gen.uniform_routing_sets(rng, T, E, k)
    logits = gen.logits_for_sets(rng, sets, E)
    ids_g, w_g = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
    ids_o, w_o = orouter.router_topk(logits, k)
    np.testing.assert_array_equal(ids_g.cpu().numpy(), ids_o)
    np.testing.assert_allclose(w_g.cpu().numpy(), w_o, rtol=_router_rtol(k), atol=0)


def test_router_without_renormalisation_and_ties(pm):
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((9, 40)).astype(np.float32)
    logits[3, :] = 0.5  # all equal: the k lowest ids, equal weights
    ids_g, w_g = pm.moe_router_topk(torch.from_numpy(logits).cuda(), 6, renormalize=False)
    ids_o, w_o = orouter.router_topk(logits, 6, renormalize=False)
    np.testing.assert_array_equal(ids_g.cpu().numpy(), ids_o)
    assert ids_o[3].tolist() == [0, 1, 2, 3, 4, 5]
    np.testing.assert_allclose(w_g.cpu().numpy(), w_o, rtol=(40 + 3) * 2.0 ** -23)
    empty = torch.empty((0, 40), dtype=torch.float32, device="cuda")
    i0, w0 = pm.moe_router_topk(empty, 6)
    assert i0.shape == (0, 6)


def _ids_tensor(sets):
    return torch.tensor(np.asarray(sets, dtype=np.int32)).cuda()


def _check_table(cache, sim, layer=0):
    exp_in, last = cache.expert_cache_slot_table(layer)
    assert exp_in.tolist() == sim.expert_in
    assert last.tolist() == sim.last_use


def test_residency_hand_trace(pm):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "lru_hand_trace.json")))
    L = hz.SyntheticLayer(0, g["E"], 128, 64, seed=1)
    cache = hz.make_cache([L], g["top_k"], g["K"], max_tokens=4)
    sim = olru.LayerLRU(g["E"], g["K"])
    for st in g["steps"]:
        ids = torch.tensor(st["ids"], dtype=torch.int32).cuda()
        waves = cache.expert_cache_ensure_resident(0, ids)
        out = sim.step(st["ids"])
        assert waves == st["waves"] == len(out["waves"])
        _check_table(cache, sim)
    s = cache.expert_cache_stats(0)
    assert (s["misses"], s["hits"], s["waves"], s["steps"]) == (10, 4, 7, 6)
    cache.close()


@pytest.mark.parametrize("K,B,E", [(40, 4, 128), (26, 4, 128), (3, 1, 16), (128, 4, 128), (1, 2, 8)])
def test_residency_matches_simulator_over_reuse_traces(pm, K, B, E):
    k = 8 if E >= 16 else 2
    rng = np.random.default_rng(K * 7 + B)
    trace = gen.reuse_routing_trace(rng, E, k, B, 256)
    L = hz.SyntheticLayer(0, E, 128, 64, seed=2)
    cache = hz.make_cache([L], k, K, max_tokens=B)
    sim = olru.LayerLRU(E, K)
    for s, sets in enumerate(trace):
        flat = [e for st in sets for e in st]
        waves = cache.expert_cache_ensure_resident(0, _ids_tensor(flat))
        out = sim.step(flat)
        assert waves == len(out["waves"]), s
        if s % 32 == 0 or s == len(trace) - 1:
            _check_table(cache, sim)
    _check_table(cache, sim)
    st = cache.expert_cache_stats(0)
    assert (st["misses"], st["hits"], st["waves"]) == (sim.misses, sim.hits, sim.waves)
    cache.close()


def test_residency_cold_prefill_worked_example(pm):
    L = hz.SyntheticLayer(0, 128, 128, 64, seed=3)
    cache = hz.make_cache([L], 8, 92, max_tokens=16)
    ids = torch.arange(128, dtype=torch.int32).cuda()
    waves = cache.expert_cache_ensure_resident(0, ids)
    assert waves == 2
    exp_in, last = cache.expert_cache_slot_table(0)
    assert exp_in.tolist() == [92 + i if i < 36 else i for i in range(92)]
    assert cache.expert_cache_stats(0)["misses"] == 128
    cache.close()


def _run_steps(cache, steps, layer=0, residual=None):
    ys = []
    for x_bits, logits in steps:
        x = hz.to_device_bf16(x_bits)
        ids, w = cache_route(logits, cache.top_k)
        y = cache.moe_paged_forward(layer, x, ids, w, residual=residual)
        ys.append(y)
    torch.cuda.synchronize()
    return [y.clone() for y in ys]


def cache_route(logits, k):
    import paged_expert_moe_gb300 as pm
    return pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)


def test_tiny_layer_parity_and_bitwise_k_invariance(pm):
    """E=8, top_k=2, H=128, I=64, 4 tokens; K=8 (no paging) against the oracle, and the
    same outputs bit for bit with K = 1, 2, 3, 4 (several waves per step)."""
    E, k, H, I, T = 8, 2, 128, 64, 4
    L = hz.SyntheticLayer(0, E, H, I, seed=0)
    rng = np.random.default_rng(0)
    steps = []
    for _ in range(3):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        steps.append(hz.step_inputs(rng, sets, E, H))
    ref_ys = []
    for x_bits, logits in steps:
        ids, w = orouter.router_topk(logits, k)
        ref_ys.append(L.oracle_y(x_bits, ids, w))
    outs = {}
    for K in (8, 1, 2, 3, 4):
        cache = hz.make_cache([L], k, K, max_tokens=T)
        outs[K] = _run_steps(cache, steps)
        cache.close()
    for i, y in enumerate(outs[8]):
        hz.assert_layer_close(hz.bf16_to_f64(y), ref_ys[i], 0)
    for K in (1, 2, 3, 4):
        for a, b in zip(outs[K], outs[8]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"K={K} differs"


def _decode_case(pm, fmt, E, K, B, n_steps, seed, mode=0, fast_int4=False, check_every=1):
    k, H, I = 8, 2048, 768
    L = hz.SyntheticLayer(fmt, E, H, I, seed=seed, fast_int4=fast_int4)
    rng = np.random.default_rng(seed)
    trace = gen.reuse_routing_trace(rng, E, k, B, n_steps)
    steps = [hz.step_inputs(rng, sets, E, H) for sets in trace]
    cache = hz.make_cache([L], k, K, max_tokens=B, mode=mode)
    ys = _run_steps(cache, steps)
    sim = olru.LayerLRU(E, K)
    for sets in trace:
        sim.step([e for st in sets for e in st])
    _check_table(cache, sim)
    st = cache.expert_cache_stats(0)
    assert (st["misses"], st["hits"]) == (sim.misses, sim.hits)
    # independence check: every slot holds exactly the bytes of the expert the table names
    exp_in, _ = cache.expert_cache_slot_table(0)
    for s, e in enumerate(exp_in.tolist()):
        if e >= 0:
            assert np.array_equal(cache.expert_cache_read_slot(0, s), L.store[e]), (s, e)
    cache.close()
    for i in range(0, n_steps, check_every):
        x_bits, logits = steps[i]
        ids, w = orouter.router_topk(logits, k)
        hz.assert_layer_close(hz.bf16_to_f64(ys[i]), L.oracle_y(x_bits, ids, w), fmt)
    return L, steps, ys


def _assert_bitwise_equal_to_all_resident(L, steps, ys, B, mode=0):
    """Paging never changes the result (section "Can paging change the model's outputs?"):
    the same steps with every expert resident (K = E) give the same bits."""
    cache = hz.make_cache([L], 8, L.E, max_tokens=B, mode=mode)
    ys_full = _run_steps(cache, steps)
    cache.close()
    for i, (a, b) in enumerate(zip(ys, ys_full)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"step {i} differs from K={L.E}"


@pytest.mark.parametrize("B", [1, 2, 4])
def test_decode_bf16_qwen3_layer(pm, B):
    """Qwen3-30B-A3B-shaped layer, bf16, K=40, p=0.8 reuse routing; against the oracle
    and bit for bit against K=128 (everything resident)."""
    L, steps, ys = _decode_case(pm, 0, 128, 40, B, 10, seed=10 + B)
    _assert_bitwise_equal_to_all_resident(L, steps, ys, B)


@pytest.mark.parametrize("B,K,mode", [(1, 40, 0), (4, 26, 1)])
def test_decode_fp8_layer(pm, B, K, mode):
    """Block-FP8 experts: against the oracle, and bit for bit against K=128; B=4 at K=26
    runs several waves in some steps."""
    L, steps, ys = _decode_case(pm, 1, 128, K, B, 8, seed=21 + B, mode=mode)
    _assert_bitwise_equal_to_all_resident(L, steps, ys, B, mode=mode)


@pytest.mark.parametrize("B,mode", [(1, 0), (2, 1), (4, 1)])
def test_decode_mxfp4_layer(pm, B, mode):
    """MXFP4 experts (E2M1 codes, E8M0 scale per 32 inputs), Qwen3 shape with 64 experts;
    B=4 at K=24 runs several waves in some steps; SM-pull mode pages the scale rows in
    with the weights. Bit for bit equal to K=64 (everything resident)."""
    L, steps, ys = _decode_case(pm, 3, 64, 24, B, 8, seed=41 + B, mode=mode)
    _assert_bitwise_equal_to_all_resident(L, steps, ys, B, mode=mode)


@pytest.mark.parametrize("B,mode", [(1, 0), (2, 1), (4, 1)])
def test_decode_nvfp4_layer(pm, B, mode):
    """NVFP4 experts (E2M1 codes, e4m3 scale per 16 inputs, fp32 tensor scale per matrix),
    Qwen3 shape with 64 experts; SM-pull mode pages the experts in inside the fused
    decode kernel (block scales with the rows, the tensor-scale headers with them). B=4 at
    K=24 runs several waves in some steps. Bit for bit equal to K=64 (everything
    resident)."""
    L, steps, ys = _decode_case(pm, 4, 64, 24, B, 8, seed=51 + B, mode=mode)
    _assert_bitwise_equal_to_all_resident(L, steps, ys, B, mode=mode)


@pytest.mark.parametrize("B,K", [(1, 40), (4, 26)])
def test_decode_int4_layer(pm, B, K):
    """B=4 at K=26 exceeds K // top_k = 3: some steps run several waves. Bit for bit
    equal to K=128 (everything resident)."""
    L, steps, ys = _decode_case(pm, 2, 128, K, B, 8, seed=31 + B)
    _assert_bitwise_equal_to_all_resident(L, steps, ys, B)


def test_sm_pull_mode_is_bitwise_identical_to_copy_engine(pm):
    L, steps, ys = _decode_case(pm, 0, 64, 12, 4, 6, seed=41)
    cache = hz.make_cache([L], 8, 12, max_tokens=4, mode=pm.PMOE_PAGEIN_SM_PULL)
    ys2 = _run_steps(cache, steps)
    st = cache.expert_cache_stats(0)
    cache.close()
    assert st["misses"] > 0
    for a, b in zip(ys, ys2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_residual_input_is_added_once(pm):
    E, k, H, I, T = 8, 2, 128, 64, 3
    L = hz.SyntheticLayer(0, E, H, I, seed=5)
    rng = np.random.default_rng(5)
    x_bits, logits = hz.step_inputs(rng, gen.uniform_routing_sets(rng, T, E, k), E, H)
    cache = hz.make_cache([L], k, 4, max_tokens=T)
    x = hz.to_device_bf16(x_bits)
    ids, w = cache_route(logits, k)
    y = cache.moe_paged_forward(0, x, ids, w, residual=x)
    ids_o, w_o = orouter.router_topk(logits, k)
    ref = gen.bf16_bits_to_float(x_bits).astype(np.float64) + L.oracle_y(x_bits, ids_o, w_o)
    hz.assert_layer_close(hz.bf16_to_f64(y), ref, 0)
    cache.close()


def test_argument_and_device_errors(pm):
    L = hz.SyntheticLayer(0, 8, 128, 64, seed=6)
    cache = hz.make_cache([L], 2, 4, max_tokens=4)
    x = torch.zeros((5, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((5, 2), dtype=torch.int32, device="cuda")
    w = torch.zeros((5, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(pm.PmoeError) as ei:
        cache.moe_paged_forward(0, x, ids, w)  # T > max_tokens
    assert ei.value.status == pm.PMOE_EINVAL
    with pytest.raises(pm.PmoeError) as ei:
        cache.moe_paged_forward(0, x[:2], ids[:2], w[:2], y=x[:2])  # y aliases x
    assert ei.value.status == pm.PMOE_EINVAL
    y = cache.moe_paged_forward(0, x[:0], ids[:0], w[:0])  # empty step
    assert y.shape == (0, 128)
    bad = torch.tensor([[1, 9]], dtype=torch.int32, device="cuda")
    with pytest.raises(pm.PmoeError) as ei:
        cache.expert_cache_ensure_resident(0, bad)
    assert ei.value.status == pm.PMOE_EDEVICE
    cache.close()
    with pytest.raises(pm.PmoeError) as ei:
        pm.ExpertCache(8, 2, 128, 64, 9)  # K > E
    assert ei.value.status == pm.PMOE_EINVAL
    with pytest.raises(pm.PmoeError) as ei:
        pm.ExpertCache(8, 2, 200, 64, 4, fmt=pm.PMOE_FP8_BLOCK128)  # FP8 needs multiples of 128
    assert ei.value.status == pm.PMOE_EUNSUPPORTED


def test_host_side_fault_injection(pm, monkeypatch):
    """Failures made on the host: the pinned allocation and the page-in copy issue."""
    monkeypatch.setenv("PMOE_INJECT_HOSTALLOC_FAIL", "1")
    with pytest.raises(pm.PmoeError) as ei:
        pm.ExpertCache(8, 2, 128, 64, 4)
    assert ei.value.status == pm.PMOE_EHOSTALLOC
    monkeypatch.delenv("PMOE_INJECT_HOSTALLOC_FAIL")
    L = hz.SyntheticLayer(0, 8, 128, 64, seed=8)
    cache = hz.make_cache([L], 2, 4, max_tokens=4)
    ids = torch.tensor([[1, 2]], dtype=torch.int32, device="cuda")
    monkeypatch.setenv("PMOE_INJECT_MEMCPY_FAIL", "1")
    with pytest.raises(pm.PmoeError) as ei:
        cache.expert_cache_ensure_resident(0, ids)
    assert ei.value.status == pm.PMOE_ECUDA
    monkeypatch.delenv("PMOE_INJECT_MEMCPY_FAIL")
    exp_in, _ = cache.expert_cache_slot_table(0)
    assert exp_in.tolist() == [-1, -1, -1, -1]  # the table was emptied, no stale slot survives
    assert cache.expert_cache_ensure_resident(0, ids) == 1
    exp_in, _ = cache.expert_cache_slot_table(0)
    for s, e in enumerate(exp_in.tolist()):
        if e >= 0:
            assert np.array_equal(cache.expert_cache_read_slot(0, s), L.store[e])
    cache.close()


@pytest.mark.parametrize("E,H,I,T,k,ids_list,Ks", [
    (16, 256, 128, 2, 4, [[3, 3, 3, 5], [3, 7, 3, 9]], [16, 4, 2]),
    (128, 2048, 768, 1, 8, [[3, 3, 5, 6, 7, 8, 9, 3]], [40, 8]),
])
def test_expert_repeated_within_a_token(pm, E, H, I, T, k, ids_list, Ks):
    """ids that name one expert several times for a token are a sum of repeated terms:
    the decode path handles an expert with more pairs than tokens, at several K."""
    L = hz.SyntheticLayer(0, E, H, I, seed=77)
    rng = np.random.default_rng(77)
    x_bits = gen.activations_bf16(rng, T, H)
    ids_np = np.asarray(ids_list, dtype=np.int32)
    w_np = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    ref = L.oracle_y(x_bits, ids_np, w_np.astype(np.float64))
    outs = []
    for K in Ks:
        cache = hz.make_cache([L], k, K, max_tokens=T)
        y = cache.moe_paged_forward(0, hz.to_device_bf16(x_bits), torch.from_numpy(ids_np).cuda(),
                                    torch.from_numpy(w_np).cuda())
        torch.cuda.synchronize()
        hz.assert_layer_close(hz.bf16_to_f64(y), ref, 0)
        outs.append(y.clone())
        cache.close()
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("fmt,mode", [("bf16", 0), ("int4", 1)])
def test_startup_independence_check(pm, fmt, mode):
    """The library's start-up check (paged == unpaged, slots hold their experts' bytes)
    passes on a small layer with more experts than slots."""
    from paged_expert_moe_gb300 import preflight as pf
    E, k, H, I, K = 16, 4, 256, 128, 5
    L = hz.SyntheticLayer(pf.FORMATS[fmt], E, H, I, seed=90)
    r = pf.independence_check(E, k, H, I, K, L.store, fmt=fmt, tokens=2, steps=5, seed=3, pagein_mode=mode)
    assert r["outputs_equal"] and r["slot_mismatches"] == [] and r["misses"] > K and r["slots_checked"] == K
