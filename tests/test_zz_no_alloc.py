"""The allocation-free decode entry point, against moe_paged_forward.

moe_decode_forward_noalloc serves callers that cannot call cudaMalloc (code inside
another framework's memory pool or allocator hooks, real-time loops that must not
enter the driver's allocator, embedders with a fixed device-memory budget): it keeps
its intermediates in the library's fixed static device scratch. This file runs last
(pytest collects it after the others) and also passes on its own in a fresh process.
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


def _experts_on_device(store, stride, order=None):
    E, nb = store.shape
    buf = np.zeros((E, stride), np.uint8)
    for slot in range(E):
        e = slot if order is None else order[slot]
        buf[slot, :nb] = store[e]
    return torch.from_numpy(buf).cuda()


@pytest.mark.parametrize("fmt", [0, 2])
def test_noalloc_matches_paged_forward_on_two_calls(pm, fmt):
    E, k, H, I, T = 32, 8, 2048, 768, 4
    L = hz.SyntheticLayer(fmt, E, H, I, seed=77)
    nb = pm.pmoe_expert_bytes(fmt, H, I)
    stride = (nb + 4095) // 4096 * 4096
    experts = _experts_on_device(L.store, stride)
    cache = hz.make_cache([L], k, E, max_tokens=T)
    rng = np.random.default_rng(78)
    for call in range(2):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        x_bits, logits = hz.step_inputs(rng, sets, E, H)
        x = hz.to_device_bf16(x_bits)
        ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
        y_ref = cache.moe_paged_forward(0, x, ids, w)
        y = pm.moe_decode_forward_noalloc(experts, stride, E, k, H, I, fmt, x, ids, w)
        torch.cuda.synchronize()
        hz.assert_layer_close(hz.bf16_to_f64(y), hz.bf16_to_f64(y_ref), fmt)
    cache.close()


def test_noalloc_with_a_slot_map_and_limits(pm):
    E, k, H, I, T = 16, 4, 256, 128, 2
    L = hz.SyntheticLayer(0, E, H, I, seed=79)
    nb = pm.pmoe_expert_bytes(0, H, I)
    stride = nb
    order = np.random.default_rng(80).permutation(E)  # slot s holds expert order[s]
    experts = _experts_on_device(L.store, stride, order)
    slot_of = torch.tensor(np.argsort(order).astype(np.int32)).cuda()
    cache = hz.make_cache([L], k, E, max_tokens=T)
    rng = np.random.default_rng(81)
    for call in range(2):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        x_bits, logits = hz.step_inputs(rng, sets, E, H)
        x = hz.to_device_bf16(x_bits)
        ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
        y_ref = cache.moe_paged_forward(0, x, ids, w)
        y = pm.moe_decode_forward_noalloc(experts, stride, E, k, H, I, 0, x, ids, w, slot_of=slot_of)
        torch.cuda.synchronize()
        hz.assert_layer_close(hz.bf16_to_f64(y), hz.bf16_to_f64(y_ref), 0)
    cache.close()
    # beyond the static scratch's limits: rejected before anything is enqueued
    x9 = torch.zeros((9, H), dtype=torch.bfloat16, device="cuda")
    ids9 = torch.zeros((9, k), dtype=torch.int32, device="cuda")
    w9 = torch.zeros((9, k), dtype=torch.float32, device="cuda")
    with pytest.raises(pm.PmoeError) as ei:
        pm.moe_decode_forward_noalloc(experts, stride, E, k, H, I, 0, x9, ids9, w9)
    assert ei.value.status == pm.PMOE_EINVAL
    with pytest.raises(pm.PmoeError) as ei:
        pm.moe_decode_forward_noalloc(experts, stride - 16, E, k, H, I, 0, x9[:1], ids9[:1], w9[:1])
    assert ei.value.status == pm.PMOE_EINVAL
