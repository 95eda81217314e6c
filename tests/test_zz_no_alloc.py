"""The allocation-free decode entry point, against the oracle and moe_paged_forward.

moe_decode_forward_noalloc serves callers that cannot call cudaMalloc (code inside
another framework's memory pool or allocator hooks, real-time loops that must not
enter the driver's allocator, embedders with a fixed device-memory budget): it keeps
its intermediates in the library's fixed static device scratch. Every case makes two
calls in a row on that shared scratch. This file runs last (pytest collects it after
the others) and also passes on its own in a fresh process.
"""

import numpy as np
import pytest

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


def _experts_on_device(store, stride, order=None):
    E, nb = store.shape
    n = E if order is None else len(order)
    buf = np.zeros((n, stride), np.uint8)
    for slot in range(n):
        e = slot if order is None else order[slot]
        buf[slot, :nb] = store[e]
    return torch.from_numpy(buf).cuda()


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_noalloc_matches_oracle_and_paged_forward_on_two_calls(pm, fmt):
    """Qwen3 shape (H=2048, I=768), 32 experts, 4 tokens, every format: each of two calls
    in a row is within the layer tolerance of the oracle and of moe_paged_forward, and
    reports no device error."""
    E, k, H, I, T = 32, 8, 2048, 768, 4
    L = hz.SyntheticLayer(fmt, E, H, I, seed=77 + fmt)
    nb = pm.pmoe_expert_bytes(fmt, H, I)
    stride = (nb + 4095) // 4096 * 4096
    experts = _experts_on_device(L.store, stride)
    cache = hz.make_cache([L], k, E, max_tokens=T)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(78 + fmt)
    for call in range(2):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        x_bits, logits = hz.step_inputs(rng, sets, E, H)
        x = hz.to_device_bf16(x_bits)
        ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
        y_paged = cache.moe_paged_forward(0, x, ids, w)
        y = pm.moe_decode_forward_noalloc(experts, stride, E, k, H, I, fmt, x, ids, w, err_out=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error bits {int(err.item())}"
        ids_o, w_o = orouter.router_topk(logits, k)
        hz.assert_layer_close(hz.bf16_to_f64(y), L.oracle_y(x_bits, ids_o, w_o), fmt)
        hz.assert_layer_close(hz.bf16_to_f64(y), hz.bf16_to_f64(y_paged), fmt)
    cache.close()


def test_noalloc_slot_map_absent_and_out_of_range_slots(pm):
    """A permuted slot map over fewer slots than experts: an expert with slot -1 and an
    expert whose slot lies past the last slot both contribute nothing (the oracle with
    their weighted terms removed); only the second raises the bad-slot error bit."""
    E, k, H, I, T = 16, 4, 256, 128, 2
    L = hz.SyntheticLayer(0, E, H, I, seed=79)
    nb = pm.pmoe_expert_bytes(0, H, I)
    stride = nb
    rng = np.random.default_rng(80)
    n_slots = E - 2
    order = rng.permutation(E)[:n_slots]  # slot s holds expert order[s]
    experts = _experts_on_device(L.store, stride, order)
    slot_np = np.full(E, -1, np.int32)
    slot_np[order] = np.arange(n_slots, dtype=np.int32)
    absent = [e for e in range(E) if slot_np[e] < 0]
    assert len(absent) == 2
    bad = absent[1]
    slot_np[bad] = n_slots  # one past the end of `experts`: must be refused on the device
    slot_of = torch.from_numpy(slot_np).cuda()
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        sets = gen.uniform_routing_sets(rng, T, E, k)
        others = [int(e) for e in rng.permutation([e for e in range(E) if e not in absent])[:k - 2]]
        sets[0] = [absent[0], bad] + others  # token 0 routes to both slotless experts
        x_bits, logits = hz.step_inputs(rng, sets, E, H)
        x = hz.to_device_bf16(x_bits)
        ids, w = pm.moe_router_topk(torch.from_numpy(logits).cuda(), k)
        y = pm.moe_decode_forward_noalloc(experts, stride, E, k, H, I, 0, x, ids, w, slot_of=slot_of,
                                          n_slots=n_slots, err_out=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 4, f"call {call}: device error bits {int(err.item())}"
        ids_o, w_o = orouter.router_topk(logits, k)
        assert absent[0] in ids_o[0] and bad in ids_o[0]
        w_kept = np.where(np.isin(ids_o, absent), 0.0, w_o)
        hz.assert_layer_close(hz.bf16_to_f64(y), L.oracle_y(x_bits, ids_o, w_kept), 0)


def test_noalloc_rejects_requests_beyond_its_limits(pm):
    E, k, H, I = 16, 4, 256, 128
    L = hz.SyntheticLayer(0, E, H, I, seed=81)
    stride = pm.pmoe_expert_bytes(0, H, I)
    experts = _experts_on_device(L.store, stride)
    x9 = torch.zeros((9, H), dtype=torch.bfloat16, device="cuda")
    ids9 = torch.zeros((9, k), dtype=torch.int32, device="cuda")
    w9 = torch.zeros((9, k), dtype=torch.float32, device="cuda")

    def status(**kw):
        with pytest.raises(pm.PmoeError) as ei:
            args = dict(experts=experts, stride=stride, E=E, top_k=k, H=H, I=I, fmt=0, x=x9[:1], ids=ids9[:1],
                        w=w9[:1])
            args.update(kw)
            pm.moe_decode_forward_noalloc(**args)
        return ei.value.status

    assert status(x=x9, ids=ids9, w=w9) == pm.PMOE_EINVAL  # T > 8: beyond the static scratch
    assert status(stride=stride - 16) == pm.PMOE_EINVAL  # a slot shorter than one expert
    assert status(n_slots=E - 1) == pm.PMOE_EINVAL  # no slot map, fewer slots than experts
    xm = torch.zeros((2 * H + 8,), dtype=torch.bfloat16, device="cuda")[1:H + 1].view(1, H)
    assert status(x=xm) == pm.PMOE_EINVAL  # x not 16-byte aligned
