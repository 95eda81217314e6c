"""The C ABI without a GPU: the library loads, exports every declared entry point, and
rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"PMOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    declared = _declared()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(pm._lib.EXPORTED)


def test_expert_sizes_from_the_library():
    import paged_expert_moe_gb300 as pm
    assert pm.pmoe_expert_bytes(pm.PMOE_BF16, 2048, 768) == 9_437_184
    assert pm.pmoe_expert_bytes(pm.PMOE_FP8_BLOCK128, 2048, 768) == 4_719_744
    assert pm.pmoe_expert_bytes(pm.PMOE_INT4_GPTQ_G128, 2048, 768) == 2_506_752
    assert pm.pmoe_expert_bytes(pm.PMOE_MXFP4, 2048, 768) == 2_506_752
    assert pm.pmoe_expert_bytes(pm.PMOE_NVFP4, 2048, 768) == 2_654_240
    assert pm.pmoe_expert_bytes(pm.PMOE_NVFP4, 2048, 200) == 0
    assert pm.pmoe_expert_bytes(pm.PMOE_FP8_BLOCK128, 200, 768) == 0
    assert pm.pmoe_expert_bytes(pm.PMOE_MXFP4, 200, 768) == 0
    assert pm.pmoe_expert_bytes(7, 2048, 768) == 0


@pytest.mark.parametrize("H,I", [(2048, 768), (128, 128), (4096, 1536), (1024, 256)])
def test_library_expert_sizes_equal_the_oracle_layout(H, I):
    import paged_expert_moe_gb300 as pm
    from oracle import formats
    for fmt in (pm.PMOE_BF16, pm.PMOE_FP8_BLOCK128, pm.PMOE_INT4_GPTQ_G128, pm.PMOE_MXFP4, pm.PMOE_NVFP4):
        assert pm.pmoe_expert_bytes(fmt, H, I) == formats.expert_nbytes(fmt, H, I), (fmt, H, I)


@pytest.mark.parametrize("desc", [
    dict(num_experts=0, top_k=1, hidden=128, intermediate=64, num_slots=1),
    dict(num_experts=8, top_k=9, hidden=128, intermediate=64, num_slots=4),
    dict(num_experts=8, top_k=2, hidden=128, intermediate=64, num_slots=9),
    dict(num_experts=8, top_k=2, hidden=130, intermediate=64, num_slots=4),
    dict(num_experts=2048, top_k=2, hidden=128, intermediate=64, num_slots=4),
    dict(num_experts=8, top_k=2, hidden=128, intermediate=64, num_slots=4, max_tokens=0),
    dict(num_experts=8, top_k=2, hidden=128, intermediate=64, num_slots=4, pagein_mode=5),
])
def test_create_rejects_bad_descriptors_before_any_cuda_call(desc):
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    full = dict(num_layers=1, format=0, max_tokens=4, pagein_mode=0, device=0)
    full.update(desc)
    d = pm._lib.pmoe_cache_desc(**full)
    h = ctypes.c_void_p()
    assert lib.expert_cache_create(ctypes.byref(d), ctypes.byref(h)) == pm.PMOE_EINVAL
    assert not h.value


def test_create_rejects_unsupported_formats():
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    d = pm._lib.pmoe_cache_desc(num_experts=8, top_k=2, hidden=192, intermediate=64, num_slots=4, num_layers=1,
                                format=pm.PMOE_INT4_GPTQ_G128, max_tokens=4, pagein_mode=0, device=0)
    h = ctypes.c_void_p()
    assert lib.expert_cache_create(ctypes.byref(d), ctypes.byref(h)) == pm.PMOE_EUNSUPPORTED


def test_create_refuses_mxfp4_shapes_off_the_128_grid():
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    for hidden, inter in ((192, 128), (128, 200)):
        d = pm._lib.pmoe_cache_desc(num_experts=8, top_k=2, hidden=hidden, intermediate=inter, num_slots=4,
                                    num_layers=1, format=pm.PMOE_MXFP4, max_tokens=16, pagein_mode=0, device=0)
        h = ctypes.c_void_p()
        assert lib.expert_cache_create(ctypes.byref(d), ctypes.byref(h)) == pm.PMOE_EUNSUPPORTED
        assert not h.value


def test_router_argument_checks_need_no_gpu():
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    nul = ctypes.c_void_p(0)
    assert lib.moe_router_topk(nul, 4, 8, 9, 1, nul, nul, nul) == pm.PMOE_EINVAL
    assert lib.moe_router_topk(nul, 4, 2000, 2, 1, nul, nul, nul) == pm.PMOE_EINVAL
    assert lib.moe_router_topk(nul, 4, 64, 33, 1, nul, nul, nul) == pm.PMOE_EINVAL
    assert lib.moe_router_topk(nul, 0, 8, 2, 1, nul, nul, nul) == pm.PMOE_OK
    assert lib.moe_router_topk(nul, 4, 8, 2, 1, nul, nul, nul) == pm.PMOE_EINVAL
    for s in (0, -1, -2, -3, -4, -5, -6, -7, 42):
        assert lib.pmoe_status_string(s)


def test_null_cache_calls_are_rejected():
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    nul = ctypes.c_void_p(0)
    assert lib.moe_paged_forward(nul, 0, nul, 1, nul, nul, nul, nul, nul) == pm.PMOE_EINVAL
    assert lib.expert_cache_ensure_resident(nul, 0, nul, 1, nul, None) == pm.PMOE_EINVAL
    assert lib.expert_cache_reset(nul, 0) == pm.PMOE_EINVAL
    lib.expert_cache_destroy(nul)


def test_noalloc_argument_checks_need_no_gpu():
    """The allocation-free decode call refuses bad sizes, slot counts and misaligned
    pointers on the host, before any CUDA call."""
    import paged_expert_moe_gb300 as pm
    lib = pm.load()
    nul = ctypes.c_void_p(0)
    p = ctypes.c_void_p
    H, I, E, k = 256, 128, 16, 4
    stride = pm.pmoe_expert_bytes(pm.PMOE_BF16, H, I)

    def call(experts=0x10000, stride=stride, n_slots=E, slot_of=0, T=2, x=0x20000, ids=0x30000, w=0x40000,
             residual=0, y=0x50000, err=0):
        return lib.moe_decode_forward_noalloc(p(experts), stride, n_slots, p(slot_of), E, k, H, I, pm.PMOE_BF16,
                                              p(x), T, p(ids), p(w), p(residual), p(y), p(err), nul)

    assert call(T=9) == pm.PMOE_EINVAL              # beyond the static scratch's token limit
    assert call(n_slots=E - 1) == pm.PMOE_EINVAL    # no slot map and fewer slots than experts
    assert call(n_slots=0, slot_of=0x60000) == pm.PMOE_EINVAL
    assert call(stride=stride - 16) == pm.PMOE_EINVAL
    assert call(x=0x20008) == pm.PMOE_EINVAL        # x, y, experts, residual: 16-byte aligned
    assert call(y=0x50004) == pm.PMOE_EINVAL
    assert call(experts=0x10008) == pm.PMOE_EINVAL
    assert call(residual=0x70002) == pm.PMOE_EINVAL
    assert call(ids=0x30002) == pm.PMOE_EINVAL      # ids, w, slot_of, err_out: 4-byte aligned
    assert call(err=0x80001) == pm.PMOE_EINVAL
    assert call(x=0x20000, y=0x20000) == pm.PMOE_EINVAL  # y aliases x
    assert call(ids=0) == pm.PMOE_EINVAL
