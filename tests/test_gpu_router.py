"""Router projection fused with the top-k (moe_router_gemm_topk) against the oracle.

The oracle computes the logits in float64 (oracle.router.router_logits) and routes them
with the same selection rule. The GPU accumulates bf16 products in fp32; each product is
exact in fp32, so its logits differ from the float64 ones by at most the accumulated
rounding H * 2^-24 * sum_c |x_c w_c| (a worst-case bound). Selection and weights are
checked exactly against the oracle applied to the GPU's own logits, and against the
oracle's float64 selection wherever its k-th/(k+1)-th gap exceeds twice that bound.
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


def _rtol(k):
    # fp32: expf within 2 ulp, k-1 additions and one division each within half an ulp
    return (k + 3) * 2.0 ** -23


@pytest.mark.parametrize("T,E,H,k", [(1, 128, 2048, 8), (5, 128, 2048, 8), (8, 8, 128, 2), (13, 160, 256, 6),
                                     (2048, 128, 2048, 8), (3, 1024, 512, 32), (9, 33, 136, 5)])
def test_router_gemm_matches_oracle(pm, T, E, H, k):
    rng = np.random.default_rng(1000 + 7 * T + E)
    x_bits = gen.activations_bf16(rng, T, H)
    w_bits = gen.bf16_bits(rng.standard_normal((E, H)) * 0.05)
    x = hz.to_device_bf16(x_bits)
    W = hz.to_device_bf16(w_bits)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids, w = pm.moe_router_gemm_topk(x, W, k, logits_out=logits)
    torch.cuda.synchronize()
    xo = gen.bf16_bits_to_float(x_bits).astype(np.float64)
    wo = gen.bf16_bits_to_float(w_bits).astype(np.float64)
    ref = orouter.router_logits(xo, wo)
    got = logits.cpu().numpy().astype(np.float64)
    bound = H * 2.0 ** -24 * (np.abs(xo) @ np.abs(wo).T)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / np.maximum(bound, 1e-300)))
    # selection and weights: the router rule on the GPU's own logits, exactly
    ids_g, w_g = ids.cpu().numpy(), w.cpu().numpy()
    ids_r, w_r = orouter.router_topk(got, k)
    assert np.array_equal(ids_g, ids_r)
    np.testing.assert_allclose(w_g, w_r, rtol=_rtol(k), atol=0)
    # the float64 selection wherever the gap leaves no doubt
    ids_o, _, _ = orouter.router_gemm_topk(xo, wo, k)
    srt = -np.sort(-ref, axis=1)
    gap = srt[:, k - 1] - srt[:, k] if k < E else np.full(T, np.inf)
    sure = gap > 2 * bound.max(axis=1)
    assert sure.mean() > 0.5
    assert np.array_equal(ids_g[sure], ids_o[sure])


def test_router_gemm_equals_projection_then_router(pm):
    """The fused call gives the same bits as its logits routed by moe_router_topk."""
    rng = np.random.default_rng(77)
    T, E, H, k = 37, 128, 2048, 8
    x = hz.to_device_bf16(gen.activations_bf16(rng, T, H))
    W = hz.to_device_bf16(gen.bf16_bits(rng.standard_normal((E, H)) * 0.05))
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids, w = pm.moe_router_gemm_topk(x, W, k, logits_out=logits)
    ids2, w2 = pm.moe_router_topk(logits, k)
    ids3, w3 = pm.moe_router_gemm_topk(x, W, k)  # without the logits output
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    assert torch.equal(ids, ids3) and torch.equal(w, w3)


def test_router_gemm_argument_errors(pm):
    x = torch.zeros((2, 12), dtype=torch.bfloat16, device="cuda")  # H = 12 is not a multiple of 8
    W = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pm.PmoeError) as ei:
        pm.moe_router_gemm_topk(x, W, 2)
    assert ei.value.status == pm.PMOE_EINVAL
