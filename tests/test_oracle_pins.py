"""Pins of the oracle against facts that do not come from the oracle itself.

Each test states what fixes the expected value: a value the pages print, a
closed form, an invariant, a library routine the case reduces to, or brute force
on a tiny input. The mutation tests at the end plant plausible mistakes in the
oracle (on the CPU) and check that some pin catches each one.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import formats, lru, moe, permute, preflight, router
from workloads import generators as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- router

def test_topk_set_is_the_max_sum_subset():
    """Brute force: with distinct logits the top-k set is the k-subset of largest sum."""
    rng = np.random.default_rng(1)
    E, k = 7, 3
    for _ in range(50):
        l = rng.standard_normal((1, E)).astype(np.float32)
        ids, _ = router.router_topk(l, k)
        best = max(itertools.combinations(range(E), k), key=lambda S: sum(float(l[0, e]) for e in S))
        assert sorted(ids[0].tolist()) == sorted(best)
        # descending logit order
        assert all(l[0, ids[0, r]] > l[0, ids[0, r + 1]] for r in range(k - 1))


def test_renormalised_weights_are_softmax_of_selected_logits():
    """Closed form: the full softmax denominator cancels, so w = softmax over S alone."""
    rng = np.random.default_rng(2)
    l = rng.standard_normal((16, 128)).astype(np.float32)
    ids, w = router.router_topk(l, 8)
    for t in range(16):
        ref = scipy.special.softmax(l[t, ids[t]].astype(np.float64))
        np.testing.assert_allclose(w[t], ref, rtol=1e-12, atol=0)


def test_router_with_k_equal_e_is_plain_softmax():
    """Special case E = k: renormalisation is the identity; compare with scipy's softmax."""
    rng = np.random.default_rng(3)
    l = rng.standard_normal((5, 6)).astype(np.float32)
    ids, w = router.router_topk(l, 6)
    for t in range(5):
        full = scipy.special.softmax(l[t].astype(np.float64))
        np.testing.assert_allclose(w[t], full[ids[t]], rtol=1e-12)
    # without renormalisation the weights are the full softmax probabilities
    ids2, w2 = router.router_topk(l, 3, renormalize=False)
    for t in range(5):
        full = scipy.special.softmax(l[t].astype(np.float64))
        np.testing.assert_allclose(w2[t], full[ids2[t]], rtol=1e-12)
        assert w2[t].sum() < 1.0


def test_router_ties_go_to_lower_id_and_shift_invariance():
    l = np.array([[0.5, 1.0, 1.0, -2.0, 1.0]], dtype=np.float32)
    ids, w = router.router_topk(l, 2)
    assert ids.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], rtol=1e-15)
    rng = np.random.default_rng(4)
    l = rng.standard_normal((8, 32)).astype(np.float32)
    i1, w1 = router.router_topk(l, 4)
    i2, w2 = router.router_topk(l + np.float32(3.0), 4)
    assert (i1 == i2).all()
    np.testing.assert_allclose(w1, w2, rtol=1e-6)


def test_logit_generator_enforces_the_gap():
    """The generator's logits select exactly the requested sets with a k/(k+1) gap > 1e-3."""
    rng = np.random.default_rng(5)
    sets = gen.uniform_routing_sets(rng, 64, 128, 8)
    l = gen.logits_for_sets(rng, sets, 128)
    ids, _ = router.router_topk(l, 8)
    for t in range(64):
        assert sorted(ids[t].tolist()) == sorted(int(e) for e in sets[t])
        v = np.sort(l[t])[::-1]
        assert float(v[7]) - float(v[8]) > 1e-3


# ----------------------------------------------------------------------------- expert math

def _dense_weights(rng, H, I, std=0.05):
    return (rng.standard_normal((I, H)) * std, rng.standard_normal((I, H)) * std,
            rng.standard_normal((H, I)) * std)


def _torch_swiglu(x, Wg, Wu, Wd):
    xt = torch.from_numpy(np.asarray(x, np.float64))
    g = torch.nn.functional.linear(xt, torch.from_numpy(Wg))
    u = torch.nn.functional.linear(xt, torch.from_numpy(Wu))
    return torch.nn.functional.linear(torch.nn.functional.silu(g) * u, torch.from_numpy(Wd)).numpy()


def test_single_expert_layer_is_a_dense_swiglu_mlp():
    """E = k = 1 reduces to one Qwen3 MLP: compare with torch.nn.functional (CPU, float64)."""
    rng = np.random.default_rng(6)
    H, I = 32, 24
    W = _dense_weights(rng, H, I)
    x = rng.standard_normal((5, H))
    y, n = moe.moe_layer(x, np.zeros((5, 1), np.int32), np.ones((5, 1)), lambda e: W)
    np.testing.assert_allclose(y, _torch_swiglu(x, *W), rtol=1e-12, atol=1e-14)
    assert n == 5


def test_identical_experts_give_one_mlp_output():
    """Weights sum to one, so identical experts combine to a single MLP output."""
    rng = np.random.default_rng(7)
    H, I, E, k = 16, 8, 6, 3
    W = _dense_weights(rng, H, I)
    l = rng.standard_normal((4, E)).astype(np.float32)
    ids, w = router.router_topk(l, k)
    x = rng.standard_normal((4, H))
    y, _ = moe.moe_layer(x, ids, w, lambda e: W)
    np.testing.assert_allclose(y, _torch_swiglu(x, *W), rtol=1e-12, atol=1e-14)


def test_layer_is_invariant_under_relabelling_experts_and_linear_in_down():
    rng = np.random.default_rng(8)
    H, I, E, k, T = 16, 8, 6, 2, 5
    Ws = [_dense_weights(rng, H, I) for _ in range(E)]
    l = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, H))
    ids, w = router.router_topk(l, k)
    y, _ = moe.moe_layer(x, ids, w, lambda e: Ws[e])
    perm = rng.permutation(E)  # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    l2 = np.empty_like(l)
    l2[:, perm] = l
    ids2, w2 = router.router_topk(l2, k)
    y2, _ = moe.moe_layer(x, ids2, w2, lambda e: Ws[inv[e]])
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-15)
    y3, _ = moe.moe_layer(x, ids, w, lambda e: (Ws[e][0], Ws[e][1], 2.5 * Ws[e][2]))
    np.testing.assert_allclose(y3, 2.5 * y, rtol=1e-12, atol=1e-15)


def test_rank_weights_enter_linearly():
    """Brute force on a tiny case: y = sum_r w_r * MLP_r(x), each MLP from torch."""
    rng = np.random.default_rng(9)
    H, I, E, k = 8, 4, 4, 2
    Ws = [_dense_weights(rng, H, I, 0.3) for _ in range(E)]
    x = rng.standard_normal((1, H))
    ids = np.array([[2, 0]])
    w = np.array([[0.7, 0.3]])
    y, _ = moe.moe_layer(x, ids, w, lambda e: Ws[e])
    ref = 0.7 * _torch_swiglu(x, *Ws[2]) + 0.3 * _torch_swiglu(x, *Ws[0])
    np.testing.assert_allclose(y, ref, rtol=1e-12)


def test_stack_activation_count_is_layers_times_top_k():
    """'Why is it fast when experts keep crossing PCIe?': one token at batch 1 activates
    48 x 8 = 384 experts."""
    rng = np.random.default_rng(10)
    H, I, E, k, L = 8, 4, 128, 8, 48
    Ws = [_dense_weights(rng, H, I, 0.1) for _ in range(4)]
    layers = []
    for _ in range(L):
        ids, w = router.router_topk(rng.standard_normal((1, E)).astype(np.float32), k)
        layers.append((ids, w, lambda e: Ws[e % 4]))
    _, n = moe.moe_stack(rng.standard_normal((1, H)), layers)
    assert n == 384 == preflight.activations_per_token(48, 8)


def test_residual_stack_with_zero_down_projections_returns_its_input():
    """With every W_d = 0 each layer adds nothing to the residual stream, so the stack is
    the identity on x (a dropped residual would return 0, a doubled one 2^L x)."""
    rng = np.random.default_rng(11)
    H, I, E, k, L = 12, 6, 5, 2, 3
    Ws = [_dense_weights(rng, H, I) for _ in range(E)]
    zeroed = [(Wg, Wu, np.zeros_like(Wd)) for Wg, Wu, Wd in Ws]
    x = rng.standard_normal((4, H))
    layers = []
    for _ in range(L):
        ids, w = router.router_topk(rng.standard_normal((4, E)).astype(np.float32), k)
        layers.append((ids, w, lambda e: zeroed[e]))
    h, n = moe.moe_stack(x, layers, residual=True)
    assert np.array_equal(h, x) and n == 4 * k * L


def test_residual_stack_matches_a_hand_built_two_layer_decoder():
    """Two layers with one expert each (k = 1, weight 1): h1 = x + MLP_0(x), h2 = h1 +
    MLP_1(h1), every MLP from torch.nn.functional (a decoder block's residual add)."""
    rng = np.random.default_rng(12)
    H, I = 16, 8
    W0, W1 = _dense_weights(rng, H, I, 0.3), _dense_weights(rng, H, I, 0.3)
    x = rng.standard_normal((3, H))
    one = (np.zeros((3, 1), np.int32), np.ones((3, 1)))
    h, n = moe.moe_stack(x, [(*one, lambda e: W0), (*one, lambda e: W1)], residual=True)
    h1 = x + _torch_swiglu(x, *W0)
    np.testing.assert_allclose(h, h1 + _torch_swiglu(h1, *W1), rtol=1e-12, atol=1e-14)
    assert n == 6


# ----------------------------------------------------------------------------- formats

def test_expert_sizes_match_the_layout_closed_forms():
    H, I = 2048, 768
    assert formats.expert_nbytes(0, H, I) == 9_437_184
    assert formats.expert_nbytes(1, H, I) == 4_719_744  # 3*2048*768 weights + 288 fp32 scales
    assert formats.expert_nbytes(2, H, I) == 2_506_752  # packed nibbles + 36,864 x (fp16 s, fp16 z)
    # the article's FP8 expert size counts the weights only, one byte each (section "Why is
    # it fast when experts keep crossing PCIe?")
    assert 3 * H * I == 4_718_592
    # NVFP4: packed codes, then per matrix 16 bytes (fp32 tensor scale + padding) and one
    # e4m3 byte per row and 16 inputs
    assert formats.expert_nbytes(4, H, I) == 2_359_296 + 16 + 196_608 + 16 + 98_304 == 2_654_240
    for f in (0, 1, 2, 3, 4):
        assert formats.expert_nbytes(f, H, I) == gen.expert_nbytes(f, H, I)


def test_e4m3_table_matches_torch_float8_for_every_code():
    """Library routine: torch's float8_e4m3fn -> float32 conversion, all 256 codes."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        if math.isnan(codes[c]):
            assert math.isnan(formats.E4M3_TABLE[c])
        else:
            assert formats.E4M3_TABLE[c] == float(codes[c]), hex(c)


def test_e4m3_printed_values():
    g = _golden("e4m3_codes.json")
    for code, v in g["codes"].items():
        got = formats.E4M3_TABLE[int(code, 16)]
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), code
    for code in g["nan_codes"]:
        assert math.isnan(formats.E4M3_TABLE[int(code, 16)])


def _fp8_expert_from_parts(qgu, qd, sgu, sd):
    return np.concatenate([qgu.ravel(), qd.ravel(), sgu.astype(np.float32).view(np.uint8).ravel(),
                           sd.astype(np.float32).view(np.uint8).ravel()])


def test_fp8_block_scale_indexing():
    """All codes 1.0 and a distinct scale per block: the weights are the scale grid
    expanded by 128 x 128 (catches a transposed or mis-strided scale index)."""
    H, I = 256, 384
    sgu = np.arange(1, (2 * I // 128) * (H // 128) + 1, dtype=np.float32).reshape(2 * I // 128, H // 128)
    sd = 100 + np.arange((H // 128) * (I // 128), dtype=np.float32).reshape(H // 128, I // 128)
    buf = _fp8_expert_from_parts(np.full((2 * I, H), 0x38, np.uint8), np.full((H, I), 0x38, np.uint8), sgu, sd)
    Wg, Wu, Wd = formats.decode_expert(buf, 1, H, I)
    Wgu = np.concatenate([Wg, Wu])
    np.testing.assert_array_equal(Wgu, np.kron(sgu, np.ones((128, 128))))
    np.testing.assert_array_equal(Wd, np.kron(sd, np.ones((128, 128))))
    assert Wu[0, 0] == sgu[I // 128, 0]  # up rows start at row I


def test_int4_nibble_order_and_group_indexing():
    """Hand-built GPTQ expert: byte 0x21 holds elements 1 (low) then 2 (high)."""
    H, I = 128, 128
    qgu = np.zeros((2 * I, H // 2), np.uint8)
    qgu[0, 0] = 0x21
    qgu[5, 63] = 0xF0  # row 5: element 126 = 0, element 127 = 15
    qd = np.zeros((H, I // 2), np.uint8)
    qd[3, 1] = 0x7A  # row 3: element 2 = 10, element 3 = 7
    szgu = np.zeros((2 * I, H // 128, 2), np.float16)
    szgu[:, :, 0] = 0.5
    szgu[:, :, 1] = 1.0
    szgu[5, 0] = (0.25, 8.0)
    szd = np.zeros((H, I // 128, 2), np.float16)
    szd[:, :, 0] = 2.0
    szd[:, :, 1] = 3.0
    buf = np.concatenate([qgu.ravel(), qd.ravel(), szgu.view(np.uint8).ravel(), szd.view(np.uint8).ravel()])
    Wg, Wu, Wd = formats.decode_expert(buf, 2, H, I)
    assert Wg[0, 0] == (1 - 1.0) * 0.5 and Wg[0, 1] == (2 - 1.0) * 0.5 and Wg[0, 2] == (0 - 1.0) * 0.5
    assert Wg[5, 126] == (0 - 8.0) * 0.25 and Wg[5, 127] == (15 - 8.0) * 0.25
    assert Wd[3, 2] == (10 - 3.0) * 2.0 and Wd[3, 3] == (7 - 3.0) * 2.0


def test_quantised_generators_round_trip_within_their_grids():
    """Closed-form error bounds: e4m3 keeps 3 mantissa bits (relative error <= 2^-4 for
    normal values); the int4 grid's error is at most half a step (s/2, plus fp16 rounding of s)."""
    H, I = 256, 128
    rng = np.random.default_rng([11, 0, 0, 1])
    wgu = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    Wg, Wu, _ = formats.decode_expert(gen.expert_bytes(1, H, I, 11), 1, H, I)
    got = np.concatenate([Wg, Wu])
    sblk = np.kron(np.abs(wgu.reshape(2 * I // 128, 128, H // 128, 128)).max(axis=(1, 3)) / 448.0, np.ones((128, 128)))
    normal = np.abs(wgu) >= sblk * 2.0 ** -6
    err = np.abs(got - wgu)
    assert (err[normal] <= np.abs(wgu[normal]) * 2.0 ** -4 * 1.0001).all()
    assert (err[~normal] <= sblk[~normal] * 2.0 ** -10 * 1.0001).all()
    rng = np.random.default_rng([12, 0, 0, 2])
    wgu = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    Wg, Wu, _ = formats.decode_expert(gen.expert_bytes(2, H, I, 12), 2, H, I)
    got = np.concatenate([Wg, Wu])
    g = wgu.reshape(2 * I, H // 128, 128)
    step = np.repeat((g.max(axis=2) - g.min(axis=2)) / 15.0, 128, axis=1)
    assert (np.abs(got - wgu) <= 0.5 * step * 1.01 + 1e-7).all()


def test_e8m0_scales_match_torch_for_every_byte():
    """The MXFP4 scale byte against torch's float8_e8m0fnu cast (a library routine)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = formats.E8M0_TABLE
    both_nan = np.isnan(ref) & np.isnan(got)
    assert both_nan[255] and not both_nan[:255].any()
    np.testing.assert_array_equal(got[:255], ref[:255])


def test_e2m1_grid_properties_and_generator_round_trip():
    """FP4 E2M1: the positive codes are strictly increasing, the sign bit negates, the
    largest value is 6 and the smallest step 0.5. The generator's own grid (a literal
    list) quantises every oracle value back to its code, and a midpoint to the code with
    the even mantissa, so the two restatements agree."""
    t = formats.E2M1_TABLE
    assert (np.diff(t[:8]) > 0).all() and t[0] == 0.0
    np.testing.assert_array_equal(t[8:], -t[:8])
    assert t[7] == 6.0 and t[1] == 0.5
    # one block of 32 holding every positive and negative grid value, amax 6: scale 2^0
    vals = np.concatenate([t[:8], t[9:], t[:8], t[9:], [6.0, -6.0]])[:32].astype(np.float32)
    packed, x = gen._mxfp4_block_quant(vals.reshape(1, 32))
    assert x.tolist() == [[127]]
    codes = np.empty(32, np.uint8)
    codes[0::2] = packed[0] & 0xF
    codes[1::2] = packed[0] >> 4
    np.testing.assert_array_equal(t[codes], vals)
    # midpoints between neighbours: ties go to the even mantissa (codes 0, 2, 2, 4, 4, 6, 6)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] + [6.0] * 25, np.float32)
    packed, x = gen._mxfp4_block_quant(mids.reshape(1, 32))
    codes[0::2] = packed[0] & 0xF
    codes[1::2] = packed[0] >> 4
    assert codes[:7].tolist() == [0, 2, 2, 4, 4, 6, 6]


def test_mxfp4_nibble_order_and_block_indexing():
    """Hand-built MXFP4 expert: byte 0x32 holds codes 2 (low, 1.0) then 3 (high, 1.5);
    scale byte 128 doubles, 126 halves, one byte per row and block of 32."""
    H, I = 128, 128
    qgu = np.zeros((2 * I, H // 2), np.uint8)
    qgu[0, 0] = 0x32
    qgu[7, 16] = 0xF9  # row 7: element 32 = code 9 (-0.5), element 33 = code 15 (-6)
    qd = np.zeros((H, I // 2), np.uint8)
    qd[4, 63] = 0x70  # row 4: element 126 = 0, element 127 = code 7 (6)
    xgu = np.full((2 * I, H // 32), 127, np.uint8)
    xgu[7, 1] = 128
    xd = np.full((H, I // 32), 127, np.uint8)
    xd[4, 3] = 126
    buf = np.concatenate([qgu.ravel(), qd.ravel(), xgu.ravel(), xd.ravel()])
    Wg, Wu, Wd = formats.decode_expert(buf, 3, H, I)
    assert Wg[0, 0] == 1.0 and Wg[0, 1] == 1.5 and Wg[0, 2] == 0.0
    assert Wg[7, 32] == -0.5 * 2.0 and Wg[7, 33] == -6.0 * 2.0 and Wg[7, 31] == 0.0
    assert Wd[4, 127] == 6.0 * 0.5 and Wd[4, 126] == 0.0
    assert formats.expert_nbytes(3, 2048, 768) == 2506752


def test_mxfp4_generator_error_bound():
    """Per block of 32, with scale X = 2^(floor(log2 amax) - 2): an element below 6X is
    off by at most half a grid step (X at most, X/4 below 2X) and one at or above 6X
    becomes +-6X (the recipe's saturation)."""
    H, I = 256, 128
    rng = np.random.default_rng([14, 0, 0, 3])
    wgu = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    Wg, Wu, _ = formats.decode_expert(gen.expert_bytes(3, H, I, 14), 3, H, I)
    got = np.concatenate([Wg, Wu])
    g = wgu.reshape(2 * I, H // 32, 32)
    X = np.repeat(2.0 ** (np.floor(np.log2(np.abs(g).max(axis=2))) - 2), 32, axis=1)
    a = np.abs(wgu)
    sat = a >= 6 * X
    assert (got[sat] == np.sign(wgu[sat]) * 6 * X[sat]).all()
    half_step = np.where(a < 2 * X, 0.25 * X, np.where(a < 4 * X, 0.5 * X, X))
    assert (np.abs(got - wgu)[~sat] <= half_step[~sat] * 1.0001).all()


def test_nvfp4_nibble_order_and_two_level_scales():
    """Hand-built NVFP4 expert. Codes: 0x32 = codes 2 (low, 1.0) then 3 (high, 1.5); 0xF9 =
    codes 9 (-0.5) then 15 (-6); 0x07 = code 7 (6) then 0; 0x70 = 0 then 6. Block scales
    (e4m3): 0x38 = 1.0, 0x40 = 2.0, 0x3C = 1.5, 0x01 = 2^-9 (the smallest subnormal).
    Tensor scales: 0.5 for gate/up, 2.0 for down. One block scale per row and 16 inputs."""
    H, I = 128, 128
    qgu = np.zeros((2 * I, H // 2), np.uint8)
    qgu[0, 0] = 0x32
    qgu[5, 8] = 0xF9          # row 5: element 16 = -0.5, element 17 = -6 (block 1)
    qgu[I + 3, 0] = 0x07      # up row 3: element 0 = 6
    qd = np.zeros((H, I // 2), np.uint8)
    qd[4, 63] = 0x70          # row 4: element 126 = 0, element 127 = 6 (block 7)
    bgu = np.full((2 * I, H // 16), 0x38, np.uint8)
    bgu[5, 1] = 0x40
    bgu[I + 3, 0] = 0x01
    bd = np.full((H, I // 16), 0x38, np.uint8)
    bd[4, 7] = 0x3C
    t = lambda v: np.concatenate([np.array([v], np.float32).view(np.uint8), np.zeros(12, np.uint8)])
    buf = np.concatenate([qgu.ravel(), qd.ravel(), t(0.5), bgu.ravel(), t(2.0), bd.ravel()])
    Wg, Wu, Wd = formats.decode_expert(buf, 4, H, I)
    assert Wg[0, 0] == 0.5 and Wg[0, 1] == 0.75 and Wg[0, 2] == 0.0
    assert Wg[5, 16] == -0.5 and Wg[5, 17] == -6.0 and Wg[5, 15] == 0.0
    assert Wu[3, 0] == 6.0 * 2.0 ** -10 and Wu[3, 1] == 0.0
    assert Wd[4, 127] == 18.0 and Wd[4, 126] == 0.0
    assert np.count_nonzero(Wg) == 4 and np.count_nonzero(Wu) == 1 and np.count_nonzero(Wd) == 1


def test_nvfp4_generator_error_bound():
    """T = amax / (6 * 448). Per block of 16 with s = e4m3(block scale) * T: an element below
    6s is off by at most half a grid step (s/4 below 2s, s/2 below 4s, s below 6s) and one at
    or above 6s becomes +-6s. No block scale exceeds 448."""
    H, I = 256, 128
    rng = np.random.default_rng([15, 0, 0, 4])
    wgu = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    buf = gen.expert_bytes(4, H, I, 15)
    Wg, Wu, _ = formats.decode_expert(buf, 4, H, I)
    got = np.concatenate([Wg, Wu])
    off = 3 * H * I // 2
    T = float(buf[off:off + 4].view(np.float32)[0])
    assert T == float(np.float32(np.abs(wgu).max() / (6.0 * 448.0)))
    b = formats.E4M3_TABLE[buf[off + 16:off + 16 + 2 * I * H // 16]].reshape(2 * I, H // 16)
    assert b.max() <= 448.0 and b.min() >= 0.0
    s_eff = np.repeat(b * T, 16, axis=1)
    a = np.abs(wgu)
    sat = a >= 6 * s_eff
    assert (got[sat] == np.sign(wgu[sat]) * 6 * s_eff[sat]).all()
    half_step = np.where(a < 2 * s_eff, 0.25 * s_eff, np.where(a < 4 * s_eff, 0.5 * s_eff, s_eff))
    assert (np.abs(got - wgu)[~sat] <= half_step[~sat] * 1.0001 + 1e-12).all()


def test_bf16_decode_matches_torch_bfloat16():
    rng = np.random.default_rng(13)
    H, I = 128, 64
    buf = gen.expert_bytes(0, H, I, 13)
    Wg, Wu, Wd = formats.decode_expert(buf, 0, H, I)
    rng = np.random.default_rng([13, 0, 0, 0])
    wgu = rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(0.02)
    ref = torch.from_numpy(wgu).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(np.concatenate([Wg, Wu]), ref)


# ----------------------------------------------------------------------------- permute

def test_grouping_matches_a_stable_library_sort():
    rng = np.random.default_rng(14)
    for T, k, E in [(1, 2, 8), (7, 3, 5), (64, 8, 128), (3, 1, 4)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
        counts, offs, perm, pos = permute.group_by_expert(ids, E)
        flat = ids.reshape(-1)
        np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
        np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
        np.testing.assert_array_equal(pos[perm], np.arange(T * k))


# ----------------------------------------------------------------------------- LRU simulator

def test_lru_hand_trace():
    g = _golden("lru_hand_trace.json")
    sim = lru.LayerLRU(g["E"], g["K"])
    for st in g["steps"]:
        out = sim.step(st["ids"])
        assert [list(m) for m in out["misses"]] == st["misses"], st["why"]
        assert len(out["waves"]) == st["waves"]
        assert out["hits"] == st["hits"]
        assert out["expert_in"] == st["expert_in"]
        assert out["last_use"] == st["last_use"]
    assert (sim.misses, sim.hits, sim.waves) == tuple(g["totals"][k] for k in ("misses", "hits", "waves"))


def test_lru_cold_prefill_worked_example():
    """K=92, all 128 experts routed, cold: wave 1 loads 0..91 into slots 0..91, wave 2
    evicts slots 0..35 (keys (0, slot)) for experts 92..127; 128 misses, 2 waves."""
    sim = lru.LayerLRU(128, 92)
    out = sim.step(list(range(128)))
    assert out["n_misses"] == 128 and len(out["waves"]) == 2
    assert out["expert_in"] == [92 + i if i < 36 else i for i in range(92)]
    assert [e for e, _ in out["waves"][0]] == list(range(92))
    assert [e for e, _ in out["waves"][1]] == list(range(92, 128))


def test_lru_never_misses_once_everything_fits():
    rng = np.random.default_rng(15)
    sim = lru.LayerLRU(16, 16)
    seen = set()
    for _ in range(50):
        ids = rng.choice(16, size=4, replace=False)
        out = sim.step(ids)
        assert out["n_misses"] == len(set(ids.tolist()) - seen)
        seen |= set(ids.tolist())


@pytest.mark.parametrize("K,printed_pct", [(92, 28), (40, 69), (26, 80)])
def test_lru_uniform_routing_miss_rate_is_one_minus_k_over_e(K, printed_pct):
    """Under uniform independent routing each step's experts are resident with
    probability K/E whatever the policy, so the steady-state miss rate is 1 - K/E;
    the article's table rounds these to 28%, 69% and 80%."""
    rng = np.random.default_rng(16 + K)
    sim = lru.LayerLRU(128, K)
    for _ in range(50):
        sim.step(rng.choice(128, size=8, replace=False))
    m0, n0 = sim.misses, sim.steps
    steps = 3000
    for _ in range(steps):
        sim.step(rng.choice(128, size=8, replace=False))
    rate = (sim.misses - m0) / (8 * (sim.steps - n0))
    exact = 1 - K / 128
    assert abs(rate - exact) < 4 * math.sqrt(exact * (1 - exact) / (8 * steps)) + 0.005
    assert round(100 * exact) == printed_pct


def test_single_wave_rule_and_batch_cap():
    """'What happens with more than one request?': one wave iff tokens x top_k <= K;
    the cap K // top_k is 11, 5 and 3 for K = 92, 40, 26 (and 3 for K = 24)."""
    assert [lru.single_wave_cap(K, 8) for K in (92, 40, 26, 24)] == [11, 5, 3, 3]
    rng = np.random.default_rng(17)
    for K in (24, 26, 40):
        sim = lru.LayerLRU(128, K)
        for B in (1, 2, 3, 4, 5):
            ids = np.concatenate([rng.choice(128, size=8, replace=False) for _ in range(B)])
            out = sim.step(ids)
            U = len(set(ids.tolist()))
            assert (len(out["waves"]) == 1) == (U <= K)
            if B * 8 <= K:
                assert len(out["waves"]) == 1
            # 4 requests x top-8 touch up to 32 distinct experts
            assert U <= 8 * B


def test_lru_prefetch_of_the_own_set_moves_every_miss_into_the_prefetch():
    """A step preceded by a step for the same set (a perfect prefetch) has no misses
    when the set fits in K. Stepping every set twice only relabels the LRU clock in the
    same order, so the total misses and the final table equal those of stepping each
    set once."""
    rng = np.random.default_rng(17)
    E, K, k = 64, 12, 4
    once, twice = lru.LayerLRU(E, K), lru.LayerLRU(E, K)
    for _ in range(300):
        ids = [int(e) for e in rng.choice(E, size=2 * k, replace=True)]
        once.step(ids)
        twice.step(ids)
        assert twice.step(ids)["n_misses"] == 0
    assert twice.misses == once.misses
    assert twice.expert_in == once.expert_in


def test_lru_evicts_only_least_recent_experts():
    """Invariant: in single-wave steps, no resident expert is older than an evicted one."""
    rng = np.random.default_rng(18)
    sim = lru.LayerLRU(32, 10)
    last = {}
    for s in range(300):
        ids = rng.choice(32, size=int(rng.integers(1, 5)), replace=False)
        before = {e for e in range(32) if sim.slot_of[e] >= 0}
        out = sim.step(ids)
        after = {e for e in range(32) if sim.slot_of[e] >= 0}
        for e in ids.tolist():
            last[e] = s
        evicted = before - after
        if evicted and len(out["waves"]) == 1:
            assert max(last[e] for e in evicted) <= min(last[e] for e in after)


# ----------------------------------------------------------------------------- preflight

def test_preflight_reproduces_the_printed_lines():
    g = _golden("preflight_printed.json")
    assert preflight.kv_bytes_per_token() == g["kv_bytes_per_token"]
    for c in g["cases"]:
        s = preflight.size_deployment(128, 8, 48, c["expert_mb"], c["K"], c["link_gbps"], c["tok_s"], g["kv_bytes_per_token"])
        p = c["printed"]
        assert round(s.slot_mb) == p["slot_mb"], c["name"]
        assert round(s.kv_tokens_per_slot) == p["kv_tokens"], c["name"]
        assert s.batch_cap == p["batch_cap"]
        assert round(100 * s.random_miss) == p["random_miss_pct"]
        assert round(100 * s.max_miss) == p["max_miss_pct"]
        assert s.reuse_implied == p["reuse_implied"]


# ----------------------------------------------------------------------------- planted mistakes

def _swiglu_pin_holds():
    rng = np.random.default_rng(6)
    H, I = 32, 24
    W = _dense_weights(rng, H, I)
    x = rng.standard_normal((5, H))
    y, _ = moe.moe_layer(x, np.zeros((5, 1), np.int32), np.ones((5, 1)), lambda e: W)
    return np.allclose(y, _torch_swiglu(x, *W), rtol=1e-9, atol=1e-12)


def test_planted_activation_mistake_is_caught(monkeypatch):
    assert _swiglu_pin_holds()
    monkeypatch.setattr(moe, "silu", lambda g: 1.0 / (1.0 + np.exp(-g)))  # sigmoid instead of silu
    assert not _swiglu_pin_holds()


def test_planted_gate_up_swap_is_caught(monkeypatch):
    orig = moe.expert_mlp
    monkeypatch.setattr(moe, "expert_mlp", lambda x, Wg, Wu, Wd: orig(x, Wu, Wg, Wd))
    assert not _swiglu_pin_holds()


def test_planted_router_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(2)
    l = rng.standard_normal((4, 16)).astype(np.float32)
    # ascending instead of descending selection
    monkeypatch.setattr(router, "select_topk", lambda row, k: sorted(range(len(row)), key=lambda e: (float(row[e]), e))[:k])
    ids, w = router.router_topk(l, 3)
    best = [sorted(max(itertools.combinations(range(16), 3), key=lambda S: sum(float(l[t, e]) for e in S))) for t in range(4)]
    assert [sorted(r) for r in ids.tolist()] != best


def test_planted_lru_tie_break_mistake_is_caught(monkeypatch):
    g = _golden("lru_hand_trace.json")
    monkeypatch.setattr(lru, "victim_key", lambda last_use, slot: (last_use, -slot))
    sim = lru.LayerLRU(g["E"], g["K"])
    mismatch = False
    for st in g["steps"]:
        out = sim.step(st["ids"])
        mismatch |= [list(m) for m in out["misses"]] != st["misses"]
    assert mismatch


def test_planted_scale_transpose_is_caught(monkeypatch):
    H, I = 256, 384
    sgu = np.arange(1, 13, dtype=np.float32).reshape(6, 2)
    sd = 100 + np.arange(6, dtype=np.float32).reshape(2, 3)
    buf = _fp8_expert_from_parts(np.full((2 * I, H), 0x38, np.uint8), np.full((H, I), 0x38, np.uint8), sgu, sd)
    real_repeat = np.repeat

    def transposed_repeat(a, reps, axis=None):
        if isinstance(a, np.ndarray) and a.shape == (6, 2) and axis == 0:
            a = a[::-1]
        return real_repeat(a, reps, axis=axis)

    monkeypatch.setattr(formats.np, "repeat", transposed_repeat)
    Wg, Wu, _ = formats.decode_expert(buf, 1, H, I)
    assert not np.array_equal(np.concatenate([Wg, Wu]), np.kron(sgu, np.ones((128, 128))))


# ---------------------------------------------------------------- router projection

def test_router_logits_of_a_one_hot_state_are_a_column():
    # x = e_j picks column j of the (E x H) router weight: logits[e] = W[e, j]
    from oracle import router as orouter
    rng = np.random.default_rng(5)
    E, H = 12, 20
    W = rng.standard_normal((E, H))
    for j in (0, 7, H - 1):
        x = np.zeros((1, H))
        x[0, j] = 1.0
        assert np.array_equal(orouter.router_logits(x, W)[0], W[:, j])
        ids, _, _ = orouter.router_gemm_topk(x, W, 3)
        assert ids[0].tolist() == sorted(range(E), key=lambda e: (-W[e, j], e))[:3]


def test_router_weights_ignore_a_feature_shared_by_all_experts():
    # a constant input feature whose weight is the same for every expert shifts all
    # logits of a token by the same amount: selection and (renormalised) weights stay
    from oracle import router as orouter
    rng = np.random.default_rng(6)
    T, E, H, k = 5, 16, 24, 4
    x = rng.standard_normal((T, H))
    W = rng.standard_normal((E, H))
    ids0, w0, _ = orouter.router_gemm_topk(x, W, k)
    x1 = np.concatenate([x, np.ones((T, 1))], axis=1)
    W1 = np.concatenate([W, np.full((E, 1), 0.75)], axis=1)
    ids1, w1, lg1 = orouter.router_gemm_topk(x1, W1, k)
    assert np.array_equal(ids0, ids1)
    np.testing.assert_allclose(w0, w1, rtol=1e-6)
    np.testing.assert_allclose(lg1 - orouter.router_logits(x, W), 0.75, atol=1e-12)


def test_router_logits_are_linear_in_the_state():
    from oracle import router as orouter
    rng = np.random.default_rng(7)
    W = rng.standard_normal((9, 11))
    a, b = rng.standard_normal((3, 11)), rng.standard_normal((3, 11))
    np.testing.assert_allclose(orouter.router_logits(a + 2 * b, W),
                               orouter.router_logits(a, W) + 2 * orouter.router_logits(b, W), atol=1e-12)
