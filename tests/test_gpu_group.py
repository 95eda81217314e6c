"""The grouping (counts, offs, the stable permutation and its inverse) through the C ABI,
bit for bit against oracle/permute.py.

Article "Running an MoE Model Larger Than Your VRAM", section "What does Paged Experts
actually do?": the routed (token, rank) pairs run expert by expert.
"""

import numpy as np
import pytest

from oracle import permute
from workloads import generators as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_expert_moe_gb300 as pm
    pm.load()
    return pm


def _run(pm, ids, E):
    import torch
    d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts, offs, perm, pos = pm.moe_group_by_expert(d, E, err_out=err)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offs.cpu().numpy(), perm.cpu().numpy(), pos.cpu().numpy(), int(err.item())


def _expect(ids, E):
    """The oracle over the valid pairs, their indices mapped back to the whole array."""
    flat = np.asarray(ids, np.int64).reshape(-1)
    valid = np.flatnonzero((flat >= 0) & (flat < E))
    counts, offs, perm_v, _ = permute.group_by_expert(flat[valid], E)
    perm = valid[perm_v].astype(np.int32)
    pos = np.full(flat.size, -1, np.int32)
    pos[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offs, perm, pos


@pytest.mark.parametrize("T,k,E,skew", [(1, 1, 1, False), (1, 8, 128, False), (33, 4, 16, True), (100, 3, 5, True),
                                        (129, 8, 128, False), (512, 8, 128, False), (1024, 8, 128, True),
                                        (640, 8, 1024, False), (1025, 8, 128, False), (2048, 8, 128, False),
                                        (2048, 8, 128, True), (1152, 8, 1024, False), (4097, 8, 128, False),
                                        (16384, 8, 128, True), (20000, 8, 128, False)])
def test_grouping_equals_oracle(pm, T, k, E, skew):
    """Uniform and skewed routing, through the kernels the forward uses: one CTA with every
    pair in shared memory up to 1024 pairs (decode), the one-CTA counting sort up to 8192,
    and four launches over per-chunk histograms beyond (2048 x 8 is the prefill workload;
    16384 x 8 = 512 chunks gives each lane of the chunk scan one full batch of 16 chunks,
    20000 x 8 = 625 chunks two batches with a ragged tail). Ragged warp ranges, chunks and
    tails."""
    rng = np.random.default_rng(7000 + T * 7 + E)
    if skew:
        p = np.arange(E, 0, -1, dtype=np.float64) ** 2
        p /= p.sum()
        ids = np.stack([rng.choice(E, size=min(k, E), replace=False, p=p) for _ in range(T)])
    else:
        ids = np.asarray(gen.uniform_routing_sets(rng, T, E, k), np.int32)
    got = _run(pm, ids, E)
    want = _expect(ids, E)
    for name, g, w in zip(("counts", "offs", "perm", "pos"), got[:4], want):
        np.testing.assert_array_equal(g, w, err_msg=name)
    assert got[4] == 0


@pytest.mark.parametrize("T", [100, 300, 2000])
def test_grouping_leaves_bad_ids_out_and_flags_them(pm, T):
    """Ids outside [0, E) get pos = -1, are not counted, and set the error word; the valid
    pairs keep their stable order (600, 1800 and 12000 pairs: each of the three kernels)."""
    rng = np.random.default_rng(7100 + T)
    E = 64
    ids = rng.integers(0, E, size=(T, 6)).astype(np.int32)
    bad = rng.choice(ids.size, size=17, replace=False)
    ids.reshape(-1)[bad[:9]] = -1
    ids.reshape(-1)[bad[9:]] = E + 3
    counts, offs, perm, pos, err = _run(pm, ids, E)
    c2, o2, p2, q2 = _expect(ids, E)
    np.testing.assert_array_equal(counts, c2)
    np.testing.assert_array_equal(offs, o2)
    np.testing.assert_array_equal(perm[:offs[E]], p2)
    np.testing.assert_array_equal(pos, q2)
    assert err == 1


def test_grouping_argument_errors(pm):
    import torch
    ids = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(pm.PmoeError):
        pm.moe_group_by_expert(ids, 0)
    with pytest.raises(pm.PmoeError):
        pm.moe_group_by_expert(ids, 1025)
    assert pm.load().moe_group_scratch_ints(8192, 128) == 0
    assert pm.load().moe_group_scratch_ints(8193, 128) == 33 * 128
    counts, offs, perm, pos = pm.moe_group_by_expert(torch.zeros(0, dtype=torch.int32, device="cuda"), 4)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == [0, 0, 0, 0] and offs.cpu().tolist() == [0, 0, 0, 0, 0]
