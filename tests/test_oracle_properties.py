"""Property-based pins of the two bit-exact parts of the oracle, on many small random cases.

- LRU simulator: on every step, the waves partition the step's distinct experts, each
  wave fits the K slots, the misses are exactly the step's experts that were not
  resident (the step loads each expert once), the table stays a consistent
  expert <-> slot map, no expert pending in the step is evicted, and a single-wave
  step evicts only experts no more recently used than any expert it keeps.
- Router: the selected set equals a brute-force search over all k-subsets (the
  largest logit sum), ordered by descending logit with ties to the lower id, and the
  weights equal the closed form softmax over the selected logits.

The hypothesis package is installed on the development box; elsewhere these tests skip.
"""

import itertools

import numpy as np
import pytest

from oracle import lru, router

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


@st.composite
def traces(draw):
    E = draw(st.integers(1, 12))
    K = draw(st.integers(1, E))
    steps = draw(st.lists(st.lists(st.integers(0, E - 1), min_size=0, max_size=10), min_size=1, max_size=25))
    return E, K, steps


@settings(max_examples=300, deadline=None)
@given(traces())
def test_lru_step_invariants(case):
    E, K, steps = case
    sim = lru.LayerLRU(E, K)
    last_seen = {}
    for s, ids in enumerate(steps):
        before = {e for e in range(E) if sim.slot_of[e] >= 0}
        out = sim.step(ids)
        U = sorted(set(ids))
        # the waves partition U, each within K slots
        flat = [e for wave in out["waves"] for e, _ in wave]
        assert sorted(flat) == U and len(flat) == len(set(flat))
        assert all(len(w) <= K for w in out["waves"])
        # every expert of a wave sat in the slot the wave names while it ran
        for wave in out["waves"]:
            assert len({v for _, v in wave}) == len(wave)
        # misses = the step's experts that were not resident; each loaded once
        assert sorted(e for e, _, _ in out["misses"]) == sorted(set(U) - before)
        # consistent table: slot_of and expert_in are inverse maps
        for v, e in enumerate(sim.expert_in):
            if e >= 0:
                assert sim.slot_of[e] == v
        for e, v in enumerate(sim.slot_of):
            if v >= 0:
                assert sim.expert_in[v] == e
        assert sum(1 for v in sim.slot_of if v >= 0) == sum(1 for e in sim.expert_in if e >= 0)
        # a single-wave step keeps every one of its experts resident, and evicts only
        # experts last used no later than any expert it keeps
        after = {e for e in range(E) if sim.slot_of[e] >= 0}
        if len(out["waves"]) == 1:
            assert set(U) <= after
            evicted = before - after
            kept_old = (before & after) - set(U)
            if evicted and kept_old:
                assert max(last_seen[e] for e in evicted) <= min(last_seen[e] for e in kept_old)
        for e in U:
            last_seen[e] = s
    assert sim.hits + sim.misses == sum(len(set(ids)) for ids in steps)


@st.composite
def logit_rows(draw):
    E = draw(st.integers(1, 9))
    k = draw(st.integers(1, E))
    # few distinct values, so that ties are common
    vals = draw(st.lists(st.sampled_from([-1.5, -0.25, 0.0, 0.5, 0.5, 2.0, 3.25]), min_size=E, max_size=E))
    return np.array(vals, dtype=np.float32), k


@settings(max_examples=400, deadline=None)
@given(logit_rows())
def test_router_selection_is_the_brute_force_optimum(case):
    row, k = case
    E = len(row)
    sel = router.select_topk(row, k)
    best = max(sum(float(row[e]) for e in c) for c in itertools.combinations(range(E), k))
    assert abs(sum(float(row[e]) for e in sel) - best) == 0.0
    # descending logits, ties to the lower id, and no lower-id expert left out at the boundary
    assert all((row[a] > row[b]) or (row[a] == row[b] and a < b) for a, b in zip(sel, sel[1:]))
    cut = float(row[sel[-1]])
    for e in range(E):
        if e not in sel:
            assert row[e] < cut or (row[e] == cut and e > sel[-1])
    ids, w = router.router_topk(row[None, :], k)
    z = np.exp(row[sel].astype(np.float64) - row[sel].max())
    np.testing.assert_allclose(w[0], z / z.sum(), rtol=1e-12)
    assert ids[0].tolist() == sel
