"""Brute-force simulator of one layer's K-slot expert table (LRU, per-step dedup, waves).

Sources:
  "Running an MoE Model Larger Than Your VRAM", TL;DR: K of the E experts of a
  layer are kept on the GPU, all E in pinned host RAM, and a step copies in only
  the routed experts that are not resident.
  Same article, "What does Paged Experts actually do?" item 3: missing experts
  are copied into slots, evicting the expert whose last use is oldest.
  Same article, "What happens with more than one request?": a decode step is one
  wave only if tokens x top_k <= K; larger steps run several waves, and every wave
  copies its own missing experts in before it computes.
  "Locality of reference helped ...", section "The fix": a hit computes from
  VRAM with no bytes moved; a miss copies that one expert and evicts the least
  recently used one.

Readings where the pages are silent (all of them matter for bit-exact slots):
  * Time is the layer's own step counter s = 0, 1, 2, ...; every expert used in a
    step gets last_use = s, so ties are common.
  * Victim order: key (last_use, slot index), smallest first; an empty slot has
    last_use = -1, so empty slots go first, in slot order.
  * An expert that is still pending in the current step is never evicted;
    experts already computed in an earlier wave of the same step may be.
  * Wave partition: the pending experts that are resident all join the wave;
    then the non-resident pending experts in ascending id fill the remaining
    K - |resident| places; every expert's tokens run in one wave.
  * The i-th miss (ascending id) goes into the i-th victim (ascending key).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""


def victim_key(last_use, slot):
    """Eviction order of an unprotected slot: least recent first, then lower slot."""
    return (last_use, slot)


class LayerLRU:
    """One layer's table: slot -> expert, slot -> last use, expert -> slot."""

    def __init__(self, E, K):
        if not (1 <= K):
            raise ValueError("K must be >= 1")
        self.E, self.K = E, K
        self.expert_in = [-1] * K
        self.last_use = [-1] * K
        self.slot_of = [-1] * E
        self.step_index = 0
        self.hits = 0
        self.misses = 0
        self.waves = 0
        self.steps = 0

    def step(self, ids):
        """Process one step's routed ids; returns a dict describing the step.

        waves: list of waves, each a list of (expert, slot) ascending by expert
        misses: list of (expert, slot, wave) in load order
        """
        E, K, s = self.E, self.K, self.step_index
        U = sorted({int(e) for e in ids})
        for e in U:
            if not (0 <= e < E):
                raise ValueError("expert id out of range")
        pending = set(U)
        resident_before = {e for e in U if self.slot_of[e] >= 0}
        waves, misses = [], []
        loads_this_step = set()
        while pending:
            R = sorted(e for e in pending if self.slot_of[e] >= 0)
            cap = K - len(R)
            nonres = sorted(e for e in pending if self.slot_of[e] < 0)
            M = nonres[:cap]
            unprotected = [v for v in range(K) if self.expert_in[v] not in pending]
            unprotected.sort(key=lambda v: victim_key(self.last_use[v], v))
            assert len(unprotected) >= len(M)
            victims = unprotected[:len(M)]
            for e, v in zip(M, victims):
                old = self.expert_in[v]
                if old >= 0:
                    self.slot_of[old] = -1
                self.expert_in[v] = e
                self.slot_of[e] = v
                assert e not in loads_this_step, "an expert was loaded twice in one step"
                loads_this_step.add(e)
                misses.append((e, v, len(waves)))
            wave = sorted(R + M)
            for e in wave:
                self.last_use[self.slot_of[e]] = s
            waves.append([(e, self.slot_of[e]) for e in wave])
            pending -= set(wave)
        n_miss = len(misses)
        # invariants of the reading
        assert n_miss == len(set(U) - resident_before)
        assert (len(waves) == 1) == (len(U) <= K) or len(U) == 0
        self.hits += len(U) - n_miss
        self.misses += n_miss
        self.waves += len(waves)
        self.steps += 1
        self.step_index += 1
        return {"unique": U, "waves": waves, "misses": misses,
                "hits": len(U) - n_miss, "n_misses": n_miss,
                "slot_of": list(self.slot_of), "expert_in": list(self.expert_in),
                "last_use": list(self.last_use)}


def single_wave_cap(K, top_k):
    """Largest decode batch served in one wave: tokens x top_k <= K, i.e. K // top_k
    ("What happens with more than one request?")."""
    return K // top_k
