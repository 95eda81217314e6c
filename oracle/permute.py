"""Token -> expert grouping oracle: histogram, exclusive scan, stable permutation.

Source: "Running an MoE Model Larger Than Your VRAM", section "What does Paged
Experts actually do?": after page-in the model's own fused-MoE kernel runs over
the resident experts, i.e. the (token, rank) pairs are grouped by expert before
the grouped projections.

Definition (pair p = t * top_k + r is token t's rank-r expert):
  counts[e]  = number of pairs routed to expert e
  offs[e]    = sum_{e' < e} counts[e']          (exclusive scan, offs[E] = T*top_k)
  perm[j]    = the pair at grouped position j: experts ascending; within one
               expert, pairs in ascending pair index (a stable grouping)
  pos[p]     = j such that perm[j] == p          (the inverse of perm)
Integer results are exact.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

import numpy as np


def group_by_expert(ids, E):
    ids = np.asarray(ids).reshape(-1)
    P = ids.size
    counts = [0] * E
    for p in range(P):
        e = int(ids[p])
        if not (0 <= e < E):
            raise ValueError("expert id out of range")
        counts[e] += 1
    offs = [0] * (E + 1)
    for e in range(E):
        offs[e + 1] = offs[e] + counts[e]
    cursor = list(offs[:E])
    perm = [0] * P
    pos = [0] * P
    for p in range(P):  # ascending pair index keeps equal experts in order
        e = int(ids[p])
        perm[cursor[e]] = p
        pos[p] = cursor[e]
        cursor[e] += 1
    return (np.array(counts, np.int32), np.array(offs, np.int32),
            np.array(perm, np.int32), np.array(pos, np.int32))
