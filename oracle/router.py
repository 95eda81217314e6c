"""Router oracle: softmax over E experts, top-k selection, renormalisation.

Source: "Running an MoE Model Larger Than Your VRAM", section "What does Paged
Experts actually do?" (first paragraph): an MoE layer routes each token to top_k
of E experts (Qwen3-30B-A3B: 8 of 128).

The pages do not spell out the score function. Reading taken (stated here and in
the design notes): softmax over all E logits, keep the top_k largest, renormalise
the kept probabilities to sum to one (Qwen3's ``norm_topk_prob``). No shared
expert. Ties: the lower expert id wins; the k outputs are ordered by descending
logit.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

import numpy as np


def select_topk(logit_row, top_k):
    """Indices of the top_k largest logits of one token, descending, ties -> lower id.

    The selection compares the fp32 logits themselves; softmax is monotone, so the
    selected set does not depend on how exp is rounded.
    """
    E = len(logit_row)
    order = sorted(range(E), key=lambda e: (-float(logit_row[e]), e))
    return order[:top_k]


def softmax_row(logit_row):
    """Numerically shifted softmax of one row, float64."""
    l = np.asarray(logit_row, dtype=np.float64)
    m = l.max()
    p = np.exp(l - m)
    return p / p.sum()


def router_topk(logits, top_k, renormalize=True):
    """Route every token: returns (ids[T, top_k] int32, w[T, top_k] float64).

    For token t: p = softmax(logits[t]) over all E; S = select_topk(logits[t]);
    w[t, r] = p[S_r] / sum_{j in S} p[j] when renormalize, else p[S_r].
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= top_k <= E):
        raise ValueError("top_k must lie in [1, E]")
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    for t in range(T):
        S = select_topk(logits[t], top_k)
        p = softmax_row(logits[t])
        sel = p[S]
        ids[t] = S
        w[t] = sel / sel.sum() if renormalize else sel
    return ids, w


def router_logits(x, router_weight):
    """The router's projection: logits[t, e] = sum_c x[t, c] * router_weight[e, c], float64.

    router_weight holds one row per expert (E x H), the layer's gate projection.
    """
    return np.asarray(x, dtype=np.float64) @ np.asarray(router_weight, dtype=np.float64).T


def router_gemm_topk(x, router_weight, top_k, renormalize=True):
    """Route every token from its hidden state: (ids, w, logits) with router_topk applied
    to router_logits(x, router_weight)."""
    logits = router_logits(x, router_weight)
    ids, w = router_topk(logits, top_k, renormalize)
    return ids, w, logits
