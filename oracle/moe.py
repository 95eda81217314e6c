"""Unpaged MoE layer oracle: SwiGLU experts and the top_k-weighted combine.

Sources:
  "Running an MoE Model Larger Than Your VRAM", section "What does Paged Experts
  actually do?": each token goes to top_k of E experts and the model's fused-MoE
  kernel runs over the resident experts.
  Same article, section "Can paging change the model's outputs?": the paged
  layer returns the same result as the unpaged one. The oracle is therefore the
  unpaged layer; residency is simulated separately (``oracle.lru``).

Expert (Qwen3 MoE MLP): g = x W_g^T, u = x W_u^T, a = silu(g) * u with
silu(g) = g * sigmoid(g), o = a W_d^T. Combine: y[t] = sum_{r=0}^{k-1} w[t,r] *
o_{ids[t,r]}(x_t), summed in rank order r = 0..k-1. All in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

import numpy as np

from .formats import decode_expert


def silu(g):
    return g / (1.0 + np.exp(-g))


def expert_mlp(x, Wg, Wu, Wd):
    """SwiGLU expert applied to the rows of x (n, H) -> (n, H), float64."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ Wg.T
    u = x @ Wu.T
    return (silu(g) * u) @ Wd.T


def expert_hidden(x, Wg, Wu):
    """The intermediate activation a = silu(x W_g^T) * (x W_u^T), (n, I)."""
    x = np.asarray(x, dtype=np.float64)
    return silu(x @ Wg.T) * (x @ Wu.T)


class ExpertSource:
    """Maps an expert id to its float64 matrices, decoding bytes on demand."""

    def __init__(self, get_bytes, fmt, H, I, cache=64):
        self._get = get_bytes
        self.fmt, self.H, self.I = fmt, H, I
        self._limit = cache
        self._cache = {}

    def __call__(self, e):
        e = int(e)
        if e in self._cache:
            m = self._cache.pop(e)
            self._cache[e] = m  # most recent last
            return m
        m = decode_expert(self._get(e), self.fmt, self.H, self.I)
        if self._limit:
            if len(self._cache) >= self._limit:
                self._cache.pop(next(iter(self._cache)))
            self._cache[e] = m
        return m


def moe_layer(x, ids, w, experts):
    """y[t] = sum_r w[t,r] * expert_{ids[t,r]}(x[t]) for every row t.

    x: (T, H) array (bf16 values given as float), ids: (T, k) ints, w: (T, k)
    floats, experts: callable e -> (W_g, W_u, W_d) float64. Tokens are
    independent, so a caller evaluates a sample of tokens by passing those rows.
    Returns y (T, H) float64 and the number of (token, rank) expert activations
    that were evaluated.
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    T, k = ids.shape
    # o[t, r] for every pair; rows that share an expert go through one matmul,
    # and each row of a matmul is the plain per-token definition.
    by_expert = {}
    for t in range(T):
        for r in range(k):
            by_expert.setdefault(int(ids[t, r]), []).append((t, r))
    o = np.zeros((T, k, x.shape[1]), dtype=np.float64)
    n_act = 0
    for e, lst in by_expert.items():
        Wg, Wu, Wd = experts(e)
        rows = np.array([t for t, _ in lst])
        out = expert_mlp(x[rows], Wg, Wu, Wd)
        for j, (t, r) in enumerate(lst):
            o[t, r] = out[j]
            n_act += 1
    y = np.zeros((T, x.shape[1]), dtype=np.float64)
    for t in range(T):
        for r in range(k):  # rank order
            y[t] += w[t, r] * o[t, r]
    return y, n_act


def moe_stack(x, layers, residual=False):
    """A stack of MoE layers with attention omitted.

    layers: list of (ids, w, experts), one per layer, routing given per layer (the
    reading for a stack with attention omitted: synthetic per-layer routing that
    does not depend on the layer's input). Without `residual` each layer feeds the
    next, x_{l+1} = moe_l(x_l); with it the layers add to a residual stream,
    x_{l+1} = x_l + moe_l(x_l), as a decoder block does. Returns the final
    activations and the total number of expert activations; for one token that is
    layers x top_k ("Why is it fast when experts keep crossing PCIe?": 48 x 8 = 384).
    """
    h = np.asarray(x, dtype=np.float64)
    n_total = 0
    for ids, w, experts in layers:
        y, n = moe_layer(h, ids, w, experts)
        h = h + y if residual else y
        n_total += n
    return h, n_total
