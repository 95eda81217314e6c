"""Seeded generators: activations, router logits with a guaranteed top-k gap, routing
traces (uniform and previous-step reuse), and expert weights encoded in the
library's byte layouts (bf16, block-FP8 e4m3, GPTQ-style int4 group 128, MXFP4).

Every expert is drawn from its own counter-style seed (seed, layer, expert,
format), so any expert can be regenerated alone, on any machine.

Encoding weights (rounding to bf16, quantising to e4m3 or int4) is input
preparation: the layer consumes already-quantised experts.
"""

import numpy as np

__all__ = [
    "bf16_bits", "bf16_bits_to_float", "activations_bf16", "uniform_routing_sets",
    "reuse_routing_trace", "logits_for_sets", "expert_bytes", "expert_nbytes",
    "layer_store", "fast_int4_expert_bytes",
]

GAP = 1e-3


def bf16_bits(a):
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_float(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations_bf16(rng, T, H):
    """x ~ N(0, 1), rounded to bf16; returns uint16 bit patterns [T, H]."""
    return bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def uniform_routing_sets(rng, T, E, top_k):
    """Each token picks top_k distinct experts uniformly at random."""
    return [list(rng.choice(E, size=top_k, replace=False)) for _ in range(T)]


def reuse_routing_trace(rng, E, top_k, B, steps, p=0.8):
    """Per decode stream: step 0 picks top_k distinct experts uniformly; at each later
    step every expert of the stream's previous set is kept with probability p, and
    each dropped one is replaced by a uniform draw from the experts outside the
    previous set. Returns sets[step][stream] -> list of top_k expert ids.
    """
    trace = []
    cur = [list(rng.choice(E, size=top_k, replace=False)) for _ in range(B)]
    trace.append([list(c) for c in cur])
    for _ in range(1, steps):
        nxt = []
        for prev in cur:
            keep = [e for e in prev if rng.random() < p]
            outside = np.setdiff1d(np.arange(E), np.array(prev))
            new = list(rng.choice(outside, size=top_k - len(keep), replace=False))
            nxt.append(keep + new)
        cur = nxt
        trace.append([list(c) for c in cur])
    return trace


def logits_for_sets(rng, sets, E, gap=GAP):
    """Router logits [T, E] float32 whose top_k set for token t is sets[t].

    Draw N(0,1)^E, sort descending, give the top_k values to the chosen experts in
    random order and the rest to the other experts in random order; redraw while
    the k-th and (k+1)-th largest values are within `gap` of each other.
    """
    T = len(sets)
    out = np.empty((T, E), dtype=np.float32)
    for t, chosen in enumerate(sets):
        k = len(chosen)
        chosen = np.asarray(chosen)
        others = np.setdiff1d(np.arange(E), chosen)
        while True:
            v = np.sort(rng.standard_normal(E).astype(np.float32))[::-1]
            if k == E or float(v[k - 1]) - float(v[k]) > gap:
                break
        row = np.empty(E, dtype=np.float32)
        row[rng.permutation(chosen)] = v[:k]
        if k < E:
            row[rng.permutation(others)] = v[k:]
        out[t] = row
    return out


def expert_nbytes(fmt, H, I):
    n_w = 3 * H * I
    if fmt == 0:
        return 2 * n_w
    if fmt == 1:
        return n_w + 4 * ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128))
    if fmt == 2:
        return n_w // 2 + 4 * ((2 * I) * (H // 128) + H * (I // 128))
    if fmt == 3:
        return n_w // 2 + (2 * I) * (H // 32) + H * (I // 32)
    if fmt == 4:
        return n_w // 2 + 16 + (2 * I) * (H // 16) + 16 + H * (I // 16)
    raise ValueError("unknown format")


def _e4m3_codes(v):
    """float32 -> e4m3 codes (uint8), round to nearest even, via torch's float8 cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _fp8_block_quant(w):
    """[R, C] float32 -> (codes [R, C] uint8, scales [R/128, C/128] float32), s = amax/448."""
    R, C = w.shape
    blk = w.reshape(R // 128, 128, C // 128, 128)
    amax = np.abs(blk).max(axis=(1, 3)).astype(np.float32)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = blk / s[:, None, :, None]
    q = np.clip(q, -448.0, 448.0).astype(np.float32)
    return _e4m3_codes(q.reshape(R, C)), s


def _int4_group_quant(w):
    """[R, C] float32 -> (packed [R, C/2] uint8, sz [R, C/128, 2] float16).

    Asymmetric GPTQ-style grid per (row, group of 128 columns): s = (max-min)/15,
    z = round(-min/s) clamped to [0, 15], q = clamp(rint(w/s) + z, 0, 15), with s
    and z stored as fp16 and q computed from the stored s.
    """
    R, C = w.shape
    g = w.reshape(R, C // 128, 128)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    s = ((mx - mn) / 15.0).astype(np.float16)
    s = np.where(s == 0, np.float16(1.0), s)
    sf = s.astype(np.float32)
    z = np.clip(np.rint(-mn / sf), 0, 15).astype(np.float16)
    q = np.clip(np.rint(g / sf[:, :, None]) + z.astype(np.float32)[:, :, None], 0, 15).astype(np.uint8)
    q = q.reshape(R, C)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    sz = np.stack([s, z], axis=2)
    return packed, sz


_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
_E2M1_MIDS = (_E2M1_MAGS[1:] + _E2M1_MAGS[:-1]) / 2


def _mxfp4_block_quant(w):
    """[R, C] float32 -> (packed E2M1 codes [R, C/2] uint8, E8M0 scales [R, C/32] uint8).

    The OCP microscaling recipe per (row, block of 32 columns): shared exponent
    floor(log2(amax)) - 2 (2 = the largest E2M1 exponent), scale 2^that; each element
    divided by the scale and rounded to the nearest E2M1 value, ties to the even
    mantissa, saturating at 6. An all-zero block gets scale 1 and zero codes.
    """
    R, C = w.shape
    g = w.reshape(R, C // 32, 32).astype(np.float32)
    amax = np.abs(g).max(axis=2)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, 0).astype(np.int32)
    e = np.clip(e, -127, 127)
    scale = np.ldexp(np.float32(1.0), e).astype(np.float32)
    a = np.abs(g) / scale[:, :, None]
    lo = np.searchsorted(_E2M1_MIDS, a, side="left")
    hi = np.searchsorted(_E2M1_MIDS, a, side="right")
    idx = np.where(lo == hi, lo, np.where(lo % 2 == 0, lo, hi))  # on a midpoint: the even code
    codes = (idx | np.where(g < 0, 8, 0)).astype(np.uint8).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def _nvfp4_quant(w):
    """[R, C] float32 -> (packed E2M1 codes [R, C/2] uint8, e4m3 block scales [R, C/16]
    uint8, fp32 tensor scale T).

    Two-level recipe: T = amax(w) / (6 * 448), so that the largest block scale is
    e4m3's largest value; per (row, block of 16 columns) the scale code is
    e4m3(amax_block / 6 / T) (round to nearest even, saturating at 448); each element
    divided by e4m3(code) * T and rounded to the nearest E2M1 value, ties to the even
    mantissa, saturating at 6. A block whose scale rounds to zero gets zero codes.
    """
    R, C = w.shape
    amax = float(np.abs(w).max())
    T = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    g = w.reshape(R, C // 16, 16).astype(np.float32)
    bamax = np.abs(g).max(axis=2)
    s_codes = _e4m3_codes(np.minimum(bamax / np.float32(6.0) / T, np.float32(448.0)))
    import torch
    s_vals = torch.from_numpy(s_codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    eff = (s_vals * T).astype(np.float32)
    a = np.where(eff[:, :, None] > 0, np.abs(g) / np.where(eff > 0, eff, 1.0)[:, :, None], 0.0)
    lo = np.searchsorted(_E2M1_MIDS, a, side="left")
    hi = np.searchsorted(_E2M1_MIDS, a, side="right")
    idx = np.where(lo == hi, lo, np.where(lo % 2 == 0, lo, hi))  # on a midpoint: the even code
    codes = (idx | np.where(g < 0, 8, 0)).astype(np.uint8).reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_codes.reshape(R, C // 16), T


def _tensor_scale_bytes(T):
    return np.concatenate([np.array([T], np.float32).view(np.uint8), np.zeros(12, np.uint8)])


def expert_bytes(fmt, H, I, seed, layer=0, expert=0, std=0.02):
    """One expert in the byte layout of `fmt`, drawn from N(0, std) master weights.

    bf16: W_gu [2I][H] (gate rows then up rows), W_d [H][I]; block-FP8 and int4 as
    in the layout contract. Returns a uint8 array.
    """
    rng = np.random.default_rng([seed, layer, expert, fmt])
    wgu = (rng.standard_normal((2 * I, H), dtype=np.float32) * np.float32(std))
    wd = (rng.standard_normal((H, I), dtype=np.float32) * np.float32(std))
    if fmt == 0:
        parts = [bf16_bits(wgu).view(np.uint8).ravel(), bf16_bits(wd).view(np.uint8).ravel()]
    elif fmt == 1:
        qgu, sgu = _fp8_block_quant(wgu)
        qd, sd = _fp8_block_quant(wd)
        parts = [qgu.ravel(), qd.ravel(), sgu.view(np.uint8).ravel(), sd.view(np.uint8).ravel()]
    elif fmt == 2:
        qgu, szgu = _int4_group_quant(wgu)
        qd, szd = _int4_group_quant(wd)
        parts = [qgu.ravel(), qd.ravel(), szgu.view(np.uint8).ravel(), szd.view(np.uint8).ravel()]
    elif fmt == 3:
        qgu, xgu = _mxfp4_block_quant(wgu)
        qd, xd = _mxfp4_block_quant(wd)
        parts = [qgu.ravel(), qd.ravel(), xgu.ravel(), xd.ravel()]
    elif fmt == 4:
        qgu, bgu, tgu = _nvfp4_quant(wgu)
        qd, bd, td = _nvfp4_quant(wd)
        parts = [qgu.ravel(), qd.ravel(), _tensor_scale_bytes(tgu), bgu.ravel(), _tensor_scale_bytes(td), bd.ravel()]
    else:
        raise ValueError("unknown format")
    out = np.concatenate(parts)
    assert out.size == expert_nbytes(fmt, H, I)
    return out


def fast_int4_expert_bytes(H, I, seed, layer=0, expert=0):
    """A GPTQ-int4 expert drawn directly in code space (for very large stores).

    Nibbles uniform in 0..15, per-(row, group) scale uniform in [0.006, 0.008]
    (fp16) and zero point uniform in {6, 7, 8, 9} (fp16): the resulting weights have
    a spread close to that of N(0, 0.02) master weights quantised with a 16-level
    grid per group of 128, and the bytes cost one random draw each.
    """
    rng = np.random.default_rng([seed, layer, expert, 2, 1])
    nq = 3 * H * I // 2
    q = np.frombuffer(rng.bytes(nq), dtype=np.uint8)
    ng = 2 * I * (H // 128) + H * (I // 128)
    s = rng.uniform(0.006, 0.008, ng).astype(np.float16)
    z = rng.integers(6, 10, ng).astype(np.float16)
    sz = np.stack([s, z], axis=1)
    out = np.concatenate([q, sz.view(np.uint8).ravel()])
    assert out.size == expert_nbytes(2, H, I)
    return out


def layer_store(fmt, H, I, E, seed, layer=0, fast=False, threads=None, out=None):
    """All E experts of one layer, [E, expert_nbytes] uint8 (experts drawn in parallel
    threads; each expert's bytes depend only on its own seed). `out` may be a
    preallocated [E, >= expert_nbytes] uint8 view (for instance a pinned store)."""
    import concurrent.futures
    import os
    nb = expert_nbytes(fmt, H, I)
    if out is None:
        out = np.empty((E, nb), dtype=np.uint8)
    else:
        out = out[:, :nb]

    def fill(e):
        if fast and fmt == 2:
            out[e] = fast_int4_expert_bytes(H, I, seed, layer, e)
        else:
            out[e] = expert_bytes(fmt, H, I, seed, layer, e)

    n = threads or min(16, len(os.sched_getaffinity(0)))
    if E * nb < (8 << 20) or n <= 1:
        for e in range(E):
            fill(e)
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(fill, range(E)))
    return out
