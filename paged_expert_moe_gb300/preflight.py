"""Deployment sizing and start-up checks for the paged-expert MoE layer.

Sizing follows the arithmetic of the article "Running an MoE Model Larger Than Your
VRAM": sections "What does a resident slot cost in context length?", "Why is it fast
when experts keep crossing PCIe?" and "A preflight script before you turn it on".

- A slot exists in every MoE layer, so one more slot costs the expert size times the
  number of layers. In KV-cache terms, that is those bytes divided by the KV bytes one
  token takes.
- A step whose distinct experts fit in K slots runs in one wave. That holds for batches
  up to K // top_k.
- A token whose every expert misses moves layers x top_k experts across the host link.
  A measured speed therefore bounds the miss rate: link bandwidth / (tokens per second
  x that traffic).
- Uniform random routing misses 1 - K/E of the time. When the speed bound sits clearly
  below that (under 0.8 of it), the speed implies reuse; otherwise the numbers are
  inconclusive.

The independence check follows the section "Can paging change the model's outputs?":
- a paged layer must return exactly what the unpaged layer returns;
- every slot must hold exactly the bytes of the expert the table names.

Everything here runs on the host, or through the library's own calls. The CLI prints
the sizing of one configuration:

    python -m paged_expert_moe_gb300.preflight --format int4 --layers 48 --slots 26 \\
        --link-gbps 15.75 --tok-s 32.6
"""

import argparse
from dataclasses import dataclass, asdict

FORMATS = {"bf16": 0, "fp8": 1, "int4": 2, "mxfp4": 3, "nvfp4": 4}


def qwen3_kv_bytes_per_token(layers=48, kv_heads=4, head_dim=128, elem_bytes=2):
    """bf16 K and V of one token over all attention layers (Qwen3-30B-A3B: 48 layers,
    4 KV heads of 128 dims)."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


@dataclass
class Sizing:
    experts: int
    top_k: int
    layers: int
    slots: int
    expert_bytes: int            # the library's byte layout of one expert (all its tensors)
    slot_stride: int             # the slot pitch in the arena (expert bytes rounded up to 4 KiB)
    arena_bytes: int             # device slot arenas of all layers
    host_store_bytes: int        # pinned host store of all layers
    slot_cost_mb: float          # one more slot, over all layers
    kv_tokens_per_slot: float    # KV-cache tokens that one slot's memory would hold
    batch_cap: int               # largest batch whose step always fits in one wave
    all_miss_gb_per_token: float
    random_miss: float           # miss rate of uniform random routing
    max_miss: float = None       # highest miss rate the measured speed allows
    reuse_implied: bool = None
    slots_fit: int = None        # the largest K whose arenas fit the given HBM budget


def size(experts, top_k, layers, slots, fmt="bf16", hidden=None, intermediate=None, expert_mb=None,
         link_gbps=None, tok_s=None, kv_bytes_per_token=None, hbm_budget_gb=None):
    """Sizing of one configuration.

    The expert size comes from the library's layout for (fmt, hidden, intermediate), or
    from expert_mb (MB = 1e6 bytes) when the layout is someone else's, as in the article's
    own script. link_gbps and tok_s (a measured speed) give the miss-rate verdict, and
    hbm_budget_gb gives the largest K that fits.
    """
    if expert_mb is None:
        from ._lib import pmoe_expert_bytes
        f = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
        eb = pmoe_expert_bytes(f, hidden, intermediate)
        if eb == 0:
            raise ValueError("unsupported expert shape for this format")
    else:
        eb = int(round(expert_mb * 1e6))
    stride = (eb + 4095) // 4096 * 4096
    kv = kv_bytes_per_token if kv_bytes_per_token is not None else qwen3_kv_bytes_per_token(layers)
    slot_cost = eb * layers / 1e6
    all_miss = eb * layers * top_k / 1e9
    s = Sizing(experts=experts, top_k=top_k, layers=layers, slots=slots, expert_bytes=eb, slot_stride=stride,
               arena_bytes=slots * stride * layers, host_store_bytes=experts * stride * layers,
               slot_cost_mb=slot_cost, kv_tokens_per_slot=eb * layers / kv, batch_cap=slots // top_k,
               all_miss_gb_per_token=all_miss, random_miss=1.0 - slots / experts)
    if link_gbps is not None and tok_s is not None:
        s.max_miss = link_gbps / (tok_s * all_miss)
        s.reuse_implied = s.max_miss < 0.8 * s.random_miss
    if hbm_budget_gb is not None:
        s.slots_fit = min(experts, int(hbm_budget_gb * 1e9 // (stride * layers)))
    return s


def report(s):
    """The three result lines of the article's preflight script, for one sizing."""
    lines = [f"slot cost: {s.slot_cost_mb:.0f} MB per slot across {s.layers} layers "
             f"= {s.kv_tokens_per_slot:.0f} KV tokens",
             f"single-wave batch cap: K // top_k = {s.slots} // {s.top_k} = {s.batch_cap}"]
    if s.max_miss is not None:
        verdict = "reuse implied" if s.reuse_implied else "inconclusive"
        lines.append(f"miss rate: random routing {100 * s.random_miss:.0f}%, allowed by the measured speed "
                     f"{100 * s.max_miss:.0f}% -> {verdict}")
    else:
        lines.append(f"miss rate: random routing {100 * s.random_miss:.0f}% (give a measured speed for a verdict)")
    return lines


def measure_link_gbps(device=0, nbytes=9_437_184, reps=40):
    """Pinned host -> device copy bandwidth of this machine's link, GB/s."""
    import torch
    dev = torch.device("cuda", device)
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize(dev)
    return nbytes * reps / (a.elapsed_time(b) / 1e3) / 1e9


def independence_check(experts, top_k, hidden, intermediate, slots, expert_store, fmt="bf16", tokens=4,
                       steps=6, seed=0, device=0, pagein_mode=0):
    """Runs the same random steps through a layer with `slots` slots and through one with
    every expert resident. The outputs must be bitwise equal, and afterwards every slot of
    the paged layer must hold exactly the bytes of the expert its table names.

    expert_store: sequence of E byte strings (uint8 numpy arrays) in the library's layout.
    Returns a dict: outputs_equal, steps, misses, slots_checked, slot_mismatches.
    """
    import numpy as np
    import torch
    from ._lib import ExpertCache
    f = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    dev = torch.device("cuda", device)
    gen = torch.Generator(device="cpu").manual_seed(seed)
    paged = ExpertCache(experts, top_k, hidden, intermediate, slots, fmt=f, max_tokens=tokens, device=device,
                        pagein_mode=pagein_mode)
    full = ExpertCache(experts, top_k, hidden, intermediate, experts, fmt=f, max_tokens=tokens, device=device,
                       pagein_mode=pagein_mode)
    try:
        paged.load_layer(0, expert_store)
        full.load_layer(0, expert_store)
        equal = True
        for _ in range(steps):
            ids = torch.stack([torch.randperm(experts, generator=gen)[:top_k] for _ in range(tokens)]).to(torch.int32)
            w = torch.softmax(torch.randn(tokens, top_k, generator=gen), dim=-1).to(torch.float32)
            x = torch.randn(tokens, hidden, generator=gen).to(torch.bfloat16)
            ids, w, x = ids.to(dev), w.to(dev), x.to(dev)
            ya = paged.moe_paged_forward(0, x, ids, w)
            yb = full.moe_paged_forward(0, x, ids, w)
            torch.cuda.synchronize(dev)
            equal = equal and bool(torch.equal(ya.view(torch.int16), yb.view(torch.int16)))
        exp_in, _ = paged.expert_cache_slot_table(0)
        mismatches = []
        checked = 0
        for s, e in enumerate(exp_in.tolist()):
            if e < 0:
                continue
            checked += 1
            if not np.array_equal(paged.expert_cache_read_slot(0, s), np.asarray(expert_store[e], dtype=np.uint8)):
                mismatches.append((s, e))
        st = paged.expert_cache_stats(0)
        return {"outputs_equal": equal, "steps": steps, "misses": st["misses"], "slots_checked": checked,
                "slot_mismatches": mismatches}
    finally:
        paged.close()
        full.close()


def main(argv=None):
    ap = argparse.ArgumentParser(description="sizing of a paged-expert MoE deployment")
    ap.add_argument("--experts", type=int, default=128)
    ap.add_argument("--top-k", type=int, default=8)
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--slots", type=int, required=True)
    ap.add_argument("--format", default="bf16", choices=sorted(FORMATS))
    ap.add_argument("--hidden", type=int, default=2048)
    ap.add_argument("--intermediate", type=int, default=768)
    ap.add_argument("--expert-mb", type=float, default=None, help="use this expert size instead of the layout's")
    ap.add_argument("--link-gbps", type=float, default=None)
    ap.add_argument("--tok-s", type=float, default=None, help="a measured decode speed")
    ap.add_argument("--hbm-gb", type=float, default=None, help="device memory available for the slot arenas")
    ap.add_argument("--measure-link", action="store_true", help="measure the pinned H2D bandwidth here")
    a = ap.parse_args(argv)
    link = measure_link_gbps() if a.measure_link else a.link_gbps
    s = size(a.experts, a.top_k, a.layers, a.slots, a.format, a.hidden, a.intermediate, a.expert_mb, link, a.tok_s,
             hbm_budget_gb=a.hbm_gb)
    for line in report(s):
        print(line)
    print({k: v for k, v in asdict(s).items() if v is not None})


if __name__ == "__main__":
    main()
