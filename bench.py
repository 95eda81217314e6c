"""Benchmark of the paged-expert MoE layer on one GB300 (or N independent replicas).

Default workload: one Qwen3-30B-A3B-shaped MoE layer (E=128, top_k=8, H=2048,
I=768), bf16 experts, K=40 slots, single-stream decode (B=1) over a 256-step routing
trace in which every expert of a stream's previous step is kept with p=0.8. A step is
one pass of the whole path over one batch: router -> residency step (dedup, LRU,
waves) -> page-in of the misses -> grouping -> gate/up + SiLU*mul -> down ->
weighted combine. B=2 and B=4 are reported alongside under "batches".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K timed steps; L2 is flushed before every
timed step, outside the events: a 256 MB write, then a read sweep of another 256 MB
buffer, so that the step finds none of its data in L2 and does not pay for writing
back the flush's own dirty lines; each step is bracketed by CUDA events
on the stream it runs on; a barrier and torch.cuda.synchronize() bracket the timed
loop; the max over ranks is reported. The reference arm times the oracle (plain
CPU float64) on the host cores on the same workload.
"""

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import generators as gen  # noqa: E402

METRIC = "MoE layer tokens/s and expert-weight HBM GB/s (% of 8 TB/s); paged decode tok/s"
E, TOPK, H, I = 128, 8, 2048, 768
K_SLOTS = 40
TRACE_STEPS = 256
SEED = 0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0



class L2Flush:
    """Evicts L2 (129 MB on GB300) before a timed step: a 256 MB write, then a read sweep
    of another 256 MB, which also retires the write's dirty lines before the step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(32 << 20, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()

FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def _peaks():
    """(HBM GB/s, bf16 TF/s burst, "measured" | "fallback")."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), \
                "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def _sustained_tflops():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p)).get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED))
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS_SUSTAINED


# --------------------------------------------------------------------------- inputs

def make_inputs(B, seed=SEED):
    rng = np.random.default_rng([seed, B])
    trace = gen.reuse_routing_trace(rng, E, TOPK, B, TRACE_STEPS, p=0.8)
    xs, logits = [], []
    for sets in trace:
        logits.append(gen.logits_for_sets(rng, sets, E))
        xs.append(gen.activations_bf16(rng, B, H))
    distinct = [len({e for st in sets for e in st}) for sets in trace]
    return trace, xs, logits, distinct


def make_store(fmt=0, seed=SEED):
    return gen.layer_store(fmt, H, I, E, seed, 0)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for t, l in self.lines if t0 - 0.15 <= t <= t1 + 0.15] or [l for _, l in self.lines[-3:]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- distributed (replicas only)

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("PMOE_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v, ws, device):
    """Max of a float over ranks (the slowest replica sets the job time)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank, time_s_per_rank):
    """Whole-job throughput of independent replicas: all units over the slowest rank's time."""
    return float(sum(units_per_rank)) / float(max(time_s_per_rank))


# --------------------------------------------------------------------------- our arm

TOUCH_STORE = True


def touch_store(torch, cache, layers, dev):
    """Pages every expert of every layer in once and empties the tables again: the state
    of a server whose host store has been read before (the start-up independence check
    does the same). The timed steps then page in the same misses as from a fresh table;
    only the first-touch cost of the store's host pages is left out of them."""
    n = min(cache.E, cache.max_tokens * cache.top_k)
    for l in range(layers):
        for e0 in range(0, cache.E, n):
            cache.expert_cache_prefetch(l, torch.arange(e0, min(cache.E, e0 + n), dtype=torch.int32, device=dev))
    torch.cuda.synchronize(dev)
    cache.expert_cache_reset(-1)
    torch.cuda.synchronize(dev)


def run_decode(pm, torch, store, B, steps, warmup, device, timed_clock=None, e2e=True, mode=0, graph=False,
               stage=False, fmt=0):
    trace, xs, logits, distinct = make_inputs(B)
    graph_launches = 0
    cache = pm.ExpertCache(E, TOPK, H, I, K_SLOTS, fmt=fmt, max_tokens=B, device=device, pagein_mode=mode)
    ebytes = pm.pmoe_expert_bytes(fmt, H, I)  # every byte of an expert the decode kernel reads
    cache.load_layer(0, store)
    dev = torch.device("cuda", device)
    if TOUCH_STORE:
        touch_store(torch, cache, 1, dev)
    x_dev = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev) for x in xs]
    l_dev = [torch.from_numpy(l).to(dev) for l in logits]
    ids = torch.empty((B, TOPK), dtype=torch.int32, device=dev)
    w = torch.empty((B, TOPK), dtype=torch.float32, device=dev)
    y = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    pre_steps = range(2) if graph else range(0)
    if graph:
        # the whole step (router, residency, SM-pull page-in, fused MoE) as one CUDA graph
        # over static buffers; each step first copies its inputs into them (device to device)
        x_s = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
        l_s = torch.empty((B, E), dtype=torch.float32, device=dev)
        for i in pre_steps:
            pm.moe_router_topk(l_dev[i], TOPK, ids_out=ids, w_out=w)
            cache.moe_paged_forward(0, x_dev[i], ids, w, y=y)
        torch.cuda.synchronize(dev)
        cache.expert_cache_set_timing(False)  # resets the launch counters
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pm.moe_router_topk(l_s, TOPK, ids_out=ids, w_out=w)
            cache.moe_paged_forward(0, x_s, ids, w, y=y)
        graph_launches = sum(v["launches"] for k_, v in cache.expert_cache_kernel_times().items()
                             if k_ not in ("copies", "pagein_copy")) + 1  # + the router

        def one(s):
            x_s.copy_(x_dev[s])
            l_s.copy_(l_dev[s])
            g.replay()
    else:
        def one(s):
            pm.moe_router_topk(l_dev[s], TOPK, ids_out=ids, w_out=w)
            if stage:
                # residency and page-in issued ahead as their own kernels (the prefetch
                # path), so the decode kernel only streams resident weights
                cache.expert_cache_ensure_resident(0, ids)
            cache.moe_paged_forward(0, x_dev[s], ids, w, y=y)

    for i in range(warmup):
        one(i % TRACE_STEPS)
    torch.cuda.synchronize(dev)
    stats0 = cache.expert_cache_stats(0)
    cache.expert_cache_set_timing(not graph)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    step_ids = [(warmup + i) % TRACE_STEPS for i in range(steps)]
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i, s in enumerate(step_ids):
        flush()
        evs[i][0].record(stream)
        one(s)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    ms = [a.elapsed_time(b) for a, b in evs]
    kt = cache.expert_cache_kernel_times()
    stats1 = cache.expert_cache_stats(0)
    total_ms = float(sum(ms))
    d_steps = [distinct[s] for s in step_ids]
    res = {
        "B": B, "steps": steps, "total_ms": total_ms, "ms_per_step": total_ms / steps,
        "step_ms_p50_p90_max": [float(np.percentile(ms, 50)), float(np.percentile(ms, 90)), float(max(ms))],
        "tokens_per_s": B * steps / (total_ms / 1e3), "t_wall": (t0, t1),
        "kernel_times": kt, "distinct_per_step": float(np.mean(d_steps)),
        "misses_per_step": (stats1["misses"] - stats0["misses"]) / steps,
        "hit_rate": (stats1["hits"] - stats0["hits"]) / max(1, (stats1["hits"] - stats0["hits"]) +
                                                            (stats1["misses"] - stats0["misses"])),
        "waves_per_step": (stats1["waves"] - stats0["waves"]) / steps,
        "bytes_paged_per_step": (stats1["bytes_paged"] - stats0["bytes_paged"]) / steps,
        "gateup_weight_bytes": sum(d * 2 * I * H * 2 for d in d_steps),
        "down_weight_bytes": sum(d * H * I * 2 for d in d_steps),
        "expert_weight_bytes": sum(d * ebytes for d in d_steps),
        "launches": (graph_launches * steps if graph else
                     sum(v["launches"] for k_, v in kt.items() if k_ not in ("copies", "pagein_copy")) + steps),
        "mode": ("SM-pull page-in inside the fused decode kernel, whole step replayed as one CUDA graph" if graph else
                 ("SM-pull page-in by a separate pull kernel, issued ahead" if (mode == 1 and stage) else
                  ("SM-pull page-in inside the fused decode kernel" if mode == 1 else
                   "copy-engine page-in (host reads the plan)"))),
    }
    cache.expert_cache_set_timing(False)
    if e2e:
        # end to end: pinned host inputs -> device, the layer, result -> pinned host, every
        # step. The table is emptied and the same warm-up replayed first, so the e2e steps
        # page in exactly what the timed steps paged in (same misses per step).
        x_h = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs]
        l_h = [torch.from_numpy(l).pin_memory() for l in logits]
        y_h = torch.empty((B, H), dtype=torch.bfloat16).pin_memory()
        x_d = x_s if graph else torch.empty((B, H), dtype=torch.bfloat16, device=dev)
        l_d = l_s if graph else torch.empty((B, E), dtype=torch.float32, device=dev)
        cache.expert_cache_reset(0)
        for i in pre_steps:
            pm.moe_router_topk(l_dev[i], TOPK, ids_out=ids, w_out=w)
            cache.moe_paged_forward(0, x_dev[i], ids, w, y=y)
        for i in range(warmup):
            one(i % TRACE_STEPS)
        torch.cuda.synchronize(dev)
        stats_e0 = cache.expert_cache_stats(0)
        evs2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i, s in enumerate(step_ids):
            flush()
            evs2[i][0].record(stream)
            x_d.copy_(x_h[s], non_blocking=True)
            l_d.copy_(l_h[s], non_blocking=True)
            if graph:
                g.replay()
            else:
                pm.moe_router_topk(l_d, TOPK, ids_out=ids, w_out=w)
                cache.moe_paged_forward(0, x_d, ids, w, y=y)
            y_h.copy_(y, non_blocking=True)
            evs2[i][1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = float(sum(a.elapsed_time(b) for a, b in evs2))
        stats_e1 = cache.expert_cache_stats(0)
        res["e2e"] = {"value": B * steps / (e2e_ms / 1e3), "unit": "tokens/s",
                      "h2d_bytes_per_step": B * H * 2 + B * E * 4, "d2h_bytes_per_step": B * H * 2,
                      "ms_per_step": e2e_ms / steps,
                      "misses_per_step": (stats_e1["misses"] - stats_e0["misses"]) / steps,
                      "timed_misses_per_step": res["misses_per_step"]}
    cache.close()
    return res


def measure_h2d(torch, dev, nbytes=9_437_184, reps=40):
    """Pinned host -> device copy bandwidth (cudaMemcpyAsync via torch), GB/s."""
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


PREFILL_T, PREFILL_K = 2048, 92


def run_prefill(pm, torch, store, steps, warmup, device, K=PREFILL_K, cold=True, n_inputs=3, mode=0, fmt=0,
                T=None):
    """Config: T-token prefill (2048 by default), uniform routing; cold = the table is emptied
    before every step."""
    T = PREFILL_T if T is None else T
    dev = torch.device("cuda", device)
    rng = np.random.default_rng([SEED, T])
    inputs = []
    for _ in range(n_inputs):
        sets = gen.uniform_routing_sets(rng, T, E, TOPK)
        inputs.append((torch.from_numpy(gen.activations_bf16(rng, T, H).view(np.int16)).view(torch.bfloat16).to(dev),
                       torch.from_numpy(gen.logits_for_sets(rng, sets, E)).to(dev)))
    cache = pm.ExpertCache(E, TOPK, H, I, K, fmt=fmt, max_tokens=T, device=device, pagein_mode=mode)
    cache.load_layer(0, store)
    ids = torch.empty((T, TOPK), dtype=torch.int32, device=dev)
    w = torch.empty((T, TOPK), dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def one(i):
        x_d, l_d = inputs[i % n_inputs]
        pm.moe_router_topk(l_d, TOPK, ids_out=ids, w_out=w)
        cache.moe_paged_forward(0, x_d, ids, w, y=y)

    for i in range(warmup):
        if cold:
            cache.expert_cache_reset(0)
        one(i)
    torch.cuda.synchronize(dev)
    s0 = cache.expert_cache_stats(0)
    cache.expert_cache_set_timing(True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if cold:
            cache.expert_cache_reset(0)
        flush()
        evs[i][0].record(stream)
        one(warmup + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    total_ms = float(sum(a.elapsed_time(b) for a, b in evs))
    kt = cache.expert_cache_kernel_times()
    s1 = cache.expert_cache_stats(0)
    cache.close()
    P = T * TOPK
    flops_gu = 2.0 * P * 2 * I * H * steps
    flops_d = 2.0 * P * H * I * steps
    return {"T": T, "K": K, "ms_per_step": total_ms / steps, "tokens_per_s": T * steps / (total_ms / 1e3),
            "misses_per_step": (s1["misses"] - s0["misses"]) / steps,
            "waves_per_step": (s1["waves"] - s0["waves"]) / steps,
            "bytes_paged_per_step": (s1["bytes_paged"] - s0["bytes_paged"]) / steps,
            "kernel_ms_per_step": {k_: v["ms"] / steps for k_, v in kt.items() if k_ != "copies"},
            "gateup_tflops": flops_gu / (kt["gateup"]["ms"] / 1e3) / 1e12,
            "down_tflops": flops_d / (kt["down"]["ms"] / 1e3) / 1e12,
            "gemm_tflops": (flops_gu + flops_d) / ((kt["gateup"]["ms"] + kt["down"]["ms"]) / 1e3) / 1e12,
            "gemm_ms_per_step": (kt["gateup"]["ms"] + kt["down"]["ms"]) / steps,
            "pagein_gbs": ((s1["bytes_paged"] - s0["bytes_paged"]) /
                           ((kt["pagein_copy"]["ms"] + kt["pull"]["ms"]) / 1e3) / 1e9
                           if kt["pagein_copy"]["ms"] + kt["pull"]["ms"] > 0 else None),
            "launches_per_step": sum(v["launches"] for k_, v in kt.items()
                                     if k_ not in ("copies", "pagein_copy")) / steps + 1}


def cpu_baseline_decode(B=1, budget_s=15.0, max_steps=400, store=None):
    """The oracle as it stands (float64 NumPy + the pure-Python LRU simulator) on the host
    cores, on the first steps of the same trace until the time budget is spent."""
    from oracle import lru as olru
    from oracle import moe as omoe
    from oracle import router as orouter
    trace, xs, logits, _ = make_inputs(B)
    store = make_store() if store is None else store
    experts = omoe.ExpertSource(lambda e: store[e], 0, H, I, cache=48)
    sim = olru.LayerLRU(E, K_SLOTS)
    t0 = time.time()
    n = 0
    while n < min(max_steps, TRACE_STEPS) and time.time() - t0 < budget_s:
        ids, w = orouter.router_topk(logits[n], TOPK)
        sim.step(ids.ravel().tolist())
        omoe.moe_layer(gen.bf16_bits_to_float(xs[n]).astype(np.float64), ids, w, experts)
        n += 1
    dt = time.time() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": B * n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} decode steps (B={B}) of the same 256-step trace: float64 NumPy router + "
                      f"SwiGLU experts decoded from the same bytes + LRU simulator, {dt:.1f} s"}


def run_prefill_sweep(pm, torch, args, local, hbm_peak, tc_peak):
    """Prefill at sizes where the grouped GEMMs are tensor-bound (AI = 512 FLOP/B at 8192
    bf16 tokens, 1024 at 16384): all experts resident (the GEMMs alone), bf16 and block FP8."""
    out = {}
    sizes = [int(t) for t in args.prefill_tokens.split(",") if t.strip()]
    for fmt, name, bpe in ((0, "bf16", 2), (1, "fp8", 1), (3, "mxfp4", 0.5)):
        store = make_store(fmt=fmt)
        runs = {f"T{T}_warm_all_resident": run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=E, cold=False,
                                                       fmt=fmt, T=T, n_inputs=2) for T in sizes}
        out[name] = _prefill_summary(runs, hbm_peak, tc_peak, wbytes_per_elem=bpe)
    out["fp8"]["note"] = ("256-pair tiles: FP8 weights dequantised to bf16 in shared memory for kind::f16 MMAs "
                          "(64-pair tiles run e4m3 kind::f8f6f4 MMAs on two-plane activations)")
    out["mxfp4"]["note"] = "MXFP4 weights (E2M1 x E8M0, exact in bf16) are dequantised in shared memory for kind::f16 MMAs"
    return out


def _summary(out):
    """A short digest of the whole line, printed as its last key."""
    def g(d, *keys):
        for k_ in keys:
            if not isinstance(d, dict) or k_ not in d:
                return None
            d = d[k_]
        return d

    def r3(v):
        return None if v is None else float(f"{v:.4g}")
    sm = {"decode_B1_tok_s": r3(out.get("value")),
          "decode_B1_kernel_hbm_frac": r3(g(out, "roofline", "frac")),
          "decode_B1_kernel_us": r3(g(out, "roofline", "avg_launch_us")),
          "e2e_B1_tok_s": r3(g(out, "e2e", "value")),
          "e2e_misses_per_step": r3(g(out, "e2e", "misses_per_step")),
          "timed_misses_per_step": r3(g(out, "e2e", "timed_misses_per_step"))}
    for B in (2, 4):
        sm[f"decode_B{B}_graph_tok_s"] = r3(g(out, "batches", f"B{B}_graph", "tokens_per_s"))
    sm["decode_B4_kernel_hbm_frac"] = r3(g(out, "batches", "B4_sm_pull_staged_no_graph", "decode_kernel_hbm_frac"))
    for name in ("cold", "warm_all_resident", "warm_all_resident_sm_pull"):
        sm[f"prefill2048_{name}_tok_s"] = r3(g(out, "prefill", name, "tokens_per_s"))
        sm[f"prefill2048_{name}_gemm_tflops"] = r3(g(out, "prefill", name, "gemm_tflops"))
        sm[f"prefill2048_{name}_bound_frac"] = r3(g(out, "prefill", name, "bound_frac"))
    for fmt in ("bf16", "fp8", "mxfp4"):
        for k_, v in (g(out, "prefill_sweep", fmt) or {}).items():
            if isinstance(v, dict) and "gemm_tflops" in v:
                sm[f"prefill_{fmt}_{k_}"] = {"gemm_tflops": r3(v["gemm_tflops"]), "tensor_frac": r3(v["tensor_frac"]),
                                             "tensor_frac_sustained": r3(v["tensor_frac_sustained"]),
                                             "bound_frac": r3(v["bound_frac"])}
    sm["fp8_decode_B1_tok_s"] = r3(g(out, "fp8", "decode_B1", "tokens_per_s"))
    sm["fp8_decode_kernel_hbm_frac"] = r3(g(out, "fp8", "decode_B1", "decode_kernel_hbm_frac"))
    sm["fp8_prefill512_gemm_tflops"] = r3(g(out, "fp8", "prefill_512_cold", "gemm_tflops"))
    sm["mxfp4_decode_B1_tok_s"] = r3(g(out, "mxfp4", "decode_B1", "tokens_per_s"))
    sm["mxfp4_decode_kernel_hbm_frac"] = r3(g(out, "mxfp4", "decode_B1", "decode_kernel_hbm_frac"))
    sm["mxfp4_prefill512_gemm_tflops"] = r3(g(out, "mxfp4", "prefill_512_cold", "gemm_tflops"))
    sm["nvfp4_decode_B1_tok_s"] = r3(g(out, "nvfp4", "decode_B1", "tokens_per_s"))
    sm["nvfp4_decode_kernel_hbm_frac"] = r3(g(out, "nvfp4", "decode_B1", "decode_kernel_hbm_frac"))
    sm["nvfp4_prefill512_gemm_tflops"] = r3(g(out, "nvfp4", "prefill_512_cold", "gemm_tflops"))
    for k_ in ("B1", "B1_graph", "B4", "B4_graph"):
        sm[f"stack_int4_{k_}_tok_s"] = r3(g(out, "stack_int4", k_, "tokens_per_s"))
        ov = g(out, "stack_int4", k_, "overlap")
        if ov is not None:
            sm[f"stack_int4_{k_}_overlap_frac"] = r3(ov.get("overlap_frac"))
    return {k_: v for k_, v in sm.items() if v is not None}


def run_ours(args):
    import torch
    ws, rank, local = dist_init()
    torch.cuda.set_device(local)
    import paged_expert_moe_gb300 as pm
    pm.load()
    store = make_store()
    hbm_peak, tc_peak, peak_kind = _peaks()
    if args.section == "fp8":
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": "ours", "section": "fp8", "fp8": run_fp8(pm, torch, args, local,
                                                                                                  hbm_peak)}))
        return
    if args.section == "mxfp4":
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": "ours", "section": "mxfp4",
                              "mxfp4": run_mxfp4(pm, torch, args, local, hbm_peak)}))
        return
    if args.section == "nvfp4":
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": "ours", "section": "nvfp4",
                              "nvfp4": run_nvfp4(pm, torch, args, local, hbm_peak)}))
        return
    if args.section in ("prefill", "stack", "decode_staged", "prefill_sweep"):
        # one part of the bench alone (for profiling); one JSON line with that part
        out = {"metric": METRIC, "impl": "ours", "section": args.section}
        if args.section == "prefill":
            out["prefill"] = _prefill_summary(
                {"cold": run_prefill(pm, torch, store, args.prefill_steps, 2, local, cold=True),
                 "warm_all_resident": run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=E, cold=False),
                 "warm_all_resident_sm_pull": run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=E,
                                                          cold=False, mode=1)},
                hbm_peak, tc_peak)
        elif args.section == "prefill_sweep":
            out["prefill_sweep"] = run_prefill_sweep(pm, torch, args, local, hbm_peak, tc_peak)
        elif args.section == "stack":
            out["stack_int4"] = run_stack_section(pm, torch, args, local, measure_h2d(torch, torch.device("cuda", local)))
        else:
            # the decode kernel alone on resident weights (page-in staged ahead): the launches
            # the roofline is measured on
            fmt = {"bf16": 0, "fp8": 1, "int4": 2, "mxfp4": 3, "nvfp4": 4}[args.format]
            st = store if fmt == 0 else make_store(fmt=fmt)
            r = run_decode(pm, torch, st, args.batch, args.steps, args.warmup, local, e2e=False, mode=1, stage=True,
                           fmt=fmt)
            dec_ms = r["kernel_times"]["decode"]["ms"]
            out["decode_staged"] = {"format": args.format, "B": args.batch, "ms_per_step": r["ms_per_step"],
                                    "decode_kernel_us": dec_ms / max(1, r["kernel_times"]["decode"]["launches"]) * 1e3,
                                    "decode_kernel_hbm_frac": r["expert_weight_bytes"] / (dec_ms / 1e3) / 1e9 / hbm_peak,
                                    "distinct_per_step": r["distinct_per_step"]}
        if rank == 0:
            print(json.dumps(out))
        return
    barrier(ws)
    torch.cuda.synchronize()
    clock = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.3)
    head = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, mode=1, graph=True)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = clock.stop(*head["t_wall"]) if clock else None
    # the same workload without the graph, with per-kernel CUDA-event timers on the
    # kernels' own streams, the page-in staged ahead by its own kernel: the decode
    # kernel's duration for the (HBM) roofline
    timed = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, stage=True)
    others = {}
    prefill = {}
    stack = {}
    fp8 = None
    mxfp4 = None
    nvfp4 = None
    sweep = None
    h2d = measure_h2d(torch, torch.device("cuda", local))
    # the other sections (batches, prefill, formats, the stack) run in single-GPU runs
    # only: replicas add nothing to them, and every rank would pin another 45 GB of host
    # memory for the stack
    if not args.headline_only and ws == 1:
        stack = run_stack_child(args, local)
        others["B1_sm_pull_staged_no_graph"] = timed
        others["B1_sm_pull_in_kernel_no_graph"] = run_decode(pm, torch, store, 1, args.steps, args.warmup, local,
                                                             e2e=False, mode=1)
        others["B1_copy_engine"] = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False)
        for B in (2, 4):
            others[f"B{B}_graph"] = run_decode(pm, torch, store, B, args.steps, args.warmup, local, e2e=False,
                                               mode=1, graph=True)
            others[B] = run_decode(pm, torch, store, B, args.steps, args.warmup, local, e2e=False)
        others["B4_sm_pull_staged_no_graph"] = run_decode(pm, torch, store, 4, args.steps, args.warmup, local,
                                                          e2e=False, mode=1, stage=True)
        prefill["cold"] = run_prefill(pm, torch, store, args.prefill_steps, 2, local, cold=True)
        prefill["cold_sm_pull"] = run_prefill(pm, torch, store, args.prefill_steps, 2, local, cold=True, mode=1)
        prefill["warm_all_resident"] = run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=E, cold=False)
        # the same step with the plan kept on the device: no host wait between the residency
        # kernel and the GEMM launches
        prefill["warm_all_resident_sm_pull"] = run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=E,
                                                           cold=False, mode=1)
        sweep = run_prefill_sweep(pm, torch, args, local, hbm_peak, tc_peak)
        fp8 = run_fp8(pm, torch, args, local, hbm_peak)
        mxfp4 = run_mxfp4(pm, torch, args, local, hbm_peak)
        nvfp4 = run_nvfp4(pm, torch, args, local, hbm_peak)
    job_ms = reduce_max(head["total_ms"], ws, torch.device("cuda", local))
    value = ws * 1 * args.steps / (job_ms / 1e3)
    if rank != 0:
        return
    kt = timed["kernel_times"]
    dec_ms = kt["decode"]["ms"]
    dec_launch = max(1, kt["decode"]["launches"])
    achieved = timed["expert_weight_bytes"] / (dec_ms / 1e3) / 1e9
    layer_gbs = achieved
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        try:
            traffic = json.load(open(tp)).get("decode_fused_bf16_B1")
        except Exception:
            traffic = None
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": job_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "Qwen3-30B-A3B-shaped MoE layer, bf16 experts, decode B=1, K=40 slots, "
                               "256-step p=0.8 reuse routing trace",
                   "E": E, "top_k": TOPK, "hidden": H, "intermediate": I, "K": K_SLOTS, "batch": 1,
                   "pagein": "SM pull from the mapped pinned host store inside the fused decode kernel (each CTA "
                             "pages in the bytes its own chunks read); the step replayed as one CUDA graph",
                   "l2": "flushed before every timed step (256 MB write, then a 256 MB read sweep; outside the events)",
                   "parallelism": f"replicas x{ws}"},
        "expert_weight_hbm_gbs": layer_gbs,
        "expert_weight_hbm_frac": layer_gbs / hbm_peak,
        "roofline": {"kernel": "decode_fused_kernel (gate/up + SiLU*mul + down + combine, one launch per wave)",
                     "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic,
                     "avg_launch_us": dec_ms / dec_launch * 1e3,
                     "algorithmic_bytes_per_launch": timed["expert_weight_bytes"] / dec_launch,
                     "measured_in": "the same workload run without the graph, page-in staged ahead by the pull kernel (per-kernel CUDA events)",
                     "algorithmic_bytes_note": "distinct routed experts x 3*H*I*2 bytes (gate, up, down weights)"},
        "headline_step_ms_p50_p90_max": head["step_ms_p50_p90_max"],
        "layer": {"misses_per_step": head["misses_per_step"], "hit_rate": head["hit_rate"],
                  "waves_per_step": head["waves_per_step"], "distinct_experts_per_step": head["distinct_per_step"],
                  "bytes_paged_per_step": head["bytes_paged_per_step"],
                  "kernel_ms_per_step_without_graph": {k_: v["ms"] / args.steps for k_, v in kt.items()
                                                       if k_ != "copies" and v["ms"]}},
        "batches": {(f"B{B}" if isinstance(B, int) else B): {"mode": r["mode"], "tokens_per_s": r["tokens_per_s"],
                              "ms_per_step": r["ms_per_step"],
                              "misses_per_step": r["misses_per_step"], "waves_per_step": r["waves_per_step"],
                              "decode_kernel_gbs": r["expert_weight_bytes"] /
                              (r["kernel_times"]["decode"]["ms"] / 1e3) / 1e9 if r["kernel_times"]["decode"]["ms"] else None,
                              "decode_kernel_hbm_frac": r["expert_weight_bytes"] /
                              (r["kernel_times"]["decode"]["ms"] / 1e3) / 1e9 / hbm_peak
                              if r["kernel_times"]["decode"]["ms"] else None,
                              "kernel_ms_per_step": {k_: v["ms"] / r["steps"] for k_, v in r["kernel_times"].items()
                                                     if k_ != "copies" and v["ms"]}}
                    for B, r in others.items()},
        "host_link": {"pinned_h2d_gbs": h2d, "chunk_bytes": 9_437_184,
                      "decode_pagein_gbs": (timed["bytes_paged_per_step"] * args.steps /
                                            (kt["pull"]["ms"] / 1e3) / 1e9) if kt["pull"]["ms"] else None,
                      "decode_pagein_kind": "SM pull kernel (CUDA-event time on the copy stream)"},
        "prefill": _prefill_summary(prefill, hbm_peak, tc_peak) if prefill else None,
        "prefill_sweep": sweep,
        "fp8": fp8,
        "mxfp4": mxfp4,
        "nvfp4": nvfp4,
        "stack_int4": ({"workload": "48-layer Qwen3-30B-A3B-shaped MoE stack (attention omitted), GPTQ-int4 g128 "
                                    "experts, K=26 slots/layer, p=0.8 reuse routing per layer, residual stream",
                        "hbm_roofline_tokens_per_s_B1": hbm_peak * 1e9 / (STACK_L * TOPK * 2_506_752),
                        "measured_in": "a child process of its own (bench.py --section stack)",
                        **stack} if stack else None),
        "e2e": head.get("e2e"),
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "impl": "ours",
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_decode(1, budget_s=args.cpu_budget, store=store)
    out["summary"] = _summary(out)
    print(json.dumps(out))


def run_fp8(pm, torch, args, local, hbm_peak):
    """The block-FP8 configuration: the same layer with e4m3 experts and fp32 128x128 scales,
    K=40, decode B=1 over the p=0.8 reuse trace, plus a cold 512-token prefill."""
    store = make_store(fmt=1)
    ebytes = pm.pmoe_expert_bytes(1, H, I)
    head = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, graph=True, fmt=1)
    staged = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, stage=True, fmt=1)
    kt = staged["kernel_times"]
    dec_gbs = staged["expert_weight_bytes"] / (kt["decode"]["ms"] / 1e3) / 1e9
    pre = run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=40, cold=True, fmt=1, T=512)
    flop = 2.0 * 512 * TOPK * 3 * H * I
    return {"workload": "Qwen3-30B-A3B-shaped MoE layer, block-FP8 e4m3 experts (fp32 128x128 scales), K=40",
            "expert_bytes": ebytes,
            "decode_B1": {"tokens_per_s": head["tokens_per_s"], "ms_per_step": head["ms_per_step"],
                          "misses_per_step": head["misses_per_step"], "mode": head["mode"],
                          "decode_kernel_gbs": dec_gbs, "decode_kernel_hbm_frac": dec_gbs / hbm_peak,
                          "decode_kernel_us": kt["decode"]["ms"] / args.steps * 1e3,
                          "decode_kernel_measured_in": "page-in staged ahead by the pull kernel"},
            "prefill_512_cold": dict(pre, FLOP_per_step=flop, weight_bytes_per_step=E * ebytes,
                                     hbm_bound_tflops=flop / (E * ebytes / (hbm_peak * 1e9)) / 1e12,
                                     hbm_bound_frac=pre["gemm_tflops"] / (flop / (E * ebytes / (hbm_peak * 1e9)) / 1e12),
                                     note="64-pair tiles: e4m3 weights into tcgen05 kind::f8f6f4 MMAs, activations "
                                          "as two e4m3 planes (hi + lo) on power-of-two scales")}


def run_mxfp4(pm, torch, args, local, hbm_peak):
    """MXFP4 experts (E2M1 codes, an E8M0 scale per 32 inputs): the same layer, K=40,
    decode B=1 over the p=0.8 reuse trace, plus a cold 512-token prefill."""
    store = make_store(fmt=3)
    ebytes = pm.pmoe_expert_bytes(3, H, I)
    head = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, graph=True, fmt=3)
    staged = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, stage=True, fmt=3)
    kt = staged["kernel_times"]
    dec_gbs = staged["expert_weight_bytes"] / (kt["decode"]["ms"] / 1e3) / 1e9
    pre = run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=40, cold=True, fmt=3, T=512)
    flop = 2.0 * 512 * TOPK * 3 * H * I
    return {"workload": "Qwen3-30B-A3B-shaped MoE layer, MXFP4 experts (E2M1, E8M0 scale per 32 inputs), K=40",
            "expert_bytes": ebytes,
            "decode_B1": {"tokens_per_s": head["tokens_per_s"], "ms_per_step": head["ms_per_step"],
                          "misses_per_step": head["misses_per_step"], "mode": head["mode"],
                          "decode_kernel_gbs": dec_gbs, "decode_kernel_hbm_frac": dec_gbs / hbm_peak,
                          "decode_kernel_us": kt["decode"]["ms"] / args.steps * 1e3,
                          "decode_kernel_measured_in": "page-in staged ahead by the pull kernel"},
            "prefill_512_cold": dict(pre, FLOP_per_step=flop, weight_bytes_per_step=E * ebytes,
                                     hbm_bound_tflops=flop / (E * ebytes / (hbm_peak * 1e9)) / 1e12,
                                     note="E2M1 x E8M0 weights are dequantised (exactly) to bf16 in shared memory "
                                          "for kind::f16 MMAs")}


def run_nvfp4(pm, torch, args, local, hbm_peak):
    """NVFP4 experts (E2M1 codes, an e4m3 scale per 16 inputs, an fp32 tensor scale per
    matrix): the same layer, K=40, decode B=1 over the p=0.8 reuse trace, plus a cold
    512-token prefill."""
    store = make_store(fmt=4)
    ebytes = pm.pmoe_expert_bytes(4, H, I)
    head = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, graph=True, fmt=4)
    staged = run_decode(pm, torch, store, 1, args.steps, args.warmup, local, e2e=False, mode=1, stage=True, fmt=4)
    kt = staged["kernel_times"]
    dec_ms = kt["decode"]["ms"]
    dec_gbs = staged["expert_weight_bytes"] / (dec_ms / 1e3) / 1e9
    pre = run_prefill(pm, torch, store, args.prefill_steps, 2, local, K=40, cold=True, fmt=4, T=512)
    flop = 2.0 * 512 * TOPK * 3 * H * I
    return {"workload": "Qwen3-30B-A3B-shaped MoE layer, NVFP4 experts (E2M1, e4m3 scale per 16 inputs, fp32 "
                        "tensor scale per matrix), K=40",
            "expert_bytes": ebytes,
            "decode_B1": {"tokens_per_s": head["tokens_per_s"], "ms_per_step": head["ms_per_step"],
                          "misses_per_step": head["misses_per_step"], "mode": head["mode"],
                          "decode_kernel_gbs": dec_gbs, "decode_kernel_hbm_frac": dec_gbs / hbm_peak,
                          "decode_kernel_us": dec_ms / args.steps * 1e3,
                          "decode_kernel_measured_in": "page-in staged ahead by the pull kernel"},
            "prefill_512_cold": dict(pre, FLOP_per_step=flop, weight_bytes_per_step=E * ebytes,
                                     hbm_bound_tflops=flop / (E * ebytes / (hbm_peak * 1e9)) / 1e12,
                                     note="E2M1 x e4m3 weights are dequantised (exactly) to bf16 in shared memory "
                                          "for kind::f16 MMAs; the fp32 tensor scale multiplies the accumulators")}


STACK_L, STACK_K = 48, 26


def _overlap(t_a, t_b, t_step):
    """Share of the shorter of two activities hidden under the longer one in a step of
    t_step: 1 when t_step = max(t_a, t_b) (fully overlapped), 0 when t_step = t_a + t_b."""
    lo = min(t_a, t_b)
    if lo <= 0:
        return None
    return float(min(1.0, max(0.0, (t_a + t_b - t_step) / lo)))


def run_stack_child(args, local):
    """The stack section in a process of its own (its 45 GB of pinned host stores do not
    share a process with the other measurements); returns its stack_int4 record."""
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK=str(local))
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--section", "stack", "--stack-steps",
                        str(args.stack_steps), "--stack-layers", str(args.stack_layers)], capture_output=True,
                       text=True, env=env)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"error": f"stack section exited {r.returncode}: {r.stderr[-300:]}"}
    return json.loads(lines[-1]).get("stack_int4")


def run_stack_section(pm, torch, args, local, h2d):
    """Config 5 in both page-in modes at B=1 and B=4: SM-pull in graphs, the same steps with
    every expert resident (the compute alone, for the overlap fraction), and copy engine."""
    stack = {}
    # the paged and the all-resident caches side by side, their runs interleaved, so that
    # both see the same host state (each 15 GB pinning slows later runs on a box)
    pull = make_stack_cache(pm, torch, local, mode=1, layers=args.stack_layers)
    res = make_stack_cache(pm, torch, local, mode=1, layers=args.stack_layers, K=E)
    runs, res_runs = {}, {}
    for B in (1, 4):
        runs[B] = run_stack(pm, torch, B, args.stack_steps, 3, local, graph=True, h2d_gbs=h2d, cache=pull)
        res_runs[B] = run_stack(pm, torch, B, args.stack_steps, 3, local, graph=True, cache=res)
    pull.close()
    res.close()
    for B in (1, 4):
        g_run, t_res = runs[B], res_runs[B]["ms_per_step"]
        t_link = g_run["overlap"]["link_ms_per_step"]
        g_run["overlap"].update({"resident_only_ms_per_step": t_res,
                                 "overlap_frac": _overlap(t_link, t_res, g_run["ms_per_step"]),
                                 "method": "page-in inside the decode kernels: (t_link + t_resident - t_step) / "
                                           "min(...), t_link = paged bytes / pinned H2D GB/s, t_resident = the "
                                           "same steps with K = E (no misses)"})
        stack[f"B{B}_graph"] = g_run
    ce = make_stack_cache(pm, torch, local, mode=0, layers=args.stack_layers)
    for B in (1, 4):
        stack[f"B{B}"] = run_stack(pm, torch, B, args.stack_steps, 3, local, h2d_gbs=h2d, cache=ce)
    ce.close()
    return stack


def make_stack_cache(pm, torch, device, mode=0, layers=STACK_L, K=STACK_K, max_tokens=4):
    """One pinned 15 GB host store for every run on it (repeated pinning of 15 GB slows
    later host-link reads on the same box). K = E: every expert of every layer paged in
    ahead, so later steps miss nothing."""
    dev = torch.device("cuda", device)
    cache = pm.ExpertCache(E, TOPK, H, I, K, num_layers=layers, fmt=pm.PMOE_INT4_GPTQ_G128, max_tokens=max_tokens,
                           device=device, pagein_mode=mode)
    for l in range(layers):
        gen.layer_store(2, H, I, E, SEED, layer=l, fast=True, out=cache.host_store(l))
    if K == E:
        n = min(E, max_tokens * TOPK)
        for l in range(layers):
            for e0 in range(0, E, n):
                cache.expert_cache_prefetch(l, torch.arange(e0, min(E, e0 + n), dtype=torch.int32, device=dev))
        torch.cuda.synchronize(dev)
    elif TOUCH_STORE:
        touch_store(torch, cache, layers, dev)
    return cache


def run_stack(pm, torch, B, steps, warmup, device, mode=0, layers=STACK_L, K=STACK_K, graph=False, h2d_gbs=None,
              cache=None):
    """48-layer MoE stack, GPTQ-int4 experts, K=26 slots per layer, decode batch B, each
    layer with its own p=0.8 reuse routing; h_{l+1} = h_l + moe_l(h_l) through
    moe_paged_stack_forward (next layer's page-in overlapped with the current layer).
    A run on a K < E cache empties its tables first (each run starts cold)."""
    dev = torch.device("cuda", device)
    own = cache is None
    if own:
        cache = make_stack_cache(pm, torch, device, mode, layers, K, max_tokens=B)
    elif cache.K != E:
        cache.expert_cache_reset(-1)
    mode, K, layers = (1 if cache.desc.pagein_mode else 0), cache.K, cache.layers
    rng = np.random.default_rng([SEED, 48, B])
    traces = [gen.reuse_routing_trace(rng, E, TOPK, B, TRACE_STEPS) for _ in range(layers)]
    n_inputs = min(TRACE_STEPS, warmup + steps)
    logits = [torch.from_numpy(np.concatenate([gen.logits_for_sets(rng, traces[l][s], E) for l in range(layers)])).to(dev)
              for s in range(n_inputs)]
    xs = [torch.from_numpy(gen.activations_bf16(rng, B, H).view(np.int16)).view(torch.bfloat16).to(dev)
          for _ in range(n_inputs)]
    distinct = [sum(len({e for st in traces[l][s] for e in st}) for l in range(layers)) for s in range(n_inputs)]
    ids = torch.empty((layers * B, TOPK), dtype=torch.int32, device=dev)
    w = torch.empty((layers * B, TOPK), dtype=torch.float32, device=dev)
    y = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    work = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    if graph:
        x_s = torch.empty((B, H), dtype=torch.bfloat16, device=dev)
        l_s = torch.empty((layers * B, E), dtype=torch.float32, device=dev)
        pm.moe_router_topk(logits[0], TOPK, ids_out=ids, w_out=w)
        cache.moe_paged_stack_forward(xs[0], ids, w, y=y, work=work)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pm.moe_router_topk(l_s, TOPK, ids_out=ids, w_out=w)
            cache.moe_paged_stack_forward(x_s, ids, w, y=y, work=work)

        def one(s):
            x_s.copy_(xs[s])
            l_s.copy_(logits[s])
            g.replay()
    else:
        def one(s):
            pm.moe_router_topk(logits[s], TOPK, ids_out=ids, w_out=w)
            cache.moe_paged_stack_forward(xs[s], ids, w, y=y, work=work)

    for i in range(warmup):
        one(i % n_inputs)
    torch.cuda.synchronize(dev)
    s0 = cache.expert_cache_stats(-1)
    cache.expert_cache_set_timing(not graph)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ids_used = [(warmup + i) % n_inputs for i in range(steps)]
    for i, si in enumerate(ids_used):
        flush()
        evs[i][0].record(stream)
        one(si)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    total_ms = float(sum(a.elapsed_time(b) for a, b in evs))
    kt = cache.expert_cache_kernel_times()
    s1 = cache.expert_cache_stats(-1)
    cache.expert_cache_set_timing(False)
    if own:
        cache.close()
    nb = pm.pmoe_expert_bytes(pm.PMOE_INT4_GPTQ_G128, H, I)
    wbytes = sum(distinct[si] for si in ids_used) * nb
    dec_ms = kt["decode"]["ms"]
    ms_step = total_ms / steps
    paged_gb = (s1["bytes_paged"] - s0["bytes_paged"]) / steps / 1e9
    overlap = None
    if h2d_gbs:
        t_link = paged_gb / h2d_gbs * 1e3  # ms the link needs for the step's page-in alone
        overlap = {"link_ms_per_step": t_link, "link_floor_frac": t_link / ms_step if ms_step else None,
                   "h2d_gbs": h2d_gbs}
        if not graph and mode == 0:
            # copy engine: the copies (copy stream) against the compute (decode + combine on
            # the compute stream), from the per-stream CUDA-event timers
            t_copy = kt["pagein_copy"]["ms"] / steps
            t_comp = (kt["decode"]["ms"] + kt["combine"]["ms"]) / steps
            overlap.update({"copy_ms_per_step": t_copy, "compute_ms_per_step": t_comp,
                            "overlap_frac": _overlap(t_copy, t_comp, ms_step),
                            "method": "per-stream CUDA-event timers: (t_copy + t_compute - t_step) / min(...)"})
    return {"B": B, "layers": layers, "K": K, "steps": steps, "ms_per_step": ms_step, "overlap": overlap,
            "mode": ("SM-pull, CUDA graph" if graph else ("SM-pull" if mode == 1 else "copy engine")),
            "tokens_per_s": B * steps / (total_ms / 1e3),
            "misses_per_token": (s1["misses"] - s0["misses"]) / (steps * B),
            "waves_per_layer_step": (s1["waves"] - s0["waves"]) / (steps * layers),
            "pagein_gb_per_step": (s1["bytes_paged"] - s0["bytes_paged"]) / steps / 1e9,
            "expert_weight_gb_per_step": wbytes / steps / 1e9,
            "decode_kernel_gbs": wbytes / (dec_ms / 1e3) / 1e9 if dec_ms else None,
            "kernel_ms_per_step": {k_: v["ms"] / steps for k_, v in kt.items() if k_ != "copies" and v["ms"]}}


def _prefill_summary(prefill, hbm_peak, tc_peak, wbytes_per_elem=2):
    """Per run: GEMM TF/s against the tensor peak (burst, and sustained for long steps) and
    against the layer's own bound min(tensor peak, AI x HBM), AI = FLOPs / weight bytes."""
    tc_sus = _sustained_tflops()
    out = {"workload": "Qwen3-30B-A3B-shaped MoE layer, prefill, uniform routing (all 128 experts routed)",
           "weight_bytes_per_step": E * 3 * H * I * wbytes_per_elem}
    for name, r in prefill.items():
        d = dict(r)
        flop = 2.0 * r["T"] * TOPK * 3 * H * I
        wb = E * 3 * H * I * wbytes_per_elem
        bound = min(tc_peak, flop / wb * hbm_peak / 1e3)
        d["FLOP_per_step"] = flop
        d["tensor_frac"] = r["gemm_tflops"] / tc_peak
        d["tensor_frac_sustained"] = r["gemm_tflops"] / tc_sus
        d["bound_tflops"] = bound
        d["bound_frac"] = r["gemm_tflops"] / bound
        d["weight_stream_frac"] = wb / (r["gemm_ms_per_step"] / 1e3) / 1e9 / hbm_peak
        out[name] = d
    out["tensor_peak_tflops"] = tc_peak
    out["tensor_peak_tflops_sustained"] = tc_sus
    out["roofline_note"] = ("AI = 2*T*top_k*3*H*I / (E*3*H*I*bytes): 128 FLOP/B at 2048 bf16 tokens (below the "
                            "ridge, HBM-bound); 512 at 8192 and 1024 at 16384 (tensor-bound)")
    return out


# --------------------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import lru as olru
    from oracle import moe as omoe
    from oracle import router as orouter
    B = 1
    trace, xs, logits, _ = make_inputs(B)
    store = make_store()
    experts = omoe.ExpertSource(lambda e: store[e], 0, H, I, cache=48)
    sim = olru.LayerLRU(E, K_SLOTS)

    def one(s):
        ids, w = orouter.router_topk(logits[s], TOPK)
        sim.step(ids.ravel().tolist())
        omoe.moe_layer(gen.bf16_bits_to_float(xs[s]).astype(np.float64), ids, w, experts)

    # each step is one decode step of the trace; the run is capped so it ends within minutes
    budget = args.cpu_budget * 6
    t_start = time.time()
    for i in range(args.warmup):
        one(i % TRACE_STEPS)
    n = 0
    t0 = time.time()
    while n < args.steps and time.time() - t0 < budget:
        one((args.warmup + n) % TRACE_STEPS)
        n += 1
    dt = time.time() - t0
    cores = len(os.sched_getaffinity(0))
    v = B * n / dt
    out = {
        "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws, "steps": n, "warmup": args.warmup,
        "ms_per_step": dt / max(n, 1) * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": "Qwen3-30B-A3B-shaped MoE layer, bf16 experts, decode B=1, K=40 slots, "
                               "256-step p=0.8 reuse routing trace", "E": E, "top_k": TOPK, "hidden": H,
                   "intermediate": I, "K": K_SLOTS, "batch": 1},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} decode steps after {args.warmup} warm-up steps, "
                                   f"{time.time() - t_start:.1f} s in all"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--prefill-steps", type=int, default=6)
    ap.add_argument("--stack-steps", type=int, default=60)
    ap.add_argument("--stack-layers", type=int, default=STACK_L,
                    help="layers of the stack section (48 for the measured workload; fewer for profiling)")
    ap.add_argument("--section", default="all",
                    choices=["all", "prefill", "prefill_sweep", "stack", "decode_staged", "fp8", "mxfp4", "nvfp4"],
                    help="run only one part (profiling); the default runs everything")
    ap.add_argument("--prefill-tokens", default="8192,16384",
                    help="token counts of the tensor-bound prefill sweep (comma-separated)")
    ap.add_argument("--batch", type=int, default=1, help="decode batch of --section decode_staged")
    ap.add_argument("--format", default="bf16", choices=["bf16", "fp8", "int4", "mxfp4", "nvfp4"],
                    help="expert format of --section decode_staged")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
