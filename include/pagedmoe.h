/*
 * pagedmoe.h — C ABI of the paged-expert MoE layer for one GB300 (sm_103a).
 *
 * The operation (article "Running an MoE Model Larger Than Your VRAM: SGLang
 * Paged Experts, the PCIe Math, and the 4-Request Cliff", TL;DR and section
 * "What does Paged Experts actually do?"): each step a router sends every token
 * to top_k of E experts; a per-layer table of K GPU slots holds K of the E
 * experts, all E live in pinned host RAM, the routed experts that are not
 * resident are copied in (the oldest-used evicted), then the fused MoE runs over
 * the slot table: gate/up projection, SiLU*mul, down projection and the
 * top_k-weighted combine. Paging never changes the result (section "Can paging
 * change the model's outputs?"): outputs are bitwise identical for every K.
 *
 * Conventions shared by every call
 *   - Every call returns a pmoe_status (0 = success). Nothing throws across the ABI.
 *   - "device" pointers are CUDA device (or managed) addresses on the cache's
 *     device; "host" pointers are ordinary host addresses. Pointers are borrowed
 *     for the duration of the call (device pointers: until the stream work that
 *     the call enqueued has finished). The caller owns everything it passes in.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls enqueue
 *     their device work on it in stream order and do not synchronise the device,
 *     except where a call says it waits (the host reads a residency plan).
 *   - Argument errors are detected on the host before any device work is
 *     enqueued and return PMOE_EINVAL with nothing enqueued.
 *   - Errors a kernel detects (an expert id outside [0, E)) are recorded in the
 *     cache's device error word; the kernel skips the bad item. The next call that
 *     reads a plan, statistics or the slot table returns PMOE_EDEVICE.
 *   - Host waits are bounded (default 10 s, env PMOE_WAIT_TIMEOUT_MS); on expiry
 *     the call returns PMOE_ETIMEOUT.
 *
 * Expert byte layouts (one contiguous byte string per expert; all of an expert's
 * tensors — weights, scales, zero points — travel together, so a paged-in expert
 * can never run with another expert's scales; section "Can paging change the
 * model's outputs?"). Sections are packed in the order listed, row-major:
 *   PMOE_BF16            W_gu bf16 [2I][H] (rows 0..I-1 gate_proj, I..2I-1 up_proj)
 *                        W_d  bf16 [H][I]
 *   PMOE_FP8_BLOCK128    Q_gu e4m3 [2I][H], Q_d e4m3 [H][I],
 *                        S_gu fp32 [2I/128][H/128], S_d fp32 [H/128][I/128];
 *                        w = e4m3(q) * s of the 128x128 block holding (row, col)
 *   PMOE_INT4_GPTQ_G128  Q_gu u8 [2I][H/2], Q_d u8 [H][I/2] (element c of a row in
 *                        byte c/2, low nibble for even c),
 *                        SZ_gu fp16 [2I][H/128][2], SZ_d fp16 [H][I/128][2]
 *                        ((scale, zero) per output row and group of 128 inputs);
 *                        w = (q - z) * s
 *   PMOE_MXFP4           Q_gu u8 [2I][H/2], Q_d u8 [H][I/2] (FP4 E2M1 codes, element
 *                        c of a row in byte c/2, low nibble for even c),
 *                        X_gu u8 [2I][H/32], X_d u8 [H][I/32] (E8M0 scale per output
 *                        row and block of 32 inputs); w = e2m1(q) * 2^(X - 127)
 *                        (X = 0xFF, NaN in the format, is read as 2^128: keep
 *                        stores free of NaN scales)
 *                        (the OCP microscaling layout; the formats of section "What
 *                        does Paged Experts actually do?", PR #45787). E2M1 times an
 *                        E8M0 scale is exact in bf16 (scales 2^-126 .. 2^125), so the
 *                        prefill path dequantises these weights without rounding.
 *   PMOE_NVFP4           Q_gu u8 [2I][H/2], Q_d u8 [H][I/2] (FP4 E2M1 codes, as MXFP4),
 *                        then T_gu fp32 + 12 bytes of padding, B_gu e4m3 [2I][H/16],
 *                        then T_d fp32 + 12 bytes of padding, B_d e4m3 [H][I/16]
 *                        (one e4m3 scale per output row and block of 16 inputs; one
 *                        fp32 tensor scale per matrix, gate and up sharing theirs);
 *                        w = e2m1(q) * e4m3(B) * T (the two-level NVFP4 encoding; the
 *                        formats of PR #45787). E2M1 times an e4m3 scale is exact in
 *                        bf16; T is applied in fp32.
 * FP8, int4, MXFP4 and NVFP4 need H and I multiples of 128; bf16 needs multiples of 8 (and,
 * for the tensor-core prefill path, H a multiple of 128 and I of 128).
 *
 * Activations x, residual and y are bf16 [T][H] row-major; router logits fp32
 * [T][E]; ids int32 [T][top_k]; routing weights fp32 [T][top_k].
 */
#ifndef PAGEDMOE_H
#define PAGEDMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PMOE_API __attribute__((visibility("default")))
#else
#define PMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PMOE_OK = 0,
  PMOE_EINVAL = -1,        /* bad argument or descriptor; nothing was enqueued        */
  PMOE_ENOMEM = -2,        /* device memory for slots or workspace could not be had   */
  PMOE_EHOSTALLOC = -3,    /* the pinned host store could not be allocated            */
  PMOE_ECUDA = -4,         /* a CUDA runtime call failed (text: pmoe_last_error)      */
  PMOE_EUNSUPPORTED = -5,  /* format / shape / device rejected at create time         */
  PMOE_ETIMEOUT = -6,      /* a bounded host wait expired                             */
  PMOE_EDEVICE = -7        /* a kernel recorded an error (bad expert id)              */
} pmoe_status;

typedef enum {
  PMOE_BF16 = 0,
  PMOE_FP8_BLOCK128 = 1,
  PMOE_INT4_GPTQ_G128 = 2,
  PMOE_MXFP4 = 3,
  PMOE_NVFP4 = 4
} pmoe_format;

typedef enum {
  /* The host reads the step's miss list back and issues one cudaMemcpyAsync per
   * missed expert (pinned host store -> slot) on the cache's copy stream. */
  PMOE_PAGEIN_COPY_ENGINE = 0,
  /* A kernel on the copy stream pulls missed experts from the mapped pinned store
   * itself (no host round trip; the step stays stream-ordered). */
  PMOE_PAGEIN_SM_PULL = 1
} pmoe_pagein_mode;

typedef struct {
  int32_t num_experts;   /* E, 1..1024                                              */
  int32_t top_k;         /* 1..min(E, 32)                                           */
  int32_t hidden;        /* H                                                        */
  int32_t intermediate;  /* I (MoE intermediate size)                                */
  int32_t num_slots;     /* K resident experts per layer, 1..E                       */
  int32_t num_layers;    /* MoE layers, each with its own table, store and arena     */
  int32_t format;        /* pmoe_format                                              */
  int32_t max_tokens;    /* largest T a forward call may pass (sizes the workspace)  */
  int32_t pagein_mode;   /* pmoe_pagein_mode                                         */
  int32_t device;        /* CUDA device ordinal                                      */
} pmoe_cache_desc;

typedef struct {
  uint64_t steps;        /* residency steps taken                                    */
  uint64_t hits;         /* distinct routed experts found resident                   */
  uint64_t misses;       /* experts copied in                                        */
  uint64_t waves;        /* waves run (a step with more than K distinct experts has several) */
  uint64_t bytes_paged;  /* host -> device bytes copied for misses                   */
} pmoe_stats;

/* Kernel classes of the per-kernel timers (expert_cache_kernel_times). */
enum {
  PMOE_K_RESIDENCY = 0,  /* residency step (copy stream)                         */
  PMOE_K_GROUP = 1,      /* histogram / scan / permutation (and tile list)       */
  PMOE_K_GATHER = 2,     /* activation row gather (tensor-core path)             */
  PMOE_K_GATEUP = 3,     /* gate/up projection + SiLU*mul                        */
  PMOE_K_DOWN = 4,       /* down projection                                      */
  PMOE_K_COMBINE = 5,    /* top_k-weighted combine                               */
  PMOE_K_PULL = 6,       /* SM-pull page-in (copy stream)                        */
  PMOE_K_COPY = 7,       /* copy-engine page-in: first to last copy of a wave    */
  PMOE_K_DECODE = 8,     /* fused decode kernel: gate/up, SiLU*mul, down (+combine) */
  PMOE_K_CLASSES = 12
};

typedef struct {
  double ms[PMOE_K_CLASSES];          /* summed device time per class (CUDA events) */
  uint64_t launches[PMOE_K_CLASSES];  /* kernel launches per class                  */
  uint64_t copies;                    /* cudaMemcpyAsync page-in copies issued      */
} pmoe_kernel_times;

typedef struct pmoe_cache pmoe_cache;  /* opaque; owned by the library */

/* Library version (major*10000 + minor*100 + patch). */
PMOE_API int pmoe_version(void);

/* Static text for a status code. */
PMOE_API const char* pmoe_status_string(int status);

/* Text of the most recent CUDA error seen by this thread (static storage). */
PMOE_API const char* pmoe_last_error(void);

/* Bytes of one expert in `format` for hidden H and intermediate I (the layouts
 * above), or 0 if the shape is invalid for the format. */
PMOE_API size_t pmoe_expert_bytes(int format, int hidden, int intermediate);

/*
 * moe_router_topk — the router (section "What does Paged Experts actually do?",
 * first paragraph: each token goes to top_k of E experts).
 * For every token t: p = softmax(logits[t]) over all E in fp32; the top_k largest
 * logits are selected, ordered by descending logit, ties to the lower expert id;
 * w[t][r] = p[ids[t][r]] / sum_r' p[ids[t][r']] when renormalize != 0, else
 * p[ids[t][r]].
 *   logits   device, fp32 [T][E]
 *   ids_out  device, int32 [T][top_k]
 *   w_out    device, fp32 [T][top_k]
 * T = 0 enqueues nothing. E in 1..1024, top_k in 1..min(E, 32), else PMOE_EINVAL.
 */
PMOE_API int moe_router_topk(const float* logits, int T, int E, int top_k, int renormalize,
                    int32_t* ids_out, float* w_out, void* stream);

/*
 * moe_router_gemm_topk — the router's projection fused in front of moe_router_topk:
 * logits[t][e] = sum_c x[t][c] * router_weight[e][c] (bf16 inputs, fp32 accumulation in a
 * fixed order), then the selection and weights of moe_router_topk on those logits.
 * The article's layer routes each token from its hidden state (section "What does Paged
 * Experts actually do?", first paragraph); this call takes that hidden state directly.
 *   x              device, bf16 [T][H], 16-byte aligned
 *   router_weight  device, bf16 [E][H] (the gate projection, one row per expert), 16-byte aligned
 *   logits_out     device, fp32 [T][E], or NULL when the logits are not wanted
 *   ids_out        device, int32 [T][top_k]
 *   w_out          device, fp32 [T][top_k]
 * T = 0 enqueues nothing. H a multiple of 8, E in 1..1024, top_k in 1..min(E, 32), else
 * PMOE_EINVAL; an H whose staging does not fit in shared memory gives PMOE_EUNSUPPORTED.
 */
PMOE_API int moe_router_gemm_topk(const void* x, const void* router_weight, int T, int H, int E, int top_k,
                                  int renormalize, float* logits_out, int32_t* ids_out, float* w_out, void* stream);

/*
 * moe_group_by_expert — the grouping in front of the fused MoE (section "What does
 * Paged Experts actually do?": the routed (token, rank) pairs run expert by expert),
 * run by the same kernels moe_paged_forward uses for it. Pair p of a flattened id
 * array (p = t * top_k + r):
 *   counts[e]  pairs with id e;   offs = exclusive scan of counts, offs[E] = valid pairs
 *   perm[j]    the pair at grouped position j: ids ascending, and pairs ascending within
 *              one id (a stable sort by id)
 *   pos[p]     j with perm[j] == p; -1 for an id outside [0, E), which is left out of
 *              the grouping and ORs 1 into *err_dev
 *   ids        device, int32 [P]
 *   counts     device, int32 [E];   offs  device, int32 [E + 1]
 *   perm, pos  device, int32 [P]; perm entries from offs[E] on are left as they were
 *   scratch    device, int32 [scratch_ints] per-chunk histograms, needed when
 *              moe_group_scratch_ints(P, E) > 0 (P above 8192), else may be NULL
 *   err_dev    device int32, or NULL
 * P in 0..2^24 and E in 1..1024, and enough scratch, else PMOE_EINVAL. P = 0 writes
 * zero counts and offs.
 */
PMOE_API int moe_group_by_expert(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offs, int32_t* perm,
                                 int32_t* pos, int32_t* scratch, size_t scratch_ints, int32_t* err_dev,
                                 void* stream);
/* The int32 scratch moe_group_by_expert needs for P pairs over E experts (0 if none). */
PMOE_API size_t moe_group_scratch_ints(int P, int E);

/*
 * expert_cache_create — build the paged-expert state for `num_layers` MoE layers:
 * a pinned host store of all E experts per layer, a device arena of K slots per
 * layer, a device LRU table per layer (all slots empty), a copy stream, events and
 * a forward workspace sized by max_tokens. The descriptor is validated before any
 * CUDA call (PMOE_EINVAL / PMOE_EUNSUPPORTED). Pinned allocation failure (for
 * instance a pinned-memory cap; rollout checklist item 2) returns PMOE_EHOSTALLOC.
 * On success *out owns everything; release it with expert_cache_destroy.
 */
PMOE_API int expert_cache_create(const pmoe_cache_desc* desc, pmoe_cache** out);

/* Release every resource of the cache after synchronising its streams. NULL is a no-op. */
PMOE_API void expert_cache_destroy(pmoe_cache* cache);

/*
 * expert_cache_host_store — the pinned host store of one layer: *host_ptr receives
 * the address of expert 0 and *stride_bytes the distance between experts (at least
 * pmoe_expert_bytes, padded to 4 KiB). The caller may fill it directly; the store
 * stays owned by the cache.
 */
PMOE_API int expert_cache_host_store(pmoe_cache* cache, int layer, void** host_ptr, size_t* stride_bytes);

/* Copy one expert's bytes (host, exactly pmoe_expert_bytes long) into the store.
 * Do not change an expert that is resident without calling expert_cache_reset. */
PMOE_API int expert_cache_load_expert(pmoe_cache* cache, int layer, int expert, const void* bytes, size_t nbytes);

/* Empty one layer's slot table (layer = -1: all layers); statistics are kept.
 * Stream-ordered after the layer's last forward and residency step. */
PMOE_API int expert_cache_reset(pmoe_cache* cache, int layer);

/*
 * expert_cache_ensure_resident — the residency step (TL;DR; section "What does
 * Paged Experts actually do?" item 3; section "What happens with more than one
 * request?"). Given the step's routed ids (device, int32, n_ids = T*top_k) for
 * `layer`: deduplicate, count hits and misses against the layer's table, choose
 * least-recently-used victims (key (last use step, slot); pending experts are
 * never evicted), split the step into waves of at most K experts when more than K
 * distinct experts are routed, and start the page-in of the first wave on the
 * copy stream. The work is ordered after the work already on `stream` (the ids'
 * producer) and after this layer's previous forward. The next moe_paged_forward
 * call for `layer` consumes this staged step and must be given the same ids.
 * In PMOE_PAGEIN_COPY_ENGINE mode the host waits (bounded) for the plan.
 * *waves_out (may be NULL) receives the number of waves (copy-engine mode) or -1
 * (SM-pull mode, where the host does not read the plan).
 */
PMOE_API int expert_cache_ensure_resident(pmoe_cache* cache, int layer, const int32_t* ids, int n_ids,
                                 void* stream, int* waves_out);

/*
 * expert_cache_prefetch — page in a predicted expert set ahead of the layer's forward
 * (the overlap of section "Why is it fast when experts keep crossing PCIe?": the
 * next layer's experts cross the link while the current layer computes; here the
 * set is a prediction, for a model whose next-layer routing is not yet known).
 * ids: device int32 [n_ids], n_ids <= max_tokens * top_k, the predicted experts
 * (repeats allowed). The call runs one residency step for them on `layer` (the
 * same LRU step as for a forward: its hits, misses and waves are counted, and the
 * experts are marked used at that step) and then the page-in of every wave, in
 * order, on the copy stream; nothing is computed. It is ordered after the work on
 * `stream` and after the layer's previous forward; the layer's next residency
 * step, and so its forward, is ordered after this page-in. A staged
 * ensure_resident that no forward consumed is completed first. Experts the
 * prediction got right are hits in the forward that follows; a wrong prediction
 * costs link time and slots, never a different result. Returns PMOE_EINVAL on bad
 * arguments, PMOE_EUNSUPPORTED under stream capture of a copy-engine cache, else
 * as ensure_resident.
 */
PMOE_API int expert_cache_prefetch(pmoe_cache* cache, int layer, const int32_t* ids, int n_ids, void* stream);

/*
 * moe_paged_forward — the fused MoE over the slot table (section "What does Paged
 * Experts actually do?" item 3; section "Can paging change the model's outputs?").
 *   x         device, bf16 [T][H]
 *   ids, w    device, int32 / fp32 [T][top_k] (from moe_router_topk)
 *   residual  device, bf16 [T][H] or NULL
 *   y         device, bf16 [T][H]; may alias residual, must not alias x
 * y[t] = bf16( residual[t] + sum_{r=0}^{top_k-1} w[t][r] * o_{ids[t][r]}(x[t]) ),
 * o_e(x) = (silu(x W_g^T) * (x W_u^T)) W_d^T; the intermediate is rounded to bf16,
 * the rank partials are summed in fp32 in rank order, then rounded once.
 * If no ensure_resident was staged for `layer`, the call runs it first. Waves run
 * in order, each after its own page-in. T in 0..max_tokens. Calls on one cache
 * share its workspace: issue them on one stream (or serialise them).
 * CUDA graphs: with PMOE_PAGEIN_SM_PULL no call waits on the host, so ensure_resident,
 * moe_paged_forward and moe_paged_stack_forward can be recorded by stream capture and
 * replayed (the single-wave decode step of section "What happens with more than one
 * request?"); a copy-engine cache returns PMOE_EUNSUPPORTED under capture. Synchronise
 * the replay stream before reading statistics or the slot table.
 */
PMOE_API int moe_paged_forward(pmoe_cache* cache, int layer, const void* x, int T, const int32_t* ids,
                      const float* w, const void* residual, void* y, void* stream);

/*
 * moe_paged_stack_forward — all num_layers MoE layers of the cache in sequence, attention
 * omitted: h_0 = x, h_{l+1} = h_l + moe_l(h_l) (the residual add of a decoder block; a
 * token at batch 1 activates layers x top_k experts, article "Running an MoE Model
 * Larger Than Your VRAM", section "Why is it fast when experts keep crossing PCIe?").
 * Each layer's residency step and page-in run on the cache's side streams while the
 * previous layer computes on `stream` (prefetch overlap; the copy/compute overlap
 * t ~ max(t_read, t_H2D)).
 *   x     device bf16 [T][H] (h_0)             y     device bf16 [T][H] (h_L)
 *   ids   device int32 [L][T][top_k]           w     device fp32 [L][T][top_k]
 *   work  device bf16 [T][H] scratch for the alternating activations (may be NULL if L == 1)
 * x, y and work must not overlap. The ids of every layer must be ready in stream order
 * at the call. Results are those of L moe_paged_forward calls with residual = input.
 */
PMOE_API int moe_paged_stack_forward(pmoe_cache* cache, const void* x, int T, const int32_t* ids, const float* w,
                                     void* y, void* work, void* stream);

/* Counters of one layer (layer = -1: summed over layers). Synchronises the cache's
 * streams; returns PMOE_EDEVICE if a kernel recorded an error. */
PMOE_API int expert_cache_stats(pmoe_cache* cache, int layer, pmoe_stats* out);

/* The layer's table after all enqueued work: expert_in_slot[K] (-1 = empty) and
 * last_use[K] (step index, -1 = never), both host int32 arrays (last_use may be
 * NULL). Synchronises the cache's streams. */
PMOE_API int expert_cache_slot_table(pmoe_cache* cache, int layer, int32_t* expert_in_slot, int32_t* last_use);

/* Copy the bytes now held in one slot (host buffer of pmoe_expert_bytes) — the
 * independence check of section "Can paging change the model's outputs?" compares
 * them with the store's bytes of the expert the table says the slot holds. */
PMOE_API int expert_cache_read_slot(pmoe_cache* cache, int layer, int slot, void* host_out, size_t nbytes);

/*
 * expert_cache_set_timing — when enable != 0, every kernel the cache launches is
 * bracketed by CUDA events on the stream it runs on, and launches are counted
 * (measurement support; timing adds two event records per launch). Resets the
 * accumulated times.
 */
PMOE_API int expert_cache_set_timing(pmoe_cache* cache, int enable);

/* Accumulated per-class device times and launch counts since timing was enabled.
 * Synchronises the cache's streams. */
PMOE_API int expert_cache_kernel_times(pmoe_cache* cache, pmoe_kernel_times* out);

/*
 * moe_decode_forward_noalloc — the decode MoE (T <= 8 tokens) over experts that are
 * already in device memory, using no device allocation of any kind. The paper has
 * no counterpart of this call; it exists for callers that cannot call cudaMalloc:
 * code running inside another framework's memory pool or allocator hooks, real-time
 * loops that must never enter the driver's allocator, and embedders whose device
 * memory is budgeted up front. For the same tokens it computes the layer that
 * moe_paged_forward computes when every routed expert is resident (same arithmetic
 * order per pair, through the library's two-kernel GEMV decode); the outputs agree
 * within the layer tolerances (bf16 and int4: relative Frobenius 1e-2; block FP8:
 * 3e-2), not necessarily bit for bit.
 *   experts   device: n_slots expert slots of pmoe_expert_bytes(format, H, I) bytes
 *             each, `stride` bytes apart (stride a multiple of 16); 16-byte aligned
 *   n_slots   slots in `experts`; at least E when slot_of is NULL
 *   slot_of   device int32 [E]: slot of each expert in `experts`, or NULL when expert
 *             e sits in slot e. A routed expert with slot -1 contributes nothing; any
 *             other slot outside [0, n_slots) is an error: the expert is skipped and
 *             error bit 4 is set
 *   x, residual, y, ids, w: as in moe_paged_forward (residual may be NULL); x,
 *             residual and y 16-byte aligned, ids and w 4-byte aligned
 *   err_out   device int32 or NULL: after the call's kernels (stream-ordered) it
 *             receives the call's device error bits: 0 = none, 1 = an id outside
 *             [0, E) was skipped, 4 = an expert's slot was outside [0, n_slots)
 * Limits: E <= 1024, T <= 8, T * top_k <= 64, and the intermediates must fit the
 * library's fixed 2 MiB static device scratch ((P*(2I + 4H)) bytes plus small
 * tables, P = T * top_k); larger requests, misaligned pointers and bad arguments
 * return PMOE_EINVAL with nothing enqueued.
 * The first call on each device (with that device current) looks up the scratch
 * address once; with lazy module loading that also loads the library's device code
 * holding the scratch, so this first call may allocate inside the driver: make it
 * during warm-up, before any stream capture. All calls share the one scratch array,
 * which keeps the last call's contents: calls that overlap on the GPU race on it, so
 * serialise them (one stream). Nothing is synchronised.
 */
PMOE_API int moe_decode_forward_noalloc(const void* experts, size_t stride, int n_slots, const int32_t* slot_of,
                                        int E, int top_k, int H, int I, int format, const void* x, int T,
                                        const int32_t* ids, const float* w, const void* residual, void* y,
                                        int32_t* err_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDMOE_H */
