// Decode path (T <= 8 tokens): one fused, weight-streaming kernel per wave.
//
// At decode batch sizes the MoE layer reads every routed expert's weights once and
// does ~1 FLOP per byte, so it is bound by HBM bandwidth (the decode-is-memory-bound
// discussion in "SGLang serving optimisation"; "Running an MoE Model Larger Than Your
// VRAM", section "Why is it fast when experts keep crossing PCIe?"). One persistent
// CTA per SM (cooperative launch, so all CTAs are resident) walks a schedule of
// chunks. A producer thread streams each chunk's weight rows into a byte ring in
// shared memory (cp.async.bulk, completion on mbarriers), a fetcher warp supplies the
// intermediate rows that down chunks need, and two groups of four consumer warps take
// the chunks in turn.
//
//   gate/up  Every expert's I row pairs (gate row j with up row j) are cut into one
//            part per CTA; CTA b takes part (b + e) mod G of the wave's e-th expert,
//            so each CTA touches every expert and the per-CTA totals differ by at
//            most one row pair. The consumers reduce the rows against the tokens' x
//            (in shared memory) and store h[pair][j] = silu(g) * u (bf16) as a 64-bit
//            word whose upper 48 bits carry the plan's tag.
//   down     CTA b owns output rows [b*H/G, (b+1)*H/G) of every expert. The W_d rows
//            stream like any other chunk; the fetcher polls the expert's h words until
//            each carries this launch's tag and stores the bf16 values next to the
//            rows. The tag makes every word self-validating, so no counter, fence or
//            grid barrier sits between the two halves, and the consumers never wait on
//            a global-memory round trip (under full HBM load one takes microseconds).
//   order    gate/up of expert e is followed, kDfLag experts later, by the down chunk
//            of expert e: by then every CTA has finished e's gate/up, so the fetch
//            overlaps the streaming of later experts.
//   combine  (single-wave steps) the CTA holds o[pair][n] for every pair of its rows,
//            so it writes y[t][n] = res + sum_r w[t,r] o[(t,r)][n] in rank order;
//            otherwise o_part is written and the combine kernel runs after the last
//            wave (same arithmetic and order, so the bits agree).
// The token -> expert grouping (stable: expert ascending, pair index ascending) is
// computed by every CTA from the ids; CTA 0 also writes pos/perm for the combine.
// Per-pair dot products have a fixed order (lane-strided 16-byte chunks, then an
// xor-shuffle tree), independent of slot, wave, grid and of how many tokens share the
// expert. Every wait is bounded; on expiry the kernel records an error and stops.
#include "decode_ring.cuh"

#include <algorithm>
#include <stdlib.h>

namespace pmoe {
namespace {

using namespace dec;


#ifdef PMOE_TRACE
// Debug builds only: per-CTA %globaltimer stamps of the last launch.
__device__ unsigned long long g_df_trace[1024][8];
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
#define DF_TRACE(slot) \
  do {                 \
    g_df_trace[blockIdx.x][slot] = gtimer(); \
  } while (0)
// per chunk: producer issue, data landed (consumer), h rows ready (down chunks), done
__device__ unsigned long long g_df_chunk[1024][256][4];
#define DF_CHUNK(k, slot)                                   \
  do {                                                      \
    if ((k) < 256) g_df_chunk[blockIdx.x][(k)][(slot)] = gtimer(); \
  } while (0)
#else
#define DF_CHUNK(k, slot) \
  do {                    \
  } while (0)
#define DF_TRACE(slot) \
  do {                 \
  } while (0)
#endif

struct DfArgs {
  const __nv_bfloat16* x;
  const int32_t* ids;
  const float* w;
  const __nv_bfloat16* residual;
  __nv_bfloat16* y;
  int T, top_k, H, I, E, wave, sub, fuse_combine;
  int ring_bytes;  // byte ring for the weight chunks
  int cg, cd;      // chunks per gate/up part and per down part
  const int32_t* plan;
  Workspace ws;
  uint8_t* arena;
  const uint8_t* store;  // the layer's mapped host store (pull != 0)
  int pull;              // page the wave's missing experts in during this launch
  size_t stride;
  ExpertLayout lay;
  int32_t* err;
};


template <int FMT, int NCH1, int NCH2>
__global__ void __launch_bounds__(kDfThreads, 1) decode_fused_kernel(const DfArgs a) {
  constexpr int EPC = Fmt<FMT>::EPC;
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ int4 s_we[kDfMaxPairs];  // per wave expert: (expert, slot, first grouped pair, end)
  __shared__ int2 s_wl[kDfMaxPairs];  // the wave's (expert, slot) list
  __shared__ int s_tok[kDfMaxPairs];  // token of each grouped pair
  __shared__ int s_pos[kDfMaxPairs];  // grouped position of each pair (t*k + r), -1 if invalid
  __shared__ int s_ids[kDfMaxPairs];
  __shared__ float s_w[kDfMaxPairs];  // routing weights (combine)
  __shared__ int s_hdr[6];
  __shared__ unsigned s_off[kDfSlots];  // ring offset of each slot's chunk
  __shared__ __align__(8) uint64_t s_full[kDfSlots];  // the chunk's weight bytes landed
  __shared__ __align__(8) uint64_t s_hrdy[kDfSlots];  // the fetcher has passed the chunk (down: h copied)
  __shared__ __align__(8) uint64_t s_empty[kDfSlots];
  __shared__ int s_abort;
  __shared__ int s_placed;  // chunks placed in the ring so far
  __shared__ int s_pulled;  // chunks whose bytes this CTA has paged in (missing experts)

  const unsigned R = (unsigned)a.ring_bytes;
  uint8_t* ring = dsm;
  uint4* x_s = reinterpret_cast<uint4*>(ring + R);
  float* o_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(x_s) + (size_t)a.T * a.H * 2);
  __nv_bfloat16* res_s = reinterpret_cast<__nv_bfloat16*>(o_s + kDfMaxPairs * kDfMaxRows);
  int4* chunks = reinterpret_cast<int4*>(res_s + kDfMaxTokens * kDfMaxRows);
  volatile int* abort_flag = &s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) DF_TRACE(0);
  const PlanLayout L{a.E};
  const int P = a.T * a.top_k;
  // The producer thread initialises the barriers and, for a launch that starts at wave
  // 0, at once streams the first gate/up chunks of the wave's leading resident experts:
  // their place in the schedule, their rows and their ring offsets follow from the plan
  // header and slot list alone, so the copies are in flight while the block groups the
  // pairs and builds the chunk list. The main loop carries on after them.
  int early_n = 0;
  unsigned early_head = 0;
  if (warp == kDfConsumerWarps && lane == 0) {
    for (int s = 0; s < kDfSlots; ++s) {
      mb_init(&s_full[s], 1);
      mb_init(&s_hrdy[s], 1);
      mb_init(&s_empty[s], kDfConsumerWarps);
    }
    s_abort = 0;
    s_pulled = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    pdl_wait();  // launched behind the residency step: its plan is complete from here on
    const int nw = a.plan[kPlanWaves], ws0 = a.plan[L.wave_start() + a.wave];
    const int ws1 = a.plan[L.wave_start() + a.wave + 1];
    static_assert(kDfLag == 3, "the entry-time slot reads below cover the first three experts");
    const int sl0 = a.plan[L.wave_slot()], sl1 = a.E > 1 ? a.plan[L.wave_slot() + 1] : -1;
    const int sl2 = a.E > 2 ? a.plan[L.wave_slot() + 2] : -1;
    const int hits0 = a.plan[L.wave_hits() + a.wave];  // the wave's experts resident before this launch
    const int D0 = ws1 - ws0;
    // (not when this launch pages experts in: the block barrier below would hold the
    // pager warps back while the producer issues, and the host link is the longer path)
    if ((a.pull == 0 || hits0 >= D0) && a.wave < nw && ws0 == 0 && a.sub == 0 && D0 > 0 &&
        D0 * (a.cg + a.cd) <= kDfMaxChunks) {
      const int nh = D0;  // (no page-in: every wave expert is resident)
      const DfSched sc0{D0, (int)gridDim.x, (int)blockIdx.x, a.I, a.H, a.cg, a.cd};
      const size_t rbg0 = (size_t)a.H * Fmt<FMT>::BPE2 / 2;
      const int rsg0 = row_scale_bytes(FMT, a.H);
      const unsigned R0 = (unsigned)a.ring_bytes;
      for (int q = 0; q < min(kDfLag, D0) * a.cg && q < kDfSlots; ++q) {
        const int4 cq = sched_entry(q, sc0);  // a gate/up chunk of wave expert q / cg
        const int slot = cq.y == 0 ? sl0 : cq.y == 1 ? sl1 : sl2;
        if (cq.y >= nh || slot < 0) break;  // (an expert paged in by this launch waits for the pagers)
        const unsigned wbytes = (unsigned)(2 * (size_t)cq.w * rbg0);
        ScaleSpan sp0{0, 0, 0}, sp1{0, 0, 0};
        if constexpr (FMT != PMOE_BF16) {
          if (cq.w > 0) {
            sp0 = scale_span<FMT>(a.lay.gu_s, rsg0, cq.z, cq.w);
            sp1 = scale_span<FMT>(a.lay.gu_s, rsg0, a.I + cq.z, cq.w);
          }
        }
        const unsigned need = (wbytes + sp0.bytes + sp1.bytes + 127u) & ~127u;
        if (early_head + need > R0) break;
        s_off[q] = early_head;
        uint64_t* fb = &s_full[q];
        if (wbytes == 0) {
          mb_arrive(fb);
        } else {
          const uint8_t* ex = a.arena + (size_t)slot * a.stride;
          uint8_t* dst = ring + early_head;
          mb_expect(fb, wbytes + sp0.bytes + sp1.bytes);
          bulk_g2s(dst, ex + a.lay.gu_w + (size_t)cq.z * rbg0, wbytes / 2, fb);
          bulk_g2s(dst + wbytes / 2, ex + a.lay.gu_w + (size_t)(a.I + cq.z) * rbg0, wbytes / 2, fb);
          if constexpr (FMT != PMOE_BF16) {
            if (sp0.bytes != 0) bulk_g2s(dst + wbytes, ex + sp0.src, sp0.bytes, fb);
            if (sp1.bytes != 0) bulk_g2s(dst + wbytes + sp0.bytes, ex + sp1.src, sp1.bytes, fb);
          }
        }
        DF_CHUNK(q, 0);
        early_head += need;
        ++early_n;
      }
    }
    s_placed = early_n;  // (published by the block barrier below)
  }
  // Launched behind the residency step (programmatic serialization), the CTAs start
  // while it runs; nothing that kernel or the ones before it write (plan, ids, weights,
  // x, the slot arena) is read before this wait. The kernel never triggers its own
  // dependents early: whatever follows it waits for its end.
  pdl_wait();
  const int r_lo = (int)((long long)a.H * blockIdx.x / gridDim.x);
  const int r_hi = (int)((long long)a.H * (blockIdx.x + 1) / gridDim.x);
  // One round of independent loads: the plan words, the ids, the first wave's list (read
  // on speculation: wave 0 starts at list index 0), the tokens' x, the routing weights and
  // the residual rows this CTA combines.
  const int nspec = min(P, a.E);
  if (tid < P) {
    s_ids[tid] = a.ids[tid];
  } else if (tid >= 64 && tid < 64 + nspec) {
    s_wl[tid - 64].x = a.plan[L.wave_exp() + tid - 64];
  } else if (tid >= 128 && tid < 128 + nspec) {
    s_wl[tid - 128].y = a.plan[L.wave_slot() + tid - 128];
  } else if (tid >= 192 && tid < 198) {
    const int q = tid - 192;
    const int at = q == 0   ? (int)kPlanWaves
                   : q == 1 ? L.wave_start() + a.wave
                   : q == 2 ? L.wave_start() + a.wave + 1
                   : q == 3 ? L.wave_hits() + a.wave
                   : q == 4 ? (int)kPlanEpochLo
                            : (int)kPlanEpochHi;
    s_hdr[q] = a.plan[at];
  } else if (tid >= 256 && tid < 256 + P) {
    s_w[tid - 256] = a.w[tid - 256];
  }
  for (int i = tid; i < a.T * (a.H / 8); i += kDfThreads) x_s[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
  if (a.residual != nullptr && a.fuse_combine != 0 && r_hi > r_lo) {
    const int rows = r_hi - r_lo;
    for (int i = tid; i < a.T * rows; i += kDfThreads) {
      const int t = i / rows;
      res_s[t * kDfMaxRows + (i - t * rows)] = a.residual[(size_t)t * a.H + r_lo + (i - t * rows)];
    }
  }
  __syncthreads();
  if (tid == 0) DF_TRACE(7);
  const int n_waves = s_hdr[0];
  if (a.wave >= n_waves) return;
  int w0 = s_hdr[1], w1 = s_hdr[2];
  if (a.sub == 1) w1 = w0 + s_hdr[3];
  else if (a.sub == 2) w0 += s_hdr[3];
  const int D = w1 - w0;
  // wave experts [n_hits, D) are paged in by this launch (the list puts resident ones first)
  const int n_hits = (a.pull != 0 && a.sub == 0) ? min(s_hdr[3], D) : D;
  if (w0 != 0) {  // not the speculated list: load this wave's part of it
    if (tid < D) s_wl[tid] = make_int2(a.plan[L.wave_exp() + w0 + tid], a.plan[L.wave_slot() + w0 + tid]);
    __syncthreads();
  }
  // tag of this launch's h words: unique per (plan epoch, wave, part of the wave)
  const unsigned long long epoch = ((unsigned long long)(uint32_t)s_hdr[5] << 32) | (uint32_t)s_hdr[4];
  const unsigned long long tag = ((epoch << 12) | ((unsigned long long)a.wave << 2) | (unsigned)a.sub) & kTagMask;

  // grouping: stable by expert id, then pair index
  if (tid < P) {
    const int p = tid, id = s_ids[p];
    int pos = -1;
    if (id >= 0 && id < a.E) {
      pos = 0;
      for (int q = 0; q < P; ++q) {
        const int o = s_ids[q];
        pos += (o >= 0 && o < a.E && (o < id || (o == id && q < p))) ? 1 : 0;
      }
      s_tok[pos] = p / a.top_k;
    }
    s_pos[p] = pos;
    if (blockIdx.x == 0 && a.sub != 2) {
      a.ws.pos[p] = pos;
      if (pos >= 0) a.ws.perm[pos] = p;
    }
  }
  if (tid < D) {
    const int2 es = s_wl[tid];
    int lo = 0, cnt = 0;
    for (int q = 0; q < P; ++q) {
      const int o = s_ids[q];
      lo += (o >= 0 && o < es.x) ? 1 : 0;
      cnt += (o == es.x) ? 1 : 0;
    }
    s_we[tid] = make_int4(es.x, es.y, lo, lo + cnt);
  }
  const DfSched sc{D, (int)gridDim.x, (int)blockIdx.x, a.I, a.H, a.cg, a.cd};
  const int n_chunks = D * (a.cg + a.cd);
  if (n_chunks > kDfMaxChunks) {  // excluded on the host; never write past the list
    if (tid == 0) atomicOr(a.err, kErrPlanOverflow);
    return;
  }
  // chunk list; .x = kind | (rows of all earlier chunks) << 2, which deals each chunk's
  // rows to the consumer warps round-robin in one sequence over the whole list
  __shared__ int s_scan[kDfThreads / 32];
  {
    int4 e0 = make_int4(0, 0, 0, 0), e1 = make_int4(0, 0, 0, 0);
    if (tid < n_chunks) e0 = sched_entry(tid, sc);
    if (tid + kDfThreads < n_chunks) e1 = sched_entry(tid + kDfThreads, sc);
    // chunks tid and tid + kDfThreads (n_chunks <= kDfMaxChunks < 2 * kDfThreads)
    const int c0 = e0.w, c1 = e1.w;
    int v = c0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) s_scan[warp] = v;
    __syncthreads();
    int before = 0, total0 = 0;
    for (int i = 0; i < kDfThreads / 32; ++i) {
      if (i < warp) before += s_scan[i];
      total0 += s_scan[i];
    }
    const int base0 = before + v - c0;
    __syncthreads();
    int v1 = c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v1, o);
      if (lane >= o) v1 += y;
    }
    if (lane == 31) s_scan[warp] = v1;
    __syncthreads();
    int before1 = 0;
    for (int i = 0; i < warp; ++i) before1 += s_scan[i];
    const int base1 = total0 + before1 + v1 - c1;
    if (tid < n_chunks) chunks[tid] = make_int4(e0.x | (base0 << 2), e0.y, e0.z, e0.w);
    if (tid + kDfThreads < n_chunks) chunks[tid + kDfThreads] = make_int4(e1.x | (base1 << 2), e1.y, e1.z, e1.w);
  }
  __syncthreads();
  if (tid == 0) DF_TRACE(1);
  const size_t rbg = (size_t)a.H * Fmt<FMT>::BPE2 / 2;  // one gate (or up) row
  const size_t rbd = (size_t)a.I * Fmt<FMT>::BPE2 / 2;  // one down row
  const int rsg = row_scale_bytes(FMT, a.H), rsd = row_scale_bytes(FMT, a.I);  // one scale row of gate/up, of down

  if (warp == kDfConsumerWarps) {
    // ---------------- producer: lane 0 places every chunk in the byte ring as soon as
    // its slot and its bytes are free (chunks are released in order) and issues its
    // bulk copies. A down chunk also reserves room for the expert's h rows, which the
    // fetcher warp fills.
    if (lane == 0) {
      unsigned head = early_head;  // the chunks streamed at entry occupy [0, early_head)
      int tail = 0, k = early_n;
      for (; k < n_chunks; ++k) {
        const int4 cd = chunks[k];
        const int kind = cd.x & 3;
        const int4 we = s_we[cd.y];
        const unsigned wbytes = kind == 1 ? (unsigned)(2 * (size_t)cd.w * rbg) : (unsigned)((size_t)cd.w * rbd);
        const unsigned hbytes = (kind == 2 && cd.w > 0) ? (unsigned)(min(we.w - we.z, a.T) * a.I * 2) : 0u;
        ScaleSpan sp0{0, 0, 0}, sp1{0, 0, 0};
        if constexpr (FMT != PMOE_BF16) {
          if (cd.w > 0) {
            if (kind == 1) {
              sp0 = scale_span<FMT>(a.lay.gu_s, rsg, cd.z, cd.w);
              sp1 = scale_span<FMT>(a.lay.gu_s, rsg, a.I + cd.z, cd.w);
            } else {
              sp0 = scale_span<FMT>(a.lay.d_s, rsd, cd.z, cd.w);
            }
          }
        }
        const unsigned need = (wbytes + hbytes + sp0.bytes + sp1.bytes + 127u) & ~127u;
        int off = -1;
        long long t0 = -1;
        while (true) {
          // place with what is known to be free; retire the oldest chunk only when
          // that fails (the wait sleeps in the barrier)
          if (k - tail < kDfSlots) {
            off = ring_place(head, s_off[tail % kDfSlots], tail == k, need, R);
            if (off >= 0) break;
          }
          if (mb_try(&s_empty[tail % kDfSlots], (uint32_t)((tail / kDfSlots) & 1))) {
            ++tail;
            continue;
          }
          if (*abort_flag) break;
          if (t0 < 0) {
            t0 = clock64();
          } else if (clock64() - t0 > kDfWaitLimit) {
            *abort_flag = 1;
            atomicOr(a.err, kErrDecodeTimeout);
            break;
          }
        }
        if (off < 0) break;
        const int s = k % kDfSlots;
        s_off[s] = (unsigned)off;
        head = (unsigned)off + need;
        uint64_t* fb = &s_full[s];
        if (wbytes != 0 && cd.y >= n_hits) {
          // an expert this launch pages in: wait until this CTA's pager has written the
          // chunk's bytes into the slot
          long long t1 = -1;
          while (ld_acquire_shared(&s_pulled) <= k && !*abort_flag) {
            if (t1 < 0) {
              t1 = clock64();
            } else if (clock64() - t1 > kDfWaitLimit) {
              *abort_flag = 1;
              atomicOr(a.err, kErrDecodeTimeout);
            }
            __nanosleep(128);
          }
          if (*abort_flag) break;
        }
        DF_CHUNK(k, 0);
        if (wbytes == 0) {
          mb_arrive(fb);
        } else {
          const uint8_t* ex = a.arena + (size_t)we.y * a.stride;
          uint8_t* dst = ring + off;
          mb_expect(fb, wbytes + sp0.bytes + sp1.bytes);
          if (kind == 1) {
            const uint32_t half = wbytes / 2;
            bulk_g2s(dst, ex + a.lay.gu_w + (size_t)cd.z * rbg, half, fb);
            bulk_g2s(dst + half, ex + a.lay.gu_w + (size_t)(a.I + cd.z) * rbg, half, fb);
          } else {
            bulk_g2s(dst, ex + a.lay.d_w + (size_t)cd.z * rbd, wbytes, fb);
          }
          if constexpr (FMT != PMOE_BF16) {
            // the scale rows go after the weights (and after a down chunk's h rows)
            uint8_t* sdst = dst + wbytes + hbytes;
            if (sp0.bytes != 0) bulk_g2s(sdst, ex + sp0.src, sp0.bytes, fb);
            if (sp1.bytes != 0) bulk_g2s(sdst + sp0.bytes, ex + sp1.src, sp1.bytes, fb);
          }
        }
        asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(su32(&s_placed)), "r"(k + 1) : "memory");
      }
      if (*abort_flag) {
        // stopped early: let the copies already issued land before the CTA exits
        const long long t1 = clock64();
        for (int q = max(0, k - kDfSlots); q < k; ++q)
          while (!mb_test(&s_full[q % kDfSlots], (uint32_t)((q / kDfSlots) & 1)) && clock64() - t1 < kDfWaitLimit) {
          }
      }
    }
  } else if (warp == kDfConsumerWarps + 1) {
    // ---------------- h fetcher: walks the chunks in order behind the producer. For a
    // down chunk it polls the expert's h words (written by every CTA's gate/up chunks)
    // until each carries this launch's tag, stores the bf16 values after the chunk's W_d
    // rows and signals s_hrdy; other chunks are passed straight through.
    for (int k = 0; k < n_chunks; ++k) {
      long long t0 = -1;
      bool ok = true;
      while (ld_acquire_shared(&s_placed) <= k) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (t0 < 0) {
          t0 = clock64();
        } else if (clock64() - t0 > kDfWaitLimit) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(a.err, kErrDecodeTimeout);
          }
          ok = false;
          break;
        }
        __nanosleep(256);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      const int s = k % kDfSlots;
      const int4 cd = chunks[k];
      if ((cd.x & 3) == 2 && cd.w > 0) {
        const int4 we = s_we[cd.y];
        const int hb = min(we.w - we.z, a.T);
        uint16_t* hdst = reinterpret_cast<uint16_t*>(ring + s_off[s] + (size_t)cd.w * rbd);
        const int n = hb * a.I;  // even
        const unsigned long long* src = a.ws.hq + (size_t)we.z * a.I;
        int bad = 0;
        for (int i0 = 2 * lane; i0 < n && !bad; i0 += 64 * 16) {
          // up to 16 16-byte loads per lane in flight; the stale ones are re-read
          // together, so each polling round costs one round trip
          ulonglong2 v[16];
          unsigned pend = 0;
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (i0 + u * 64 < n) {
              v[u] = ld_relaxed_u64x2(src + i0 + u * 64);
              pend |= 1u << u;
            }
          long long t1 = -1;
          while (true) {
#pragma unroll
            for (int u = 0; u < 16; ++u)
              if ((pend >> u) & 1u) {
                if ((v[u].x >> 16) == tag && (v[u].y >> 16) == tag) {
                  *reinterpret_cast<uint32_t*>(hdst + i0 + u * 64) =
                      (uint32_t)(v[u].x & 0xffffu) | ((uint32_t)(v[u].y & 0xffffu) << 16);
                  pend &= ~(1u << u);
                }
              }
            if (pend == 0) break;
            if (*abort_flag) {
              bad = 1;
              break;
            }
            if (t1 < 0) {
              t1 = clock64();
            } else if (clock64() - t1 > kDfWaitLimit) {
              *abort_flag = 1;
              atomicOr(a.err, kErrDecodeTimeout);
              bad = 1;
              break;
            }
            __nanosleep(256);
#pragma unroll
            for (int u = 0; u < 16; ++u)
              if ((pend >> u) & 1u) v[u] = ld_relaxed_u64x2(src + i0 + u * 64);
          }
        }
        if (__any_sync(0xffffffffu, bad)) break;
        // these generic stores share the ring with later bulk copies (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) DF_CHUNK(k, 2);
      }
      __syncwarp();
      if (lane == 0) mb_arrive(&s_hrdy[s]);
    }
  } else if (warp >= kDfConsumerWarps + 2) {
    // ---------------- pagers: for every chunk of an expert this launch pages in, copy the
    // bytes the chunk reads (its weight rows and the scale rows they use) from the mapped
    // host store into the expert's slot, in schedule order, then publish the progress.
    // Every CTA copies what its own chunks read; together they fill the slot.
    if (a.pull != 0) {
      const int vl = tid - (kDfConsumerWarps + 2) * 32, nl = kDfPagerWarps * 32;
      const int hb = a.H / 128, ib = a.I / 128;
      for (int k = 0; k < n_chunks; ++k) {
        const int4 cd = chunks[k];
        if (cd.y < n_hits || cd.w == 0) continue;
        if (pagers_any(*abort_flag)) break;  // every pager warp sees the same answer
        const int4 we = s_we[cd.y];
        const uint8_t* src = a.store + (size_t)we.x * a.stride;
        uint8_t* dst = a.arena + (size_t)we.y * a.stride;
        const int z = cd.z, n = cd.w;
        // NVFP4: the matrix's 16-byte tensor-scale header (just before its block scales),
        // loaded first so that its host-link round trip overlaps the rows' and stored last
        uint32_t hdr = 0;
        const size_t hdr_off = ((cd.x & 3) == 1 ? a.lay.gu_s : a.lay.d_s) - 16;
        if constexpr (FMT == PMOE_NVFP4)
          if (vl < 4) hdr = *reinterpret_cast<const uint32_t*>(src + hdr_off + 4 * vl);
        if ((cd.x & 3) == 1) {
          lanes_copy16x2(src, dst, a.lay.gu_w + (size_t)z * rbg, (size_t)n * rbg, a.lay.gu_w + (size_t)(a.I + z) * rbg,
                         (size_t)n * rbg, vl, nl);
          if constexpr (FMT == PMOE_FP8_BLOCK128) {
            const size_t row = 4 * (size_t)hb;  // one block row of scales
            lanes_copy4x2(src, dst, a.lay.gu_s + (size_t)(z >> 7) * row,
                          (size_t)(((z + n - 1) >> 7) - (z >> 7) + 1) * row, a.lay.gu_s + (size_t)((a.I + z) >> 7) * row,
                          (size_t)(((a.I + z + n - 1) >> 7) - ((a.I + z) >> 7) + 1) * row, vl, nl);
          } else if constexpr (FMT == PMOE_INT4_GPTQ_G128 || FMT == PMOE_MXFP4 || FMT == PMOE_NVFP4) {
            // one row's scale bytes: (s, z) pairs, E8M0 per 32 inputs, or e4m3 per 16
            const size_t row = (size_t)row_scale_bytes(FMT, a.H);
            lanes_copy4x2(src, dst, a.lay.gu_s + (size_t)z * row, (size_t)n * row, a.lay.gu_s + (size_t)(a.I + z) * row,
                          (size_t)n * row, vl, nl);
          }
        } else {
          lanes_copy16x2(src, dst, a.lay.d_w + (size_t)z * rbd, (size_t)n * rbd, 0, 0, vl, nl);
          if constexpr (FMT == PMOE_FP8_BLOCK128) {
            const size_t row = 4 * (size_t)ib;
            lanes_copy4x2(src, dst, a.lay.d_s + (size_t)(z >> 7) * row,
                          (size_t)(((z + n - 1) >> 7) - (z >> 7) + 1) * row, 0, 0, vl, nl);
          } else if constexpr (FMT == PMOE_INT4_GPTQ_G128 || FMT == PMOE_MXFP4 || FMT == PMOE_NVFP4) {
            const size_t row = (size_t)row_scale_bytes(FMT, a.I);
            lanes_copy4x2(src, dst, a.lay.d_s + (size_t)z * row, (size_t)n * row, 0, 0, vl, nl);
          }
        }
        if constexpr (FMT == PMOE_NVFP4)
          if (vl < 4) *reinterpret_cast<uint32_t*>(dst + hdr_off + 4 * vl) = hdr;
        // the stores (generic proxy) are read next by bulk copies (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        pagers_sync();
        if (vl == 0) asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(su32(&s_pulled)), "r"(k + 1) : "memory");
      }
    }
  } else {
    // ---------------- consumers (warps 0 .. kDfConsumerWarps-1): every warp walks every
    // chunk; the rows of the whole list are dealt to the warps round-robin (row i of the
    // list goes to warp i mod kDfConsumerWarps), so a warp holds about one row of a chunk
    // and moves on to the next chunk at once. Each warp waits on the chunk's barriers
    // itself and releases it (the empty barrier counts one arrival per warp).
    const int nv = a.H / 8;
    const int nch1 = (int)(rbg / 16), nch2 = (int)(rbd / 16);
    const bool fuse = a.fuse_combine != 0 && a.sub == 0 && n_waves == 1;
    bool first_down = true;
    for (int k = 0; k < n_chunks; ++k) {
      const int s = k % kDfSlots;
      const int4 cd = chunks[k];
      const int kind = cd.x & 3;
      const int first = ((warp - (cd.x >> 2)) % kDfConsumerWarps + kDfConsumerWarps) % kDfConsumerWarps;  // this warp's first row
      const uint32_t par = (uint32_t)((k / kDfSlots) & 1);
      // every chunk's s_hrdy phase is waited for (not only down chunks'), so that a warp
      // never waits on a phase two ahead of the barrier's (parity would alias)
      bool got = mb_wait(&s_full[s], par, abort_flag, a.err);
      if (got) got = mb_wait(&s_hrdy[s], par, abort_flag, a.err);
      if (!__all_sync(0xffffffffu, got)) break;
      if (k == 0 && lane == 0 && warp == 0) DF_TRACE(2);
      if (warp == 0 && lane == 0) DF_CHUNK(k, 1);
      const int4 we = s_we[cd.y];
      const uint8_t* st = ring + s_off[s];
      bool ok = true;
      // NVFP4: the chunk's matrix's tensor scale, in the 16-byte header before its block
      // scales in the slot (an expert this launch pages in: written by this CTA's pagers
      // before the chunk's progress, which the producer acquired before its copies)
      float tsc = 1.f;
      if constexpr (FMT == PMOE_NVFP4) {
        if (cd.w > 0) {
          const uint8_t* hdr = a.arena + (size_t)we.y * a.stride + (kind == 1 ? a.lay.gu_s : a.lay.d_s) - 16;
          asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(tsc) : "l"(hdr));
        }
      }
      if (kind == 1) {
        if (warp == 0 && lane == 0) DF_TRACE(6);  // (the last write is the last gate/up chunk)
        for (int rp = first; rp < cd.w; rp += kDfConsumerWarps) {
          const uint4* grow = reinterpret_cast<const uint4*>(st + (size_t)rp * rbg);
          const uint4* urow = reinterpret_cast<const uint4*>(st + (size_t)(cd.w + rp) * rbg);
          uint4 gw[NCH1], uw[NCH1];
#pragma unroll
          for (int c = 0; c < NCH1; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nch1) {
              gw[c] = lds128(grow + idx);
              uw[c] = lds128(urow + idx);
            }
          }
          const int j = cd.z + rp;
          for (int gp = we.z; gp < we.w; ++gp) {
            const uint4* xr = x_s + (size_t)s_tok[gp] * nv;
            float g = 0.f, u = 0.f;
            if constexpr (FMT == PMOE_BF16) {
#pragma unroll
              for (int c = 0; c < NCH1; ++c) {
                const int idx = lane + 32 * c;
                if (idx < nch1) {
                  const float2 d = gu_dot_bf16(gw[c], uw[c], lds128(xr + idx));
                  g += d.x;
                  u += d.y;
                }
              }
            } else {
              // this row pair's scale rows, in the ring after the chunk's weight rows
              const ScaleSpan sg = scale_span<FMT>(a.lay.gu_s, rsg, cd.z, cd.w);
              const ScaleSpan su = scale_span<FMT>(a.lay.gu_s, rsg, a.I + cd.z, cd.w);
              const uint8_t* sgr = st + 2 * (size_t)cd.w * rbg + sg.first +
                                   (size_t)(scale_row<FMT>(j) - scale_row<FMT>(cd.z)) * rsg;
              const uint8_t* sur = st + 2 * (size_t)cd.w * rbg + sg.bytes + su.first +
                                   (size_t)(scale_row<FMT>(a.I + j) - scale_row<FMT>(a.I + cd.z)) * rsg;
#pragma unroll
              for (int c = 0; c < NCH1; ++c) {
                const int idx = lane + 32 * c;
                if (idx < nch1) {
                  const ChunkQ qg = chunk_q_ring<FMT>(sgr, idx, tsc);
                  const ChunkQ qu = chunk_q_ring<FMT>(sur, idx, tsc);
                  g += chunk_dot<FMT, kSrcShared>(gw[c], xr + idx * (EPC / 8), qg);
                  u += chunk_dot<FMT, kSrcShared>(uw[c], xr + idx * (EPC / 8), qu);
                }
              }
            }
            g = warp_sum(g);
            u = warp_sum(u);
            if (lane == 0) {
              const __nv_bfloat16 hb = __float2bfloat16_rn(silu_mul(g, u));
              const unsigned long long bits = (unsigned long long)__bfloat16_as_ushort(hb);
              st_relaxed_u64(a.ws.hq + (size_t)gp * a.I + j, (tag << 16) | bits);
            }
          }
        }
      } else if (cd.w > 0) {
        if (first_down && warp == 0 && lane == 0) DF_TRACE(3);
        first_down = false;
        // the fetcher stored the h rows of the expert's first T pairs after the W_d
        // rows; further pairs (an expert routed twice by one token) read theirs here
        const uint4* hsv = reinterpret_cast<const uint4*>(st + (size_t)cd.w * rbd);
        const uint8_t* sdb = st + (size_t)cd.w * rbd + (size_t)min(we.w - we.z, a.T) * a.I * 2;
        for (int rr = first; rr < cd.w && ok; rr += kDfConsumerWarps) {
          const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)rr * rbd);
          const int n_out = cd.z + rr;
          const uint8_t* sdr = nullptr;
          if constexpr (FMT != PMOE_BF16)
            sdr = sdb + scale_span<FMT>(a.lay.d_s, rsd, cd.z, cd.w).first +
                  (size_t)(scale_row<FMT>(n_out) - scale_row<FMT>(cd.z)) * rsd;
          for (int gp = we.z; gp < we.w && ok; ++gp) {
            const int pi = gp - we.z;
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < NCH2; ++c) {
              const int idx = lane + 32 * c;
              if (idx < nch2) {
                const ChunkQ q = chunk_q_ring<FMT>(sdr, idx, tsc);
                if (pi < a.T) {
                  acc += chunk_dot<FMT, kSrcShared>(lds128(row + idx), hsv + (size_t)pi * (a.I / 8) + idx * (EPC / 8), q);
                } else {
                  uint4 hv[EPC / 8];
                  ok = ok && fetch_h_direct(a.ws.hq + (size_t)gp * a.I + (size_t)idx * EPC, tag, hv, EPC / 8,
                                            abort_flag, a.err);
                  acc += chunk_dot<FMT, kSrcRegs>(lds128(row + idx), hv, q);
                }
              }
            }
            acc = warp_sum(acc);
            if (lane == 0) {
              if (fuse) o_s[gp * kDfMaxRows + (n_out - r_lo)] = acc;
              else a.ws.o_part[(size_t)gp * a.H + n_out] = acc;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (warp == 0) DF_CHUNK(k, 3);
        mb_arrive(&s_empty[s]);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    consumers_sync();
    if (tid == 0) DF_TRACE(4);
    if (fuse && !*abort_flag) {
      const int rows = r_hi - r_lo;
      for (int idx = tid; idx < a.T * rows; idx += kDfConsumerWarps * 32) {
        const int t = idx / rows, nl = idx - t * rows;
        float acc = 0.f;
        for (int r = 0; r < a.top_k; ++r) {
          const int gp = s_pos[t * a.top_k + r];
          if (gp < 0) continue;
          acc = fmaf(s_w[t * a.top_k + r], o_s[gp * kDfMaxRows + nl], acc);
        }
        if (a.residual != nullptr) acc = __bfloat162float(res_s[t * kDfMaxRows + nl]) + acc;
        a.y[(size_t)t * a.H + r_lo + nl] = __float2bfloat16_rn(acc);
      }
    }
    if (tid == 0) DF_TRACE(5);
  }
}

template <int FMT, int NCH1, int NCH2>
cudaError_t launch_df(const DfArgs& a, int grid, size_t smem, cudaStream_t s, int pdl) {
  auto k = decode_fused_kernel<FMT, NCH1, NCH2>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative (all CTAs co-resident: the down chunks wait for other CTAs' gate/up
  // rows), launched through cudaLaunchKernelEx so that it can be recorded into a graph;
  // optionally with programmatic serialization behind the residency step
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDfThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

__global__ void pdl_probe_kernel(int* out) {
  pdl_wait();
  if (threadIdx.x == 0) out[blockIdx.x] = 1;
}

size_t fmt_row_bytes(int fmt, int n) {
  return fmt == PMOE_BF16 ? (size_t)n * 2 : fmt == PMOE_FP8_BLOCK128 ? (size_t)n : (size_t)n / 2;
}

// Launch geometry: chunks per gate/up part (cg) and per down part (cd), each at most
// kDfMaxChunkBytes, the fixed shared-memory areas and the byte ring that fills the rest.
struct DfGeom {
  int cg, cd;
  size_t fixed, ring;
  size_t max_chunk;  // ring bytes of the largest chunk (weights, h rows, scale rows)
};

bool df_geometry(int fmt, int T, int top_k, int H, int I, int G, DfGeom* g) {
  // formats the fused kernel streams (NVFP4 decodes through the GEMV kernels)
  if (fmt != PMOE_BF16 && fmt != PMOE_FP8_BLOCK128 && fmt != PMOE_INT4_GPTQ_G128 && fmt != PMOE_MXFP4 &&
      fmt != PMOE_NVFP4)
    return false;
  if (T < 1 || T * top_k > kDfMaxPairs || G < 1 || G > 1024 || H % 8 != 0 || I % 8 != 0) return false;
  if (H >= (1 << 20) || I >= (1 << 20)) return false;  // the schedule's 32-bit products
  const size_t rbg = fmt_row_bytes(fmt, H), rbd = fmt_row_bytes(fmt, I);
  if (rbg % 16 != 0 || rbd % 16 != 0) return false;
  if (2 * rbg > (size_t)kDfMaxChunkBytes || rbd > (size_t)kDfMaxChunkBytes) return false;
  const int nch1 = (int)(rbg / 16), nch2 = (int)(rbd / 16);
  if (nch1 > 32 * 8 || nch2 > 32 * 4) return false;
  const long long gu_rows = (I + G - 1) / G, d_rows = (H + G - 1) / G;
  if (d_rows > kDfMaxRows) return false;
  const long long rj = kDfMaxChunkBytes / (2 * (long long)rbg), rd = kDfMaxChunkBytes / (long long)rbd;
  g->cg = (int)std::max(1LL, (gu_rows + rj - 1) / rj);
  g->cd = (int)std::max(1LL, (d_rows + rd - 1) / rd);
  if ((long long)T * top_k * (g->cg + g->cd) > kDfMaxChunks) return false;
  if (T > kDfMaxTokens) return false;
  g->fixed = (size_t)T * H * 2 + (size_t)kDfMaxPairs * kDfMaxRows * 4 + (size_t)kDfMaxTokens * kDfMaxRows * 2 +
             (size_t)kDfMaxChunks * sizeof(int4);
  // a quantised chunk carries its scale rows, copied in 16-byte units: the scale regions
  // must start and end on 16-byte boundaries
  size_t scale_max = 0;
  if (fmt != PMOE_BF16) {
    if (H % 128 != 0 || I % 128 != 0) return false;
    const ExpertLayout lay = expert_layout(fmt, H, I);
    if (lay.gu_s % 16 != 0 || lay.d_s % 16 != 0 || lay.bytes % 16 != 0) return false;
    const size_t rsg = (size_t)row_scale_bytes(fmt, H), rsd = (size_t)row_scale_bytes(fmt, I);
    scale_max = 2 * ((size_t)(rj + 1) * rsg + 32) + (size_t)(kDfMaxRows + 1) * rsd + 32;
  }
  // a down chunk also holds the h rows of up to T pairs
  const size_t max_chunk = (size_t)kDfMaxChunkBytes + (size_t)T * I * 2 + 128 + scale_max;
  g->max_chunk = max_chunk;
  if (g->fixed + 2 * max_chunk > kDfSmemBudget) return false;
  g->ring = ((kDfSmemBudget - g->fixed) / 128) * 128;
  return true;
}

}  // namespace

#ifdef PMOE_TRACE
extern "C" __attribute__((visibility("default"))) int pmoe_debug_decode_trace(unsigned long long* out, int n_ctas) {
  return cudaMemcpyFromSymbol(out, g_df_trace, (size_t)n_ctas * 8 * sizeof(unsigned long long)) == cudaSuccess ? 0 : -4;
}
extern "C" __attribute__((visibility("default"))) int pmoe_debug_decode_chunks(unsigned long long* out, int n_ctas) {
  return cudaMemcpyFromSymbol(out, g_df_chunk, (size_t)n_ctas * 256 * 4 * sizeof(unsigned long long)) == cudaSuccess
             ? 0
             : -4;
}
#endif

bool decode_pdl_supported(int device) {
  // 0 = not probed yet, 1 = accepted, -1 = refused (per device; the first cache created
  // on a device probes it, outside any stream capture)
  static int state[64] = {};
  if (device < 0 || device >= 64) return false;
  if (state[device] != 0) return state[device] > 0;
  const char* off = getenv("PMOE_NO_PDL");  // deployment switch: plain stream order
  if (off != nullptr && off[0] == '1') {
    state[device] = -1;
    return false;
  }
  int ok = 0;
  int* out = nullptr;
  cudaStream_t st = nullptr;
  if (cudaMalloc(&out, 2 * sizeof(int)) == cudaSuccess && cudaMemset(out, 0, 2 * sizeof(int)) == cudaSuccess &&
      cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int host[2] = {0, 0};
    if (cudaLaunchKernelEx(&cfg, pdl_probe_kernel, out) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess &&
        cudaMemcpy(host, out, sizeof(host), cudaMemcpyDeviceToHost) == cudaSuccess)
      ok = host[0] == 1 && host[1] == 1;
  }
  (void)cudaGetLastError();  // a refused attribute combination is not a sticky error
  if (st != nullptr) cudaStreamDestroy(st);
  if (out != nullptr) cudaFree(out);
  state[device] = ok ? 1 : -1;
  return ok != 0;
}

bool decode_chunking(int fmt, int T, int top_k, int H, int I, int num_sms, int* cg, int* cd, size_t* max_chunk) {
  DfGeom g;
  if (!df_geometry(fmt, T, top_k, H, I, num_sms, &g)) return false;
  *cg = g.cg;
  *cd = g.cd;
  *max_chunk = g.max_chunk;
  return true;
}

bool decode_fused_supported(int fmt, int T, int top_k, int H, int I, int num_sms) {
  DfGeom g;
  return df_geometry(fmt, T, top_k, H, I, num_sms, &g);
}

cudaError_t launch_decode_fused(int fmt, const __nv_bfloat16* x, const int32_t* ids, const float* w,
                                const __nv_bfloat16* residual, __nv_bfloat16* y, int T, int top_k, int H, int I,
                                const int32_t* plan, int E, int wave, int sub, int fuse_combine, const Workspace& ws,
                                uint8_t* arena, const uint8_t* store, int pull, size_t stride, int32_t* err, int num_sms,
                                cudaStream_t s, int pdl) {
  DfGeom g;
  if (!df_geometry(fmt, T, top_k, H, I, num_sms, &g)) return cudaErrorInvalidValue;
  DfArgs a;
  a.x = x;
  a.ids = ids;
  a.w = w;
  a.residual = residual;
  a.y = y;
  a.T = T;
  a.top_k = top_k;
  a.H = H;
  a.I = I;
  a.E = E;
  a.wave = wave;
  a.sub = sub;
  a.fuse_combine = fuse_combine;
  a.ring_bytes = (int)g.ring;
  a.cg = g.cg;
  a.cd = g.cd;
  a.plan = plan;
  a.ws = ws;
  a.arena = arena;
  a.store = store;
  a.pull = (pull != 0 && store != nullptr) ? 1 : 0;
  a.stride = stride;
  a.lay = expert_layout(fmt, H, I);
  if (fmt == PMOE_NVFP4) {  // the kernel's scale regions start after the 16-byte tensor-scale headers
    a.lay.gu_s += 16;
    a.lay.d_s += 16;
  }
  a.err = err;
  const size_t smem = g.ring + g.fixed;
  const int nch1 = (int)(fmt_row_bytes(fmt, H) / 16), nch2 = (int)(fmt_row_bytes(fmt, I) / 16);
#define PMOE_DF(F, A, B) return launch_df<F, A, B>(a, num_sms, smem, s, pdl)
  if (fmt == PMOE_BF16) {
    if (nch1 <= 32 * 4 && nch2 <= 32 * 1) PMOE_DF(PMOE_BF16, 4, 1);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 3) PMOE_DF(PMOE_BF16, 8, 3);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 4) PMOE_DF(PMOE_BF16, 8, 4);
  } else if (fmt == PMOE_FP8_BLOCK128) {
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_DF(PMOE_FP8_BLOCK128, 4, 2);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 4) PMOE_DF(PMOE_FP8_BLOCK128, 8, 4);
  } else if (fmt == PMOE_INT4_GPTQ_G128) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_DF(PMOE_INT4_GPTQ_G128, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_DF(PMOE_INT4_GPTQ_G128, 4, 2);
  } else if (fmt == PMOE_MXFP4) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_DF(PMOE_MXFP4, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_DF(PMOE_MXFP4, 4, 2);
  } else if (fmt == PMOE_NVFP4) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_DF(PMOE_NVFP4, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_DF(PMOE_NVFP4, 4, 2);
  }
#undef PMOE_DF
  return cudaErrorInvalidValue;
}

}  // namespace pmoe
