// Persistent decode of a whole stack of MoE layers: one cooperative launch per token step
// walks every layer, h_{l+1} = h_l + moe_l(h_l) (article "Running an MoE Model Larger Than
// Your VRAM", section "Why is it fast when experts keep crossing PCIe?": a token at batch 1
// activates layers x top_k experts, and the page-in of later layers' experts overlaps the
// current layer's compute).
//
// Same block as the fused single-layer decode kernel (11 consumer warps, a producer, an h
// fetcher, 3 pager warps; a shared-memory byte ring fed by bulk copies), with the layer
// loop inside:
//   * every layer's plan is made beforehand (one residency launch for all layers); the
//     kernel runs only when every layer's step is one wave (T * top_k <= K), so a layer's
//     slots are never reused within the launch;
//   * the producer, fetcher, pagers and consumers each walk the same chunk sequence, all
//     layers in order; the ring, its slots and its barriers run on across layers, so the
//     next layer's weights stream in while the current one finishes;
//   * the pagers run ahead through every layer's missing experts (each CTA copies the
//     bytes its own chunks read, as in the single-layer kernel): the host link works while
//     earlier layers compute;
//   * layer l's combine writes, for this CTA's rows, h_{l+1} = h_l + sum_r w_r o_r (rank
//     order, fp32, one bf16 rounding) as tagged 64-bit words; the fetcher gathers all H
//     values of h_{l+1} (every CTA's rows) before the consumers start layer l+1's gate/up
//     chunks. The intermediate h words and these words alternate between two buffers by
//     layer parity.
// The arithmetic of every output element is that of the fused single-layer kernel (same
// dot products, same rank-ordered combine), so the result equals L single-layer forward
// calls with residual = input, bit for bit. Every wait is bounded.
#include "decode_ring.cuh"

namespace pmoe {
namespace {

constexpr int kStMaxTokens = 2;
constexpr int kStMaxPairs = 16;   // T * top_k
constexpr int kStMaxLayers = 128;
constexpr int kStMetaHdr = 8;     // D, resident experts, epoch lo/hi, arena (2 words), store (2 words)

// Words of one layer's metadata in shared memory: the header, the wave's experts
// (expert, slot, first grouped pair, end), each grouped pair's token, each pair's grouped
// position and routing weight.
// (A multiple of 4 words: the expert records are 16-byte vectors, the pointers 8 bytes.)
#ifdef PMOE_TRACE
// Debug builds only: per CTA and layer, %globaltimer at (0) the fetcher starting the input
// gather, (1) the input gathered, (2) the consumers' first chunk landed, (3) the last chunk
// consumed, (4) the combine published.
__device__ unsigned long long g_st_trace[1024][kStMaxLayers][5];
__device__ __forceinline__ unsigned long long st_gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
#define ST_TRACE(l, slot)                                    \
  do {                                                       \
    g_st_trace[blockIdx.x][(l)][(slot)] = st_gtimer();       \
  } while (0)
// per chunk (the first 128 of the launch): issued, landed (consumers), passed by the
// fetcher, consumed
__device__ unsigned long long g_st_chunk[1024][128][4];
#define ST_CHUNK(k, slot)                                             \
  do {                                                                \
    if ((k) < 128) g_st_chunk[blockIdx.x][(k)][(slot)] = st_gtimer(); \
  } while (0)
#else
#define ST_CHUNK(k, slot) \
  do {                    \
  } while (0)
#define ST_TRACE(l, slot) \
  do {                    \
  } while (0)
#endif

__host__ __device__ constexpr int st_meta_words(int P) { return (kStMetaHdr + 4 * P + 3 * P + 3) & ~3; }

// This CTA's chunk schedule for a wave of D experts (entries (kind, expert index, first
// row, rows), the single-layer kernel's order) does not depend on the layer: one table per
// D in 1..P, built at entry, stands in for the per-chunk arithmetic. Table D starts at
// entry (cg + cd) * D * (D - 1) / 2.
__host__ __device__ constexpr int st_sched_entries(int P, int per) { return per * P * (P + 1) / 2; }
__device__ __forceinline__ int st_sched_base(int D, int per) { return per * D * (D - 1) / 2; }

struct StArgs {
  const __nv_bfloat16* x;          // [T][H] h_0
  __nv_bfloat16* y;                // [T][H] h_L
  const int32_t* ids;              // [L][T][top_k]
  const float* w;                  // [L][T][top_k]
  const int32_t* plan0;            // layer l's plan at plan0 + l * plan_words
  int plan_words;
  uint8_t* const* arenas;          // [L] slot arenas (device array of device pointers)
  const uint8_t* const* stores;    // [L] mapped host stores (device pointers)
  unsigned long long* hq;          // [2][P][I] tagged intermediate words, by layer parity
  unsigned long long* xq;          // [2][T][H] tagged h_{l} words, by layer parity
  int T, top_k, H, I, E, L;
  int ring_bytes, cg, cd;
  size_t stride;
  ExpertLayout lay;
  int32_t* err;
};

// Barrier of the consumer warps that ORs a predicate over them (so that they leave a
// loop together: a warp missing from the next barrier would stall the others).
__device__ __forceinline__ int consumers_any(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred), "n"(kDfConsumerWarps * 32)
      : "memory");
  return r;
}

__device__ __forceinline__ void st_release_shared(int* p, int v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(su32(p)), "r"(v) : "memory");
}

// Waits until the shared counter *p reaches at least v (bounded; the abort flag also ends it).
__device__ __forceinline__ bool wait_shared_at_least(const int* p, int v, volatile int* abort_flag, int32_t* err) {
  long long t0 = -1;
  while (ld_acquire_shared(p) < v) {
    if (*abort_flag) return false;
    if (t0 < 0) {
      t0 = clock64();
    } else if (clock64() - t0 > kDfWaitLimit) {
      *abort_flag = 1;
      atomicOr(err, kErrDecodeTimeout);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// One warp gathers n tagged 64-bit words (n even; bf16 value in the low 16 bits, the tag
// above) into n bf16 values at dst, waiting until each carries `tag`: up to 16 16-byte
// loads per lane in flight, the stale ones re-read together. Returns false on abort.
__device__ __noinline__ bool warp_gather_tagged(const unsigned long long* src, int n, unsigned long long tag, uint16_t* dst,
                                   volatile int* abort_flag, int32_t* err) {
  const int lane = threadIdx.x & 31;
  int bad = 0;
  for (int i0 = 2 * lane; i0 < n && !bad; i0 += 64 * 16) {
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
            *reinterpret_cast<uint32_t*>(dst + i0 + u * 64) =
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
        atomicOr(err, kErrDecodeTimeout);
        bad = 1;
        break;
      }
      __nanosleep(256);
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if ((pend >> u) & 1u) v[u] = ld_relaxed_u64x2(src + i0 + u * 64);
    }
  }
  return !__any_sync(0xffffffffu, bad);
}

template <int FMT, int NCH1, int NCH2>
__global__ void __launch_bounds__(kDfThreads, 1) decode_stack_kernel(const StArgs a) {
  constexpr int EPC = Fmt<FMT>::EPC;
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ unsigned s_off[kDfSlots];                // ring offset of each slot's chunk
  __shared__ __align__(8) uint64_t s_full[kDfSlots];  // the chunk's weight bytes landed
  __shared__ __align__(8) uint64_t s_hrdy[kDfSlots];  // the fetcher has passed the chunk (down: h copied)
  __shared__ __align__(8) uint64_t s_empty[kDfSlots];
  __shared__ int s_abort;
  __shared__ int s_placed;  // chunks placed in the ring so far (all layers, in order)
  __shared__ int s_pulled;  // chunks whose bytes this CTA has paged in
  __shared__ int s_xready;  // the last layer whose input h_l is in x_s
  __shared__ int s_cons;    // the last layer whose combine this CTA's consumers have finished

  const int P = a.T * a.top_k;
  const int MW = st_meta_words(P);
  const unsigned R = (unsigned)a.ring_bytes;
  uint8_t* ring = dsm;
  uint4* x_s = reinterpret_cast<uint4*>(ring + R);  // [2][T][H] bf16, h_l in buffer l & 1
  float* o_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(x_s) + (size_t)2 * a.T * a.H * 2);
  int* meta = reinterpret_cast<int*>(o_s + kStMaxPairs * kDfMaxRows);
  int4* sched = reinterpret_cast<int4*>(meta + (size_t)a.L * MW);  // [st_sched_entries(P, cg + cd)]
  volatile int* abort_flag = &s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PlanLayout L{a.E};
  if (warp == kDfConsumerWarps && lane == 0) {
    for (int s = 0; s < kDfSlots; ++s) {
      mb_init(&s_full[s], 1);
      mb_init(&s_hrdy[s], 1);
      mb_init(&s_empty[s], kDfConsumerWarps);
    }
    s_abort = 0;
    s_placed = 0;
    s_pulled = 0;
    s_xready = 0;
    s_cons = -1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Every layer's metadata, one warp per layer: the wave's experts and slots from the
  // plan, the pairs grouped stably by expert id then pair index, the routing weights.
  for (int l = warp; l < a.L; l += kDfThreads / 32) {
    int* m = meta + (size_t)l * MW;
    int4* we = reinterpret_cast<int4*>(m + kStMetaHdr);
    int* tok = m + kStMetaHdr + 4 * P;
    int* pos = tok + P;
    float* wr = reinterpret_cast<float*>(pos + P);
    const int32_t* plan = a.plan0 + (size_t)l * a.plan_words;
    const int id = lane < P ? a.ids[(size_t)l * P + lane] : -1;
    const float wt = lane < P ? a.w[(size_t)l * P + lane] : 0.f;
    const int nw = plan[kPlanWaves];
    const int D = nw > 0 ? plan[L.wave_start() + 1] - plan[L.wave_start()] : 0;
    const int e = lane < D ? plan[L.wave_exp() + lane] : -1;
    const int slot = lane < D ? plan[L.wave_slot() + lane] : -1;
    int p_pos = -1, lo = 0, cnt = 0;
    const bool valid = id >= 0 && id < a.E;
    if (valid) p_pos = 0;
    for (int q = 0; q < P; ++q) {
      const int o = __shfl_sync(0xffffffffu, id, q);
      const bool ov = o >= 0 && o < a.E;
      if (valid && ov && (o < id || (o == id && q < lane))) ++p_pos;
      if (lane < D) {
        lo += (ov && o < e) ? 1 : 0;
        cnt += (o == e) ? 1 : 0;
      }
    }
    if (lane < P) {
      pos[lane] = p_pos;
      wr[lane] = wt;
      if (p_pos >= 0) tok[p_pos] = lane / a.top_k;
    }
    if (lane < D) we[lane] = make_int4(e, slot, lo, lo + cnt);
    if (lane == 0) {
      m[0] = nw > 1 ? -1 : D;  // (several waves: refused below)
      m[1] = nw > 0 ? min(plan[L.wave_hits()], D) : 0;
      m[2] = plan[kPlanEpochLo];
      m[3] = plan[kPlanEpochHi];
      *reinterpret_cast<uint8_t**>(m + 4) = a.arenas[l];
      *reinterpret_cast<const uint8_t**>(m + 6) = a.stores[l];
    }
  }
  {
    const int per = a.cg + a.cd, n_tab = st_sched_entries(P, per);
    for (int i = tid; i < n_tab; i += kDfThreads) {
      int D = 1;
      while (st_sched_base(D + 1, per) <= i) ++D;
      const DfSched sc{D, (int)gridDim.x, (int)blockIdx.x, a.I, a.H, a.cg, a.cd};
      sched[i] = sched_entry(i - st_sched_base(D, per), sc);
    }
  }
  for (int i = tid; i < a.T * (a.H / 8); i += kDfThreads) x_s[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
  __syncthreads();
  // a layer with several waves (excluded on the host) would reuse slots within the launch
  if (tid == 0) {
    for (int l = 0; l < a.L; ++l)
      if (meta[(size_t)l * MW] < 0) {
        atomicOr(a.err, kErrPlanOverflow);
        s_abort = 1;
      }
  }
  __syncthreads();
  if (s_abort) return;

  const int G = (int)gridDim.x;
  const int r_lo = (int)((long long)a.H * blockIdx.x / G);
  const int r_hi = (int)((long long)a.H * (blockIdx.x + 1) / G);
  const size_t rbg = (size_t)a.H * Fmt<FMT>::BPE2 / 2;  // one gate (or up) row
  const size_t rbd = (size_t)a.I * Fmt<FMT>::BPE2 / 2;  // one down row
  const int rsg = row_scale_bytes(FMT, a.H), rsd = row_scale_bytes(FMT, a.I);  // one scale row of gate/up, of down
  // tags: layer l's h words carry its plan epoch (wave 0, part 0, as in the single-layer
  // kernel); the words of h_l carry the same epoch with part 3, which no h word uses
  auto layer_epoch = [&](int l) {
    const int* m = meta + (size_t)l * MW;
    return ((unsigned long long)(uint32_t)m[3] << 32) | (uint32_t)m[2];
  };
  auto h_tag = [&](int l) { return (layer_epoch(l) << 12) & kTagMask; };
  auto x_tag = [&](int l) { return ((layer_epoch(l) << 12) | 3ull) & kTagMask; };

  if (warp == kDfConsumerWarps) {
    // ---------------- producer: lane 0 places every chunk of every layer in the byte ring
    // as soon as its slot and its bytes are free and issues its bulk copies (after the
    // pagers, for an expert this launch pages in). A down chunk also reserves room for
    // the expert's h rows, which the fetcher fills.
    if (lane == 0) {
      unsigned head = 0;
      int tail = 0, kk = 0;
      bool stop = false;
      for (int l = 0; l < a.L && !stop; ++l) {
        const int* m = meta + (size_t)l * MW;
        const int D = m[0], n_hits = m[1];
        const int4* we_l = reinterpret_cast<const int4*>(m + kStMetaHdr);
        const uint8_t* arena = *reinterpret_cast<uint8_t* const*>(m + 4);
        const int4* sc = sched + st_sched_base(D, a.cg + a.cd);
        const int n_chunks = D * (a.cg + a.cd);
        for (int q = 0; q < n_chunks; ++q, ++kk) {
          const int4 cd = sc[q];
          const int kind = cd.x & 3;
          const int4 we = we_l[cd.y];
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
            if (kk - tail < kDfSlots) {
              off = ring_place(head, s_off[tail % kDfSlots], tail == kk, need, R);
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
          if (off < 0) {
            stop = true;
            break;
          }
          const int s = kk % kDfSlots;
          s_off[s] = (unsigned)off;
          head = (unsigned)off + need;
          uint64_t* fb = &s_full[s];
          if (wbytes != 0 && cd.y >= n_hits) {
            // an expert this launch pages in: wait until this CTA's pagers have copied the
            // chunk's bytes into the slot
            if (!wait_shared_at_least(&s_pulled, kk + 1, abort_flag, a.err)) {
              stop = true;
              break;
            }
          }
          if (wbytes == 0) {
            mb_arrive(fb);
          } else {
            const uint8_t* ex = arena + (size_t)we.y * a.stride;
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
          ST_CHUNK(kk, 0);
          st_release_shared(&s_placed, kk + 1);
        }
      }
      if (*abort_flag) {
        // stopped early: let the copies already issued land before the CTA exits
        const long long t1 = clock64();
        for (int q = max(0, kk - kDfSlots); q < kk; ++q)
          while (!mb_test(&s_full[q % kDfSlots], (uint32_t)((q / kDfSlots) & 1)) && clock64() - t1 < kDfWaitLimit) {
          }
      }
    }
  } else if (warp == kDfConsumerWarps + 1) {
    // ---------------- fetcher: walks the chunks in order behind the producer. At the start
    // of layer l > 0 it gathers h_l (every CTA's combined rows of layer l - 1) into its x
    // buffer; for a down chunk it gathers the expert's h rows (written by every CTA's
    // gate/up chunks) after the chunk's W_d rows. Each chunk is then passed to the consumers.
    int kk = 0;
    bool ok = true;
    for (int l = 0; l < a.L && ok; ++l) {
      const int* m = meta + (size_t)l * MW;
      const int D = m[0];
      const int4* we_l = reinterpret_cast<const int4*>(m + kStMetaHdr);
      if (l > 0) {
        // h_l is complete only after this CTA's own combine of layer l - 1: start polling
        // then (polling earlier, 152 CTAs re-reading the words, loads the memory system
        // the weight copies need). The buffer's previous content, h_{l-2}, is dead by then.
        ok = wait_shared_at_least(&s_cons, l - 1, abort_flag, a.err);
        if (lane == 0) ST_TRACE(l, 0);
        if (!__all_sync(0xffffffffu, ok)) break;
        uint16_t* xd = reinterpret_cast<uint16_t*>(x_s + (size_t)(l & 1) * a.T * (a.H / 8));
        ok = warp_gather_tagged(a.xq + (size_t)(l & 1) * a.T * a.H, a.T * a.H, x_tag(l), xd, abort_flag, a.err);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) ST_TRACE(l, 1);
        if (lane == 0) st_release_shared(&s_xready, l);
      }
      const int4* sc = sched + st_sched_base(D, a.cg + a.cd);
      const int n_chunks = D * (a.cg + a.cd);
      for (int q = 0; q < n_chunks; ++q, ++kk) {
        ok = wait_shared_at_least(&s_placed, kk + 1, abort_flag, a.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const int s = kk % kDfSlots;
        const int4 cd = sc[q];
        if ((cd.x & 3) == 2 && cd.w > 0) {
          const int4 we = we_l[cd.y];
          const int hb = min(we.w - we.z, a.T);
          uint16_t* hdst = reinterpret_cast<uint16_t*>(ring + s_off[s] + (size_t)cd.w * rbd);
          const unsigned long long* src = a.hq + ((size_t)(l & 1) * kStMaxPairs + we.z) * a.I;
          ok = warp_gather_tagged(src, hb * a.I, h_tag(l), hdst, abort_flag, a.err);
          if (!ok) break;
          // these generic stores share the ring with later bulk copies (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) ST_CHUNK(kk, 2);
        if (lane == 0) mb_arrive(&s_hrdy[s]);
      }
    }
  } else if (warp >= kDfConsumerWarps + 2) {
    // ---------------- pagers: for every chunk of an expert the launch pages in, in chunk
    // order over all layers, copy the bytes the chunk reads (its weight rows and their
    // scale rows) from the layer's mapped host store into the expert's slot, then publish
    // the progress. They wait for nothing else, so they run ahead into later layers.
    const int vl = tid - (kDfConsumerWarps + 2) * 32, nl = kDfPagerWarps * 32;
    const int hb = a.H / 128, ib = a.I / 128;
    int kk = 0;
    bool stop = false;
    for (int l = 0; l < a.L && !stop; ++l) {
      const int* m = meta + (size_t)l * MW;
      const int D = m[0], n_hits = m[1];
      const int4* we_l = reinterpret_cast<const int4*>(m + kStMetaHdr);
      uint8_t* arena = *reinterpret_cast<uint8_t* const*>(m + 4);
      const uint8_t* store = *reinterpret_cast<const uint8_t* const*>(m + 6);
      const int4* sc = sched + st_sched_base(D, a.cg + a.cd);
      const int n_chunks = D * (a.cg + a.cd);
      for (int q = 0; q < n_chunks; ++q, ++kk) {
        const int4 cd = sc[q];
        if (cd.y < n_hits || cd.w == 0) continue;
        if (pagers_any(*abort_flag)) {  // every pager warp sees the same answer
          stop = true;
          break;
        }
        const int4 we = we_l[cd.y];
        const uint8_t* src = store + (size_t)we.x * a.stride;
        uint8_t* dst = arena + (size_t)we.y * a.stride;
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
            lanes_copy4(src, dst, a.lay.gu_s + (size_t)(z >> 7) * row,
                        (size_t)(((z + n - 1) >> 7) - (z >> 7) + 1) * row, vl, nl);
            lanes_copy4(src, dst, a.lay.gu_s + (size_t)((a.I + z) >> 7) * row,
                        (size_t)(((a.I + z + n - 1) >> 7) - ((a.I + z) >> 7) + 1) * row, vl, nl);
          } else if constexpr (FMT == PMOE_INT4_GPTQ_G128 || FMT == PMOE_MXFP4) {
            const size_t row = 4 * (size_t)hb;  // one row's scale bytes
            lanes_copy4(src, dst, a.lay.gu_s + (size_t)z * row, (size_t)n * row, vl, nl);
            lanes_copy4(src, dst, a.lay.gu_s + (size_t)(a.I + z) * row, (size_t)n * row, vl, nl);
          } else if constexpr (FMT == PMOE_NVFP4) {
            // twice those rows' bytes (an e4m3 scale per 16 inputs): 8 loads in flight per lane
            const size_t row = (size_t)row_scale_bytes(FMT, a.H);
            lanes_copy4x2(src, dst, a.lay.gu_s + (size_t)z * row, (size_t)n * row, a.lay.gu_s + (size_t)(a.I + z) * row,
                          (size_t)n * row, vl, nl);
          }
        } else {
          lanes_copy16x2(src, dst, a.lay.d_w + (size_t)z * rbd, (size_t)n * rbd, 0, 0, vl, nl);
          if constexpr (FMT == PMOE_FP8_BLOCK128) {
            const size_t row = 4 * (size_t)ib;
            lanes_copy4(src, dst, a.lay.d_s + (size_t)(z >> 7) * row,
                        (size_t)(((z + n - 1) >> 7) - (z >> 7) + 1) * row, vl, nl);
          } else if constexpr (FMT == PMOE_INT4_GPTQ_G128 || FMT == PMOE_MXFP4) {
            const size_t row = 4 * (size_t)ib;
            lanes_copy4(src, dst, a.lay.d_s + (size_t)z * row, (size_t)n * row, vl, nl);
          } else if constexpr (FMT == PMOE_NVFP4) {
            const size_t row = (size_t)row_scale_bytes(FMT, a.I);
            lanes_copy4x2(src, dst, a.lay.d_s + (size_t)z * row, (size_t)n * row, 0, 0, vl, nl);
          }
        }
        if constexpr (FMT == PMOE_NVFP4)
          if (vl < 4) *reinterpret_cast<uint32_t*>(dst + hdr_off + 4 * vl) = hdr;
        // the stores (generic proxy) are read next by bulk copies (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        pagers_sync();
        if (vl == 0) st_release_shared(&s_pulled, kk + 1);
      }
    }
  } else {
    // ---------------- consumers (warps 0 .. kDfConsumerWarps-1): every warp walks every
    // chunk of every layer; rows are dealt round-robin over the whole sequence. A layer's
    // gate/up chunks wait until its input h_l is in x_s; after its last chunk the warps
    // combine this CTA's rows of h_{l+1}.
    const int nv = a.H / 8;
    const int nch1 = (int)(rbg / 16), nch2 = (int)(rbd / 16);
    int kk = 0, rows_before = 0;
    for (int l = 0; l < a.L; ++l) {
      const int* m = meta + (size_t)l * MW;
      const int D = m[0];
      const int4* we_l = reinterpret_cast<const int4*>(m + kStMetaHdr);
      const int* tok = m + kStMetaHdr + 4 * P;
      const int* pos = tok + P;
      const float* wr = reinterpret_cast<const float*>(pos + P);
      bool ok = true;
      if (l > 0) ok = __all_sync(0xffffffffu, wait_shared_at_least(&s_xready, l, abort_flag, a.err));
      const uint4* xl = x_s + (size_t)(l & 1) * a.T * nv;
      unsigned long long* hq = a.hq + (size_t)(l & 1) * kStMaxPairs * a.I;
      const unsigned long long tag = h_tag(l);
      const int4* sc = sched + st_sched_base(D, a.cg + a.cd);
      const int n_chunks = D * (a.cg + a.cd);
      for (int q = 0; q < n_chunks && ok; ++q, ++kk) {
        const int s = kk % kDfSlots;
        const int4 cd = sc[q];
        const int kind = cd.x & 3;
        const int first = ((warp - rows_before) % kDfConsumerWarps + kDfConsumerWarps) % kDfConsumerWarps;
        rows_before += cd.w;
        const uint32_t par = (uint32_t)((kk / kDfSlots) & 1);
        // every chunk's s_hrdy phase is waited for, so that a warp never waits on a phase
        // two ahead of the barrier's (parity would alias)
        bool got = mb_wait(&s_full[s], par, abort_flag, a.err);
        if (got) got = mb_wait(&s_hrdy[s], par, abort_flag, a.err);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (q == 0 && tid == 0) ST_TRACE(l, 2);
        if (tid == 0) ST_CHUNK(kk, 1);
        const int4 we = we_l[cd.y];
        const uint8_t* st = ring + s_off[s];
        // NVFP4: the chunk's matrix's tensor scale, in the 16-byte header before its block
        // scales in the slot (an expert this launch pages in: written by this CTA's pagers
        // before the chunk's progress, which the producer acquired before its copies)
        float tsc = 1.f;
        if constexpr (FMT == PMOE_NVFP4) {
          if (cd.w > 0) {
            const uint8_t* arena_l = *reinterpret_cast<uint8_t* const*>(m + 4);
            const uint8_t* hdr = arena_l + (size_t)we.y * a.stride + (kind == 1 ? a.lay.gu_s : a.lay.d_s) - 16;
            asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(tsc) : "l"(hdr));
          }
        }
        if (kind == 1) {
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
              const uint4* xr = xl + (size_t)tok[gp] * nv;
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
                st_relaxed_u64(hq + (size_t)gp * a.I + j, (tag << 16) | bits);
              }
            }
          }
        } else if (cd.w > 0) {
          // the fetcher stored the h rows of the expert's first T pairs after the W_d rows;
          // further pairs (an expert routed twice by one token) read theirs here
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
                  const ChunkQ qd = chunk_q_ring<FMT>(sdr, idx, tsc);
                  if (pi < a.T) {
                    acc += chunk_dot<FMT, kSrcShared>(lds128(row + idx), hsv + (size_t)pi * (a.I / 8) + idx * (EPC / 8),
                                                      qd);
                  } else {
                    uint4 hv[EPC / 8];
                    ok = ok && fetch_h_direct(hq + (size_t)gp * a.I + (size_t)idx * EPC, tag, hv, EPC / 8,
                                              abort_flag, a.err);
                    acc += chunk_dot<FMT, kSrcRegs>(lds128(row + idx), hv, qd);
                  }
                }
              }
              acc = warp_sum(acc);
              if (lane == 0) o_s[gp * kDfMaxRows + (n_out - r_lo)] = acc;
            }
          }
        }
        __syncwarp();
        if (tid == 0) ST_CHUNK(kk, 3);
        if (lane == 0) mb_arrive(&s_empty[s]);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
      // the consumer warps leave together (after a wait that gave up, the flag is raised)
      if (consumers_any(!ok || *abort_flag)) break;
      if (tid == 0) ST_TRACE(l, 3);
      // combine this CTA's rows: h_{l+1} = h_l + sum_r w_r o_r in rank order (fp32), rounded
      // once to bf16, then published for every CTA (or written out after the last layer)
      const int rows = r_hi - r_lo;
      const __nv_bfloat16* xh = reinterpret_cast<const __nv_bfloat16*>(xl);
      const unsigned long long xt = l + 1 < a.L ? x_tag(l + 1) : 0ull;
      unsigned long long* xq = a.xq + (size_t)((l + 1) & 1) * a.T * a.H;
      for (int idx = tid; idx < a.T * rows; idx += kDfConsumerWarps * 32) {
        const int t = idx / rows, nl = idx - t * rows;
        float acc = 0.f;
        for (int r = 0; r < a.top_k; ++r) {
          const int gp = pos[t * a.top_k + r];
          if (gp < 0) continue;
          acc = fmaf(wr[t * a.top_k + r], o_s[gp * kDfMaxRows + nl], acc);
        }
        acc = __bfloat162float(xh[(size_t)t * a.H + r_lo + nl]) + acc;
        const __nv_bfloat16 v = __float2bfloat16_rn(acc);
        if (l + 1 < a.L) st_relaxed_u64(xq + (size_t)t * a.H + r_lo + nl, (xt << 16) | __bfloat16_as_ushort(v));
        else a.y[(size_t)t * a.H + r_lo + nl] = v;
      }
      // (o_s is rewritten by the next layer's down chunks)
      consumers_sync();
      if (tid == 0) ST_TRACE(l, 4);
      if (tid == 0) st_release_shared(&s_cons, l);
    }
  }
}

struct StGeom {
  int cg, cd;
  size_t fixed, ring;
};

bool st_geometry(int fmt, int T, int top_k, int H, int I, int L, int G, StGeom* g) {
  if (T < 1 || T > kStMaxTokens || T * top_k > kStMaxPairs || L < 1 || L > kStMaxLayers) return false;
  size_t max_chunk = 0;
  if (!decode_chunking(fmt, T, top_k, H, I, G, &g->cg, &g->cd, &max_chunk)) return false;
  g->fixed = (size_t)2 * T * H * 2 + (size_t)kStMaxPairs * kDfMaxRows * 4 + (size_t)L * st_meta_words(T * top_k) * 4 +
             (size_t)st_sched_entries(T * top_k, g->cg + g->cd) * sizeof(int4);
  if (g->fixed + 2 * max_chunk > kDfSmemBudget) return false;
  g->ring = ((kDfSmemBudget - g->fixed) / 128) * 128;
  return true;
}

template <int FMT, int NCH1, int NCH2>
cudaError_t launch_st(const StArgs& a, int grid, size_t smem, cudaStream_t s) {
  auto k = decode_stack_kernel<FMT, NCH1, NCH2>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative: every CTA waits for the others' intermediate and combined rows
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDfThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

size_t st_row_bytes(int fmt, int n) {
  return fmt == PMOE_BF16 ? (size_t)n * 2 : fmt == PMOE_FP8_BLOCK128 ? (size_t)n : (size_t)n / 2;
}

}  // namespace

#ifdef PMOE_TRACE
extern "C" __attribute__((visibility("default"))) int pmoe_debug_stack_trace(unsigned long long* out, int n_ctas) {
  return cudaMemcpyFromSymbol(out, g_st_trace, (size_t)n_ctas * kStMaxLayers * 5 * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? 0
             : -4;
}
extern "C" __attribute__((visibility("default"))) int pmoe_debug_stack_chunks(unsigned long long* out, int n_ctas) {
  return cudaMemcpyFromSymbol(out, g_st_chunk, (size_t)n_ctas * 128 * 4 * sizeof(unsigned long long)) == cudaSuccess
             ? 0
             : -4;
}
#endif

bool decode_stack_supported(int fmt, int T, int top_k, int H, int I, int L, int num_sms) {
  StGeom g;
  return st_geometry(fmt, T, top_k, H, I, L, num_sms, &g);
}

cudaError_t launch_decode_stack(int fmt, const __nv_bfloat16* x, __nv_bfloat16* y, const int32_t* ids, const float* w,
                                int T, int top_k, int H, int I, int E, int L, const int32_t* plan0, int plan_words,
                                uint8_t* const* arenas, const uint8_t* const* stores, unsigned long long* hq,
                                unsigned long long* xq, size_t stride, int32_t* err, int num_sms, cudaStream_t s) {
  StGeom g;
  if (!st_geometry(fmt, T, top_k, H, I, L, num_sms, &g)) return cudaErrorInvalidValue;
  StArgs a{};
  a.x = x;
  a.y = y;
  a.ids = ids;
  a.w = w;
  a.plan0 = plan0;
  a.plan_words = plan_words;
  a.arenas = arenas;
  a.stores = stores;
  a.hq = hq;
  a.xq = xq;
  a.T = T;
  a.top_k = top_k;
  a.H = H;
  a.I = I;
  a.E = E;
  a.L = L;
  a.ring_bytes = (int)g.ring;
  a.cg = g.cg;
  a.cd = g.cd;
  a.stride = stride;
  a.lay = expert_layout(fmt, H, I);
  if (fmt == PMOE_NVFP4) {  // the kernel's scale regions start after the 16-byte tensor-scale headers
    a.lay.gu_s += 16;
    a.lay.d_s += 16;
  }
  a.err = err;
  const size_t smem = g.ring + g.fixed;
  const int nch1 = (int)(st_row_bytes(fmt, H) / 16), nch2 = (int)(st_row_bytes(fmt, I) / 16);
#define PMOE_ST(F, A, B) return launch_st<F, A, B>(a, num_sms, smem, s)
  if (fmt == PMOE_BF16) {
    if (nch1 <= 32 * 4 && nch2 <= 32 * 1) PMOE_ST(PMOE_BF16, 4, 1);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 3) PMOE_ST(PMOE_BF16, 8, 3);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 4) PMOE_ST(PMOE_BF16, 8, 4);
  } else if (fmt == PMOE_FP8_BLOCK128) {
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_ST(PMOE_FP8_BLOCK128, 4, 2);
    if (nch1 <= 32 * 8 && nch2 <= 32 * 4) PMOE_ST(PMOE_FP8_BLOCK128, 8, 4);
  } else if (fmt == PMOE_INT4_GPTQ_G128) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_ST(PMOE_INT4_GPTQ_G128, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_ST(PMOE_INT4_GPTQ_G128, 4, 2);
  } else if (fmt == PMOE_MXFP4) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_ST(PMOE_MXFP4, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_ST(PMOE_MXFP4, 4, 2);
  } else if (fmt == PMOE_NVFP4) {
    if (nch1 <= 32 * 2 && nch2 <= 32 * 1) PMOE_ST(PMOE_NVFP4, 2, 1);
    if (nch1 <= 32 * 4 && nch2 <= 32 * 2) PMOE_ST(PMOE_NVFP4, 4, 2);
  }
#undef PMOE_ST
  return cudaErrorInvalidValue;
}

}  // namespace pmoe
