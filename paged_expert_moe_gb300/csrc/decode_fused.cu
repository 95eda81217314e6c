// Decode path (T <= 8 tokens): one fused, weight-streaming kernel per wave.
//
// At decode batch sizes the MoE layer reads every routed expert's weights once and
// does ~1 FLOP per byte, so it is bound by HBM bandwidth (the decode-is-memory-bound
// discussion in "SGLang serving optimisation"; "Running an MoE Model Larger Than Your
// VRAM", section "Why is it fast when experts keep crossing PCIe?"). One persistent
// CTA per SM (cooperative launch, so all CTAs are resident) does, for the wave's
// experts in order:
//   phase 1  gate/up + SiLU*mul: the wave's row pairs, cut into chunks that never cross
//            an expert, are dealt out in one contiguous range per CTA; a producer
//            thread streams each chunk's gate rows and the matching up rows into a
//            shared-memory ring (cp.async.bulk, completion on mbarriers); consumer
//            warps reduce them against the tokens' x (in shared memory), write
//            h[pair][j] (bf16) and then add the finished row count to the expert's
//            completion counter.
//   phase 2  down: CTA b owns output rows [b*H/G, (b+1)*H/G) of every expert. The
//            producer streams those W_d rows (they do not depend on h), waits until the
//            expert's counter shows all I rows of h are written, and then bulk-copies
//            the expert's h rows into the same stage (no grid-wide barrier).
//   phase 3  combine (single-wave steps): the CTA holds o[pair][n] for every pair of
//            its rows, so it writes y[t][n] = res + sum_r w[t,r] o[(t,r)][n] in rank
//            order; otherwise o_part is written and the combine kernel runs after the
//            last wave (same arithmetic and order, so the bits agree).
// The token -> expert grouping (stable: expert ascending, pair index ascending) is
// computed by every CTA from the ids; CTA 0 also writes pos/perm for the combine.
// Per-pair dot products have a fixed order (lane-strided 16-byte chunks, then an
// xor-shuffle tree), independent of slot, wave and of how many tokens share the
// expert. Every wait is bounded; on expiry the kernel records an error and stops.
#include "decode_common.cuh"

namespace pmoe {
namespace {

using namespace dec;

constexpr int kDfThreads = 288;  // warps 0-7 consume (two groups of four), warp 8 produces
constexpr int kDfStageBytes = 32 * 1024;
constexpr int kDfMaxStages = 6;
constexpr int kDfMaxPairs = 64;   // T * top_k
constexpr int kDfMaxRows = 32;    // phase-2 output rows per CTA (H / grid)
constexpr int kDfMaxChunks = 512;
constexpr long long kDfWaitLimit = 4000000000LL;
constexpr int32_t kErrDecodeTimeout = 32;

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
#else
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
  int T, top_k, H, I, E, wave, sub, stages, fuse_combine;
  const int32_t* plan;
  Workspace ws;
  const uint8_t* arena;
  size_t stride;
  ExpertLayout lay;
  int32_t* err;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t par, volatile int* abort_flag, int32_t* err) {
  if (mb_try(b, par)) return true;
  const long long t0 = clock64();
  while (!mb_try(b, par)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kDfWaitLimit) {
      *abort_flag = 1;
      atomicOr(err, kErrDecodeTimeout);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_acq_rel_add(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void group_sync(int grp) { asm volatile("bar.sync %0, 128;" ::"r"(2 + grp) : "memory"); }
// Group barrier that ORs a predicate over the group's 128 threads: a failed wait in any
// warp makes the whole group leave together (no warp is left at a named barrier).
__device__ __forceinline__ int group_bar_or(int grp, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %2, 0;\n\tbar.red.or.pred q, %1, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(2 + grp), "r"(pred)
      : "memory");
  return r;
}

struct ChunkList {
  int n1, n2, n_lo, n_hi;
};

// Chunks of one CTA. Phase 1: every expert's I row pairs are cut into cpe = ceil(I/rj1)
// chunks of rj1 rows; the n_we*cpe chunks are dealt out in one contiguous range per CTA
// (so a CTA streams long contiguous runs and no chunk crosses an expert). Phase 2:
// (expert index, first output row, count) over the CTA's output rows, every expert.
// Entry q is computed by thread q from its index alone.
__device__ ChunkList chunk_bounds(int b, int G, int n_we, int I, int H, int rj1, int rd, int* g0, int* c2) {
  ChunkList cl;
  const int cpe = (I + rj1 - 1) / rj1;
  const long long total = (long long)n_we * cpe;
  *g0 = (int)(total * b / G);
  cl.n1 = (int)(total * (b + 1) / G) - *g0;
  cl.n_lo = (int)((long long)H * b / G);
  cl.n_hi = (int)((long long)H * (b + 1) / G);
  *c2 = (cl.n_hi - cl.n_lo + rd - 1) / rd;
  cl.n2 = n_we * *c2;
  if (cl.n1 + cl.n2 > kDfMaxChunks) {  // excluded on the host; never write past the list
    cl.n1 = 0;
    cl.n2 = 0;
  }
  return cl;
}

__device__ int4 chunk_entry(int q, const ChunkList& cl, int g0, int c2, int I, int rj1, int rd) {
  if (q < cl.n1) {
    const int cpe = (I + rj1 - 1) / rj1;
    const int g = g0 + q, i = g / cpe, j = (g - i * cpe) * rj1;
    return make_int4(1, i, j, min(rj1, I - j));
  }
  const int qq = q - cl.n1, i = qq / c2, r = cl.n_lo + (qq - i * c2) * rd;
  return make_int4(2, i, r, min(rd, cl.n_hi - r));
}

template <int FMT, int NCH1, int NCH2>
__global__ void __launch_bounds__(kDfThreads, 1) decode_fused_kernel(const DfArgs a) {
  constexpr int EPC = Fmt<FMT>::EPC;
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ ChunkList s_cl;
  __shared__ int4 s_we[kDfMaxPairs];  // per wave expert: (expert, slot, first grouped pair, end)
  __shared__ int s_tok[kDfMaxPairs];  // token of each grouped pair
  __shared__ int s_pos[kDfMaxPairs];  // grouped position of each pair (t*k + r), -1 if invalid
  __shared__ int s_ids[kDfMaxPairs];

  const int S = a.stages;
  uint8_t* ring = dsm;
  uint4* x_s = reinterpret_cast<uint4*>(ring + (size_t)S * kDfStageBytes);
  float* o_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(x_s) + (size_t)a.T * a.H * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(o_s + kDfMaxPairs * kDfMaxRows);
  uint64_t* empty = full + kDfMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kDfMaxStages);
  int4* chunks = reinterpret_cast<int4*>(empty + kDfMaxStages + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) DF_TRACE(0);
  const PlanLayout L{a.E};
  const int P = a.T * a.top_k;
  // one round of independent loads: the plan words this launch needs and the ids
  __shared__ int s_hdr[4];
  if (threadIdx.x == 0) s_hdr[0] = a.plan[kPlanWaves];
  if (threadIdx.x == 32) s_hdr[1] = a.plan[L.wave_start() + a.wave];
  if (threadIdx.x == 64) s_hdr[2] = a.plan[L.wave_start() + a.wave + 1];
  if (threadIdx.x == 96) s_hdr[3] = a.plan[L.wave_hits() + a.wave];
  if (threadIdx.x >= 128 && threadIdx.x < 128 + P) s_ids[threadIdx.x - 128] = a.ids[threadIdx.x - 128];
  __syncthreads();
  if (a.wave >= s_hdr[0]) return;
  int w0 = s_hdr[1], w1 = s_hdr[2];
  if (a.sub == 1) w1 = w0 + s_hdr[3];
  else if (a.sub == 2) w0 = w0 + s_hdr[3];
  const int n_we = w1 - w0;
  const size_t rbg = (size_t)a.H * Fmt<FMT>::BPE2 / 2;  // one gate (or up) row
  const size_t rbd = (size_t)a.I * Fmt<FMT>::BPE2 / 2;  // one down row
  const size_t hrow = (size_t)a.I * 2;                  // one h row (bf16)
  const int rj1 = (int)(kDfStageBytes / (2 * rbg));
  const size_t h_room = (size_t)a.T * hrow;              // an expert has at most T pairs
  const int rd = (int)((kDfStageBytes - h_room) / rbd);
  const size_t h_off = ((size_t)rd * rbd + 15) & ~(size_t)15;
  unsigned* done = a.ws.done;

  // grouping: stable by expert id, then pair index
  __shared__ int2 s_wl[kDfMaxPairs];  // the launch's wave experts and slots, loaded in parallel
  if (threadIdx.x < n_we)
    s_wl[threadIdx.x] = make_int2(a.plan[L.wave_exp() + w0 + threadIdx.x], a.plan[L.wave_slot() + w0 + threadIdx.x]);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mb_init(&full[s], 1);
      mb_init(&empty[s], 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  int g0, c2;
  const ChunkList clb = chunk_bounds(blockIdx.x, gridDim.x, n_we, a.I, a.H, rj1, rd, &g0, &c2);
  for (int q = threadIdx.x; q < clb.n1 + clb.n2; q += blockDim.x) chunks[q] = chunk_entry(q, clb, g0, c2, a.I, rj1, rd);
  if (threadIdx.x == 0) s_cl = clb;
  __syncthreads();
  if (threadIdx.x < P) {
    const int p = threadIdx.x, id = s_ids[p];
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
  if (threadIdx.x < n_we) {
    const int2 es = s_wl[threadIdx.x];
    int lo = 0, cnt = 0;
    for (int q = 0; q < P; ++q) {
      const int o = s_ids[q];
      lo += (o >= 0 && o < es.x) ? 1 : 0;
      cnt += (o == es.x) ? 1 : 0;
    }
    s_we[threadIdx.x] = make_int4(es.x, es.y, lo, lo + cnt);
  }
  __syncthreads();
  if (threadIdx.x == 0) DF_TRACE(1);
  const ChunkList ch = s_cl;
  const int n_chunks = ch.n1 + ch.n2;

  if (warp == 8) {
    // ---------------- producer warp. Lane 0 issues each chunk's weight copies as soon as
    // its stage is free (phase-2 chunks announce their h bytes too); meanwhile the lanes
    // poll the completion counters of up to 32 issued phase-2 chunks at once, and lane i
    // issues the h copy of the chunk whose completion it observed.
    __shared__ int s_ready[kDfMaxPairs];  // expert index -> its h is complete (observed)
    for (int i = lane; i < n_we; i += 32) s_ready[i] = 0;
    __syncwarp();
    int k = 0, kh = ch.n1;
    long long last = clock64();
    while (true) {
      // every branch below is decided by lane 0 (or a ballot) and broadcast, so the warp
      // stays converged
      int stop = ((k >= n_chunks && kh >= n_chunks) || *abort_flag) ? 1 : 0;
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (stop) break;
      // issue every chunk whose stage is free (weights; phase-2 chunks also announce h)
      int n_issued = 0;
      if (lane == 0) {
        while (k + n_issued < n_chunks &&
               mb_try(&empty[(k + n_issued) % S], (uint32_t)(((k + n_issued) / S) & 1) ^ 1u)) {
          const int kk = k + n_issued, s = kk % S;
          const int4 cd = chunks[kk];
          const int4 we = s_we[cd.y];
          const uint8_t* ex = a.arena + (size_t)we.y * a.stride;
          uint8_t* st = ring + (size_t)s * kDfStageBytes;
          if (cd.x == 1) {
            const uint32_t bytes = (uint32_t)(cd.w * rbg);
            mb_expect(&full[s], 2 * bytes);
            bulk_g2s(st, ex + a.lay.gu_w + (size_t)cd.z * rbg, bytes, &full[s]);
            bulk_g2s(st + (size_t)rj1 * rbg, ex + a.lay.gu_w + (size_t)(a.I + cd.z) * rbg, bytes, &full[s]);
          } else {
            const uint32_t wbytes = (uint32_t)(cd.w * rbd);
            const uint32_t hbytes = (uint32_t)((we.w - we.z) * hrow);
            mb_expect(&full[s], wbytes + hbytes);
            bulk_g2s(st, ex + a.lay.d_w + (size_t)cd.z * rbd, wbytes, &full[s]);
          }
          ++n_issued;
        }
      }
      n_issued = __shfl_sync(0xffffffffu, n_issued, 0);
      k += n_issued;
      bool progressed = n_issued > 0;
      // h copies of issued phase-2 chunks whose expert is complete; the completion
      // counters are read (one L2 round trip) only when nothing else could be issued
      if (kh < k) {
        const int q = kh + lane;
        int ready = 0;
        int4 we = make_int4(0, 0, 0, 0);
        if (q < k) {
          const int ei = chunks[q].y;
          we = s_we[ei];
          ready = s_ready[ei];
          if (!ready && n_issued == 0) {
            ready = ld_acquire(done + we.x) >= (unsigned)a.I ? 1 : 0;
            if (ready) s_ready[ei] = 1;
          }
        }
        const unsigned m = __ballot_sync(0xffffffffu, ready);
        const int n_ready = (m == 0xffffffffu) ? 32 : (__ffs(~m) - 1);  // leading run of ready chunks
        if (lane < n_ready) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          const uint32_t hbytes = (uint32_t)((we.w - we.z) * hrow);
          if (hbytes > 0) {
            const int s = q % S;
            bulk_g2s(ring + (size_t)s * kDfStageBytes + h_off, a.ws.h + (size_t)we.z * a.I, hbytes, &full[s]);
          }
        }
        __syncwarp();
        if (n_ready > 0) {
          kh += n_ready;
          progressed = true;
        }
      }
      if (progressed) {
        last = clock64();
      } else {
        int expired = (clock64() - last > kDfWaitLimit) ? 1 : 0;
        expired = __shfl_sync(0xffffffffu, expired, 0);
        if (expired) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(a.err, kErrDecodeTimeout);
          }
          break;
        }
      }
    }
  } else {
    // ---------------- consumers (warps 0-7): group grp takes chunks k = grp, grp+2, ...
    const int nv = a.H / 8;
    for (int i = threadIdx.x; i < a.T * nv; i += 256) x_s[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
    consumers_sync();
    const int grp = warp >> 2, wl = warp & 3;
    const int nch1 = (int)(rbg / 16), nch2 = (int)(rbd / 16);
    const bool fuse = a.fuse_combine != 0 && a.sub == 0 && a.plan[kPlanWaves] == 1;
    int pending_rows = 0;
    for (int k = grp; k < n_chunks; k += 2) {
      const int s = k % S;
      const bool got = mb_wait(&full[s], (uint32_t)((k / S) & 1), abort_flag, a.err);
      if (group_bar_or(grp, got ? 0 : 1)) break;
      if (k == 0 && lane == 0) DF_TRACE(2);
      if (k == ch.n1 && lane == 0) DF_TRACE(3);
      if (k == ch.n1 - 1 && lane == 0) DF_TRACE(6);  // wait for this CTA's last phase-1 chunk
      const int4 cd = chunks[k];
      const int4 we = s_we[cd.y];
      const uint8_t* ex = a.arena + (size_t)we.y * a.stride;
      const uint8_t* st = ring + (size_t)s * kDfStageBytes;
      if (cd.x == 1) {
        for (int rp = wl; rp < cd.w; rp += 4) {
          const uint4* grow = reinterpret_cast<const uint4*>(st + (size_t)rp * rbg);
          const uint4* urow = reinterpret_cast<const uint4*>(st + (size_t)(rj1 + rp) * rbg);
          uint4 gw[NCH1], uw[NCH1];
#pragma unroll
          for (int c = 0; c < NCH1; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nch1) {
              gw[c] = grow[idx];
              uw[c] = urow[idx];
            }
          }
          const int j = cd.z + rp;
          for (int gp = we.z; gp < we.w; ++gp) {
            const uint4* xr = x_s + (size_t)s_tok[gp] * nv;
            float g = 0.f, u = 0.f;
#pragma unroll
            for (int c = 0; c < NCH1; ++c) {
              const int idx = lane + 32 * c;
              if (idx < nch1) {
                const ChunkQ qg = chunk_q<FMT>(ex + a.lay.gu_s, j, idx, a.H);
                const ChunkQ qu = chunk_q<FMT>(ex + a.lay.gu_s, a.I + j, idx, a.H);
                g += chunk_dot<FMT, true>(gw[c], xr + idx * (EPC / 8), qg);
                u += chunk_dot<FMT, true>(uw[c], xr + idx * (EPC / 8), qu);
              }
            }
            g = warp_sum(g);
            u = warp_sum(u);
            if (lane == 0) a.ws.h[(size_t)gp * a.I + j] = __float2bfloat16_rn(silu_mul(g, u));
          }
        }
        group_sync(grp);
        if (wl == 0 && lane == 0) {
          mb_arrive(&empty[s]);
          // publish this group's finished rows once per expert (a release costs a round
          // trip to L2): when its next chunk is another expert or not a phase-1 chunk
          pending_rows += cd.w;
          const int kn = k + 2;
          if (kn >= ch.n1 || chunks[kn].y != cd.y) {
            red_release_add(done + we.x, (unsigned)pending_rows);
            pending_rows = 0;
          }
        }
      } else {
        const uint4* hs = reinterpret_cast<const uint4*>(st + h_off);
        for (int gp = we.z; gp < we.w; ++gp) {
          const uint4* hq = hs + (size_t)(gp - we.z) * (a.I / 8);
          for (int rr = wl; rr < cd.w; rr += 4) {
            const uint4* row = reinterpret_cast<const uint4*>(st + (size_t)rr * rbd);
            const int n = cd.z + rr;
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < NCH2; ++c) {
              const int idx = lane + 32 * c;
              if (idx < nch2) {
                const ChunkQ q = chunk_q<FMT>(ex + a.lay.d_s, n, idx, a.I);
                acc += chunk_dot<FMT, true>(row[idx], hq + idx * (EPC / 8), q);
              }
            }
            acc = warp_sum(acc);
            if (lane == 0) {
              if (fuse) o_s[gp * kDfMaxRows + (n - ch.n_lo)] = acc;
              else a.ws.o_part[(size_t)gp * a.H + n] = acc;
            }
          }
        }
        group_sync(grp);
        if (wl == 0 && lane == 0) mb_arrive(&empty[s]);
      }
    }
    consumers_sync();
    if (threadIdx.x == 0) DF_TRACE(4);
    if (fuse && !*abort_flag) {
      const int rows = ch.n_hi - ch.n_lo;
      for (int idx = threadIdx.x; idx < a.T * rows; idx += 256) {
        const int t = idx / rows, nl = idx - t * rows;
        float acc = 0.f;
        for (int r = 0; r < a.top_k; ++r) {
          const int gp = s_pos[t * a.top_k + r];
          if (gp < 0) continue;
          acc = fmaf(a.w[t * a.top_k + r], o_s[gp * kDfMaxRows + nl], acc);
        }
        const size_t off = (size_t)t * a.H + ch.n_lo + nl;
        if (a.residual != nullptr) acc = __bfloat162float(a.residual[off]) + acc;
        a.y[off] = __float2bfloat16_rn(acc);
      }
    }
  }
  // the last CTA out resets the completion counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atom_acq_rel_add(a.ws.gbar, 1u);
    if (prev == gridDim.x - 1) {
      for (int i = 0; i < n_we; ++i) done[s_we[i].x] = 0u;
      atomicExch(a.ws.gbar, 0u);
      __threadfence();
    }
    DF_TRACE(5);
  }
}

template <int FMT, int NCH1, int NCH2>
cudaError_t launch_df(const DfArgs& a, int grid, size_t smem, cudaStream_t s) {
  auto k = decode_fused_kernel<FMT, NCH1, NCH2>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // cooperative (all CTAs co-resident), launched through cudaLaunchKernelEx so that the
  // launch can also be recorded into a CUDA graph
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

size_t fmt_row_bytes(int fmt, int n) {
  return fmt == PMOE_BF16 ? (size_t)n * 2 : fmt == PMOE_FP8_BLOCK128 ? (size_t)n : (size_t)n / 2;
}

size_t df_fixed_smem(int T, int H) {
  return (size_t)T * H * 2 + kDfMaxPairs * kDfMaxRows * 4 + 2 * kDfMaxStages * 8 + 16 + kDfMaxChunks * sizeof(int4);
}

}  // namespace

#ifdef PMOE_TRACE
extern "C" __attribute__((visibility("default"))) int pmoe_debug_decode_trace(unsigned long long* out, int n_ctas) {
  return cudaMemcpyFromSymbol(out, g_df_trace, (size_t)n_ctas * 8 * sizeof(unsigned long long)) == cudaSuccess ? 0 : -4;
}
#endif

bool decode_fused_supported(int fmt, int T, int top_k, int H, int I, int num_sms) {
  if (T < 1 || T * top_k > kDfMaxPairs || num_sms < 1 || num_sms > 1024) return false;
  if ((H + num_sms - 1) / num_sms > kDfMaxRows) return false;
  const size_t rbg = fmt_row_bytes(fmt, H), rbd = fmt_row_bytes(fmt, I);
  if (rbg % 16 != 0 || rbd % 16 != 0) return false;
  if (2 * rbg > (size_t)kDfStageBytes) return false;
  const size_t h_room = (size_t)T * I * 2;
  if (h_room + rbd > (size_t)kDfStageBytes) return false;
  const int nch1 = (int)(rbg / 16), nch2 = (int)(rbd / 16);
  if (nch1 > 32 * 8 || nch2 > 32 * 4) return false;
  const size_t budget = 225 * 1024;  // leaves room for the static shared arrays
  if (df_fixed_smem(T, H) + 2 * (size_t)kDfStageBytes > budget) return false;
  // chunk list bound: every expert contributes ceil(rows/rj1) + ceil(out rows/rd) chunks
  const long long n_we = (long long)T * top_k;
  const long long rj1 = kDfStageBytes / (2 * (long long)rbg);
  const long long rd = (kDfStageBytes - (long long)h_room) / (long long)rbd;
  const long long nrows = (H + num_sms - 1) / num_sms;
  const long long bound = (n_we * ((I + rj1 - 1) / rj1) + num_sms - 1) / num_sms + n_we * ((nrows + rd - 1) / rd);
  return bound <= kDfMaxChunks;
}

cudaError_t launch_decode_fused(int fmt, const __nv_bfloat16* x, const int32_t* ids, const float* w,
                                const __nv_bfloat16* residual, __nv_bfloat16* y, int T, int top_k, int H, int I,
                                const int32_t* plan, int E, int wave, int sub, int fuse_combine, const Workspace& ws,
                                const uint8_t* arena, size_t stride, int32_t* err, int num_sms, cudaStream_t s) {
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
  a.plan = plan;
  a.ws = ws;
  a.arena = arena;
  a.stride = stride;
  a.lay = expert_layout(fmt, H, I);
  a.err = err;
  const size_t fixed = df_fixed_smem(T, H);
  const size_t budget = 225 * 1024;  // leaves room for the static shared arrays
  int stages = (int)((budget - fixed) / kDfStageBytes);
  if (stages > kDfMaxStages) stages = kDfMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  a.stages = stages;
  const size_t smem = (size_t)stages * kDfStageBytes + fixed;
  const int nch1 = (int)(fmt_row_bytes(fmt, H) / 16), nch2 = (int)(fmt_row_bytes(fmt, I) / 16);
#define PMOE_DF(F, A, B) return launch_df<F, A, B>(a, num_sms, smem, s)
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
  }
#undef PMOE_DF
  return cudaErrorInvalidValue;
}

}  // namespace pmoe
