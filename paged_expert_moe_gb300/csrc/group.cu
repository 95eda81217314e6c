// Token -> expert grouping: histogram, exclusive scan, stable permutation, the
// per-wave tile list of the tensor-core path, and the row gather of activations.
//
// Article "Running an MoE Model Larger Than Your VRAM", section "What does Paged
// Experts actually do?": once the routed experts are resident the fused MoE runs
// over them, i.e. the (token, rank) pairs are grouped by expert. Pair p = t*top_k + r.
//   counts[e]  pairs routed to e;   offs = exclusive scan of counts (offs[E] = P)
//   perm[j]    pairs grouped by expert ascending, ascending pair index inside one
//              expert (stable), so the grouping is deterministic;   pos = perm^-1
// Large P: per-chunk histograms, a per-expert scan over chunks, then each pair's
// stable position from its chunk's prefix and its rank among equal ids before it.
// A pair whose id is outside [0, E) is left out (pos = -1) and flagged.
// Block-FP8 layers on the tensor path gather x as two e4m3 planes on a per-row
// power-of-two scale instead (fp8_planes.cuh).
#include "fp8_planes.cuh"
#include "pmoe_internal.h"

namespace pmoe {
namespace {

constexpr int kChunk = 256;  // pairs per CTA in the large-P grouping

// Pass 1 (one CTA per chunk of 256 pairs): per-chunk histogram chunk_cnt[chunk][e].
__global__ void __launch_bounds__(kChunk) group_chunk_hist(const int32_t* __restrict__ ids, int P, int E,
                                                           int32_t* __restrict__ chunk_cnt, int32_t* __restrict__ err) {
  __shared__ int s_cnt[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int p = blockIdx.x * kChunk + threadIdx.x;
  if (p < P) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    else if (err != nullptr) atomicOr(err, kErrBadExpertId);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_cnt[(size_t)blockIdx.x * E + e] = s_cnt[e];
}

// Pass 2 (one warp per expert): counts[e] and, in place, the exclusive prefix of
// chunk_cnt[.][e] over chunks (the pairs of e in earlier chunks). Lane l takes the
// chunks [l * seg, (l + 1) * seg): their sum, a warp scan of the lane sums, then the
// prefixes. Loads go 16 at a time, so a lane's segment costs a few L2 round trips
// instead of one per chunk.
__global__ void __launch_bounds__(256) group_chunk_scan(int n_chunks, int E, int32_t* __restrict__ chunk_cnt,
                                                        int32_t* __restrict__ counts) {
  constexpr int kBatch = 16;
  const int e = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;  // e is the same for the whole warp
  const int seg = (n_chunks + 31) / 32;
  const int c0 = min(n_chunks, lane * seg), c1 = min(n_chunks, c0 + seg);
  int sum = 0;
  for (int b = c0; b < c1; b += kBatch) {
    int v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) v[i] = (b + i < c1) ? chunk_cnt[(size_t)(b + i) * E + e] : 0;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) sum += v[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) counts[e] = incl;
  int run = incl - sum;
  for (int b = c0; b < c1; b += kBatch) {
    int v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) v[i] = (b + i < c1) ? chunk_cnt[(size_t)(b + i) * E + e] : 0;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (b + i < c1) chunk_cnt[(size_t)(b + i) * E + e] = run;
      run += v[i];
    }
  }
}

// Pass 4 (one CTA per chunk): stable position of every pair:
// pos = offs[e] + (pairs of e in earlier chunks) + (pairs of e earlier in this chunk).
__global__ void __launch_bounds__(kChunk) group_chunk_place(const int32_t* __restrict__ ids, int P, int E,
                                                            const int32_t* __restrict__ chunk_pre, Workspace ws) {
  __shared__ int s_ids[kChunk];
  const int p = blockIdx.x * kChunk + threadIdx.x;
  const int id = (p < P) ? ids[p] : -1;
  s_ids[threadIdx.x] = id;
  __syncthreads();
  if (p >= P) return;
  if (id < 0 || id >= E) {
    ws.pos[p] = -1;
    return;
  }
  int before = 0;
  for (int i = 0; i < (int)threadIdx.x; ++i) before += (s_ids[i] == id);
  const int j = ws.offs[id] + chunk_pre[(size_t)blockIdx.x * E + id] + before;
  ws.perm[j] = p;
  ws.pos[p] = j;
}

// offs = scan(counts); per-wave tiles of at most tile_n pairs. One CTA of 1024 threads,
// counts already in ws.counts (written by this CTA before a barrier, or by an earlier
// launch).
__device__ void offs_and_tiles(int E, const int32_t* __restrict__ plan, const Workspace& ws, int tile_n,
                               int32_t* __restrict__ err) {
  __shared__ int s_v[kMaxExperts + 1];
  __shared__ int s_t[kMaxExperts + 1];
  const int tid = threadIdx.x;
  const PlanLayout L{E};
  // offs: inclusive Hillis-Steele scan (E <= 1024, fixed order -> deterministic)
  s_v[tid] = (tid < E) ? ws.counts[tid] : 0;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int add = (tid >= off) ? s_v[tid - off] : 0;
    __syncthreads();
    s_v[tid] += add;
    __syncthreads();
  }
  if (tid < E) ws.offs[tid + 1] = s_v[tid];
  if (tid == 0) ws.offs[0] = 0;
  if (plan == nullptr || tile_n <= 0) return;
  // tiles, in the plan's wave order (ascending expert id within a wave)
  const int n_waves = plan[kPlanWaves];
  const int n_wexp = plan[L.wave_start() + n_waves];
  int my_tiles = 0, e = -1, cnt = 0;
  if (tid < n_wexp) {
    e = plan[L.wave_exp() + tid];
    cnt = ws.counts[e];
    my_tiles = (cnt + tile_n - 1) / tile_n;
  }
  s_t[tid] = my_tiles;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int add = (tid >= off) ? s_t[tid - off] : 0;
    __syncthreads();
    s_t[tid] += add;
    __syncthreads();
  }
  const int first = s_t[tid] - my_tiles;
  if (tid < n_wexp && my_tiles > 0) {
    const int slot = plan[L.wave_slot() + tid];
    const int e_off = (e == 0) ? 0 : s_v[e - 1];  // offs[e]
    // even split, chunk rounded up to a multiple of 16 pairs
    int chunk = (cnt + my_tiles - 1) / my_tiles;
    chunk = (chunk + 15) & ~15;
    for (int i = 0; i < my_tiles; ++i) {
      const int idx = first + i;
      if (idx >= ws.max_tiles) {
        atomicOr(err, kErrPlanOverflow);
        break;
      }
      const int start = i * chunk;
      const int n = (cnt - start < chunk) ? (cnt - start) : chunk;
      ws.tiles[3 * idx + 0] = slot;
      ws.tiles[3 * idx + 1] = e_off + start;
      ws.tiles[3 * idx + 2] = n > 0 ? n : 0;
    }
  }
  __syncthreads();
  if (tid <= n_waves) {
    const int j = plan[L.wave_start() + tid];  // first wave-list index of wave tid
    int t = (j == 0) ? 0 : s_t[j - 1];
    if (t > ws.max_tiles) t = ws.max_tiles;
    ws.tile_wave[tid] = t;
    const int jh = j + (tid < n_waves ? plan[L.wave_hits() + tid] : 0);  // first non-resident expert
    int th = (jh == 0) ? 0 : s_t[jh - 1];
    if (th > ws.max_tiles) th = ws.max_tiles;
    ws.tile_split[tid] = th;
  }
}

__global__ void __launch_bounds__(1024) group_scan_tiles(int E, const int32_t* __restrict__ plan, Workspace ws,
                                                         int tile_n, int32_t* __restrict__ err) {
  offs_and_tiles(E, plan, ws, tile_n, err);
}

// Single CTA, the whole grouping in one launch: a stable counting sort. The ids, the
// per-warp histograms and perm live in shared memory (4 P + 128 E + 4 P bytes). The
// ranking within a batch costs ~140 cycles per warp, so four launches over many CTAs
// beat it beyond kGroupOneCtaMaxPairs. Warp w
// takes the pairs [w * per, (w + 1) * per) in batches of 32; lanes of a batch with the
// same id are ranked by lane (match + popcount), so an expert's pairs keep ascending
// order. s_hist[w][e] first counts warp w's pairs of e, then holds their next position
// relative to offs[e]. err may be null (bad ids then only get pos = -1).
__global__ void __launch_bounds__(1024) group_one_cta(const int32_t* __restrict__ ids, int P, int E,
                                                      const int32_t* __restrict__ plan, Workspace ws, int tile_n,
                                                      int32_t* __restrict__ err) {
  extern __shared__ int s_dyn[];
  int* s_hist = s_dyn;            // [32][E]
  int* s_ids = s_hist + 32 * E;   // [P]
  int* s_perm = s_ids + P;        // [P]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < P; i += blockDim.x) s_ids[i] = ids[i];
  for (int i = tid; i < 32 * E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int per = (P + 31) / 32;
  const int p0 = warp * per, p1 = min(P, p0 + per);
  int* h = s_hist + warp * E;
  const unsigned below = (1u << lane) - 1u;
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    const int id = p < p1 ? s_ids[p] : -1;
    const bool ok = p < p1 && id >= 0 && id < E;
    if (p < p1 && !ok) {
      ws.pos[p] = -1;
      if (err != nullptr) atomicOr(err, kErrBadExpertId);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1);
    if (ok && (peers & below) == 0) h[id] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = s_hist[w * E + e];
      s_hist[w * E + e] = run;
      run += v;
    }
    ws.counts[e] = run;
  }
  __syncthreads();
  offs_and_tiles(E, plan, ws, tile_n, err);
  __syncthreads();
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    const int id = p < p1 ? s_ids[p] : -1;
    const bool ok = p < p1 && id >= 0 && id < E;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1);
    if (ok) {
      const int j = ws.offs[id] + h[id] + __popc(peers & below);
      s_perm[j] = p;
      ws.pos[p] = j;
    }
    __syncwarp();
    if (ok && (peers & below) == 0) h[id] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  const int n_valid = ws.offs[E];
  for (int j = tid; j < n_valid; j += blockDim.x) ws.perm[j] = s_perm[j];
}

// Single CTA for small P: everything in one launch (decode). Thread e owns expert e.
__global__ void __launch_bounds__(1024) group_small(const int32_t* __restrict__ ids, int P, int E,
                                                    const int32_t* __restrict__ plan, Workspace ws,
                                                    int32_t* __restrict__ err) {
  __shared__ int s_ids[1024];
  __shared__ int s_v[kMaxExperts];
  const int tid = threadIdx.x;
  for (int p = tid; p < P; p += blockDim.x) {
    const int id = ids[p];
    s_ids[p] = id;
    if (id < 0 || id >= E) {
      ws.pos[p] = -1;
      if (err != nullptr) atomicOr(err, kErrBadExpertId);
    }
  }
  __syncthreads();
  int cnt = 0;
  if (tid < E)
    for (int p = 0; p < P; ++p) cnt += (s_ids[p] == tid);
  s_v[tid] = cnt;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int add = (tid >= off) ? s_v[tid - off] : 0;
    __syncthreads();
    s_v[tid] += add;
    __syncthreads();
  }
  if (tid < E) {
    const int base = s_v[tid] - cnt;
    ws.counts[tid] = cnt;
    ws.offs[tid] = base;
    if (tid == E - 1) ws.offs[E] = s_v[tid];
    int j = base;
    for (int p = 0; p < P; ++p)
      if (s_ids[p] == tid) {
        ws.perm[j] = p;
        ws.pos[p] = j;
        ++j;
      }
  }
}

// x_perm[j] = x[perm[j] / top_k]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int P, int top_k,
                                                          int H, __nv_bfloat16* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nvec = H / 8;
  for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < P; j += nwarps) {
    const int t = perm[j] / top_k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)j * H);
    // eight 16-byte loads per lane before their stores: a 4 KB row in flight per warp
    for (int c0 = lane; c0 < nvec; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + 32 * i < nvec) v[i] = __ldg(src + c0 + 32 * i);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + 32 * i < nvec) dst[c0 + 32 * i] = v[i];
    }
  }
}

// Row j of x_perm as two e4m3 planes: hi at xq[j][.], lo at xq[p_cap + j][.], and the
// row's scale sx[j] (x_perm row j ~= sx[j] * (hi + lo)). One warp per row: a pass for the
// row's largest magnitude, then one that splits every value.
__global__ void __launch_bounds__(256) gather_rows_fp8x2_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const int32_t* __restrict__ perm, int P, int top_k,
                                                                int H, size_t p_cap, uint8_t* __restrict__ xq,
                                                                float* __restrict__ sx) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nvec = H / 8;
  for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < P; j += nwarps) {
    const int t = perm[j] / top_k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    float amax = 0.f;
    for (int c = lane; c < nvec; c += 32) {
      const uint4 v = __ldg(src + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float s, inv;
    plane_scale(amax, &s, &inv);
    uint2* hi_row = reinterpret_cast<uint2*>(xq + (size_t)j * H);
    uint2* lo_row = reinterpret_cast<uint2*>(xq + (p_cap + (size_t)j) * H);
    for (int c = lane; c < nvec; c += 32) {
      const uint4 v = __ldg(src + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint16_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        split_e4m3x2(f.x * inv, f.y * inv, &hi[i], &lo[i]);
      }
      hi_row[c] = make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
      lo_row[c] = make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
    }
    if (lane == 0) sx[j] = s;
  }
}

}  // namespace

cudaError_t launch_group_one_cta(const int32_t* ids, int P, int E, const int32_t* plan, Workspace ws, int tile_n,
                                 int32_t* err, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(group_one_cta, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(8 * (size_t)kGroupOneCtaMaxPairs + 128 * (size_t)kMaxExperts));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  group_one_cta<<<1, 1024, 8 * (size_t)P + 128 * (size_t)E, s>>>(ids, P, E, plan, ws, tile_n, err);
  return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, int P, int E, const int32_t* plan, Workspace ws, int tile_n,
                         int32_t* err, cudaStream_t s) {
  if (P <= 1024 && tile_n <= 0) {
    group_small<<<1, 1024, 0, s>>>(ids, P, E, plan, ws, err);
    return cudaGetLastError();
  }
  if (P <= kGroupOneCtaMaxPairs) return launch_group_one_cta(ids, P, E, plan, ws, tile_n, err, s);
  const int n_chunks = (P + kChunk - 1) / kChunk;
  if ((size_t)n_chunks * E > (size_t)ws.chunk_cap) return cudaErrorInvalidValue;
  group_chunk_hist<<<n_chunks, kChunk, 0, s>>>(ids, P, E, ws.chunk_cnt, err);
  group_chunk_scan<<<(32 * E + 255) / 256, 256, 0, s>>>(n_chunks, E, ws.chunk_cnt, ws.counts);
  group_scan_tiles<<<1, 1024, 0, s>>>(E, plan, ws, tile_n, err);
  group_chunk_place<<<n_chunks, kChunk, 0, s>>>(ids, P, E, ws.chunk_cnt, ws);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* perm, int P, int top_k, int H,
                               __nv_bfloat16* x_perm, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  int blocks = (P + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  gather_rows_kernel<<<blocks, 256, 0, s>>>(x, perm, P, top_k, H, x_perm);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_fp8x2(const __nv_bfloat16* x, const int32_t* perm, int P, int top_k, int H,
                                     size_t p_cap, uint8_t* xq, float* sx, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  if (H % 8 != 0 || (size_t)P > p_cap) return cudaErrorInvalidValue;
  int blocks = (P + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  gather_rows_fp8x2_kernel<<<blocks, 256, 0, s>>>(x, perm, P, top_k, H, p_cap, xq, sx);
  return cudaGetLastError();
}

}  // namespace pmoe
