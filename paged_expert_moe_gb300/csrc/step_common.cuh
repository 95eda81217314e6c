// Device pieces of a decode step: the router's per-token top-k (one warp per token) and
// the residency step's LRU planning over a table held in shared memory (one block of up
// to 1024 threads, one thread per expert id and per slot).
//
// Article "Running an MoE Model Larger Than Your VRAM": section "What does Paged Experts
// actually do?" (the router picks top_k experts per token; routed experts that are not
// resident are copied in, evicting the oldest-used) and section "What happens with more
// than one request?" (more distinct experts than slots -> several waves).
#pragma once

#include "pmoe_internal.h"

#include <math.h>

namespace pmoe {
namespace step {

// Top-k of one token's E logits by one warp; lane l holds logits e = l + 32 * i, i < NPL.
// Selection by descending logit, ties to the lower id; weights are the softmax over the
// selected logits (renorm) or over all E. row, ids_row and w_row may point to global or
// shared memory.
template <int NPL>
__device__ __forceinline__ void warp_topk(const float* row, int E, int top_k, int renorm, int32_t* ids_row,
                                          float* w_row) {
  const int lane = threadIdx.x & 31;
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;

  float my_sel = -INFINITY;  // lane r keeps the r-th selected logit
  int my_id = -1;
  float vmax = 0.f;
  for (int r = 0; r < top_k; ++r) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && (v[i] > bv || be == 0x7fffffff)) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be) || (be == 0x7fffffff && oe != 0x7fffffff)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane && be != 0x7fffffff) taken |= 1u << (be >> 5);
    if (r == 0) vmax = bv;
    if (lane == r) {
      my_sel = bv;
      my_id = be;
    }
  }
  // softmax pieces: the full denominator (only needed without renormalisation)
  float denom;
  const float e_sel = (lane < top_k) ? expf(my_sel - vmax) : 0.f;
  if (renorm) {
    denom = e_sel;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  } else {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i < E) sum += expf(v[i] - vmax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    denom = sum;
  }
  if (lane < top_k) {
    ids_row[lane] = my_id;
    w_row[lane] = e_sel / denom;
  }
}

// Exclusive prefix sum over the NT threads of the block, one int each; *total receives
// the sum. s_warp holds at least 33 ints.
template <int NT>
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "whole warps, at most 32 of them");
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < NW ? s_warp[lane] : 0;
    int wx = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wx, off);
      if (lane >= off) wx += y;
    }
    s_warp[lane] = wx - w;  // exclusive warp offsets
    if (lane == 31) s_warp[32] = wx;
  }
  __syncthreads();
  const int r = s_warp[warp] + x - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

// Shared-memory table and scratch of one residency step (E, K <= the block's threads).
struct LruSmem {
  int* pend;      // [E] routed this step and not yet placed in a wave
  int* slot_of;   // [E] slot of each expert, -1 absent
  int* exp_in;    // [K] expert in each slot, -1 empty
  int* last;      // [K] step of each slot's last use, -1 empty
  int* unprot;    // [K] slot may be evicted in the current wave
  int* rank_exp;  // [E] the wave's misses in ascending id
  int* warp;      // [33] scan scratch
  int* bad;       // [1] an id outside [0, E) was routed
};

struct LruCounts {
  int unique, misses, waves;
};

// One residency step over the table in m (slot_of, exp_in, last loaded; pend zeroed;
// *bad = 0), every thread of an NT-thread block taking part. Rules (the readings where
// the pages are silent):
//   * every expert used in the step gets last_use = step;
//   * victims are unprotected slots (empty, or holding an expert not pending in this
//     step) in ascending (last_use, slot) order; empty slots have last_use = -1;
//   * a wave holds every pending resident expert plus the lowest-id non-resident
//     pending experts that fit in the remaining K - |resident| slots;
//   * the i-th miss (ascending expert id) takes the i-th victim;
//   * the wave list puts the experts that were resident (hits) first, then the wave's
//     misses, each part in ascending id.
// Thread t owns expert id t and slot t. The table in m is updated in place; the wave
// and miss lists, wave_of and the per-wave starts and hit counts go to plan (global or
// shared memory); the header words are the caller's.
template <int NT>
__device__ LruCounts lru_plan_core(const int32_t* ids, int n_ids, int E, int K, int step, const LruSmem& m,
                                   int32_t* plan) {
  const PlanLayout L{E};
  const int tid = threadIdx.x;
  if (tid < E) plan[L.wave_of() + tid] = -1;
  for (int p = tid; p < n_ids; p += NT) {
    const int e = ids[p];
    if (e < 0 || e >= E) *m.bad = 1;
    else m.pend[e] = 1;
  }
  __syncthreads();
  LruCounts out{0, 0, 0};
  out.unique = __syncthreads_count(tid < E && m.pend[tid]);

  int wave = 0, n_miss = 0, n_wexp = 0;
  while (true) {
    const bool pend = tid < E && m.pend[tid] != 0;
    if (__syncthreads_count(pend) == 0 || wave >= E) break;
    const bool res = pend && m.slot_of[tid] >= 0;
    const bool nonres = pend && !res;
    const int n_res = __syncthreads_count(res);
    const int cap = K - n_res;
    int n_nonres;
    const int rank = block_exclusive_scan<NT>(nonres ? 1 : 0, m.warp, &n_nonres);
    const int n_load = n_nonres < cap ? n_nonres : cap;
    if (nonres && rank < n_load) m.rank_exp[rank] = tid;
    bool unprot = false;
    if (tid < K) {
      const int x = m.exp_in[tid];
      unprot = (x < 0) || (m.pend[x] == 0);
      m.unprot[tid] = unprot ? 1 : 0;
    }
    __syncthreads();
    if (unprot) {
      const int my_last = m.last[tid];
      int vr = 0;
      for (int v = 0; v < K; ++v)
        vr += (m.unprot[v] && (m.last[v] < my_last || (m.last[v] == my_last && v < tid))) ? 1 : 0;
      if (vr < n_load) {
        const int e_new = m.rank_exp[vr];
        const int old = m.exp_in[tid];
        if (old >= 0) m.slot_of[old] = -1;
        m.exp_in[tid] = e_new;
        m.slot_of[e_new] = tid;
        plan[L.miss_exp() + n_miss + vr] = e_new;
        plan[L.miss_slot() + n_miss + vr] = tid;
      }
    }
    __syncthreads();
    const bool inw = tid < E && m.pend[tid] != 0 && m.slot_of[tid] >= 0;
    const bool inw_hit = inw && res;
    int n_w, n_h;
    const int hrank = block_exclusive_scan<NT>(inw_hit ? 1 : 0, m.warp, &n_h);
    const int mrank = block_exclusive_scan<NT>((inw && !inw_hit) ? 1 : 0, m.warp, &n_w);
    n_w += n_h;
    if (inw) {
      const int slot = m.slot_of[tid];
      const int at = n_wexp + (inw_hit ? hrank : n_h + mrank);
      plan[L.wave_exp() + at] = tid;
      plan[L.wave_slot() + at] = slot;
      plan[L.wave_of() + tid] = wave;
      m.last[slot] = step;
    }
    if (tid == 0) {
      plan[L.wave_start() + wave] = n_wexp;
      plan[L.miss_start() + wave] = n_miss;
      plan[L.wave_hits() + wave] = n_h;
    }
    __syncthreads();
    if (inw) m.pend[tid] = 0;
    n_wexp += n_w;
    n_miss += n_load;
    ++wave;
    __syncthreads();
  }
  if (tid == 0) {
    plan[L.wave_start() + wave] = n_wexp;
    plan[L.miss_start() + wave] = n_miss;
    plan[L.wave_hits() + wave] = 0;
  }
  out.misses = n_miss;
  out.waves = wave;
  return out;
}

}  // namespace step
}  // namespace pmoe
