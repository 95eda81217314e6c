// Residency step of one layer's K-slot expert table, on the device (one CTA).
//
// Article "Running an MoE Model Larger Than Your VRAM": TL;DR (copy in only the
// routed experts that are not resident), section "What does Paged Experts actually
// do?" item 3 (least recently used out) and section "What happens with more than one
// request?" (more distinct experts than slots -> several waves, each with its own
// page-in). Post "Locality of reference helped ...", section "The fix": a hit moves
// no bytes, a miss copies one expert and evicts the least recently used one.
//
// Rules (the readings where the pages are silent):
//   * every expert used in a step gets last_use = the layer's step counter;
//   * victims are unprotected slots (empty, or holding an expert not pending in this
//     step) in ascending (last_use, slot) order; empty slots have last_use = -1;
//   * a wave holds every pending resident expert plus the lowest-id non-resident
//     pending experts that fit in the remaining K - |resident| slots;
//   * the i-th miss (ascending expert id) takes the i-th victim.
// One thread owns one expert id and one slot (E, K <= 1024 = blockDim.x).
#include "pmoe_internal.h"

namespace pmoe {
namespace {

constexpr int kThreads = 1024;

// Exclusive block-wide prefix sum of one int per thread; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
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
    int w = s_warp[lane];
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

__device__ __forceinline__ void residency_body(const int32_t* __restrict__ ids, int n_ids, int E, int K,
                                               LayerState st, int32_t* __restrict__ plan, int32_t* __restrict__ err,
                                               unsigned long long* __restrict__ epoch) {
  __shared__ int s_pend[kMaxExperts];
  __shared__ int s_slot_of[kMaxExperts];
  __shared__ int s_exp_in[kMaxExperts];
  __shared__ int s_last[kMaxExperts];
  __shared__ int s_unprot[kMaxExperts];
  __shared__ int s_rank_exp[kMaxExperts];
  __shared__ int s_warp[33];
  __shared__ int s_bad;

  const PlanLayout L{E};
  const int tid = threadIdx.x;
  // The kernel that consumes the plan may launch now and wait for this one to end. The
  // table was last written by this layer's previous residency step, which ended before
  // anything after it in the stream began; the ids and the plan (which the previous
  // step's compute reads) are touched only after the wait for the kernel before this
  // one (the router) to complete.
  pdl_trigger();
  const int step = *st.step;
  if (tid < E) {
    s_pend[tid] = 0;
    s_slot_of[tid] = st.slot_of[tid];
  }
  if (tid < K) {
    s_exp_in[tid] = st.expert_in[tid];
    s_last[tid] = st.last_use[tid];
  }
  if (tid == 0) s_bad = 0;
  pdl_wait();
  if (tid < E) plan[L.wave_of() + tid] = -1;
  __syncthreads();
  for (int p = tid; p < n_ids; p += kThreads) {
    const int e = ids[p];
    if (e < 0 || e >= E) s_bad = 1;
    else s_pend[e] = 1;
  }
  __syncthreads();
  const int n_unique = __syncthreads_count(tid < E && s_pend[tid]);

  int wave = 0, n_miss = 0, n_wexp = 0;
  while (true) {
    const bool pend = tid < E && s_pend[tid] != 0;
    if (__syncthreads_count(pend) == 0 || wave >= E) break;
    const bool res = pend && s_slot_of[tid] >= 0;
    const bool nonres = pend && !res;
    const int n_res = __syncthreads_count(res);
    const int cap = K - n_res;
    int n_nonres;
    const int rank = block_exclusive_scan(nonres ? 1 : 0, s_warp, &n_nonres);
    const int n_load = n_nonres < cap ? n_nonres : cap;
    if (nonres && rank < n_load) s_rank_exp[rank] = tid;
    bool unprot = false;
    if (tid < K) {
      const int x = s_exp_in[tid];
      unprot = (x < 0) || (s_pend[x] == 0);
      s_unprot[tid] = unprot ? 1 : 0;
    }
    __syncthreads();
    if (unprot) {
      const int my_last = s_last[tid];
      int vr = 0;
      for (int v = 0; v < K; ++v)
        vr += (s_unprot[v] && (s_last[v] < my_last || (s_last[v] == my_last && v < tid))) ? 1 : 0;
      if (vr < n_load) {
        const int e_new = s_rank_exp[vr];
        const int old = s_exp_in[tid];
        if (old >= 0) s_slot_of[old] = -1;
        s_exp_in[tid] = e_new;
        s_slot_of[e_new] = tid;
        plan[L.miss_exp() + n_miss + vr] = e_new;
        plan[L.miss_slot() + n_miss + vr] = tid;
      }
    }
    __syncthreads();
    // wave list: the experts that were resident (hits) first, then this wave's misses,
    // each part in ascending id, so compute on the hits can start before the page-in
    const bool inw = tid < E && s_pend[tid] != 0 && s_slot_of[tid] >= 0;
    const bool inw_hit = inw && res;
    int n_w, n_h;
    const int hrank = block_exclusive_scan(inw_hit ? 1 : 0, s_warp, &n_h);
    const int mrank = block_exclusive_scan((inw && !inw_hit) ? 1 : 0, s_warp, &n_w);
    n_w += n_h;
    if (inw) {
      const int slot = s_slot_of[tid];
      const int at = n_wexp + (inw_hit ? hrank : n_h + mrank);
      plan[L.wave_exp() + at] = tid;
      plan[L.wave_slot() + at] = slot;
      plan[L.wave_of() + tid] = wave;
      s_last[slot] = step;
    }
    if (tid == 0) {
      plan[L.wave_start() + wave] = n_wexp;
      plan[L.miss_start() + wave] = n_miss;
      plan[L.wave_hits() + wave] = n_h;
    }
    __syncthreads();
    if (inw) s_pend[tid] = 0;
    n_wexp += n_w;
    n_miss += n_load;
    ++wave;
    __syncthreads();
  }
  if (tid == 0) {
    plan[L.wave_start() + wave] = n_wexp;
    plan[L.miss_start() + wave] = n_miss;
    plan[L.wave_hits() + wave] = 0;
    plan[kPlanUnique] = n_unique;
    plan[kPlanWaves] = wave;
    plan[kPlanMisses] = n_miss;
    plan[kPlanError] = s_bad ? kErrBadExpertId : 0;
    plan[kPlanStep] = step;
    const unsigned long long ep = atomicAdd(epoch, 1ull) + 1ull;
    plan[kPlanEpochLo] = (int32_t)(uint32_t)(ep & 0xffffffffull);
    plan[kPlanEpochHi] = (int32_t)(uint32_t)(ep >> 32);
    if (s_bad) atomicOr(err, kErrBadExpertId);
    *st.step = step + 1;
    st.counters[0] += (unsigned long long)(n_unique - n_miss);
    st.counters[1] += (unsigned long long)n_miss;
    st.counters[2] += (unsigned long long)wave;
    st.counters[3] += 1ull;
  }
  if (tid < E) st.slot_of[tid] = s_slot_of[tid];
  if (tid < K) {
    st.expert_in[tid] = s_exp_in[tid];
    st.last_use[tid] = s_last[tid];
  }
}

__global__ void __launch_bounds__(kThreads) residency_kernel(const int32_t* __restrict__ ids, int n_ids, int E,
                                                             int K, LayerState st, int32_t* __restrict__ plan,
                                                             int32_t* __restrict__ err,
                                                             unsigned long long* __restrict__ epoch) {
  residency_body(ids, n_ids, E, K, st, plan, err, epoch);
}

// Every layer of a stack at once: CTA l plans layer l (the layers' tables are independent,
// and their states and plans lie at fixed strides from layer 0's).
__global__ void __launch_bounds__(kThreads) residency_layers_kernel(const int32_t* __restrict__ ids, int n_ids,
                                                                    int E, int K, LayerState st0, size_t state_stride,
                                                                    int32_t* __restrict__ plan0, int plan_words,
                                                                    int32_t* __restrict__ err,
                                                                    unsigned long long* __restrict__ epoch) {
  const int l = blockIdx.x;
  const size_t d = state_stride * (size_t)l;
  LayerState st;
  st.slot_of = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(st0.slot_of) + d);
  st.expert_in = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(st0.expert_in) + d);
  st.last_use = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(st0.last_use) + d);
  st.step = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(st0.step) + d);
  st.counters = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(st0.counters) + d);
  residency_body(ids + (size_t)l * n_ids, n_ids, E, K, st, plan0 + (size_t)l * plan_words, err, epoch);
}

}  // namespace

cudaError_t launch_residency(const int32_t* ids, int n_ids, int E, int K, LayerState st, int32_t* plan,
                             int32_t* err, unsigned long long* epoch, cudaStream_t s, bool pdl) {
  static bool carveout_set = false;  // keep room for a decode CTA on the same SM
  if (!carveout_set) {
    cudaFuncSetAttribute(residency_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    carveout_set = true;
  }
  if (!pdl) {
    residency_kernel<<<1, kThreads, 0, s>>>(ids, n_ids, E, K, st, plan, err, epoch);
    return cudaGetLastError();
  }
  // may start while the kernel before it (the router) drains; it waits for it before
  // reading the ids
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residency_kernel, ids, n_ids, E, K, st, plan, err, epoch);
}

cudaError_t launch_residency_layers(const int32_t* ids, int n_ids, int layers, int E, int K, LayerState st0,
                                    size_t state_stride, int32_t* plan0, int plan_words, int32_t* err,
                                    unsigned long long* epoch, cudaStream_t s) {
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaFuncSetAttribute(residency_layers_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    carveout_set = true;
  }
  residency_layers_kernel<<<layers, kThreads, 0, s>>>(ids, n_ids, E, K, st0, state_stride, plan0, plan_words, err,
                                                      epoch);
  return cudaGetLastError();
}

}  // namespace pmoe
