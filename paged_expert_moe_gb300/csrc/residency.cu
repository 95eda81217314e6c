// Residency step of one layer's K-slot expert table, on the device (one CTA).
//
// Article "Running an MoE Model Larger Than Your VRAM": TL;DR (copy in only the
// routed experts that are not resident), section "What does Paged Experts actually
// do?" item 3 (the oldest-used expert is evicted) and section "What happens with more than one
// request?" (more distinct experts than slots -> several waves, every one
// copying its own missing experts in). Post "Locality of reference helped ...", section "The fix": a hit moves
// no bytes, a miss copies one expert and evicts the least recently used one.
//
// The planning itself is step::lru_plan_core (step_common.cuh, which states the rules
// taken where the pages are silent); this kernel loads the layer's table, plans the step
// and writes the table, the plan header and the counters back. One thread owns one
// expert id and one slot (E, K <= 1024 = blockDim.x).
#include "step_common.cuh"

namespace pmoe {
namespace {

constexpr int kThreads = 1024;

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
  const step::LruSmem m{s_pend, s_slot_of, s_exp_in, s_last, s_unprot, s_rank_exp, s_warp, &s_bad};
  const step::LruCounts n = step::lru_plan_core<kThreads>(ids, n_ids, E, K, step, m, plan);
  if (tid == 0) {
    plan[kPlanUnique] = n.unique;
    plan[kPlanWaves] = n.waves;
    plan[kPlanMisses] = n.misses;
    plan[kPlanError] = s_bad ? kErrBadExpertId : 0;
    plan[kPlanStep] = step;
    const unsigned long long ep = atomicAdd(epoch, 1ull) + 1ull;
    plan[kPlanEpochLo] = (int32_t)(uint32_t)(ep & 0xffffffffull);
    plan[kPlanEpochHi] = (int32_t)(uint32_t)(ep >> 32);
    if (s_bad) atomicOr(err, kErrBadExpertId);
    *st.step = step + 1;
    st.counters[0] += (unsigned long long)(n.unique - n.misses);
    st.counters[1] += (unsigned long long)n.misses;
    st.counters[2] += (unsigned long long)n.waves;
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
