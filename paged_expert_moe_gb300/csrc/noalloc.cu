// moe_decode_forward_noalloc: the decode MoE over experts that already sit in device
// memory, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another framework's
// memory pool or allocator hooks, real-time loops that must never reach the
// driver's allocator, and embedders whose device memory is budgeted and handed out
// up front. This entry point needs no allocation at all: its intermediates (the
// one-wave plan, the token grouping, the bf16 intermediate h and the fp32 per-pair
// outputs) live in one file-scope device array of fixed size, g_noalloc_scratch.
// Every GPU that loads the library holds this array until the process exits.
//
// Host code never names g_noalloc_scratch as an address: in host code that name is a
// host-side stand-in, and a kernel given it would fault or read the wrong memory.
// The first call on each device, with that device current, looks the device
// address up once with cudaGetSymbolAddress and keeps it; with lazy module loading
// that lookup is also what loads this file's device code and its array, so the
// first call can enter the driver's allocator: make it during warm-up, before any
// stream capture. Every call shares the one array, which keeps the last call's
// contents: calls that overlap on the GPU (different streams, or different host
// threads on one device) race on it and must be serialised by the caller. The
// per-call error word at the start of the array is cleared each call and, when the
// caller passes err_out, copied there after the call's kernels.
#include "pmoe_internal.h"

#include <mutex>

namespace pmoe {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(2) << 20;  // 2 MiB
constexpr int kNoallocMaxPairs = 64;                      // T * top_k
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct DeviceSetup {
  std::once_flag once;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  cudaError_t status = cudaSuccess;
};
DeviceSetup g_setup[kMaxDevices];

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Offsets of the scratch sections for (E, P, H, I); total is the bytes needed.
struct ScratchMap {
  size_t err, plan, counts, offs, perm, pos, h, o_part, total;
};

ScratchMap scratch_map(int E, int P, int H, int I) {
  ScratchMap m{};
  size_t off = 0;
  m.err = off;
  off = align256(off + 4);
  m.plan = off;
  off = align256(off + 4 * (size_t)PlanLayout{E}.words());
  m.counts = off;
  off = align256(off + 4 * (size_t)E);
  m.offs = off;
  off = align256(off + 4 * (size_t)(E + 1));
  m.perm = off;
  off = align256(off + 4 * (size_t)P);
  m.pos = off;
  off = align256(off + 4 * (size_t)P);
  m.h = off;
  off = align256(off + 2 * (size_t)P * I);
  m.o_part = off;
  off = align256(off + 4 * (size_t)P * H);
  m.total = off;
  return m;
}

// Slot of a routed expert: slot_of[e], or e when there is no map. -1 marks an expert
// the caller holds no slot for; any other value outside [0, n_slots) is an error.
__device__ __forceinline__ int expert_slot(const int32_t* __restrict__ slot_of, int e) {
  return slot_of != nullptr ? slot_of[e] : e;
}

// One-wave plan for experts that are all resident: the distinct routed ids in
// ascending order with their slots. An expert without a valid slot is left out of
// the plan; a slot other than -1 outside [0, n_slots) is also flagged.
__global__ void __launch_bounds__(1024) resident_plan_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                             const int32_t* __restrict__ slot_of, int n_slots,
                                                             int32_t* __restrict__ plan, int32_t* __restrict__ err) {
  __shared__ int s_used[kMaxExperts];
  __shared__ int s_scan[kMaxExperts];
  const int tid = threadIdx.x;
  const PlanLayout L{E};
  s_used[tid] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) s_used[e] = 1;
    else atomicOr(err, kErrBadExpertId);
  }
  __syncthreads();
  int used = (tid < E) ? s_used[tid] : 0;
  const int slot = used ? expert_slot(slot_of, tid) : -1;
  if (used && (slot < 0 || slot >= n_slots)) {
    if (slot != -1) atomicOr(err, kErrBadSlot);
    used = 0;
  }
  s_scan[tid] = used;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int add = (tid >= off) ? s_scan[tid - off] : 0;
    __syncthreads();
    s_scan[tid] += add;
    __syncthreads();
  }
  const int n = s_scan[1023];
  if (used) {
    const int r = s_scan[tid] - 1;
    plan[L.wave_exp() + r] = tid;
    plan[L.wave_slot() + r] = slot;
    plan[L.wave_of() + tid] = 0;
  } else if (tid < E) {
    plan[L.wave_of() + tid] = -1;
  }
  if (tid == 0) {
    plan[kPlanUnique] = n;
    plan[kPlanWaves] = n > 0 ? 1 : 0;
    plan[kPlanMisses] = 0;
    plan[kPlanError] = 0;
    plan[L.wave_start() + 0] = 0;
    plan[L.wave_start() + 1] = n;
    plan[L.miss_start() + 0] = 0;
    plan[L.miss_start() + 1] = 0;
    plan[L.wave_hits() + 0] = n;
    plan[L.wave_hits() + 1] = 0;
  }
}

// Pairs whose expert has no valid slot are left out of the combine (pos = -1).
__global__ void drop_unslotted_kernel(const int32_t* __restrict__ ids, int P, int E,
                                      const int32_t* __restrict__ slot_of, int n_slots, Workspace ws) {
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e < 0 || e >= E) continue;
    const int slot = expert_slot(slot_of, e);
    if (slot < 0 || slot >= n_slots) ws.pos[p] = -1;
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

int setup_device(int dev, DeviceSetup** out) {
  if (dev < 0 || dev >= kMaxDevices) return PMOE_EUNSUPPORTED;
  DeviceSetup& s = g_setup[dev];
  std::call_once(s.once, [&] {
    void* p = nullptr;
    s.status = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (s.status == cudaSuccess) s.scratch = (unsigned char*)p;
    if (s.status == cudaSuccess) s.status = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
  });
  if (s.status != cudaSuccess) return PMOE_ECUDA;
  *out = &s;
  return PMOE_OK;
}

}  // namespace
}  // namespace pmoe

using namespace pmoe;

extern "C" int moe_decode_forward_noalloc(const void* experts, size_t stride, int n_slots, const int32_t* slot_of,
                                          int E, int top_k, int H, int I, int format, const void* x, int T,
                                          const int32_t* ids, const float* w, const void* residual, void* y,
                                          int32_t* err_out, void* stream) {
  if (E < 1 || E > kMaxExperts || top_k < 1 || top_k > E || T < 0 || T > kGemvMaxTokens) return PMOE_EINVAL;
  if (n_slots < 1 || (slot_of == nullptr && n_slots < E)) return PMOE_EINVAL;
  if (H <= 0 || I <= 0 || H % 8 != 0 || I % 8 != 0 || H > 4096 || I > 1536) return PMOE_EINVAL;
  if (format != PMOE_BF16 && format != PMOE_FP8_BLOCK128 && format != PMOE_INT4_GPTQ_G128 && format != PMOE_MXFP4 &&
      format != PMOE_NVFP4)
    return PMOE_EUNSUPPORTED;
  if (format != PMOE_BF16 && (H % 128 != 0 || I % 128 != 0)) return PMOE_EUNSUPPORTED;
  const ExpertLayout lay = expert_layout(format, H, I);
  if (stride < lay.bytes || stride % 16 != 0) return PMOE_EINVAL;
  const int P = T * top_k;
  if (P > kNoallocMaxPairs) return PMOE_EINVAL;  // larger steps: use moe_paged_forward
  const ScratchMap m = scratch_map(E, P, H, I);
  if (m.total > kNoallocScratchBytes) return PMOE_EINVAL;  // the static scratch is 2 MiB
  if (T > 0 && (experts == nullptr || x == nullptr || ids == nullptr || w == nullptr || y == nullptr || x == y))
    return PMOE_EINVAL;
  // the kernels move experts, x, residual and y in 16-byte vectors
  if (!aligned16(experts) || !aligned16(x) || !aligned16(y) || (residual != nullptr && !aligned16(residual)) ||
      !aligned4(ids) || !aligned4(w) || (slot_of != nullptr && !aligned4(slot_of)) ||
      (err_out != nullptr && !aligned4(err_out)))
    return PMOE_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PMOE_ECUDA;
  DeviceSetup* ds = nullptr;
  const int r = setup_device(dev, &ds);
  if (r != PMOE_OK) return r;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char* base = ds->scratch;
  int32_t* err = (int32_t*)(base + m.err);
  int32_t* plan = (int32_t*)(base + m.plan);
  Workspace ws{};
  ws.counts = (int32_t*)(base + m.counts);
  ws.offs = (int32_t*)(base + m.offs);
  ws.perm = (int32_t*)(base + m.perm);
  ws.pos = (int32_t*)(base + m.pos);
  ws.h = (__nv_bfloat16*)(base + m.h);
  ws.o_part = (float*)(base + m.o_part);
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess) return PMOE_ECUDA;
  if (T > 0) {
    resident_plan_kernel<<<1, 1024, 0, s>>>(ids, P, E, slot_of, n_slots, plan, err);
    if (cudaGetLastError() != cudaSuccess) return PMOE_ECUDA;
    if (launch_group(ids, P, E, plan, ws, 0, err, s) != cudaSuccess) return PMOE_ECUDA;
    if (slot_of != nullptr || n_slots < E) {
      drop_unslotted_kernel<<<1, 128, 0, s>>>(ids, P, E, slot_of, n_slots, ws);
      if (cudaGetLastError() != cudaSuccess) return PMOE_ECUDA;
    }
    const uint8_t* arena = (const uint8_t*)experts;
    if (launch_gemv_gateup(format, (const __nv_bfloat16*)x, T, top_k, H, I, plan, E, 0, ws, arena, stride,
                           ds->num_sms, s) != cudaSuccess)
      return PMOE_ECUDA;
    if (launch_gemv_down(format, H, I, plan, E, 0, ws, arena, stride, ds->num_sms, s) != cudaSuccess)
      return PMOE_ECUDA;
    if (launch_combine(ws, w, (const __nv_bfloat16*)residual, (__nv_bfloat16*)y, T, top_k, H, s) != cudaSuccess)
      return PMOE_ECUDA;
  }
  // the call's device error bits, for a caller that wants them (stream-ordered)
  if (err_out != nullptr && cudaMemcpyAsync(err_out, err, 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return PMOE_ECUDA;
  return PMOE_OK;
}
