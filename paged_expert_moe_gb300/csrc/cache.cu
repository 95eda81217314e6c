// Host runtime of the paged-expert MoE layer and the C ABI (include/pagedmoe.h).
//
// Owns, per MoE layer: the pinned host store of all E experts, the device arena of K
// slots, the device LRU table and the residency plan; per cache: the copy stream, the
// events that order page-in against compute, the forward workspace and the device
// error word. The residency decision itself runs on the device (residency.cu); in
// copy-engine mode the host reads the plan back and issues one cudaMemcpyAsync per
// missed expert on the copy stream, in SM-pull mode a kernel pulls the experts over
// the host link itself and the host never waits.
//
// Ordering (article "Running an MoE Model Larger Than Your VRAM", sections "What
// does Paged Experts actually do?" and "What happens with more than one request?";
// the copy/compute overlap follows the read/transfer overlap arithmetic of the KV
// offload discussion, t_overlapped ~ max(t_read, t_H2D)):
//   residency(l) waits for the ids' producer and for layer l's previous forward;
//   wave 0's page-in follows it on the copy stream; the forward waits for the page-in;
//   wave w > 0 copies wait for wave w-1's compute (they overwrite its slots).
#include "pmoe_internal.h"
#include "tc_gemm.h"

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

using namespace pmoe;

namespace {

thread_local char g_last_error[256] = "";

void set_cuda_error(cudaError_t e, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
  cudaGetLastError();  // a non-sticky error must not resurface at the next launch check
}

#define PMOE_CUDA(call)                                   \
  do {                                                    \
    const cudaError_t e_ = (call);                        \
    if (e_ != cudaSuccess) {                              \
      set_cuda_error(e_, #call);                          \
      return PMOE_ECUDA;                                  \
    }                                                     \
  } while (0)

bool env_flag(const char* name) {
  const char* v = getenv(name);
  return v != nullptr && v[0] != '\0' && v[0] != '0';
}

long wait_timeout_ms() {
  const char* v = getenv("PMOE_WAIT_TIMEOUT_MS");
  if (v == nullptr) return 10000;
  const long t = strtol(v, nullptr, 10);
  return t > 0 ? t : 10000;
}

// Poll an event until it completes or the deadline passes.
int wait_event_bounded(cudaEvent_t ev) {
  const auto t0 = std::chrono::steady_clock::now();
  const long limit = wait_timeout_ms();
  int spins = 0;
  while (true) {
    const cudaError_t q = cudaEventQuery(ev);
    if (q == cudaSuccess) return PMOE_OK;
    if (q != cudaErrorNotReady) {
      set_cuda_error(q, "cudaEventQuery");
      return PMOE_ECUDA;
    }
    if (++spins > 2000) {
      const long ms = (long)std::chrono::duration_cast<std::chrono::milliseconds>(
                          std::chrono::steady_clock::now() - t0).count();
      if (ms > limit) return PMOE_ETIMEOUT;
      std::this_thread::yield();
    }
  }
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return st == cudaStreamCaptureStatusActive;
}

int validate_shape(int fmt, int H, int I) {
  if (H <= 0 || I <= 0 || H % 8 != 0 || I % 8 != 0) return PMOE_EINVAL;
  if (fmt != PMOE_BF16 && fmt != PMOE_FP8_BLOCK128 && fmt != PMOE_INT4_GPTQ_G128 && fmt != PMOE_MXFP4 &&
      fmt != PMOE_NVFP4)
    return PMOE_EUNSUPPORTED;
  if (fmt != PMOE_BF16 && (H % 128 != 0 || I % 128 != 0)) return PMOE_EUNSUPPORTED;
  // decode kernels hold a row in registers: H <= 4096 (bf16) / 4096 (fp8, int4), I <= 1536
  if (H > 4096 || I > 1536) return PMOE_EUNSUPPORTED;
  return PMOE_OK;
}

}  // namespace

struct pmoe_cache {
  pmoe_cache_desc d{};
  int num_sms = 0;
  ExpertLayout lay{};
  size_t stride = 0;
  size_t expert_bytes = 0;
  int words = 0;
  bool use_tc = false;  // tensor-core prefill path available
  cudaStream_t copy_stream = nullptr;
  cudaStream_t plan_stream = nullptr;  // residency kernels + plan read-back (copy-engine mode)
  std::vector<uint8_t*> host_store, host_store_dev, arena;
  std::vector<LayerState> st;
  std::vector<int32_t*> plan_dev;
  int32_t* plan_host = nullptr;
  int32_t* state_buf = nullptr;
  size_t state_stride = 0;  // bytes between consecutive layers' LRU states in state_buf
  int32_t* plan_buf = nullptr;
  int32_t* err_dev = nullptr;
  std::vector<cudaEvent_t> ev_plan, ev_layer_done, ev_ready;
  std::vector<int> staged, staged_waves, layer_used;
  std::vector<int> pull_deferred;  // the staged step's wave-0 page-in is left to the fused decode kernel
  std::vector<int> plan_on_compute;  // the staged step was planned on the compute stream
  bool pdl = false;  // cooperative launches with programmatic serialization are accepted
  cudaEvent_t ev_ids = nullptr, ev_wave_done = nullptr, ev_stack = nullptr;
  Workspace ws{};
  void* ws_buf = nullptr;
  // persistent stack decode (SM-pull caches of several layers; inside ws_buf)
  unsigned long long* stack_hq = nullptr;  // [2][16][I]
  unsigned long long* stack_xq = nullptr;  // [2][2][H]
  uint8_t** stack_arenas = nullptr;        // [L] device copy of arena
  const uint8_t** stack_stores = nullptr;  // [L] device copy of host_store_dev
  std::vector<TcMaps> maps;  // per layer tensor maps (bf16 prefill path)
  TcMaps ws_maps{};
  // per-kernel timers
  bool timing = false;
  bool in_capture = false;  // the current call is being recorded into a CUDA graph
  struct Mark {
    int cls;
    cudaEvent_t a, b;
  };
  std::vector<Mark> marks;       // recorded, not yet resolved
  std::vector<cudaEvent_t> pool; // free events
  double ms[PMOE_K_CLASSES] = {};
  uint64_t launches[PMOE_K_CLASSES] = {};
  uint64_t copies = 0;

  int32_t* plan_h(int layer) { return plan_host + (size_t)layer * words; }
};

namespace {

cudaEvent_t pool_get(pmoe_cache* c) {
  if (!c->pool.empty()) {
    cudaEvent_t e = c->pool.back();
    c->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Resolve every recorded mark (waits for them) and return the events to the pool.
int resolve_marks(pmoe_cache* c) {
  for (auto& m : c->marks) {
    if (cudaEventSynchronize(m.b) != cudaSuccess) return PMOE_ECUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, m.a, m.b) == cudaSuccess) c->ms[m.cls] += t;
    c->pool.push_back(m.a);
    c->pool.push_back(m.b);
  }
  c->marks.clear();
  return PMOE_OK;
}

// Brackets one kernel launch with timing events when timing is on; counts launches.
struct KernelMark {
  pmoe_cache* c;
  int cls;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  KernelMark(pmoe_cache* c_, int cls_, cudaStream_t s_) : c(c_), cls(cls_), s(s_) {
    c->launches[cls] += 1;
    if (c->timing && !c->in_capture) {
      if (c->marks.size() >= 2048) resolve_marks(c);
      a = pool_get(c);
      if (a) cudaEventRecord(a, s);
    }
  }
  ~KernelMark() {
    if (a) {
      cudaEvent_t b = pool_get(c);
      if (b) {
        cudaEventRecord(b, s);
        c->marks.push_back({cls, a, b});
      } else {
        c->pool.push_back(a);
      }
    }
  }
};

void free_cache(pmoe_cache* c) {
  if (c == nullptr) return;
  if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
  if (c->plan_stream) cudaStreamSynchronize(c->plan_stream);
  for (cudaEvent_t e : c->ev_layer_done)
    if (e) cudaEventSynchronize(e);
  resolve_marks(c);
  for (cudaEvent_t e : c->pool)
    if (e) cudaEventDestroy(e);
  for (auto p : c->host_store)
    if (p) cudaFreeHost(p);
  for (auto p : c->arena)
    if (p) cudaFree(p);
  if (c->plan_host) cudaFreeHost(c->plan_host);
  if (c->state_buf) cudaFree(c->state_buf);
  if (c->plan_buf) cudaFree(c->plan_buf);
  if (c->err_dev) cudaFree(c->err_dev);
  if (c->ws_buf) cudaFree(c->ws_buf);
  for (auto& v : {&c->ev_plan, &c->ev_layer_done, &c->ev_ready})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  if (c->ev_ids) cudaEventDestroy(c->ev_ids);
  if (c->ev_wave_done) cudaEventDestroy(c->ev_wave_done);
  if (c->ev_stack) cudaEventDestroy(c->ev_stack);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  if (c->plan_stream) cudaStreamDestroy(c->plan_stream);
  delete c;
}

int issue_copies(pmoe_cache* c, int layer, int wave) {
  const int32_t* plan = c->plan_h(layer);
  const PlanLayout L{c->d.num_experts};
  const int m0 = plan[L.miss_start() + wave], m1 = plan[L.miss_start() + wave + 1];
  if (env_flag("PMOE_INJECT_MEMCPY_FAIL") && m1 > m0) {
    snprintf(g_last_error, sizeof(g_last_error), "injected page-in copy failure");
    return PMOE_ECUDA;
  }
  if (m1 == m0) return PMOE_OK;
  KernelMark km(c, PMOE_K_COPY, c->copy_stream);
  for (int m = m0; m < m1; ++m) {
    const int e = plan[L.miss_exp() + m], s = plan[L.miss_slot() + m];
    PMOE_CUDA(cudaMemcpyAsync(c->arena[layer] + (size_t)s * c->stride, c->host_store[layer] + (size_t)e * c->stride,
                              c->expert_bytes, cudaMemcpyHostToDevice, c->copy_stream));
    c->copies += 1;
  }
  return PMOE_OK;
}

// A staged step that no forward consumed still owes the page-in of its later waves:
// finish them in order (no compute in between), so the arena matches the table.
int flush_staged(pmoe_cache* c, int layer) {
  if (!c->staged[layer]) return PMOE_OK;
  c->staged[layer] = 0;
  // (a step planned on a compute stream is always consumed by the forward that planned
  // it, so it never reaches here)
  c->plan_on_compute[layer] = 0;
  const int first = c->pull_deferred[layer] ? 0 : 1;
  c->pull_deferred[layer] = 0;
  for (int wv = first; wv < c->staged_waves[layer]; ++wv) {
    if (c->d.pagein_mode == PMOE_PAGEIN_COPY_ENGINE) {
      const int r = issue_copies(c, layer, wv);
      if (r != PMOE_OK) return r;
    } else {
      KernelMark km(c, PMOE_K_PULL, c->copy_stream);
      PMOE_CUDA(launch_pull_pages(c->plan_dev[layer], c->d.num_experts, wv, c->host_store_dev[layer], c->stride,
                                  c->expert_bytes, c->arena[layer], c->err_dev, c->copy_stream));
    }
  }
  if (!c->in_capture) PMOE_CUDA(cudaEventRecord(c->ev_layer_done[layer], c->copy_stream));
  return PMOE_OK;
}

int max_waves(const pmoe_cache* c, int n_ids) {
  const int u = n_ids < c->d.num_experts ? n_ids : c->d.num_experts;
  return (u + c->d.num_slots - 1) / c->d.num_slots;
}

}  // namespace

extern "C" {

int pmoe_version(void) { return 100; }

const char* pmoe_status_string(int status) {
  switch (status) {
    case PMOE_OK: return "ok";
    case PMOE_EINVAL: return "invalid argument";
    case PMOE_ENOMEM: return "out of device memory";
    case PMOE_EHOSTALLOC: return "pinned host allocation failed";
    case PMOE_ECUDA: return "CUDA error";
    case PMOE_EUNSUPPORTED: return "unsupported configuration";
    case PMOE_ETIMEOUT: return "timed out waiting for the device";
    case PMOE_EDEVICE: return "a kernel recorded an error (bad expert id)";
    default: return "unknown status";
  }
}

const char* pmoe_last_error(void) { return g_last_error; }

size_t pmoe_expert_bytes(int format, int hidden, int intermediate) {
  if (validate_shape(format, hidden, intermediate) != PMOE_OK) return 0;
  return expert_layout(format, hidden, intermediate).bytes;
}

int moe_router_topk(const float* logits, int T, int E, int top_k, int renormalize, int32_t* ids_out, float* w_out,
                    void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > E || top_k > kMaxTopK) return PMOE_EINVAL;
  if (T == 0) return PMOE_OK;
  if (logits == nullptr || ids_out == nullptr || w_out == nullptr) return PMOE_EINVAL;
  PMOE_CUDA(launch_router_topk(logits, T, E, top_k, renormalize ? 1 : 0, ids_out, w_out, (cudaStream_t)stream));
  return PMOE_OK;
}

int moe_group_by_expert(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offs, int32_t* perm,
                        int32_t* pos, int32_t* scratch, size_t scratch_ints, int32_t* err_dev, void* stream) {
  if (P < 0 || P > (1 << 24) || E < 1 || E > kMaxExperts) return PMOE_EINVAL;
  if (counts == nullptr || offs == nullptr || (P > 0 && (ids == nullptr || perm == nullptr || pos == nullptr)))
    return PMOE_EINVAL;
  if (P > kGroupOneCtaMaxPairs && (scratch == nullptr || scratch_ints < moe_group_scratch_ints(P, E)))
    return PMOE_EINVAL;
  Workspace ws{};
  ws.counts = counts;
  ws.offs = offs;
  ws.perm = perm;
  ws.pos = pos;
  ws.chunk_cnt = scratch;
  ws.chunk_cap = (int)std::min(scratch_ints, (size_t)INT32_MAX);
  PMOE_CUDA(launch_group(ids, P, E, nullptr, ws, 0, err_dev, (cudaStream_t)stream));
  return PMOE_OK;
}

size_t moe_group_scratch_ints(int P, int E) {
  if (P <= kGroupOneCtaMaxPairs) return 0;
  return (size_t)((P + 255) / 256) * (size_t)E;
}

int moe_router_gemm_topk(const void* x, const void* router_weight, int T, int H, int E, int top_k, int renormalize,
                         float* logits_out, int32_t* ids_out, float* w_out, void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > E || top_k > kMaxTopK || H < 8 || H % 8 != 0)
    return PMOE_EINVAL;
  if (T == 0) return PMOE_OK;
  if (x == nullptr || router_weight == nullptr || ids_out == nullptr || w_out == nullptr) return PMOE_EINVAL;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(router_weight) % 16 != 0)
    return PMOE_EINVAL;
  if (router_gemm_smem(H, E) > 200 * 1024) return PMOE_EUNSUPPORTED;
  PMOE_CUDA(launch_router_gemm_topk((const __nv_bfloat16*)x, (const __nv_bfloat16*)router_weight, T, H, E, top_k,
                                    renormalize ? 1 : 0, logits_out, ids_out, w_out, (cudaStream_t)stream));
  return PMOE_OK;
}

int expert_cache_create(const pmoe_cache_desc* desc, pmoe_cache** out) {
  if (desc == nullptr || out == nullptr) return PMOE_EINVAL;
  *out = nullptr;
  const pmoe_cache_desc d = *desc;
  if (d.num_experts < 1 || d.num_experts > kMaxExperts) return PMOE_EINVAL;
  if (d.top_k < 1 || d.top_k > d.num_experts || d.top_k > kMaxTopK) return PMOE_EINVAL;
  if (d.num_slots < 1 || d.num_slots > d.num_experts) return PMOE_EINVAL;
  if (d.num_layers < 1 || d.max_tokens < 1 || d.device < 0) return PMOE_EINVAL;
  if ((long long)d.max_tokens * d.top_k > (1LL << 24)) return PMOE_EINVAL;
  if (d.pagein_mode != PMOE_PAGEIN_COPY_ENGINE && d.pagein_mode != PMOE_PAGEIN_SM_PULL) return PMOE_EINVAL;
  {
    const int v = validate_shape(d.format, d.hidden, d.intermediate);
    if (v != PMOE_OK) return v;
  }
  PMOE_CUDA(cudaSetDevice(d.device));
  cudaDeviceProp prop;
  PMOE_CUDA(cudaGetDeviceProperties(&prop, d.device));
  if (prop.major != 10 || prop.minor != 3) {
    snprintf(g_last_error, sizeof(g_last_error), "device is sm_%d%d; this library is built for sm_103a",
             prop.major, prop.minor);
    return PMOE_EUNSUPPORTED;
  }
  pmoe_cache* c = new (std::nothrow) pmoe_cache();
  if (c == nullptr) return PMOE_ENOMEM;
  c->d = d;
  c->num_sms = prop.multiProcessorCount;
  c->pdl = decode_pdl_supported(d.device);
  c->lay = expert_layout(d.format, d.hidden, d.intermediate);
  c->expert_bytes = c->lay.bytes;
  c->stride = round_up(c->expert_bytes, 4096);
  c->words = PlanLayout{d.num_experts}.words();
  const int E = d.num_experts, K = d.num_slots, Lr = d.num_layers;
  c->host_store.assign(Lr, nullptr);
  c->host_store_dev.assign(Lr, nullptr);
  c->arena.assign(Lr, nullptr);
  c->st.resize(Lr);
  c->plan_dev.assign(Lr, nullptr);
  c->ev_plan.assign(Lr, nullptr);
  c->ev_layer_done.assign(Lr, nullptr);
  c->ev_ready.assign(Lr, nullptr);
  c->staged.assign(Lr, 0);
  c->staged_waves.assign(Lr, 0);
  c->pull_deferred.assign(Lr, 0);
  c->plan_on_compute.assign(Lr, 0);
  c->layer_used.assign(Lr, 0);
  int status = PMOE_OK;
#define PMOE_TRY(call)              \
  do {                              \
    const cudaError_t e_ = (call);  \
    if (e_ != cudaSuccess) {        \
      set_cuda_error(e_, #call);    \
      status = PMOE_ECUDA;          \
      goto fail;                    \
    }                               \
  } while (0)
  PMOE_TRY(cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking));
  PMOE_TRY(cudaStreamCreateWithFlags(&c->plan_stream, cudaStreamNonBlocking));
  PMOE_TRY(cudaEventCreateWithFlags(&c->ev_ids, cudaEventDisableTiming));
  PMOE_TRY(cudaEventCreateWithFlags(&c->ev_wave_done, cudaEventDisableTiming));
  PMOE_TRY(cudaEventCreateWithFlags(&c->ev_stack, cudaEventDisableTiming));
  for (int l = 0; l < Lr; ++l) {
    PMOE_TRY(cudaEventCreateWithFlags(&c->ev_plan[l], cudaEventDisableTiming));
    PMOE_TRY(cudaEventCreateWithFlags(&c->ev_layer_done[l], cudaEventDisableTiming));
    PMOE_TRY(cudaEventCreateWithFlags(&c->ev_ready[l], cudaEventDisableTiming));
  }
  // pinned host store (mapped, so the SM-pull kernel can read it)
  for (int l = 0; l < Lr; ++l) {
    if (env_flag("PMOE_INJECT_HOSTALLOC_FAIL")) {
      snprintf(g_last_error, sizeof(g_last_error), "injected pinned allocation failure");
      status = PMOE_EHOSTALLOC;
      goto fail;
    }
    void* p = nullptr;
    const cudaError_t e = cudaHostAlloc(&p, (size_t)E * c->stride, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      set_cuda_error(e, "cudaHostAlloc (expert store)");
      cudaGetLastError();
      status = PMOE_EHOSTALLOC;
      goto fail;
    }
    c->host_store[l] = (uint8_t*)p;
    void* pd = nullptr;
    PMOE_TRY(cudaHostGetDevicePointer(&pd, p, 0));
    c->host_store_dev[l] = (uint8_t*)pd;
  }
  for (int l = 0; l < Lr; ++l) {
    void* p = nullptr;
    const cudaError_t e = cudaMalloc(&p, (size_t)K * c->stride);
    if (e != cudaSuccess) {
      set_cuda_error(e, "cudaMalloc (slot arena)");
      cudaGetLastError();
      status = PMOE_ENOMEM;
      goto fail;
    }
    c->arena[l] = (uint8_t*)p;
  }
  {
    // LRU state: per layer slot_of[E], expert_in[K], last_use[K], step[1], pad, counters (4 x u64)
    const size_t per = round_up((size_t)E + 2 * K + 2, 2) * 4 + 4 * 8;
    c->state_stride = per;
    PMOE_TRY(cudaMalloc(&c->state_buf, per * Lr));
    PMOE_TRY(cudaMemset(c->state_buf, 0xFF, per * Lr));
    for (int l = 0; l < Lr; ++l) {
      uint8_t* b = (uint8_t*)c->state_buf + per * l;
      LayerState& s = c->st[l];
      s.slot_of = (int32_t*)b;
      s.expert_in = s.slot_of + E;
      s.last_use = s.expert_in + K;
      s.step = s.last_use + K;
      s.counters = (unsigned long long*)(b + per - 4 * 8);
      PMOE_TRY(cudaMemset(s.step, 0, 4));
      PMOE_TRY(cudaMemset(s.counters, 0, 4 * 8));
    }
    PMOE_TRY(cudaMalloc(&c->plan_buf, (size_t)c->words * 4 * Lr));
    PMOE_TRY(cudaMemset(c->plan_buf, 0, (size_t)c->words * 4 * Lr));
    for (int l = 0; l < Lr; ++l) c->plan_dev[l] = c->plan_buf + (size_t)c->words * l;
    PMOE_TRY(cudaHostAlloc((void**)&c->plan_host, (size_t)c->words * 4 * Lr, cudaHostAllocPortable));
    memset(c->plan_host, 0, (size_t)c->words * 4 * Lr);
    PMOE_TRY(cudaMalloc(&c->err_dev, 4));
    PMOE_TRY(cudaMemset(c->err_dev, 0, 4));
  }
  {
    // forward workspace
    const size_t P = (size_t)d.max_tokens * d.top_k;
    c->use_tc = d.max_tokens > kGemvMaxTokens && tc_supported(d.hidden, d.intermediate);
    c->ws.max_tiles = (int)(E + P / 16 + 1);
    size_t off = 0;
    auto carve = [&](size_t bytes) {
      const size_t o = off;
      off = round_up(off + bytes, 256);
      return o;
    };
    const size_t o_counts = carve(4 * (size_t)E), o_offs = carve(4 * (size_t)(E + 1)), o_perm = carve(4 * P),
                 o_pos = carve(4 * P), o_tiles = carve(12 * (size_t)c->ws.max_tiles),
                 o_tw = carve(4 * (size_t)(E + 2)), o_ts = carve(4 * (size_t)(E + 2)),
                 o_h = carve(2 * P * d.intermediate),
                 o_o = carve(4 * P * d.hidden), o_x = c->use_tc ? carve(2 * P * d.hidden) : 0;
    const size_t chunk_cap = ((P + 255) / 256) * (size_t)E;
    const size_t o_ch = carve(4 * chunk_cap);
    // block-FP8 on the tensor path: the activation planes' scales (the planes themselves
    // take the bytes of x_perm and h)
    const bool f8_tc = c->use_tc && d.format == PMOE_FP8_BLOCK128;
    const size_t o_sx = f8_tc ? carve(4 * P) : 0;
    const size_t o_hsc = f8_tc ? carve(4 * P * (size_t)(d.intermediate / 64)) : 0;
    const size_t o_ep = carve(8);
    const size_t o_hq = carve(8 * std::min(P, (size_t)kDecodeMaxPairs) * d.intermediate);
    // the persistent stack decode: tagged exchange words (two layers' worth each) and the
    // layers' arena and host-store pointers
    const bool stack_bufs = Lr > 1 && d.pagein_mode == PMOE_PAGEIN_SM_PULL;
    const size_t o_shq = stack_bufs ? carve(8 * 2 * 16 * (size_t)d.intermediate) : 0;
    const size_t o_sxq = stack_bufs ? carve(8 * 2 * 2 * (size_t)d.hidden) : 0;
    const size_t o_tab = stack_bufs ? carve(2 * 8 * (size_t)Lr) : 0;
    const cudaError_t e = cudaMalloc(&c->ws_buf, off);
    if (e != cudaSuccess) {
      set_cuda_error(e, "cudaMalloc (workspace)");
      cudaGetLastError();
      status = PMOE_ENOMEM;
      goto fail;
    }
    uint8_t* b = (uint8_t*)c->ws_buf;
    c->ws.counts = (int32_t*)(b + o_counts);
    c->ws.offs = (int32_t*)(b + o_offs);
    c->ws.perm = (int32_t*)(b + o_perm);
    c->ws.pos = (int32_t*)(b + o_pos);
    c->ws.tiles = (int32_t*)(b + o_tiles);
    c->ws.tile_wave = (int32_t*)(b + o_tw);
    c->ws.tile_split = (int32_t*)(b + o_ts);
    c->ws.h = (__nv_bfloat16*)(b + o_h);
    c->ws.o_part = (float*)(b + o_o);
    c->ws.x_perm = c->use_tc ? (__nv_bfloat16*)(b + o_x) : nullptr;
    c->ws.sx = f8_tc ? (float*)(b + o_sx) : nullptr;
    c->ws.hsc = f8_tc ? (float*)(b + o_hsc) : nullptr;
    c->ws.p_cap = P;
    c->ws.chunk_cnt = (int32_t*)(b + o_ch);
    c->ws.chunk_cap = (int)chunk_cap;
    c->ws.epoch = (unsigned long long*)(b + o_ep);
    PMOE_TRY(cudaMemset(c->ws.epoch, 0, 8));
    c->ws.hq = (unsigned long long*)(b + o_hq);
    if (stack_bufs) {
      c->stack_hq = (unsigned long long*)(b + o_shq);
      c->stack_xq = (unsigned long long*)(b + o_sxq);
      PMOE_TRY(cudaMemset(c->stack_hq, 0, 8 * 2 * 16 * (size_t)d.intermediate));
      PMOE_TRY(cudaMemset(c->stack_xq, 0, 8 * 2 * 2 * (size_t)d.hidden));
      c->stack_arenas = (uint8_t**)(b + o_tab);
      c->stack_stores = (const uint8_t**)(b + o_tab + 8 * (size_t)Lr);
      PMOE_TRY(cudaMemcpy(c->stack_arenas, c->arena.data(), 8 * (size_t)Lr, cudaMemcpyHostToDevice));
      PMOE_TRY(cudaMemcpy((void*)c->stack_stores, c->host_store_dev.data(), 8 * (size_t)Lr, cudaMemcpyHostToDevice));
    }
    PMOE_TRY(cudaMemset(c->ws.hq, 0, 8 * std::min(P, (size_t)kDecodeMaxPairs) * d.intermediate));
  }
  if (c->use_tc) {
    c->maps.resize(Lr);
    for (int l = 0; l < Lr; ++l) {
      const int r = tc_make_weight_maps(c->arena[l], c->stride, K, d.hidden, d.intermediate, d.format, &c->maps[l]);
      if (r != PMOE_OK) {
        status = r;
        goto fail;
      }
    }
    const int r = tc_make_act_maps(d.format, c->ws.x_perm, c->ws.h, (size_t)d.max_tokens * d.top_k, d.hidden, d.intermediate,
                                   &c->ws_maps);
    if (r != PMOE_OK) {
      status = r;
      goto fail;
    }
  }
#undef PMOE_TRY
  *out = c;
  return PMOE_OK;
fail:
  free_cache(c);
  return status;
}

void expert_cache_destroy(pmoe_cache* cache) { free_cache(cache); }

int expert_cache_host_store(pmoe_cache* c, int layer, void** host_ptr, size_t* stride_bytes) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || host_ptr == nullptr) return PMOE_EINVAL;
  *host_ptr = c->host_store[layer];
  if (stride_bytes) *stride_bytes = c->stride;
  return PMOE_OK;
}

int expert_cache_load_expert(pmoe_cache* c, int layer, int expert, const void* bytes, size_t nbytes) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || expert < 0 || expert >= c->d.num_experts ||
      bytes == nullptr || nbytes != c->expert_bytes)
    return PMOE_EINVAL;
  memcpy(c->host_store[layer] + (size_t)expert * c->stride, bytes, nbytes);
  return PMOE_OK;
}

int expert_cache_reset(pmoe_cache* c, int layer) {
  if (c == nullptr || layer < -1 || layer >= c->d.num_layers) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? c->d.num_layers : layer + 1;
  for (int l = l0; l < l1; ++l) {
    {
      const int r = flush_staged(c, l);
      if (r != PMOE_OK) return r;
    }
    // the table is updated on the stream the residency kernels run on
    cudaStream_t ps = c->d.pagein_mode == PMOE_PAGEIN_COPY_ENGINE ? c->plan_stream : c->copy_stream;
    PMOE_CUDA(cudaStreamWaitEvent(ps, c->ev_layer_done[l], 0));
    const LayerState& s = c->st[l];
    PMOE_CUDA(cudaMemsetAsync(s.slot_of, 0xFF, 4 * (size_t)c->d.num_experts, ps));
    PMOE_CUDA(cudaMemsetAsync(s.expert_in, 0xFF, 4 * (size_t)c->d.num_slots, ps));
    PMOE_CUDA(cudaMemsetAsync(s.last_use, 0xFF, 4 * (size_t)c->d.num_slots, ps));
  }
  return PMOE_OK;
}

}  // extern "C"

namespace {

// The residency step of `layer`, ordered after `ids_ready` (the ids' producer) and after
// the layer's previous forward. defer_pull (SM-pull mode): leave the page-in of the
// step's waves to the fused decode kernel, which copies each missing expert's bytes as
// its chunks need them. compute (SM-pull with defer_pull only): plan on that stream,
// directly ahead of the decode kernel, instead of on the copy stream.
int ensure_resident_impl(pmoe_cache* c, int layer, const int32_t* ids, int n_ids, cudaEvent_t ids_ready,
                         int* waves_out, bool defer_pull = false, cudaStream_t compute = nullptr,
                         bool on_compute = false);

}  // namespace

extern "C" {

int expert_cache_ensure_resident(pmoe_cache* c, int layer, const int32_t* ids, int n_ids, void* stream,
                                 int* waves_out) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || n_ids < 0 ||
      n_ids > c->d.max_tokens * c->d.top_k || (n_ids > 0 && ids == nullptr))
    return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  c->in_capture = stream_capturing((cudaStream_t)stream);
  PMOE_CUDA(cudaEventRecord(c->ev_ids, (cudaStream_t)stream));
  return ensure_resident_impl(c, layer, ids, n_ids, c->ev_ids, waves_out);
}

int expert_cache_prefetch(pmoe_cache* c, int layer, const int32_t* ids, int n_ids, void* stream) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || n_ids < 0 ||
      n_ids > c->d.max_tokens * c->d.top_k || (n_ids > 0 && ids == nullptr))
    return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  c->in_capture = stream_capturing((cudaStream_t)stream);
  PMOE_CUDA(cudaEventRecord(c->ev_ids, (cudaStream_t)stream));
  // one residency step for the predicted ids (an LRU step like any other), then the
  // page-in of every wave, in order, on the copy stream; nothing is computed
  const int r = ensure_resident_impl(c, layer, ids, n_ids, c->ev_ids, nullptr);
  if (r != PMOE_OK && r != PMOE_EDEVICE) return r;
  const int f = flush_staged(c, layer);
  return f != PMOE_OK ? f : r;
}

}  // extern "C"

namespace {

int ensure_resident_impl(pmoe_cache* c, int layer, const int32_t* ids, int n_ids, cudaEvent_t ids_ready,
                         int* waves_out, bool defer_pull, cudaStream_t compute, bool on_compute) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || n_ids < 0 ||
      n_ids > c->d.max_tokens * c->d.top_k || (n_ids > 0 && ids == nullptr))
    return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  {
    const int r = flush_staged(c, layer);  // a previous staged step that was never consumed
    if (r != PMOE_OK) return r;
  }
  const bool ce = c->d.pagein_mode == PMOE_PAGEIN_COPY_ENGINE;
  // copy-engine mode plans on its own stream, so planning the next layer never queues
  // behind this layer's copies; SM-pull plans and pulls in one stream order. A step
  // whose page-in the decode kernel does itself plans on the compute stream, right
  // before that kernel: router, residency and decode then follow one another in one
  // stream, and each may launch while the one before it drains.
  on_compute = on_compute && !ce && defer_pull && compute != nullptr;
  cudaStream_t ps = ce ? c->plan_stream : on_compute ? compute : c->copy_stream;
  if (c->in_capture && ce) {
    snprintf(g_last_error, sizeof(g_last_error),
             "graph capture needs PMOE_PAGEIN_SM_PULL (copy-engine page-in reads the plan on the host)");
    return PMOE_EUNSUPPORTED;
  }
  if (!on_compute) PMOE_CUDA(cudaStreamWaitEvent(ps, ids_ready, 0));
  // inside a captured graph the layer's previous forward precedes this step by graph order
  if (!c->in_capture) PMOE_CUDA(cudaStreamWaitEvent(ps, c->ev_layer_done[layer], 0));
  c->plan_on_compute[layer] = on_compute ? 1 : 0;
  {
    KernelMark km(c, PMOE_K_RESIDENCY, ps);
    // programmatic serialization only where nothing but the router precedes it in the
    // stream (the timers put events between kernels outside graph capture)
    const bool pdl = on_compute && c->pdl && !(c->timing && !c->in_capture);
    PMOE_CUDA(launch_residency(ids, n_ids, c->d.num_experts, c->d.num_slots, c->st[layer], c->plan_dev[layer],
                               c->err_dev, c->ws.epoch, ps, pdl));
  }
  c->layer_used[layer] = 1;
  int waves = -1;
  int status = PMOE_OK;
  if (ce) {
    PMOE_CUDA(cudaMemcpyAsync(c->plan_h(layer), c->plan_dev[layer], (size_t)c->words * 4, cudaMemcpyDeviceToHost, ps));
    PMOE_CUDA(cudaEventRecord(c->ev_plan[layer], ps));
    // the copies overwrite victim slots: they follow the plan (which followed this
    // layer's previous forward)
    PMOE_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ev_plan[layer], 0));
    const int r = wait_event_bounded(c->ev_plan[layer]);
    if (r != PMOE_OK) return r;
    const int32_t* plan = c->plan_h(layer);
    waves = plan[kPlanWaves];
    if (plan[kPlanError] != 0) status = PMOE_EDEVICE;
    if (waves > 0) {
      const int r2 = issue_copies(c, layer, 0);
      if (r2 != PMOE_OK) {
        // the table already names experts whose bytes never arrived: empty it, so the
        // next step pages everything in again rather than computing with stale slots
        const LayerState& ls = c->st[layer];
        cudaMemsetAsync(ls.slot_of, 0xFF, 4 * (size_t)c->d.num_experts, ps);
        cudaMemsetAsync(ls.expert_in, 0xFF, 4 * (size_t)c->d.num_slots, ps);
        cudaMemsetAsync(ls.last_use, 0xFF, 4 * (size_t)c->d.num_slots, ps);
        return r2;
      }
    }
  } else {
    // the plan is on the device now: compute on the resident experts may start while the
    // pull kernel brings the missing ones
    if (!on_compute) PMOE_CUDA(cudaEventRecord(c->ev_plan[layer], c->copy_stream));
    c->pull_deferred[layer] = defer_pull ? 1 : 0;
    if (!defer_pull) {
      KernelMark km(c, PMOE_K_PULL, c->copy_stream);
      PMOE_CUDA(launch_pull_pages(c->plan_dev[layer], c->d.num_experts, 0, c->host_store_dev[layer], c->stride,
                                  c->expert_bytes, c->arena[layer], c->err_dev, c->copy_stream));
    }
  }
  if (!on_compute) PMOE_CUDA(cudaEventRecord(c->ev_ready[layer], c->copy_stream));
  c->staged[layer] = 1;
  c->staged_waves[layer] = waves >= 0 ? waves : max_waves(c, n_ids);
  if (waves_out) *waves_out = waves;
  return status;
}

}  // namespace

extern "C" {

int moe_paged_forward(pmoe_cache* c, int layer, const void* x, int T, const int32_t* ids, const float* w,
                      const void* residual, void* y, void* stream) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || T < 0 || T > c->d.max_tokens) return PMOE_EINVAL;
  if (T == 0) return PMOE_OK;
  if (x == nullptr || ids == nullptr || w == nullptr || y == nullptr || x == y) return PMOE_EINVAL;
  if (T > kGemvMaxTokens && !c->use_tc) return PMOE_EUNSUPPORTED;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  cudaStream_t s = (cudaStream_t)stream;
  c->in_capture = stream_capturing(s);
  const int k = c->d.top_k, P = T * k, E = c->d.num_experts, H = c->d.hidden, I = c->d.intermediate;
  int status = PMOE_OK;
  const bool tc = c->use_tc && T > kGemvMaxTokens;
  const bool fused = !tc && decode_fused_supported(c->d.format, T, k, H, I, c->num_sms);
  const bool ce = c->d.pagein_mode == PMOE_PAGEIN_COPY_ENGINE;
  if (!c->staged[layer]) {
    // no step was staged ahead: plan it now; in SM-pull mode the fused decode kernel then
    // pages the missing experts in itself, overlapping the host link with the resident
    // experts' weight streaming
    PMOE_CUDA(cudaEventRecord(c->ev_ids, s));
    const int r = ensure_resident_impl(c, layer, ids, P, c->ev_ids, nullptr, fused && !ce, s, true);
    if (r == PMOE_EDEVICE) status = r;
    else if (r != PMOE_OK) return r;
  }
  c->staged[layer] = 0;
  const bool pull_in_kernel = c->pull_deferred[layer] != 0;
  c->pull_deferred[layer] = 0;
  // the plan was made on this stream, right before the decode kernel
  const bool planned_here = c->plan_on_compute[layer] != 0;
  c->plan_on_compute[layer] = 0;
  const int nw = c->staged_waves[layer];
  // Copy-engine steps whose first wave has both resident and paged-in experts compute
  // the resident ones while the copies are still in flight (the plan lists them first).
  // (SM-pull mode: the host does not know the split, and launching both parts
  // unconditionally cost more than the overlap gained, so the wave runs whole.)
  bool split0 = false;
  if (ce && (tc || fused) && nw > 0) {
    const int32_t* plan = c->plan_h(layer);
    const PlanLayout L{E};
    const int hits0 = plan[L.wave_hits() + 0];
    const int size0 = plan[L.wave_start() + 1] - plan[L.wave_start() + 0];
    split0 = hits0 > 0 && hits0 < size0;
  }
  // the fused decode kernel forms y itself when the step has a single unsplit wave
  const int fuse_combine = (fused && !split0) ? (ce ? (nw == 1 ? 1 : 0) : 1) : 0;
  const bool need_combine = !fused || nw > 1 || split0;

  auto compute = [&](int wv, int sub) -> int {
    if (tc) {
      {
        KernelMark km(c, PMOE_K_GATEUP, s);
        PMOE_CUDA(tc_gateup(c->d.format, c->maps[layer], c->ws_maps, c->plan_dev[layer], E, wv, sub, c->ws, I, H,
                            c->arena[layer], c->stride, c->num_sms, c->err_dev, tc_tile_n(T, k, E), s));
      }
      KernelMark km(c, PMOE_K_DOWN, s);
      PMOE_CUDA(tc_down(c->d.format, c->maps[layer], c->ws_maps, c->plan_dev[layer], E, wv, sub, c->ws, I, H,
                        c->arena[layer], c->stride, c->num_sms, c->err_dev, tc_tile_n(T, k, E), s));
    } else if (fused) {
      KernelMark km(c, PMOE_K_DECODE, s);
      // launched behind the residency step it follows directly (wave 0 of a step planned
      // on this stream), so that its CTAs start while the plan is being made
      const int pdl = (planned_here && wv == 0 && sub == 0 && c->pdl && !(c->timing && !c->in_capture)) ? 1 : 0;
      PMOE_CUDA(launch_decode_fused(c->d.format, (const __nv_bfloat16*)x, ids, w, (const __nv_bfloat16*)residual,
                                    (__nv_bfloat16*)y, T, k, H, I, c->plan_dev[layer], E, wv, sub, fuse_combine,
                                    c->ws, c->arena[layer], c->host_store_dev[layer], pull_in_kernel ? 1 : 0,
                                    c->stride, c->err_dev, c->num_sms, s, pdl));
    } else {
      {
        KernelMark km(c, PMOE_K_GATEUP, s);
        PMOE_CUDA(launch_gemv_gateup(c->d.format, (const __nv_bfloat16*)x, T, k, H, I, c->plan_dev[layer], E, wv,
                                     c->ws, c->arena[layer], c->stride, c->num_sms, s));
      }
      KernelMark km(c, PMOE_K_DOWN, s);
      PMOE_CUDA(launch_gemv_down(c->d.format, H, I, c->plan_dev[layer], E, wv, c->ws, c->arena[layer], c->stride,
                                 c->num_sms, s));
    }
    return PMOE_OK;
  };

  // grouping needs only the ids and the plan; in copy-engine mode the plan is ready
  // once the host has read it, before the copies land
  if (!planned_here) PMOE_CUDA(cudaStreamWaitEvent(s, split0 ? c->ev_plan[layer] : c->ev_ready[layer], 0));
  if (!fused) {  // the fused decode kernel groups the pairs itself
    KernelMark km(c, PMOE_K_GROUP, s);
    PMOE_CUDA(launch_group(ids, P, E, c->plan_dev[layer], c->ws, tc ? tc_tile_n(T, k, E) : 0, c->err_dev, s));
  }
  if (tc) {
    KernelMark km(c, PMOE_K_GATHER, s);
    if (tc_fp8_planes(c->d.format, tc_tile_n(T, k, E)))
      PMOE_CUDA(launch_gather_rows_fp8x2((const __nv_bfloat16*)x, c->ws.perm, P, k, H, c->ws.p_cap,
                                         reinterpret_cast<uint8_t*>(c->ws.x_perm), c->ws.sx, s));
    else
      PMOE_CUDA(launch_gather_rows((const __nv_bfloat16*)x, c->ws.perm, P, k, H, c->ws.x_perm, s));
  }
  for (int wv = 0; wv < nw; ++wv) {
    if (wv > 0 && !pull_in_kernel) {
      PMOE_CUDA(cudaEventRecord(c->ev_wave_done, s));
      PMOE_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ev_wave_done, 0));
      if (ce) {
        const int r = issue_copies(c, layer, wv);
        if (r != PMOE_OK) return r;
      } else {
        KernelMark km(c, PMOE_K_PULL, c->copy_stream);
        PMOE_CUDA(launch_pull_pages(c->plan_dev[layer], E, wv, c->host_store_dev[layer], c->stride, c->expert_bytes,
                                    c->arena[layer], c->err_dev, c->copy_stream));
      }
      PMOE_CUDA(cudaEventRecord(c->ev_ready[layer], c->copy_stream));
      PMOE_CUDA(cudaStreamWaitEvent(s, c->ev_ready[layer], 0));
    }
    if (wv == 0 && split0) {
      int r = compute(0, 1);  // resident experts, overlapping the page-in
      if (r != PMOE_OK) return r;
      PMOE_CUDA(cudaStreamWaitEvent(s, c->ev_ready[layer], 0));
      r = compute(0, 2);  // the experts just paged in
      if (r != PMOE_OK) return r;
    } else {
      const int r = compute(wv, 0);
      if (r != PMOE_OK) return r;
    }
  }
  if (need_combine) {
    // SM-pull steps that may have several waves: the combine skips itself if the step
    // turned out to have one wave (the fused kernel then already wrote y)
    KernelMark km(c, PMOE_K_COMBINE, s);
    PMOE_CUDA(launch_combine(c->ws, w, (const __nv_bfloat16*)residual, (__nv_bfloat16*)y, T, k, H, s,
                             (fused && !ce && !split0) ? c->plan_dev[layer] : nullptr,
                             tc && tc_o_part_bf16(c->d.format, tc_tile_n(T, k, E))));
  }
  // (under graph capture the graph's own order takes this event's place, and an event
  // recorded into a graph could not be waited on or queried outside it)
  if (!c->in_capture) PMOE_CUDA(cudaEventRecord(c->ev_layer_done[layer], s));
  return status;
}

int moe_paged_stack_forward(pmoe_cache* c, const void* x, int T, const int32_t* ids, const float* w, void* y,
                            void* work, void* stream) {
  if (c == nullptr || T < 0 || T > c->d.max_tokens) return PMOE_EINVAL;
  if (T == 0) return PMOE_OK;
  const int L = c->d.num_layers;
  if (x == nullptr || ids == nullptr || w == nullptr || y == nullptr || x == y) return PMOE_EINVAL;
  if (L > 1 && (work == nullptr || work == x || work == y)) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  cudaStream_t s = (cudaStream_t)stream;
  c->in_capture = stream_capturing(s);
  const int P = T * c->d.top_k;
  const size_t act = (size_t)T * c->d.hidden * 2;
  // every layer's ids are ready once the work already on `stream` is done
  PMOE_CUDA(cudaEventRecord(c->ev_stack, s));
  int status = PMOE_OK;
  // SM-pull decode: each layer's fused decode kernel pages its own missing experts in,
  // overlapping the host link with that layer's resident weights (a separate pull
  // kernel could not run beside it: the decode kernel holds every SM); the residency
  // steps are still planned one layer ahead
  const bool tc = c->use_tc && T > kGemvMaxTokens;
  const bool defer = c->d.pagein_mode == PMOE_PAGEIN_SM_PULL && !tc &&
                     decode_fused_supported(c->d.format, T, c->d.top_k, c->d.hidden, c->d.intermediate, c->num_sms);
  bool none_staged = true;
  for (int l = 0; l < L && none_staged; ++l) none_staged = !c->staged[l];
  if (defer && none_staged && L > 1) {
    // every layer's routing is known: plan all layers in one launch (one CTA per layer),
    // each layer's decode kernel then pages its own missing experts in
    cudaStream_t ps = c->copy_stream;
    PMOE_CUDA(cudaStreamWaitEvent(ps, c->ev_stack, 0));
    // (inside a captured graph each layer's previous forward precedes this by graph order)
    if (!c->in_capture)
      for (int l = 0; l < L; ++l) PMOE_CUDA(cudaStreamWaitEvent(ps, c->ev_layer_done[l], 0));
    {
      KernelMark km(c, PMOE_K_RESIDENCY, ps);
      PMOE_CUDA(launch_residency_layers(ids, P, L, c->d.num_experts, c->d.num_slots, c->st[0], c->state_stride,
                                        c->plan_dev[0], c->words, c->err_dev, c->ws.epoch, ps));
    }
    // Every layer's step one wave (T * top_k <= K): all layers in one persistent launch,
    // which pages each layer's misses in ahead of its compute and hands h_{l+1} from layer
    // to layer on the device
    if (c->stack_hq != nullptr && P <= c->d.num_slots &&
        decode_stack_supported(c->d.format, T, c->d.top_k, c->d.hidden, c->d.intermediate, L, c->num_sms)) {
      PMOE_CUDA(cudaEventRecord(c->ev_ready[0], ps));
      PMOE_CUDA(cudaStreamWaitEvent(s, c->ev_ready[0], 0));
      for (int l = 0; l < L; ++l) c->layer_used[l] = 1;
      {
        KernelMark km(c, PMOE_K_DECODE, s);
        PMOE_CUDA(launch_decode_stack(c->d.format, (const __nv_bfloat16*)x, (__nv_bfloat16*)y, ids, w, T, c->d.top_k,
                                      c->d.hidden, c->d.intermediate, c->d.num_experts, L, c->plan_dev[0], c->words,
                                      c->stack_arenas, c->stack_stores, c->stack_hq, c->stack_xq, c->stride,
                                      c->err_dev, c->num_sms, s));
      }
      if (!c->in_capture)
        for (int l = 0; l < L; ++l) PMOE_CUDA(cudaEventRecord(c->ev_layer_done[l], s));
      return status;
    }
    for (int l = 0; l < L; ++l) {
      PMOE_CUDA(cudaEventRecord(c->ev_ready[l], ps));
      c->layer_used[l] = 1;
      c->staged[l] = 1;
      c->staged_waves[l] = max_waves(c, P);
      c->pull_deferred[l] = 1;
    }
  } else if (!c->staged[0]) {
    const int r = ensure_resident_impl(c, 0, ids, P, c->ev_stack, nullptr, defer);
    if (r == PMOE_EDEVICE) status = r;
    else if (r != PMOE_OK) return r;
  }
  const uint8_t* in = (const uint8_t*)x;
  for (int l = 0; l < L; ++l) {
    // h_{l+1} = h_l + moe_l(h_l); the buffers alternate so that the last layer writes y
    uint8_t* out = (((L - 1 - l) & 1) == 0) ? (uint8_t*)y : (uint8_t*)work;
    (void)act;
    int r = moe_paged_forward(c, l, in, T, ids + (size_t)l * P, w + (size_t)l * P, in, out, stream);
    if (r == PMOE_EDEVICE) status = r;
    else if (r != PMOE_OK) return r;
    if (l + 1 < L && !c->staged[l + 1]) {
      // plan and page in layer l+1 while layer l computes (the host's plan read-back in
      // copy-engine mode overlaps the kernels just enqueued)
      r = ensure_resident_impl(c, l + 1, ids + (size_t)(l + 1) * P, P, c->ev_stack, nullptr, defer);
      if (r == PMOE_EDEVICE) status = r;
      else if (r != PMOE_OK) return r;
    }
    in = out;
  }
  return status;
}

int expert_cache_stats(pmoe_cache* c, int layer, pmoe_stats* out) {
  if (c == nullptr || out == nullptr || layer < -1 || layer >= c->d.num_layers) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  PMOE_CUDA(cudaStreamSynchronize(c->plan_stream));
  PMOE_CUDA(cudaStreamSynchronize(c->copy_stream));
  for (int l = 0; l < c->d.num_layers; ++l) {
    const int r = wait_event_bounded(c->ev_layer_done[l]);
    if (r != PMOE_OK) return r;
  }
  memset(out, 0, sizeof(*out));
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? c->d.num_layers : layer + 1;
  for (int l = l0; l < l1; ++l) {
    unsigned long long cnt[4];
    PMOE_CUDA(cudaMemcpy(cnt, c->st[l].counters, sizeof(cnt), cudaMemcpyDeviceToHost));
    out->hits += cnt[0];
    out->misses += cnt[1];
    out->waves += cnt[2];
    out->steps += cnt[3];
  }
  out->bytes_paged = out->misses * (uint64_t)c->expert_bytes;
  int32_t err = 0;
  PMOE_CUDA(cudaMemcpy(&err, c->err_dev, 4, cudaMemcpyDeviceToHost));
  return err ? PMOE_EDEVICE : PMOE_OK;
}

int expert_cache_slot_table(pmoe_cache* c, int layer, int32_t* expert_in_slot, int32_t* last_use) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || expert_in_slot == nullptr) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  PMOE_CUDA(cudaStreamSynchronize(c->plan_stream));
  PMOE_CUDA(cudaStreamSynchronize(c->copy_stream));
  PMOE_CUDA(cudaMemcpy(expert_in_slot, c->st[layer].expert_in, 4 * (size_t)c->d.num_slots, cudaMemcpyDeviceToHost));
  if (last_use)
    PMOE_CUDA(cudaMemcpy(last_use, c->st[layer].last_use, 4 * (size_t)c->d.num_slots, cudaMemcpyDeviceToHost));
  int32_t err = 0;
  PMOE_CUDA(cudaMemcpy(&err, c->err_dev, 4, cudaMemcpyDeviceToHost));
  return err ? PMOE_EDEVICE : PMOE_OK;
}

int expert_cache_read_slot(pmoe_cache* c, int layer, int slot, void* host_out, size_t nbytes) {
  if (c == nullptr || layer < 0 || layer >= c->d.num_layers || slot < 0 || slot >= c->d.num_slots ||
      host_out == nullptr || nbytes != c->expert_bytes)
    return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  PMOE_CUDA(cudaStreamSynchronize(c->copy_stream));
  PMOE_CUDA(cudaEventSynchronize(c->ev_layer_done[layer]));
  PMOE_CUDA(cudaMemcpy(host_out, c->arena[layer] + (size_t)slot * c->stride, nbytes, cudaMemcpyDeviceToHost));
  return PMOE_OK;
}

int expert_cache_set_timing(pmoe_cache* c, int enable) {
  if (c == nullptr) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  const int r = resolve_marks(c);
  if (r != PMOE_OK) return r;
  c->timing = enable != 0;
  for (int i = 0; i < PMOE_K_CLASSES; ++i) {
    c->ms[i] = 0.0;
    c->launches[i] = 0;
  }
  c->copies = 0;
  return PMOE_OK;
}

int expert_cache_kernel_times(pmoe_cache* c, pmoe_kernel_times* out) {
  if (c == nullptr || out == nullptr) return PMOE_EINVAL;
  PMOE_CUDA(cudaSetDevice(c->d.device));
  const int r = resolve_marks(c);
  if (r != PMOE_OK) return r;
  for (int i = 0; i < PMOE_K_CLASSES; ++i) {
    out->ms[i] = c->ms[i];
    out->launches[i] = c->launches[i];
  }
  out->copies = c->copies;
  return PMOE_OK;
}

}  // extern "C"
