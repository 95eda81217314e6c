// Internal declarations shared by the library's translation units (host + device).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/pagedmoe.h"

namespace pmoe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kGemvMaxTokens = 8;  // decode (weight-streaming) path for T <= this
constexpr int kDecodeMaxPairs = 64;  // T * top_k of the fused decode kernel

// Programmatic dependent launch (sm_90 and later). A kernel launched with the
// programmatic-serialization attribute may start while the kernel before it in the
// stream is still running; pdl_wait() blocks until that kernel has completed and its
// writes are visible, so a dependent kernel reads nothing its predecessor writes before
// it. pdl_trigger() lets the dependent kernel launch before this one ends. Both are no-ops
// for kernels launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Device error word bits.
enum : int32_t { kErrBadExpertId = 1, kErrPlanOverflow = 2, kErrBadSlot = 4, kErrPullTimeout = 8 };

// Layout of a layer's residency plan (int32 words), written by the residency kernel
// and mirrored to pinned host memory in copy-engine mode.
struct PlanLayout {
  int E;
  __host__ __device__ int header() const { return 0; }                 // 8 words
  __host__ __device__ int wave_start() const { return 8; }             // E + 1
  __host__ __device__ int wave_exp() const { return 8 + (E + 1); }     // E
  __host__ __device__ int wave_slot() const { return 8 + 2 * E + 1; }  // E
  __host__ __device__ int miss_start() const { return 8 + 3 * E + 1; } // E + 1
  __host__ __device__ int miss_exp() const { return 8 + 4 * E + 2; }   // E
  __host__ __device__ int miss_slot() const { return 8 + 5 * E + 2; }  // E
  __host__ __device__ int wave_of() const { return 8 + 6 * E + 2; }    // E
  __host__ __device__ int wave_hits() const { return 8 + 7 * E + 2; }  // E + 1: resident experts first in each wave
  __host__ __device__ int words() const { return 8 + 8 * E + 3; }
};
// header words
// kPlanEpochLo/Hi: a number the residency kernel draws from a cache-wide counter on
// every call, unique per plan; the fused decode kernel tags its intermediate rows with it.
enum { kPlanUnique = 0, kPlanWaves = 1, kPlanMisses = 2, kPlanError = 3, kPlanStep = 4, kPlanEpochLo = 5,
       kPlanEpochHi = 6 };

// One layer's device LRU state.
struct LayerState {
  int32_t* slot_of;     // [E]  slot holding expert e, -1 if absent
  int32_t* expert_in;   // [K]  expert in slot s, -1 if empty
  int32_t* last_use;    // [K]  step of last use, -1 if never
  int32_t* step;        // [1]  the layer's step counter
  unsigned long long* counters;  // [4] hits, misses, waves, steps
};

// Forward workspace (device), shared by all layers of a cache.
struct Workspace {
  int32_t* counts;      // [E]
  int32_t* offs;        // [E + 1]
  int32_t* perm;        // [P]  grouped position -> pair
  int32_t* pos;         // [P]  pair -> grouped position
  int32_t* tiles;       // [3 * max_tiles] (slot, pair start, pair count) per tile, grouped by wave
  int32_t* tile_wave;   // [E + 2] tile range of each wave
  int32_t* tile_split;  // [E + 2] first tile of each wave's non-resident (just paged-in) experts
  __nv_bfloat16* h;     // [P][I] intermediate activations, grouped order
  float* o_part;        // [P][H] per-pair down-projection outputs, grouped order: fp32, or
                        // bf16 in the first half of the bytes where tc_o_part_bf16 says so
  __nv_bfloat16* x_perm;  // [P][H] tokens gathered in grouped order (tensor-core path)
  // Block-FP8 layers on the tensor path hold x_perm and h as two e4m3 planes each, in the
  // same bytes: x planes [2][p_cap][H], h planes [2][p_cap][I] (fp8_planes.cuh), with
  // power-of-two scales sx[p_cap] (one per row) and hsc[I/64][p_cap] (one per 64 columns).
  float* sx;
  float* hsc;
  size_t p_cap;         // rows the tensor-core activation buffers hold (max_tokens * top_k)
  int32_t* chunk_cnt;   // [ceil(P/256)][E] per-chunk histograms / prefixes (large-P grouping)
  // [min(P, 64)][I] fused-decode intermediate rows, one 64-bit word per element: bf16 bits
  // in the low 16, the launch's 48-bit tag above (zeroed once; tag 0 is never issued)
  unsigned long long* hq;
  unsigned long long* epoch;  // [1] counter the residency kernel draws plan epochs from
  int chunk_cap;        // entries of chunk_cnt
  int max_tiles;
};

// Kernel launchers (each returns cudaError_t of the launch).
cudaError_t launch_router_topk(const float* logits, int T, int E, int top_k, int renorm,
                               int32_t* ids, float* w, cudaStream_t s);
// Layers 0..layers-1 at once; layer l's ids are ids[l * n_ids ...], its state lies
// l * state_stride bytes after layer 0's, its plan l * plan_words words after plan0.
cudaError_t launch_residency_layers(const int32_t* ids, int n_ids, int layers, int E, int K, LayerState st0,
                                    size_t state_stride, int32_t* plan0, int plan_words, int32_t* err,
                                    unsigned long long* epoch, cudaStream_t s);
size_t router_gemm_smem(int H, int E);
cudaError_t launch_router_gemm_topk(const __nv_bfloat16* x, const __nv_bfloat16* wr, int T, int H, int E, int top_k,
                                    int renorm, float* logits_out, int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_residency(const int32_t* ids, int n_ids, int E, int K, LayerState st,
                             int32_t* plan, int32_t* err, unsigned long long* epoch, cudaStream_t s,
                             bool pdl = false);
cudaError_t launch_group(const int32_t* ids, int P, int E, const int32_t* plan, Workspace ws,
                         int tile_n, int32_t* err, cudaStream_t s);
// The whole grouping in one CTA (ids, histograms and perm in shared memory), which
// launch_group takes for 1024 < P <= kGroupOneCtaMaxPairs (and P <= 1024 with tiles);
// beyond it, four launches over per-chunk histograms (ws.chunk_cnt).
constexpr int kGroupOneCtaMaxPairs = 8192;
cudaError_t launch_group_one_cta(const int32_t* ids, int P, int E, const int32_t* plan, Workspace ws, int tile_n,
                                 int32_t* err, cudaStream_t s);
cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* perm, int P, int top_k, int H,
                               __nv_bfloat16* x_perm, cudaStream_t s);
cudaError_t launch_gather_rows_fp8x2(const __nv_bfloat16* x, const int32_t* perm, int P, int top_k, int H,
                                     size_t p_cap, uint8_t* xq, float* sx, cudaStream_t s);
cudaError_t launch_gemv_gateup(int fmt, const __nv_bfloat16* x, int T, int top_k, int H, int I,
                               const int32_t* plan, int E, int wave, const Workspace& ws,
                               const uint8_t* arena, size_t stride, int num_sms, cudaStream_t s);
cudaError_t launch_gemv_down(int fmt, int H, int I, const int32_t* plan, int E, int wave,
                             const Workspace& ws, const uint8_t* arena, size_t stride, int num_sms,
                             cudaStream_t s);
cudaError_t launch_combine(const Workspace& ws, const float* w, const __nv_bfloat16* residual,
                           __nv_bfloat16* y, int T, int top_k, int H, cudaStream_t s,
                           const int32_t* skip_if_single_wave_plan = nullptr, bool bf16_part = false);
bool decode_fused_supported(int fmt, int T, int top_k, int H, int I, int num_sms);
// The fused decode kernels' chunking of one CTA's rows: chunks per gate/up part (cg) and
// per down part (cd), and the ring bytes of the largest chunk.
bool decode_chunking(int fmt, int T, int top_k, int H, int I, int num_sms, int* cg, int* cd, size_t* max_chunk);
// Persistent decode of all L layers of a stack in one cooperative launch, every layer's
// step planned beforehand and one wave each (T * top_k <= K). x: h_0 [T][H], y: h_L;
// ids, w: [L][T][top_k]; plan0: layer l's plan at plan0 + l * plan_words; arenas,
// stores: device arrays of the layers' slot arenas and mapped host stores; hq
// [2][16][I] and xq [2][T][H]: tagged exchange words (zeroed once).
bool decode_stack_supported(int fmt, int T, int top_k, int H, int I, int L, int num_sms);
cudaError_t launch_decode_stack(int fmt, const __nv_bfloat16* x, __nv_bfloat16* y, const int32_t* ids, const float* w,
                                int T, int top_k, int H, int I, int E, int L, const int32_t* plan0, int plan_words,
                                uint8_t* const* arenas, const uint8_t* const* stores, unsigned long long* hq,
                                unsigned long long* xq, size_t stride, int32_t* err, int num_sms, cudaStream_t s);
cudaError_t launch_decode_fused(int fmt, const __nv_bfloat16* x, const int32_t* ids, const float* w,
                                const __nv_bfloat16* residual, __nv_bfloat16* y, int T, int top_k, int H, int I,
                                const int32_t* plan, int E, int wave, int sub, int fuse_combine, const Workspace& ws,
                                uint8_t* arena, const uint8_t* store, int pull, size_t stride, int32_t* err,
                                int num_sms, cudaStream_t s, int pdl = 0);
// Whether this device accepts a cooperative launch with programmatic serialization
// (probed once per device with an empty kernel, outside any stream capture).
bool decode_pdl_supported(int device);
cudaError_t launch_pull_pages(const int32_t* plan, int E, int wave, const uint8_t* host_store_dev,
                              size_t stride, size_t expert_bytes, uint8_t* arena, int32_t* err,
                              cudaStream_t s);

// Expert section offsets within an expert's bytes.
struct ExpertLayout {
  size_t gu_w, d_w, gu_s, d_s, bytes;
};
ExpertLayout expert_layout(int fmt, int H, int I);

}  // namespace pmoe
