// Router: softmax over E experts, top-k selection, renormalisation (one warp per token).
//
// Article "Running an MoE Model Larger Than Your VRAM", section "What does Paged
// Experts actually do?": each token is routed to top_k of E experts. Selection
// compares the fp32 logits themselves (descending, ties to the lower id), so the
// chosen ids never depend on how exp is rounded.
#include "pmoe_internal.h"

#include <math.h>

namespace pmoe {
namespace {

// Lane l holds logits e = l + 32 * i, i < NPL.
template <int NPL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                          int top_k, int renorm, int32_t* __restrict__ ids,
                                                          float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
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
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - vmax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    denom = s;
  }
  if (lane < top_k) {
    ids[(size_t)t * top_k + lane] = my_id;
    w[(size_t)t * top_k + lane] = e_sel / denom;
  }
}

}  // namespace

cudaError_t launch_router_topk(const float* logits, int T, int E, int top_k, int renorm, int32_t* ids,
                               float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int threads = 256, per_block = threads / 32;
  const int blocks = (T + per_block - 1) / per_block;
  const int npl = (E + 31) / 32;
#define PMOE_ROUTER_CASE(N) \
  router_topk_kernel<N><<<blocks, threads, 0, s>>>(logits, T, E, top_k, renorm, ids, w)
  if (npl <= 1) PMOE_ROUTER_CASE(1);
  else if (npl <= 2) PMOE_ROUTER_CASE(2);
  else if (npl <= 4) PMOE_ROUTER_CASE(4);
  else if (npl <= 8) PMOE_ROUTER_CASE(8);
  else if (npl <= 16) PMOE_ROUTER_CASE(16);
  else PMOE_ROUTER_CASE(32);
#undef PMOE_ROUTER_CASE
  return cudaGetLastError();
}

}  // namespace pmoe
