// Router: softmax over E experts, top-k selection, renormalisation (one warp per token);
// and the same preceded by the router GEMM (hidden state -> E logits) in one kernel.
//
// Article "Running an MoE Model Larger Than Your VRAM", section "What does Paged
// Experts actually do?": each token is routed to top_k of E experts. Selection
// compares the fp32 logits themselves (descending, ties to the lower id), so the
// chosen ids never depend on how exp is rounded.
#include "step_common.cuh"

#include <math.h>

namespace pmoe {
namespace {

using step::warp_topk;

template <int NPL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                          int top_k, int renorm, int32_t* __restrict__ ids,
                                                          float* __restrict__ w) {
  pdl_trigger();  // the residency step may launch now; it waits for these ids itself
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk<NPL>(logits + (size_t)t * E, E, top_k, renorm, ids + (size_t)t * top_k, w + (size_t)t * top_k);
}

// Router GEMM fused with the top-k: logits[t][e] = sum_c x[t][c] * W[e][c] for a tile of
// kRgTokens tokens (their rows staged in shared memory; each router row is read once per
// tile), then one warp per token selects and weights its experts from the tile's logits.
// Each logit is one warp's reduction: lane-strided 16-byte chunks accumulated in fp32 in
// chunk order, then an xor-shuffle tree - the same order for every tile and launch.
constexpr int kRgTokens = 8;

template <int NPL>
__global__ void __launch_bounds__(256) router_gemm_topk_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const __nv_bfloat16* __restrict__ wr, int T, int H,
                                                               int E, int top_k, int renorm,
                                                               float* __restrict__ logits_out,
                                                               int32_t* __restrict__ ids, float* __restrict__ w) {
  extern __shared__ __align__(16) uint8_t rg_smem[];
  uint4* xs = reinterpret_cast<uint4*>(rg_smem);                                   // [kRgTokens][H/8]
  float* ls = reinterpret_cast<float*>(rg_smem + (size_t)kRgTokens * H * 2);       // [kRgTokens][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int t0 = blockIdx.x * kRgTokens, nt = min(kRgTokens, T - t0);
  const int nv = H / 8;
  for (int i = threadIdx.x; i < nt * nv; i += blockDim.x)
    xs[i] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t0 * H) + i);
  __syncthreads();
  for (int e = warp; e < E; e += nwarps) {
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    float acc[kRgTokens];
#pragma unroll
    for (int t = 0; t < kRgTokens; ++t) acc[t] = 0.f;
    for (int c = lane; c < nv; c += 32) {
      const uint4 wv = __ldg(wrow + c);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int t = 0; t < kRgTokens; ++t) {
        if (t < nt) {
          const uint4 xv = xs[t * nv + c];
          const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
          float a = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            a = fmaf(__uint_as_float(ww[q] << 16), __uint_as_float(xx[q] << 16), a);
            a = fmaf(__uint_as_float(ww[q] & 0xffff0000u), __uint_as_float(xx[q] & 0xffff0000u), a);
          }
          acc[t] += a;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRgTokens; ++t) {
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && t < nt) {
        ls[t * E + e] = v;
        if (logits_out != nullptr) logits_out[(size_t)(t0 + t) * E + e] = v;
      }
    }
  }
  __syncthreads();
  if (warp < nt)
    warp_topk<NPL>(ls + warp * E, E, top_k, renorm, ids + (size_t)(t0 + warp) * top_k,
                   w + (size_t)(t0 + warp) * top_k);
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

size_t router_gemm_smem(int H, int E) { return (size_t)kRgTokens * H * 2 + (size_t)kRgTokens * E * 4; }

cudaError_t launch_router_gemm_topk(const __nv_bfloat16* x, const __nv_bfloat16* wr, int T, int H, int E, int top_k,
                                    int renorm, float* logits_out, int32_t* ids, float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const size_t smem = router_gemm_smem(H, E);
  const int blocks = (T + kRgTokens - 1) / kRgTokens;
  const int npl = (E + 31) / 32;
#define PMOE_RG_CASE(N)                                                                                       \
  do {                                                                                                        \
    cudaError_t e_ = cudaFuncSetAttribute(router_gemm_topk_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                          (int)smem);                                                         \
    if (e_ != cudaSuccess) return e_;                                                                         \
    router_gemm_topk_kernel<N><<<blocks, 256, smem, s>>>(x, wr, T, H, E, top_k, renorm, logits_out, ids, w); \
  } while (0)
  if (npl <= 1) PMOE_RG_CASE(1);
  else if (npl <= 2) PMOE_RG_CASE(2);
  else if (npl <= 4) PMOE_RG_CASE(4);
  else if (npl <= 8) PMOE_RG_CASE(8);
  else if (npl <= 16) PMOE_RG_CASE(16);
  else PMOE_RG_CASE(32);
#undef PMOE_RG_CASE
  return cudaGetLastError();
}

}  // namespace pmoe
