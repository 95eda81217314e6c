// Decode path (T <= 8 tokens): weight-streaming GEMV kernels over the slot table,
// the top_k-weighted combine, and the SM-pull page-in kernel.
//
// At batch 1..4 the MoE layer reads each routed expert's weights once and does ~1
// FLOP per byte, so it is bound by HBM bandwidth (the decode-is-memory-bound
// discussion of "SGLang serving optimisation" and "Running an MoE Model Larger Than
// Your VRAM", section "Why is it fast when experts keep crossing PCIe?"). Every
// weight byte is read once per step for all tokens routed to the expert.
//
// Work split: a warp owns whole rows (gate/up: RJ row pairs; down: R rows) of one
// expert; lane l reads the 16-byte chunks l, l+32, ... of each row with
// non-allocating vector loads, so a warp keeps 2-8 KB in flight; the partial sums
// are reduced by a fixed xor-shuffle tree. The per-pair reduction order depends only
// on the row length, never on the slot, the wave or how many tokens share the
// expert, which keeps outputs bitwise identical for every K.
#include "decode_common.cuh"

namespace pmoe {
namespace {

using namespace dec;

// h[p][j] = bf16(silu(x_t . Wg[j]) * (x_t . Wu[j])) for every pair p of every expert of the wave.
template <int FMT, int NCH, int RJ>
__global__ void __launch_bounds__(256) gemv_gateup_kernel(const __nv_bfloat16* __restrict__ x, int T, int top_k,
                                                          int H, int I, const int32_t* __restrict__ plan, int E,
                                                          int wave, Workspace ws, const uint8_t* __restrict__ arena,
                                                          size_t stride, ExpertLayout lay) {
  extern __shared__ uint4 x_s[];
  constexpr int EPC = Fmt<FMT>::EPC;
  const int nv = H / 8;
  for (int i = threadIdx.x; i < T * nv; i += blockDim.x) x_s[i] = __ldg(reinterpret_cast<const uint4*>(x) + i);
  __syncthreads();
  const PlanLayout L{E};
  if (wave >= plan[kPlanWaves]) return;
  const int w0 = plan[L.wave_start() + wave], w1 = plan[L.wave_start() + wave + 1];
  const int jb = I / RJ;
  const int n_items = (w1 - w0) * jb;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nch = H / EPC;
  const size_t row_bytes = (size_t)H * Fmt<FMT>::BPE2 / 2;
  for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < n_items; item += nwarps) {
    const int i = item / jb;
    const int j0 = (item - i * jb) * RJ;
    const int e = plan[L.wave_exp() + w0 + i];
    const int slot = plan[L.wave_slot() + w0 + i];
    const uint8_t* ex = arena + (size_t)slot * stride;
    uint4 gw[RJ][NCH], uw[RJ][NCH];
#pragma unroll
    for (int r = 0; r < RJ; ++r) {
      const uint8_t* grow = ex + lay.gu_w + (size_t)(j0 + r) * row_bytes;
      const uint8_t* urow = ex + lay.gu_w + (size_t)(I + j0 + r) * row_bytes;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nch) {
          gw[r][c] = ld_stream(grow + (size_t)idx * 16);
          uw[r][c] = ld_stream(urow + (size_t)idx * 16);
        }
      }
    }
    const int p0 = ws.offs[e], p1 = ws.offs[e + 1];
    for (int p = p0; p < p1; ++p) {
      const int t = ws.perm[p] / top_k;
      const uint4* xr = x_s + (size_t)t * nv;
#pragma unroll
      for (int r = 0; r < RJ; ++r) {
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int idx = lane + 32 * c;
          if (idx < nch) {
            const ChunkQ qg = chunk_q<FMT>(ex + lay.gu_s, j0 + r, idx, H);
            const ChunkQ qu = chunk_q<FMT>(ex + lay.gu_s, I + j0 + r, idx, H);
            g += chunk_dot<FMT, kSrcShared>(gw[r][c], xr + idx * (EPC / 8), qg);
            u += chunk_dot<FMT, kSrcShared>(uw[r][c], xr + idx * (EPC / 8), qu);
          }
        }
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == r) ws.h[(size_t)p * I + j0 + r] = __float2bfloat16_rn(silu_mul(g, u));
      }
    }
  }
}

// o_part[p][n] = h[p] . Wd[n] (fp32) for every pair p of every expert of the wave.
template <int FMT, int NCH, int R>
__global__ void __launch_bounds__(256) gemv_down_kernel(int H, int I, const int32_t* __restrict__ plan, int E,
                                                        int wave, Workspace ws, const uint8_t* __restrict__ arena,
                                                        size_t stride, ExpertLayout lay) {
  constexpr int EPC = Fmt<FMT>::EPC;
  const PlanLayout L{E};
  if (wave >= plan[kPlanWaves]) return;
  const int w0 = plan[L.wave_start() + wave], w1 = plan[L.wave_start() + wave + 1];
  const int nb = H / R;
  const int n_items = (w1 - w0) * nb;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nch = I / EPC;
  const size_t row_bytes = (size_t)I * Fmt<FMT>::BPE2 / 2;
  for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < n_items; item += nwarps) {
    const int i = item / nb;
    const int n0 = (item - i * nb) * R;
    const int e = plan[L.wave_exp() + w0 + i];
    const int slot = plan[L.wave_slot() + w0 + i];
    const uint8_t* ex = arena + (size_t)slot * stride;
    uint4 wr[R][NCH];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint8_t* row = ex + lay.d_w + (size_t)(n0 + r) * row_bytes;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nch) wr[r][c] = ld_stream(row + (size_t)idx * 16);
      }
    }
    const int p0 = ws.offs[e], p1 = ws.offs[e + 1];
    for (int p = p0; p < p1; ++p) {
      const uint4* hr = reinterpret_cast<const uint4*>(ws.h + (size_t)p * I);
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        acc[r] = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int idx = lane + 32 * c;
          if (idx < nch) {
            const ChunkQ q = chunk_q<FMT>(ex + lay.d_s, n0 + r, idx, I);
            acc[r] += chunk_dot<FMT, kSrcGlobal>(wr[r][c], hr + idx * (EPC / 8), q);
          }
        }
        acc[r] = warp_sum(acc[r]);
      }
      float mine = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (lane == r) mine = acc[r];
      if (lane < R) ws.o_part[(size_t)p * H + n0 + lane] = mine;
    }
  }
}

// y[t][n] = bf16(residual[t][n] + sum_r w[t][r] * o_part[pos[t*k+r]][n]), ranks in order.
// o_part rows are fp32 (decode kernels) or bf16 (tensor-core prefill kernels: BF16_PART).
template <bool BF16_PART>
__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ o_part, const int32_t* __restrict__ pos,
                                                      const float* __restrict__ w,
                                                      const __nv_bfloat16* __restrict__ residual,
                                                      __nv_bfloat16* __restrict__ y, int T, int top_k, int H,
                                                      const int32_t* __restrict__ skip_plan) {
  if (skip_plan != nullptr && skip_plan[kPlanWaves] == 1) return;  // the fused decode kernel already wrote y
  const int nv = H / 8;
  const int total = T * nv;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int t = idx / nv, c = idx - t * nv;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int r = 0; r < top_k; ++r) {
      const int p = pos[t * top_k + r];
      if (p < 0) continue;
      const float wr = w[t * top_k + r];
      float o[8];
      if (BF16_PART) {
        const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o_part) +
                                                        (size_t)p * H + (size_t)c * 8);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[2 * i] = bf_lo(qw[i]);
          o[2 * i + 1] = bf_hi(qw[i]);
        }
      } else {
        const float4* op = reinterpret_cast<const float4*>(static_cast<const float*>(o_part) + (size_t)p * H +
                                                           (size_t)c * 8);
        const float4 a = op[0], b = op[1];
        o[0] = a.x, o[1] = a.y, o[2] = a.z, o[3] = a.w, o[4] = b.x, o[5] = b.y, o[6] = b.z, o[7] = b.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wr, o[i], acc[i]);
    }
    if (residual != nullptr) {
      const uint4 rv = *reinterpret_cast<const uint4*>(residual + (size_t)t * H + (size_t)c * 8);
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = bf_lo(rw[i]) + acc[2 * i];
        acc[2 * i + 1] = bf_hi(rw[i]) + acc[2 * i + 1];
      }
    }
    uint32_t outw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      outw[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * H + (size_t)c * 8) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
}

// SM-pull page-in: copy the wave's missed experts from the mapped pinned store.
__global__ void __launch_bounds__(256) pull_pages_kernel(const int32_t* __restrict__ plan, int E, int wave,
                                                         const uint8_t* __restrict__ store, size_t stride,
                                                         uint8_t* __restrict__ arena) {
  const PlanLayout L{E};
  if (wave >= plan[kPlanWaves]) return;
  const int m0 = plan[L.miss_start() + wave], m1 = plan[L.miss_start() + wave + 1];
  const size_t vec_per = stride / 16;
  const size_t total = (size_t)(m1 - m0) * vec_per;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  constexpr int U = 8;
  for (size_t base = (size_t)blockIdx.x * blockDim.x + threadIdx.x; base < total; base += nthreads * U) {
    uint4 v[U];
    size_t idx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      idx[u] = base + (size_t)u * nthreads;
      if (idx[u] < total) {
        const size_t m = idx[u] / vec_per, off = idx[u] - m * vec_per;
        const int e = plan[L.miss_exp() + m0 + (int)m];
        v[u] = ld_stream(store + (size_t)e * stride + off * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (idx[u] < total) {
        const size_t m = idx[u] / vec_per, off = idx[u] - m * vec_per;
        const int slot = plan[L.miss_slot() + m0 + (int)m];
        *reinterpret_cast<uint4*>(arena + (size_t)slot * stride + off * 16) = v[u];
      }
    }
  }
}

template <int FMT, int NCH, int RJ>
cudaError_t gateup_t(const __nv_bfloat16* x, int T, int top_k, int H, int I, const int32_t* plan, int E, int wave,
                     const Workspace& ws, const uint8_t* arena, size_t stride, ExpertLayout lay, int grid,
                     cudaStream_t s) {
  const size_t smem = (size_t)T * H * 2;
  auto k = gemv_gateup_kernel<FMT, NCH, RJ>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k<<<grid, 256, smem, s>>>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay);
  return cudaGetLastError();
}

template <int FMT, int NCH, int R>
cudaError_t down_t(int H, int I, const int32_t* plan, int E, int wave, const Workspace& ws, const uint8_t* arena,
                   size_t stride, ExpertLayout lay, int grid, cudaStream_t s) {
  gemv_down_kernel<FMT, NCH, R><<<grid, 256, 0, s>>>(H, I, plan, E, wave, ws, arena, stride, lay);
  return cudaGetLastError();
}

}  // namespace

ExpertLayout expert_layout(int fmt, int H, int I) {
  ExpertLayout l{};
  const size_t n_gu = (size_t)2 * I * H, n_d = (size_t)H * I;
  if (fmt == PMOE_BF16) {
    l.gu_w = 0;
    l.d_w = 2 * n_gu;
    l.gu_s = l.d_s = 0;
    l.bytes = 2 * (n_gu + n_d);
  } else if (fmt == PMOE_FP8_BLOCK128) {
    l.gu_w = 0;
    l.d_w = n_gu;
    l.gu_s = n_gu + n_d;
    l.d_s = l.gu_s + 4 * (size_t)(2 * I / 128) * (H / 128);
    l.bytes = l.d_s + 4 * (size_t)(H / 128) * (I / 128);
  } else if (fmt == PMOE_MXFP4) {
    l.gu_w = 0;
    l.d_w = n_gu / 2;
    l.gu_s = l.d_w + n_d / 2;
    l.d_s = l.gu_s + (size_t)(2 * I) * (H / 32);  // one E8M0 byte per row and 32 inputs
    l.bytes = l.d_s + (size_t)H * (I / 32);
  } else if (fmt == PMOE_NVFP4) {
    // each scale section: fp32 tensor scale, 12 bytes of padding, one e4m3 byte per row
    // and block of 16 inputs
    l.gu_w = 0;
    l.d_w = n_gu / 2;
    l.gu_s = l.d_w + n_d / 2;
    l.d_s = l.gu_s + 16 + (size_t)(2 * I) * (H / 16);
    l.bytes = l.d_s + 16 + (size_t)H * (I / 16);
  } else {
    l.gu_w = 0;
    l.d_w = n_gu / 2;
    l.gu_s = l.d_w + n_d / 2;
    l.d_s = l.gu_s + 4 * (size_t)(2 * I) * (H / 128);
    l.bytes = l.d_s + 4 * (size_t)H * (I / 128);
  }
  return l;
}

cudaError_t launch_gemv_gateup(int fmt, const __nv_bfloat16* x, int T, int top_k, int H, int I,
                               const int32_t* plan, int E, int wave, const Workspace& ws, const uint8_t* arena,
                               size_t stride, int num_sms, cudaStream_t s) {
  const ExpertLayout lay = expert_layout(fmt, H, I);
  const int grid = num_sms * 4;
  if (fmt == PMOE_BF16) {
    const int nch = H / 8;
    if (nch <= 32 * 4) return gateup_t<PMOE_BF16, 4, 1>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 8) return gateup_t<PMOE_BF16, 8, 1>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 16) return gateup_t<PMOE_BF16, 16, 1>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_FP8_BLOCK128) {
    const int nch = H / 16;
    if (nch <= 32 * 4) return gateup_t<PMOE_FP8_BLOCK128, 4, 2>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 8) return gateup_t<PMOE_FP8_BLOCK128, 8, 2>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_INT4_GPTQ_G128) {
    const int nch = H / 32;
    if (nch <= 32 * 2) return gateup_t<PMOE_INT4_GPTQ_G128, 2, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 4) return gateup_t<PMOE_INT4_GPTQ_G128, 4, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_MXFP4) {
    const int nch = H / 32;
    if (nch <= 32 * 2) return gateup_t<PMOE_MXFP4, 2, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 4) return gateup_t<PMOE_MXFP4, 4, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_NVFP4) {
    const int nch = H / 32;
    if (nch <= 32 * 2) return gateup_t<PMOE_NVFP4, 2, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 4) return gateup_t<PMOE_NVFP4, 4, 4>(x, T, top_k, H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_down(int fmt, int H, int I, const int32_t* plan, int E, int wave, const Workspace& ws,
                             const uint8_t* arena, size_t stride, int num_sms, cudaStream_t s) {
  const ExpertLayout lay = expert_layout(fmt, H, I);
  const int grid = num_sms * 4;
  if (fmt == PMOE_BF16) {
    const int nch = I / 8;
    if (nch <= 32 * 1) return down_t<PMOE_BF16, 1, 8>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 3) return down_t<PMOE_BF16, 3, 4>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 6) return down_t<PMOE_BF16, 6, 2>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_FP8_BLOCK128) {
    const int nch = I / 16;
    if (nch <= 32 * 2) return down_t<PMOE_FP8_BLOCK128, 2, 4>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 4) return down_t<PMOE_FP8_BLOCK128, 4, 2>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_INT4_GPTQ_G128) {
    const int nch = I / 32;
    if (nch <= 32 * 1) return down_t<PMOE_INT4_GPTQ_G128, 1, 8>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 2) return down_t<PMOE_INT4_GPTQ_G128, 2, 4>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_MXFP4) {
    const int nch = I / 32;
    if (nch <= 32 * 1) return down_t<PMOE_MXFP4, 1, 8>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 2) return down_t<PMOE_MXFP4, 2, 4>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  } else if (fmt == PMOE_NVFP4) {
    const int nch = I / 32;
    if (nch <= 32 * 1) return down_t<PMOE_NVFP4, 1, 8>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
    if (nch <= 32 * 2) return down_t<PMOE_NVFP4, 2, 4>(H, I, plan, E, wave, ws, arena, stride, lay, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const Workspace& ws, const float* w, const __nv_bfloat16* residual, __nv_bfloat16* y,
                           int T, int top_k, int H, cudaStream_t s, const int32_t* skip_plan, bool bf16_part) {
  if (T == 0) return cudaSuccess;
  const int total = T * (H / 8);
  int blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (bf16_part)
    combine_kernel<true><<<blocks, 256, 0, s>>>(ws.o_part, ws.pos, w, residual, y, T, top_k, H, skip_plan);
  else
    combine_kernel<false><<<blocks, 256, 0, s>>>(ws.o_part, ws.pos, w, residual, y, T, top_k, H, skip_plan);
  return cudaGetLastError();
}

cudaError_t launch_pull_pages(const int32_t* plan, int E, int wave, const uint8_t* host_store_dev, size_t stride,
                              size_t expert_bytes, uint8_t* arena, int32_t* err, cudaStream_t s) {
  (void)expert_bytes;
  (void)err;
  // at most one small CTA per SM on half of the SMs: the pull then leaves room for the
  // (cooperative, one CTA per SM) decode kernel to run beside it, and 8 x 16-byte loads
  // per thread keep ~2 MB in flight over the host link
  // The SMs it runs on keep the largest shared-memory carveout, so a decode CTA (which
  // needs most of the shared memory) can be placed beside a pull CTA.
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaFuncSetAttribute(pull_pages_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    carveout_set = true;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  pull_pages_kernel<<<sms / 2, 256, 0, s>>>(plan, E, wave, host_store_dev, stride, arena);
  return cudaGetLastError();
}

}  // namespace pmoe
