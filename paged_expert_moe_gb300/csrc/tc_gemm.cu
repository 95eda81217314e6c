// Prefill path: grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged in shared memory by TMA, one persistent CTA per SM.
//
// Article "Running an MoE Model Larger Than Your VRAM", sections "What does Paged
// Experts actually do?" (the fused MoE runs over the resident slots) and "Why do
// short prompts get slower first tokens?" (a prefill touches nearly every expert).
// With ~128 pairs per expert the contraction is dense enough for the tensor cores.
//
// Tiles (swap-AB: the weight rows are the MMA's M side, the expert's pairs the N side):
//   gate/up  D_g[128 rows j][N pairs] = W_g[j0:j0+128, :] . x_perm[pairs, :]^T and the
//            same for W_u into a second accumulator; the epilogue writes
//            h[pair][j] = bf16(silu(D_g) * D_u).           K = H, BK = 64
//   down     D[128 rows n][N pairs] = W_d[n0:n0+128, :] . h[pairs, :]^T; the epilogue
//            writes the fp32 partial o_part[pair][n].      K = I, BK = 64
// N = the tile's pair count rounded up to 16 (<= 256): the instruction descriptor is
// built per tile, so no MMA work is spent on other experts' pairs beyond that.
// Warp roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues tcgen05.mma (warp 1 owns
// the TMEM allocation), warps 2-5 drain TMEM (32 lanes each) in the epilogue.
// Every mbarrier wait is bounded; on expiry the CTA records kErrTcTimeout, stops,
// waits (bounded) for its copies in flight, frees its TMEM and returns.
#include "tc_gemm.h"

#include <cuda.h>
#include <cstdio>

namespace pmoe {
namespace {

constexpr int kBK = 64;             // K elements per stage (128 bytes of bf16 = one swizzle row)
constexpr int kTileRowsB = 32;      // rows per TMA box of the pair operand
constexpr int kThreads = 192;       // 6 warps
constexpr long long kWaitLimit = 4000000000LL;  // clock64 cycles (~2 s) before a wait gives up
constexpr int32_t kErrTcTimeout = 16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the limit passed or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimit) {
      *abort_flag = 1;
      atomicOr(err, kErrTcTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 accumulator, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

template <bool GATEUP>
struct TcCfg {
  static constexpr int kA = GATEUP ? 2 : 1;                 // A tiles per stage (gate + up)
  static constexpr int kABytes = 128 * kBK * 2;             // 16 KB
  static constexpr int kBBytes = 256 * kBK * 2;             // 32 KB (room for N = 256)
  static constexpr int kStageBytes = kA * kABytes + kBBytes;
  static constexpr int kStages = GATEUP ? 3 : 4;
  static constexpr int kTmemCols = GATEUP ? 512 : 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align slack*/ + 256 /*barriers*/;
};

// One persistent CTA per SM loops over (tile, m-tile) items of one wave.
template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b,
                      const int32_t* __restrict__ plan, int E, int wave, Workspace ws, int I, int H,
                      int32_t* __restrict__ err) {
  using C = TcCfg<GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (wave >= plan[kPlanWaves]) return;
  const int t0 = ws.tile_wave[wave], t1 = ws.tile_wave[wave + 1];
  const int m_tiles = GATEUP ? (I / 128) : (H / 128);
  const int n_items = (t1 - t0) * m_tiles;
  if ((int)blockIdx.x >= n_items) return;
  const int kdim = GATEUP ? H : I;
  const int n_kb = kdim / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w);
    prefetch_map(&map_b);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = t0 + item / m_tiles, mt = item % m_tiles;
        const int slot = ws.tiles[3 * tile + 0], pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
        const int nb = (np + kTileRowsB - 1) / kTileRowsB;
        const uint32_t bytes = C::kA * C::kABytes + nb * kTileRowsB * kBK * 2;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          if (GATEUP) {
            tma_load_3d(st, &map_w, &full[s], kb * kBK, mt * 128, slot);
            tma_load_3d(st + C::kABytes, &map_w, &full[s], kb * kBK, I + mt * 128, slot);
          } else {
            tma_load_3d(st, &map_w, &full[s], kb * kBK, mt * 128, slot);
          }
          uint8_t* bst = st + C::kA * C::kABytes;
          for (int b = 0; b < nb; ++b)
            tma_load_2d(bst + b * kTileRowsB * kBK * 2, &map_b, &full[s], kb * kBK, pstart + b * kTileRowsB);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain: every stage's last load consumed and its MMAs committed (bounded)
      for (int i = 0; i < C::kStages; ++i) {
        mbar_wait(&empty[s], ph ^ 1u, abort_flag, err);
        if (++s == C::kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int tile = t0 + item / m_tiles;
        const int np = ws.tiles[3 * tile + 2];
        const int n_mma = (np + 15) & ~15;
        const uint32_t idesc = idesc_bf16(128, n_mma < 16 ? 16 : n_mma);
        if (it > 0) {
          if (!mbar_wait(acc_empty, acc_ph, abort_flag, err)) break;
          acc_ph ^= 1u;
          fence_after();
        }
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, err)) {
            ok = false;
            break;
          }
          fence_after();
          const uint8_t* st = smem + s * C::kStageBytes;
          const uint32_t a0 = smem_u32(st);
          const uint32_t bb = smem_u32(st + C::kA * C::kABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            mma_bf16(tmem, sw128_desc(a0 + kk * 32), sw128_desc(bb + kk * 32), idesc, acc);
            if (GATEUP) mma_bf16(tmem + 256, sw128_desc(a0 + C::kABytes + kk * 32), sw128_desc(bb + kk * 32), idesc, acc);
          }
          mma_commit(&empty[s]);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) mma_commit(acc_full);
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
    const int q = warp & 3;
    const int row = q * 32 + lane;
    uint32_t acc_ph = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int tile = t0 + item / m_tiles, mt = item % m_tiles;
      const int pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
      const int n_mma = (np + 15) & ~15;
      if (!mbar_wait(acc_full, acc_ph, abort_flag, err)) break;
      acc_ph ^= 1u;
      fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = 0; c < n_mma; c += 16) {
        if (GATEUP) {
          uint32_t g[16], u[16];
          tmem_ld16(tbase + c, g);
          tmem_ld16(tbase + 256 + c, u);
          tmem_wait_ld();
          const int j = mt * 128 + row;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (c + i < np) {
              const float gv = __uint_as_float(g[i]), uv = __uint_as_float(u[i]);
              const float hv = gv / (1.f + expf(-gv)) * uv;
              ws.h[(size_t)(pstart + c + i) * I + j] = __float2bfloat16_rn(hv);
            }
          }
        } else {
          uint32_t o[16];
          tmem_ld16(tbase + c, o);
          tmem_wait_ld();
          const int n = mt * 128 + row;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < np) ws.o_part[(size_t)(pstart + c + i) * H + n] = __uint_as_float(o[i]);
        }
      }
      fence_before();
      mbar_arrive(acc_empty);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

int encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
           const cuuint32_t* box) {
  EncodeTiledFn fn = get_encode();
  if (fn == nullptr) return PMOE_ECUDA;
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides_bytes, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PMOE_OK : PMOE_ECUDA;
}

template <bool GATEUP>
cudaError_t launch_tc(const CUtensorMap& mw, const CUtensorMap& mb, const int32_t* plan, int E, int wave,
                      const Workspace& ws, int I, int H, int num_sms, int32_t* err, cudaStream_t s) {
  using C = TcCfg<GATEUP>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(tc_grouped_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc_grouped_kernel<GATEUP><<<num_sms, kThreads, C::kSmemBytes, s>>>(mw, mb, plan, E, wave, ws, I, H, err);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(int H, int I) {
  return H % 128 == 0 && I % 128 == 0 && H >= 128 && I >= 128 && get_encode() != nullptr;
}

int tc_make_weight_maps(uint8_t* arena, size_t stride, int K, int H, int I, TcMaps* out) {
  if (stride % 16 != 0) return PMOE_EUNSUPPORTED;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)(2 * I), (cuuint64_t)K};
    const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)stride};
    const cuuint32_t box[3] = {(cuuint32_t)kBK, 128, 1};
    if (encode(&out->gu, arena, 3, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)K};
    const cuuint64_t strides[2] = {(cuuint64_t)I * 2, (cuuint64_t)stride};
    const cuuint32_t box[3] = {(cuuint32_t)kBK, 128, 1};
    uint8_t* base = arena + (size_t)2 * 2 * I * H;  // W_d follows W_gu in a bf16 expert
    if (encode(&out->d, base, 3, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  return PMOE_OK;
}

int tc_make_act_maps(__nv_bfloat16* x_perm, __nv_bfloat16* h, size_t P, int H, int I, TcMaps* out) {
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)P};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kTileRowsB};
    if (encode(&out->x, x_perm, 2, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)P};
    const cuuint64_t strides[1] = {(cuuint64_t)I * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kTileRowsB};
    if (encode(&out->h, h, 2, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  return PMOE_OK;
}

cudaError_t tc_gateup(const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, const Workspace& ws,
                      int I, int H, int num_sms, int32_t* err, cudaStream_t s) {
  return launch_tc<true>(wm.gu, am.x, plan, E, wave, ws, I, H, num_sms, err, s);
}

cudaError_t tc_down(const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, const Workspace& ws,
                    int I, int H, int num_sms, int32_t* err, cudaStream_t s) {
  return launch_tc<false>(wm.d, am.h, plan, E, wave, ws, I, H, num_sms, err, s);
}

}  // namespace pmoe
