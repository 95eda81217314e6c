// Prefill path: grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged in shared memory by TMA, one persistent CTA per SM.
//
// Article "Running an MoE Model Larger Than Your VRAM", sections "What does Paged
// Experts actually do?" (the fused MoE runs over the resident slots) and "Why do
// short prompts get slower first tokens?" (a prompt's tokens route to almost all
// of a layer's experts).
// With ~128 pairs per expert the contraction is dense enough for the tensor cores.
//
// Tiles (swap-AB: the weight rows are the MMA's M side, the expert's pairs the N side):
//   gate/up  D[128][N pairs] = [W_g[j0:j0+64]; W_u[j0:j0+64]] . x_perm[pairs]^T: TMEM
//            lanes 0-63 hold gate, 64-127 the matching up rows; the epilogue exchanges
//            them through shared memory and writes h[pair][j0:j0+64] =
//            bf16(silu(gate) * up) as 16-byte rows.           K = H, BK = 64
//   down     D[128 rows n][N pairs] = W_d[n0:n0+128, :] . h[pairs, :]^T; the epilogue
//            writes the pair's expert output o_part[pair][n]: bf16 weights as bf16
//            rows (half the bytes for the combine to read), staged through shared
//            memory two pairs to a word; quantised ones (converter warps) as fp32
//            rows.                                             K = I, BK = 64
// The two TMEM accumulator buffers (2 x 256 columns) let the epilogue of one item run
// while the MMAs of the next fill the other buffer; 4 TMA stages of 48 KB. Every TMA
// instruction costs time of its own, so a bf16 stage is few boxes: gate/up's weight tile
// as one 4-D box (64 gate rows, then the 64 up rows), a tile of more than 64 pairs in
// 128-row boxes.
// N = the tile's pair count rounded up to 16 (<= 256): the instruction descriptor is
// built per tile, so no MMA work is spent on other experts' pairs beyond that.
// Warp roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues tcgen05.mma (warp 1 owns
// the TMEM allocation), warps 2-5 drain TMEM (32 lanes each) in the epilogue. Quantised
// weights: warp 0 streams the raw weight tiles into a deep ring of their own, warp 14
// the activation tiles, and converter warps 6-13 dequantise each raw tile (loaded with the
// TMA swizzle of its 64- or 32-byte rows, so that their reads are conflict-free) into a
// shallow ring of bf16 operand tiles (the raw bytes, not the operand tiles, are what must
// be in flight from HBM).
// Every mbarrier wait is bounded; on expiry the CTA records kErrTcTimeout, stops,
// waits (bounded) for its copies in flight, frees its TMEM and returns.
#include "tc_gemm.h"

#include "fp8_planes.cuh"

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cstdio>

namespace pmoe {
namespace {

constexpr int kBK = 64;             // K elements per stage (128 bytes of bf16 = one swizzle row)
constexpr int kTileRowsB = 32;      // rows per TMA box of the pair operand
constexpr int kBigRowsB = 128;      // rows per box of a tile's whole 128-pair chunks (tiles of >= 128 pairs)
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

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
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

// Instruction descriptor, kind::f8f6f4: e4m3 A and B (format code 0, K-major), fp32 accumulator.
__device__ __forceinline__ uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One FP8 MMA, K = 32 (32 bytes of each K-major row).
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n"
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

// Stage: A = 128 weight rows x 64 K (16 KB) + B = up to NMAX pair rows x 64 K (NMAX = 256:
// 32 KB; NMAX = 64, used when a forward has few tokens per expert: 8 KB, which leaves room
// for twice the stages and so hides twice the latency).
// Gate/up A tiles hold 64 gate rows (TMEM lanes 0-63) then the matching 64 up rows
// (lanes 64-127), so one M=128 MMA feeds both halves of SiLU*mul.
template <int FMT, int NMAX>
struct TcCfg {
  static constexpr bool kQuant = FMT != PMOE_BF16;
  static constexpr int kABytes = 128 * kBK * 2;            // bf16 A tile (MMA operand)
  static constexpr int kBBytes = NMAX * kBK * 2;           // bf16 B tile (up to NMAX pairs)
  // quantised A tile as loaded by TMA, before the converter warps dequantise it
  static constexpr int kQBytes = FMT == PMOE_FP8_BLOCK128                           ? 128 * kBK
                                 : (FMT == PMOE_INT4_GPTQ_G128 || FMT == PMOE_MXFP4 || FMT == PMOE_NVFP4)
                                     ? 128 * kBK / 2
                                                                                     : 0;
  static constexpr int kStagingFloats = 128 * 17;
  // quantised formats: each converter thread's copy of its row's scales (<= 16 words), padded
  static constexpr int kScaleWords = kQuant ? 256 * 17 : 0;
  static constexpr int kFixedBytes = kStagingFloats * 4 + kScaleWords * 4 + 1024 + 1024;
  static constexpr int kBudget = 220 * 1024 - kFixedBytes;
  // bf16: stages of (A + B) as deep as fit, at most 8
  static constexpr int kStagesFit = kBudget / (kABytes + kBBytes);
  static constexpr int kStages = kQuant ? 0 : (kStagesFit < 8 ? kStagesFit : 8);
  // quantised: three rings. The raw weight tiles stream from HBM and set the pace, so
  // they get most of the memory (deep: many tiles in flight); the converted bf16 A tiles
  // only bridge the converters and the MMAs (shallow); the activation tiles (B) sit in
  // between.
  static constexpr int kAStages = kQuant ? (NMAX > 64 ? 3 : 5) : 0;
  static constexpr int kBStages = kQuant ? (NMAX > 64 ? 3 : 6) : 0;
  static constexpr int kQFit = kQuant ? (kBudget - kAStages * kABytes - kBStages * kBBytes) / kQBytes : 0;
  static constexpr int kQStages = kQFit < 24 ? kQFit : 24;
  static constexpr int kRingBytes =
      kQuant ? kAStages * kABytes + kBStages * kBBytes + kQStages * kQBytes : kStages * (kABytes + kBBytes);
  static constexpr int kAccCols = 256;   // one accumulator buffer (N <= 256 fp32 columns)
  static constexpr int kTmemCols = 512;  // two buffers: the epilogue of tile i overlaps the MMAs of tile i+1
  static constexpr int kSmemBytes = kRingBytes + kFixedBytes;
  // + 8 converter warps (two threads per A-tile row) and a second producer warp (activation tiles)
  static constexpr int kThreads = kQuant ? 480 : 192;
  static_assert((kQuant ? (kAStages >= 2 && kQStages >= 4) : kStages >= 2) && kSmemBytes <= 227 * 1024,
                "shared memory");
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Down epilogue, one chunk of 16 pairs c..c+15 of an item (m-tile mt). Thread `row` (the
// TMEM lane: weight row n = mt * 128 + row) holds v[i] for pair c + i; it rounds them to
// bf16 and stages them two pairs to a word, stg[row * 9 + j] = (pair 2j, pair 2j + 1).
// After a barrier, thread et (0..127) reads the words of pairs 2 (et & 7) and + 1 for
// rows (et >> 3) * 8 .. +7 and writes each pair's 8 outputs as one 16-byte store. Half
// the shared-memory traffic of fp32 staging; both sides hit 32 distinct banks.
__device__ __forceinline__ void stage_o_chunk(uint32_t* stg, int row, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    stg[row * 9 + j] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

__device__ __forceinline__ void store_o_rows(const uint32_t* stg, int et, int c, int np, int pstart, int mt,
                                             int H, float* o_part) {
  const int pp = et & 7, rb = et >> 3;
  const int p0 = c + 2 * pp;
  if (p0 >= np) return;
  uint32_t w[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) w[r] = stg[(rb * 8 + r) * 9 + pp];
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    lo[k] = (w[2 * k] & 0xffffu) | (w[2 * k + 1] << 16);
    hi[k] = (w[2 * k] >> 16) | (w[2 * k + 1] & 0xffff0000u);
  }
  __nv_bfloat16* o16 = reinterpret_cast<__nv_bfloat16*>(o_part);
  const size_t col = (size_t)mt * 128 + rb * 8;
  *reinterpret_cast<uint4*>(o16 + (size_t)(pstart + p0) * H + col) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  if (p0 + 1 < np)
    *reinterpret_cast<uint4*>(o16 + (size_t)(pstart + p0 + 1) * H + col) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

// Named barrier over the 128 epilogue threads that also ORs a predicate across them,
// so a failed wait in any epilogue thread makes all of them leave together.
__device__ __forceinline__ int epi_bar_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred)
      : "memory");
  return r;
}

// One persistent CTA per SM loops over (tile, m-tile) items of one wave.
template <bool GATEUP, int FMT, int NMAX>
__global__ void __launch_bounds__(TcCfg<FMT, NMAX>::kThreads, 1)
    tc_grouped_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b,
                      const __grid_constant__ CUtensorMap map_bb,
                      const int32_t* __restrict__ plan, int E, int wave, int sub, Workspace ws, int I, int H,
                      const uint8_t* __restrict__ arena, size_t stride, ExpertLayout lay, int32_t* __restrict__ err) {
  using C = TcCfg<FMT, NMAX>;
  constexpr bool kQuant = C::kQuant;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // bf16: smem = kStages x (A | B). Quantised: A ring, then B ring, then Q ring.
  uint8_t* aring = smem;
  uint8_t* bring = aring + C::kAStages * C::kABytes;
  uint8_t* qring = bring + C::kBStages * C::kBBytes;
  float* staging = reinterpret_cast<float*>(smem + C::kRingBytes);
  uint32_t* scale_cache = reinterpret_cast<uint32_t*>(staging + C::kStagingFloats);
  uint64_t* bars = reinterpret_cast<uint64_t*>(scale_cache + C::kScaleWords);
  // bf16 stages
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  // quantised rings: raw tile landed / read by the converters; B tile landed / used by
  // the MMAs; converted A tile written / used by the MMAs
  uint64_t* qfull = empty + C::kStages;
  uint64_t* qempty = qfull + C::kQStages;
  uint64_t* bfull = qempty + C::kQStages;
  uint64_t* bempty = bfull + C::kBStages;
  uint64_t* afull = bempty + C::kBStages;
  uint64_t* aempty = afull + C::kAStages;
  uint64_t* acc_full = aempty + C::kAStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;         // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (wave >= plan[kPlanWaves]) return;
  int t0 = ws.tile_wave[wave], t1 = ws.tile_wave[wave + 1];
  if (sub == 1) t1 = ws.tile_split[wave];       // experts resident before the step
  else if (sub == 2) t0 = ws.tile_split[wave];  // experts paged in for this wave
  const int m_tiles = GATEUP ? (I / 64) : (H / 128);
  const int n_items = (t1 - t0) * m_tiles;
  if ((int)blockIdx.x >= n_items) return;
  const int kdim = GATEUP ? H : I;
  const int n_kb = kdim / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], 256);
    }
    for (int s = 0; s < C::kBStages; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < C::kAStages; ++s) {
      mbar_init(&afull[s], 256);
      mbar_init(&aempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w);
    prefetch_map(&map_b);
    prefetch_map(&map_bb);
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
  // a tile's pair rows (bf16 operand tiles): more than 64 of them in 128-row boxes, the
  // last box reading past the tile (rows no MMA column uses; at most NMAX rows in all),
  // fewer in 32-row boxes
  auto b_boxes = [&](int np, int* nbig, int* nsmall) {
    const bool big = NMAX >= kBigRowsB && np > 64;
    *nbig = big ? (np + kBigRowsB - 1) / kBigRowsB : 0;
    *nsmall = big ? 0 : (np + kTileRowsB - 1) / kTileRowsB;
  };

  if (warp == 0 && !kQuant) {
    if (lane == 0) {
      // ---------------- TMA producer (bf16): A and B tiles of one stage
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = t0 + item / m_tiles, mt = item % m_tiles;
        const int slot = ws.tiles[3 * tile + 0], pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
        int nbig, nsmall;
        b_boxes(np, &nbig, &nsmall);
        const int r0 = nbig * kBigRowsB;
        const uint32_t bytes = C::kABytes + (r0 + nsmall * kTileRowsB) * kBK * 2;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * (C::kABytes + C::kBBytes);
          mbar_arrive_expect_tx(&full[s], bytes);
          if (GATEUP) {
            tma_load_4d(st, &map_w, &full[s], kb * kBK, mt * 64, 0, slot);  // 64 gate rows, then the 64 up rows
          } else {
            tma_load_3d(st, &map_w, &full[s], kb * kBK, mt * 128, slot);
          }
          uint8_t* bst = st + C::kABytes;
          for (int b = 0; b < nbig; ++b)
            tma_load_2d(bst + b * kBigRowsB * kBK * 2, &map_bb, &full[s], kb * kBK, pstart + b * kBigRowsB);
          for (int b = 0; b < nsmall; ++b)
            tma_load_2d(bst + (r0 + b * kTileRowsB) * kBK * 2, &map_b, &full[s], kb * kBK, pstart + r0 + b * kTileRowsB);
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
  } else if (warp == 0 && kQuant) {
    if (lane == 0) {
      // ---------------- TMA producer of the raw weight tiles (quantised formats)
      int q = 0;
      uint32_t qph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = t0 + item / m_tiles, mt = item % m_tiles;
        const int slot = ws.tiles[3 * tile + 0];
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&qempty[q], qph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* dst = qring + q * C::kQBytes;
          mbar_arrive_expect_tx(&qfull[q], C::kQBytes);
          const int kc = FMT == PMOE_FP8_BLOCK128 ? kb * kBK : kb * kBK / 2;  // bytes along K
          if (GATEUP) {
            tma_load_3d(dst, &map_w, &qfull[q], kc, mt * 64, slot);
            tma_load_3d(dst + C::kQBytes / 2, &map_w, &qfull[q], kc, I + mt * 64, slot);
          } else {
            tma_load_3d(dst, &map_w, &qfull[q], kc, mt * 128, slot);
          }
          if (++q == C::kQStages) {
            q = 0;
            qph ^= 1u;
          }
        }
      }
      for (int i = 0; i < C::kQStages; ++i) {  // drain: every raw tile read by the converters
        mbar_wait(&qempty[q], qph ^ 1u, abort_flag, err);
        if (++q == C::kQStages) {
          q = 0;
          qph ^= 1u;
        }
      }
    }
  } else if (kQuant && warp == 14) {
    if (lane == 0) {
      // ---------------- TMA producer of the activation tiles (quantised formats)
      int b = 0;
      uint32_t bph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = t0 + item / m_tiles;
        const int pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
        // 32-row boxes here (128-row ones measured 2-3% slower with the converter stage)
        const int nb = (np + kTileRowsB - 1) / kTileRowsB;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&bempty[b], bph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* bst = bring + b * C::kBBytes;
          mbar_arrive_expect_tx(&bfull[b], (uint32_t)(nb * kTileRowsB * kBK * 2));
          for (int t = 0; t < nb; ++t)
            tma_load_2d(bst + t * kTileRowsB * kBK * 2, &map_b, &bfull[b], kb * kBK, pstart + t * kTileRowsB);
          if (++b == C::kBStages) {
            b = 0;
            bph ^= 1u;
          }
        }
      }
      for (int i = 0; i < C::kBStages; ++i) {  // drain: every B tile used by its MMAs
        mbar_wait(&bempty[b], bph ^ 1u, abort_flag, err);
        if (++b == C::kBStages) {
          b = 0;
          bph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int s = 0, qb = 0;
      uint32_t ph = 0, qbph = 0;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int tile = t0 + item / m_tiles;
        const int np = ws.tiles[3 * tile + 2];
        const int n_mma = (np + 15) & ~15;
        const uint32_t idesc = idesc_bf16(128, n_mma < 16 ? 16 : n_mma);
        const int ab = it & 1, use = it >> 1;
        if (use > 0) {
          if (!mbar_wait(&acc_empty[ab], (uint32_t)((use - 1) & 1), abort_flag, err)) break;
          fence_after();
        }
        const uint32_t d = tmem + (uint32_t)(ab * C::kAccCols);
        for (int kb = 0; kb < n_kb; ++kb) {
          uint32_t a0, bb;
          if constexpr (kQuant) {
            // s / ph walk the A ring, qb / qbph the B ring
            if (!mbar_wait(&afull[s], ph, abort_flag, err) || !mbar_wait(&bfull[qb], qbph, abort_flag, err)) {
              ok = false;
              break;
            }
            a0 = smem_u32(aring + s * C::kABytes);
            bb = smem_u32(bring + qb * C::kBBytes);
          } else {
            if (!mbar_wait(&full[s], ph, abort_flag, err)) {
              ok = false;
              break;
            }
            const uint8_t* st = smem + s * (C::kABytes + C::kBBytes);
            a0 = smem_u32(st);
            bb = smem_u32(st + C::kABytes);
          }
          fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(d, sw128_desc(a0 + kk * 32), sw128_desc(bb + kk * 32), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          if constexpr (kQuant) {
            mma_commit(&aempty[s]);
            mma_commit(&bempty[qb]);
            if (++qb == C::kBStages) {
              qb = 0;
              qbph ^= 1u;
            }
            if (++s == C::kAStages) {
              s = 0;
              ph ^= 1u;
            }
          } else {
            mma_commit(&empty[s]);
            if (++s == C::kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        if (ok) mma_commit(&acc_full[ab]);
      }
    }
  } else if (kQuant && warp >= 6 && warp <= 13) {
    // ---------------- converters: warps 6..13, two threads per row of the A tile (thread
    // ct owns row ct % 128, K half ct / 128 of each stage). Each
    // quantised row (64 K values) is dequantised with its scale (block-FP8: the fp32
    // scale of its 128x128 block; int4: (q - z) * s of its group of 128; MXFP4: the E2M1
    // value times 2^(X - 127) of its block of 32, exact in bf16) to bf16 and written in
    // the 128-byte-swizzled K-major layout TMA would have produced.
    const int ct = threadIdx.x - 192, r = ct & 127, hf = ct >> 7;
    int q = 0, s = 0;  // raw tile (Q ring) and converted tile (A ring) of the current step
    uint32_t qph = 0, ph = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int tile = t0 + item / m_tiles, mt = item % m_tiles;
      const int slot = ws.tiles[3 * tile + 0];
      const uint8_t* ex = arena + (size_t)slot * stride;
      const int grow = GATEUP ? (r < 64 ? mt * 64 + r : I + mt * 64 + (r - 64)) : mt * 128 + r;
      const int cols = GATEUP ? H : I;
      const uint8_t* sc = ex + (GATEUP ? lay.gu_s : lay.d_s);
      // this row's scales (block-FP8: one fp32 per 128-column block of its block row;
      // int4: one (s, z) pair per group; MXFP4: one E8M0 byte per 32 columns, four to a
      // word), read once per item instead of once per stage
      // (NVFP4: one word = the four e4m3 block scales of a 64-input stage, after the
      // 16-byte tensor-scale header; the tensor scale itself is applied in the epilogue)
      const int nblk = FMT == PMOE_NVFP4 ? (cols >> 6) : (cols >> 7);
      const uint32_t* srow =
          FMT == PMOE_NVFP4 ? reinterpret_cast<const uint32_t*>(sc + 16 + (size_t)grow * (cols >> 4))
                            : reinterpret_cast<const uint32_t*>(sc) +
                                  (FMT == PMOE_FP8_BLOCK128 ? (size_t)(grow >> 7) * nblk : (size_t)grow * nblk);
      uint32_t* my_sc = scale_cache + ct * 17;
      const bool cached = nblk <= 16;
      if (cached)
        for (int j = 0; j < nblk; ++j) my_sc[j] = __ldg(srow + j);
      for (int kb = 0; kb < n_kb; ++kb) {
        if (!mbar_wait(&qfull[q], qph, abort_flag, err) || !mbar_wait(&aempty[s], ph ^ 1u, abort_flag, err)) {
          ok = false;
          break;
        }
        const uint8_t* qt = qring + q * C::kQBytes;  // row r at qt + r * (kQBytes / 128)
        uint4* arow = reinterpret_cast<uint4*>(aring + s * C::kABytes + r * 128);
        // this thread's 32 (e4m3) or 16 (4-bit) bytes of its row: 16-byte chunks at their
        // swizzled places (64-byte rows: chunk k at k ^ ((r >> 1) & 3); 32-byte rows: chunk
        // k at k ^ ((r >> 2) & 1)), conflict-free across the warp's 32 rows
        uint32_t qw[8];
        if (FMT == PMOE_FP8_BLOCK128) {
          const uint8_t* qrow = qt + r * kBK;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + (((2 * hf + k) ^ ((r >> 1) & 3)) << 4));
            qw[4 * k + 0] = v.x, qw[4 * k + 1] = v.y, qw[4 * k + 2] = v.z, qw[4 * k + 3] = v.w;
          }
        } else {
          const uint4 v = *reinterpret_cast<const uint4*>(qt + r * (kBK / 2) + ((hf ^ ((r >> 2) & 1)) << 4));
          qw[0] = v.x, qw[1] = v.y, qw[2] = v.z, qw[3] = v.w;
        }
        if (FMT == PMOE_FP8_BLOCK128) {
          const float sv = __uint_as_float(cached ? my_sc[(kb * kBK) >> 7] : __ldg(srow + ((kb * kBK) >> 7)));
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            const int c = 4 * hf + ci;
            const uint32_t wv[2] = {qw[2 * ci], qw[2 * ci + 1]};
            uint32_t out[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[h] & 0xffffu), __NV_E4M3);
              const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[h] >> 16), __NV_E4M3);
              const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
              const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
              const __nv_bfloat162 b0 = __floats2bfloat162_rn(f0.x * sv, f0.y * sv);
              const __nv_bfloat162 b1 = __floats2bfloat162_rn(f1.x * sv, f1.y * sv);
              out[2 * h] = *reinterpret_cast<const uint32_t*>(&b0);
              out[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&b1);
            }
            arow[c ^ (r & 7)] = make_uint4(out[0], out[1], out[2], out[3]);
          }
        } else if (FMT == PMOE_NVFP4) {
          // 64 codes = four blocks of 16, each with its own e4m3 byte; E2M1 times e4m3
          // is exact in bf16
          const uint32_t bw = cached ? my_sc[kb] : __ldg(srow + kb);
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            const int c = 4 * hf + ci;
            const uint32_t word = qw[ci];  // 8 codes, low nibble first
            const __half_raw sh = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)((bw >> (8 * (c >> 1))) & 0xffu), __NV_E4M3);
            const float sv = __half2float(*reinterpret_cast<const __half*>(&sh));
            uint32_t out[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const __half2_raw pr =
                  __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * h)) & 0xffu), __NV_E2M1);
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pr));
              const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sv, f.y * sv);
              out[h] = *reinterpret_cast<const uint32_t*>(&bv);
            }
            arow[c ^ (r & 7)] = make_uint4(out[0], out[1], out[2], out[3]);
          }
        } else if (FMT == PMOE_MXFP4) {
          // 64 codes = two blocks of 32, each with its own E8M0 byte
          const uint32_t xw = cached ? my_sc[(kb * kBK) >> 7] : __ldg(srow + ((kb * kBK) >> 7));
          const int xb = ((kb * kBK) >> 5) & 3;  // first of the stage's two scale bytes in the word
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            const int c = 4 * hf + ci;
            const uint32_t word = qw[ci];  // 8 codes, low nibble first
            const uint32_t xbyte = (xw >> (8 * (xb + (c >> 2)))) & 0xffu;
            const float sv = xbyte ? __uint_as_float(xbyte << 23) : __uint_as_float(0x00400000u);
            uint32_t out[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const __half2_raw pr =
                  __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * h)) & 0xffu), __NV_E2M1);
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pr));
              const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sv, f.y * sv);
              out[h] = *reinterpret_cast<const uint32_t*>(&bv);
            }
            arow[c ^ (r & 7)] = make_uint4(out[0], out[1], out[2], out[3]);
          }
        } else {
          const uint32_t szw = cached ? my_sc[(kb * kBK) >> 7] : __ldg(srow + ((kb * kBK) >> 7));
          const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&szw));
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            const int c = 4 * hf + ci;
            const uint32_t word = qw[ci];  // 8 nibbles, low first
            uint32_t out[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float w0 = ((float)((word >> (8 * h)) & 0xFu) - sz.y) * sz.x;
              const float w1 = ((float)((word >> (8 * h + 4)) & 0xFu) - sz.y) * sz.x;
              const __nv_bfloat162 bv = __floats2bfloat162_rn(w0, w1);
              out[h] = *reinterpret_cast<const uint32_t*>(&bv);
            }
            arow[c ^ (r & 7)] = make_uint4(out[0], out[1], out[2], out[3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&afull[s]);
        mbar_arrive(&qempty[q]);
        if (++q == C::kQStages) {
          q = 0;
          qph ^= 1u;
        }
        if (++s == C::kAStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const int tile = t0 + item / m_tiles, mt = item % m_tiles;
      const int pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
      const int n_mma = (np + 15) & ~15;
      const int ab = it & 1, use = it >> 1;
      // NVFP4: the matrix's fp32 tensor scale, applied to the fp32 accumulators
      const float tsc = FMT == PMOE_NVFP4 ? __ldg(reinterpret_cast<const float*>(
                                                arena + (size_t)ws.tiles[3 * tile + 0] * stride +
                                                (GATEUP ? lay.gu_s : lay.d_s)))
                                          : 1.f;
      const bool got = mbar_wait(&acc_full[ab], (uint32_t)(use & 1), abort_flag, err);
      if (epi_bar_or(got ? 0 : 1)) break;
      fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kAccCols);
      for (int c = 0; c < n_mma; c += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + c, v);
        tmem_wait_ld();
        if (GATEUP) {
          // stage gate (rows 0-63) and up (rows 64-127) values, then each thread forms
          // 8 consecutive h values of one pair: one 16-byte store, 128 B per pair row
#pragma unroll
          for (int i = 0; i < 16; ++i) staging[row * 17 + i] = __uint_as_float(v[i]) * tsc;
          epi_bar();
          const int pl = et >> 3, js = (et & 7) * 8;
          if (c + pl < np) {
            uint32_t packed[4];
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2) {
              const float g0 = staging[(js + jj) * 17 + pl], u0 = staging[(64 + js + jj) * 17 + pl];
              const float g1 = staging[(js + jj + 1) * 17 + pl], u1 = staging[(64 + js + jj + 1) * 17 + pl];
              const __nv_bfloat162 hv = __floats2bfloat162_rn(g0 / (1.f + expf(-g0)) * u0, g1 / (1.f + expf(-g1)) * u1);
              packed[jj >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(ws.h + (size_t)(pstart + c + pl) * I + mt * 64 + js) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
          epi_bar();
        } else if (!kQuant) {
          float f[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
          stage_o_chunk(reinterpret_cast<uint32_t*>(staging), row, f);
          epi_bar();
          store_o_rows(reinterpret_cast<const uint32_t*>(staging), et, c, np, pstart, mt, H, ws.o_part);
          epi_bar();
        } else {
          // the converter warps bound this kernel on issue slots: fp32 rows straight from
          // the registers cost the epilogue the fewest instructions
          const int n = mt * 128 + row;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < np) ws.o_part[(size_t)(pstart + c + i) * H + n] = __uint_as_float(v[i]) * tsc;
        }
      }
      fence_before();
      mbar_arrive(&acc_empty[ab]);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- block-FP8 on kind::f8f6f4
//
// The e4m3 weight tiles go from TMA straight to the tensor cores. The activations come as
// two e4m3 planes on power-of-two scales (fp8_planes.cuh), and a K step multiplies both:
// gate/up stacks them as one operand of 2N rows (one MMA; the hi and lo columns of the
// partial are added in the promotion), down issues two MMAs (hi, then lo) into one
// partial. Either way it costs what one bf16 MMA costs. The weights' 128x128 block
// scale changes every 128 K and the h scales every 64 K, so the MMAs accumulate one K unit
// (gate/up: a 128-K stage; down: half a stage) per TMEM partial buffer, and promotion
// warps fold each partial into fp32 registers:
//   gate/up  acc += partial * s_w[row block][k block]; the epilogue multiplies by the row's
//            x scale sx[pair], forms h = silu(gate) * up and writes h as two planes with
//            one scale per (pair, 64 columns), hsc[m-tile][pair]
//   down     acc += partial * s_w[row block][k block] * hsc[k unit][pair]; the epilogue
//            writes o_part[pair][n] rounded to bf16, as the kernel above does
// Tiles as in tc_grouped_kernel (swap-AB: 128 weight rows on M, the tile's pairs on N),
// at most kTcSmallN = 64 pairs. Two promotion groups of four warps take the items in turn,
// each with its own ring of partial buffers, so one group's epilogue overlaps the other's
// MMAs. The weight tiles (the HBM stream) and the activation planes (re-read by every
// m-tile, from L2) have rings and producers of their own, the weights' the deeper one; a
// stage is one TMA box in each (gate/up's weights as a 4-D box of gate and up rows; both
// planes as one box of 32 or 64 rows each, the lo rows after the hi rows).
// Warps: 0 TMA weights, 1 MMA issuer (owns the TMEM), 2-5 and 6-9 promotion groups 0 and 1
// (TMEM lanes 32*(warp%4)..), 10 TMA activation planes.
struct F8Cfg {
  // TMEM partial buffers per group: gate/up stacks the hi and lo planes as one 2N-row
  // operand (one MMA per K step, 2 x 128 columns); down keeps them apart (two MMAs per
  // K step into 4 x 64 columns: it has two K units per stage)
  static constexpr int parts(bool gateup) { return gateup ? 2 : 4; }
  static constexpr int part_cols(bool gateup) { return gateup ? 128 : 64; }
  static constexpr int kN = 64;                   // pairs per tile (MMA N at most)
  static constexpr int kBK = 128;                 // K per stage (one byte each)
  static constexpr int kWBytes = 128 * kBK;       // weight tile, 128 rows
  static constexpr int kPlaneBytes = kN * kBK;    // one activation plane
  static constexpr int kXBytes = 2 * kPlaneBytes;
  static constexpr int kStagingFloats = 128 * 17;  // per group
  static constexpr int kHscUnits = 16;            // down: h scales staged per window of 16 K units
  static constexpr int kHscFloats = kHscUnits * kN;
  static constexpr int kFixedBytes = 2 * (kStagingFloats + kHscFloats + kN) * 4 + 1024 + 1024;
  static constexpr int kRingStages = (220 * 1024 - kFixedBytes) / kWBytes;  // 16 KB each
  static constexpr int kXStages = 4;
  static constexpr int kWStages = kRingStages - kXStages;
  static constexpr int kTmemCols = 512;           // 2 groups x (4 x 64 or 2 x 128 columns)
  static constexpr int kSmemBytes = (kWStages + kXStages) * kWBytes + kFixedBytes;
  static constexpr int kGroupThreads = 128;
  static constexpr int kThreads = 352;
  static_assert(kWBytes == kXBytes && kWStages >= 6 && kSmemBytes <= 227 * 1024, "fp8 tiles");
};

// Named barriers of the two promotion groups (ids 1 and 2, 128 threads each).
__device__ __forceinline__ void grp_bar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }

__device__ __forceinline__ int grp_bar_or(int g, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %2, 0;\n\t"
      "bar.red.or.pred q, %1, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(1 + g), "r"(pred)
      : "memory");
  return r;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

template <bool GATEUP>
__global__ void __launch_bounds__(F8Cfg::kThreads, 1)
    tc_fp8_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b,
                  const __grid_constant__ CUtensorMap map_bb,
                  const int32_t* __restrict__ plan, int E, int wave, int sub, Workspace ws, int I, int H,
                  const uint8_t* __restrict__ arena, size_t stride, ExpertLayout lay, int32_t* __restrict__ err) {
  using C = F8Cfg;
  constexpr int kN = C::kN;
  constexpr int kUnits = GATEUP ? 1 : 2;  // partial buffers per stage
  constexpr int kSteps = 4 / kUnits;      // K = 32 MMA steps per unit
  constexpr int kParts = C::parts(GATEUP), kPartCols = C::part_cols(GATEUP);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = wring + C::kWStages * C::kWBytes;
  float* staging0 = reinterpret_cast<float*>(xring + C::kXStages * C::kXBytes);  // [2][128 * 17]
  float* hsc0 = staging0 + 2 * C::kStagingFloats;                                // [2][kHscUnits * kN]
  float* sx0 = hsc0 + 2 * C::kHscFloats;                                         // [2][kN]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(sx0 + 2 * kN);
  uint64_t* wempty = wfull + C::kWStages;
  uint64_t* xfull = wempty + C::kWStages;
  uint64_t* xempty = xfull + C::kXStages;
  uint64_t* pfull = xempty + C::kXStages;     // [2][kParts] partial buffer written by the MMAs
  uint64_t* pempty = pfull + 2 * kParts;  // [2][kParts] partial buffer read by its group
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(pempty + 2 * kParts);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (wave >= plan[kPlanWaves]) return;
  int t0 = ws.tile_wave[wave], t1 = ws.tile_wave[wave + 1];
  if (sub == 1) t1 = ws.tile_split[wave];
  else if (sub == 2) t0 = ws.tile_split[wave];
  const int m_tiles = GATEUP ? (I / 64) : (H / 128);
  const int n_items = (t1 - t0) * m_tiles;
  if ((int)blockIdx.x >= n_items) return;
  const int kdim = GATEUP ? H : I;
  const int n_kb = kdim / C::kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < C::kXStages; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int r = 0; r < 2 * kParts; ++r) {
      mbar_init(&pfull[r], 1);
      mbar_init(&pempty[r], C::kGroupThreads);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w);
    prefetch_map(&map_b);
    prefetch_map(&map_bb);
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
  // rows of each activation plane a tile's stage holds: 32 or 64 (one box of both planes)
  auto plane_rows = [](int np) { return np <= 32 ? 32 : 64; };

  if (warp == 0 || warp == 10) {
    if (lane == 0) {
      // ---------------- TMA producers: weight tiles (warp 0) and activation planes (warp 10)
      const bool wts = warp == 0;
      const int depth = wts ? C::kWStages : C::kXStages;
      uint64_t* fullb = wts ? wfull : xfull;
      uint64_t* emptyb = wts ? wempty : xempty;
      uint8_t* ring = wts ? wring : xring;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int tile = t0 + item / m_tiles, mt = item % m_tiles;
        const int slot = ws.tiles[3 * tile + 0], pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
        const int nst = plane_rows(np);
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&emptyb[s], ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + s * C::kWBytes;
          if (wts) {
            mbar_arrive_expect_tx(&fullb[s], (uint32_t)C::kWBytes);
            if (GATEUP)
              tma_load_4d(st, &map_w, &fullb[s], kb * C::kBK, mt * 64, 0, slot);  // 64 gate rows, then the 64 up rows
            else
              tma_load_3d(st, &map_w, &fullb[s], kb * C::kBK, mt * 128, slot);
          } else {
            // one box: nst hi rows, then nst lo rows (rows past the tile feed MMA columns no
            // one reads)
            mbar_arrive_expect_tx(&fullb[s], (uint32_t)(2 * nst * C::kBK));
            tma_load_3d(st, nst == 32 ? &map_b : &map_bb, &fullb[s], kb * C::kBK, pstart, 0);
          }
          if (++s == depth) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain: every stage's last load consumed and its MMAs committed (bounded)
      for (int i = 0; i < depth; ++i) {
        mbar_wait(&emptyb[s], ph ^ 1u, abort_flag, err);
        if (++s == depth) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: per unit, hi and lo planes into one partial buffer of
      // the item's group
      int sw = 0, sx = 0;
      uint32_t wph = 0, xph = 0;
      int r0 = 0, r1 = 0;  // next partial buffer of each group's ring, and its phase
      uint32_t rph0 = 0u, rph1 = 0u;
      bool ok = true;
      int it = 0;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
        const int g = it & 1;
        const int tile = t0 + item / m_tiles;
        const int np = ws.tiles[3 * tile + 2];
        const int n_mma = (np + 15) & ~15;
        const int nst = plane_rows(np);
        const uint32_t idesc = idesc_e4m3(128, GATEUP ? 2 * nst : (n_mma < 16 ? 16 : n_mma));
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&wfull[sw], wph, abort_flag, err) || !mbar_wait(&xfull[sx], xph, abort_flag, err)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t a0 = smem_u32(wring + sw * C::kWBytes);
          const uint32_t bh = smem_u32(xring + sx * C::kXBytes), bl = bh + (uint32_t)(nst * C::kBK);
          for (int u = 0; u < kUnits; ++u) {
            int rr = g ? r1 : r0;
            uint32_t rp = g ? rph1 : rph0;
            const int pb = g * kParts + rr;
            if (!mbar_wait(&pempty[pb], rp ^ 1u, abort_flag, err)) {
              ok = false;
              break;
            }
            fence_after();
            const uint32_t d = tmem + (uint32_t)(pb * kPartCols);
#pragma unroll
            for (int j = 0; j < kSteps; ++j) {
              const uint32_t ko = (uint32_t)((u * kSteps + j) * 32);
              mma_e4m3(d, sw128_desc(a0 + ko), sw128_desc(bh + ko), idesc, j > 0 ? 1u : 0u);
              if (!GATEUP) mma_e4m3(d, sw128_desc(a0 + ko), sw128_desc(bl + ko), idesc, 1u);
            }
            mma_commit(&pfull[pb]);
            if (++rr == kParts) {
              rr = 0;
              rp ^= 1u;
            }
            if (g) {
              r1 = rr;
              rph1 = rp;
            } else {
              r0 = rr;
              rph0 = rp;
            }
          }
          if (!ok) break;
          mma_commit(&wempty[sw]);
          mma_commit(&xempty[sx]);
          if (++sw == C::kWStages) {
            sw = 0;
            wph ^= 1u;
          }
          if (++sx == C::kXStages) {
            sx = 0;
            xph ^= 1u;
          }
        }
      }
    }
  } else {
    // ---------------- promotion and epilogue: group g = warps 2-5 (g = 0) or 6-9 (g = 1)
    // takes the items it = g, g + 2, ... of this CTA
    const int g = (warp - 2) >> 2, qtr = warp & 3;
    const int row = qtr * 32 + lane;                  // TMEM lane = weight row of the tile
    const int et = (warp - 2 - 4 * g) * 32 + lane;    // 0..127 within the group
    float* staging = staging0 + g * C::kStagingFloats;
    float* hsc_sm = hsc0 + g * C::kHscFloats;
    float* sx_sm = sx0 + g * kN;
    const uint32_t tlane = (uint32_t)(qtr * 32) << 16;
    const int n_units = n_kb * kUnits;
    int r = 0;
    uint32_t rph = 0;
    bool bad = false;
    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      if ((it & 1) != g) continue;
      const int tile = t0 + item / m_tiles, mt = item % m_tiles;
      const int slot = ws.tiles[3 * tile + 0], pstart = ws.tiles[3 * tile + 1], np = ws.tiles[3 * tile + 2];
      const int n_mma = (np + 15) & ~15;
      if (GATEUP && et < kN) sx_sm[et] = et < np ? ws.sx[pstart + et] : 0.f;  // read after grp_bar_or below
      // this row's 128x128 weight-block scales: gate rows (lanes 0-63) and up rows (64-127)
      // of a gate/up tile lie in one block row each
      const int rb = GATEUP ? ((row < 64 ? mt * 64 : I + mt * 64) >> 7) : mt;
      const float* sw_row = reinterpret_cast<const float*>(arena + (size_t)slot * stride +
                                                           (GATEUP ? lay.gu_s : lay.d_s)) +
                            (size_t)rb * n_kb;
      float acc[kN];
#pragma unroll
      for (int i = 0; i < kN; ++i) acc[i] = 0.f;
      for (int kb = 0; kb < n_kb; ++kb) {
        const float sw = __ldg(sw_row + kb);
        for (int u = 0; u < kUnits; ++u) {
          const int ku = kb * kUnits + u;
          if (!GATEUP && ku % C::kHscUnits == 0) {
            // stage the h scales of the next window of K units for this tile's pairs
            const int w = n_units - ku < C::kHscUnits ? n_units - ku : C::kHscUnits;
            grp_bar(g);
            for (int i = et; i < w * kN; i += C::kGroupThreads) {
              const int uu = i / kN, c = i % kN;
              hsc_sm[i] = c < np ? ws.hsc[(size_t)(ku + uu) * ws.p_cap + pstart + c] : 0.f;
            }
            grp_bar(g);
          }
          const int pb = g * kParts + r;
          // tcgen05.ld is warp-collective: the warp goes on only if all its lanes' waits did
          const bool got = __all_sync(0xffffffffu, !bad && mbar_wait(&pfull[pb], rph, abort_flag, err));
          if (!got) bad = true;
          fence_after();
          if (got) {
            // two halves of 32 columns (the second only if the MMAs wrote it)
            const float* hs = hsc_sm + (ku % C::kHscUnits) * kN;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              if (h2 == 0 || n_mma > 32) {
                uint32_t v[32];
                tmem_ld32(tmem + tlane + (uint32_t)(pb * kPartCols + 32 * h2), v);
                if (GATEUP) {
                  uint32_t u[32];  // the lo plane's columns, plane_rows(np) after the hi plane's
                  tmem_ld32(tmem + tlane + (uint32_t)(pb * kPartCols + plane_rows(np) + 32 * h2), u);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    acc[32 * h2 + i] = fmaf(__uint_as_float(v[i]) + __uint_as_float(u[i]), sw, acc[32 * h2 + i]);
                } else {
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    acc[32 * h2 + i] = fmaf(__uint_as_float(v[i]), sw * hs[32 * h2 + i], acc[32 * h2 + i]);
                }
              }
            }
          }
          fence_before();
          mbar_arrive(&pempty[pb]);
          if (++r == kParts) {
            r = 0;
            rph ^= 1u;
          }
        }
      }
      if (grp_bar_or(g, bad ? 1 : 0)) break;
      if (GATEUP) {
        // exchange 16 pairs at a time through shared memory (gate rows 0-63, up rows
        // 64-127); 8 threads per pair then form 8 consecutive h values each, take the
        // scale of the pair's 64 columns and write both planes
        uint8_t* hq = reinterpret_cast<uint8_t*>(ws.h);
        const int pl = et >> 3, js = (et & 7) * 8;
#pragma unroll
        for (int cc = 0; cc < kN; cc += 16) {
          if (cc < n_mma) {
#pragma unroll
            for (int i = 0; i < 16; ++i) staging[row * 17 + i] = acc[cc + i] * sx_sm[cc + i];
            grp_bar(g);
            float hv[8], amax = 0.f;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float gt = staging[(js + jj) * 17 + pl], up = staging[(64 + js + jj) * 17 + pl];
              hv[jj] = gt / (1.f + expf(-gt)) * up;
              amax = fmaxf(amax, fabsf(hv[jj]));
            }
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            float sc, inv;
            plane_scale(amax, &sc, &inv);
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) split_e4m3x2(hv[2 * q] * inv, hv[2 * q + 1] * inv, &hi[q], &lo[q]);
            if (cc + pl < np) {
              const size_t prow = (size_t)pstart + cc + pl;
              *reinterpret_cast<uint2*>(hq + prow * I + mt * 64 + js) =
                  make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
              *reinterpret_cast<uint2*>(hq + (ws.p_cap + prow) * I + mt * 64 + js) =
                  make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
              if ((et & 7) == 0) ws.hsc[(size_t)mt * ws.p_cap + prow] = sc;
            }
            grp_bar(g);
          }
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < kN; cc += 16) {
          if (cc < np) {
            stage_o_chunk(reinterpret_cast<uint32_t*>(staging), row, acc + cc);
            grp_bar(g);
            store_o_rows(reinterpret_cast<const uint32_t*>(staging), et, cc, np, pstart, mt, H, ws.o_part);
            grp_bar(g);
          }
        }
      }
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

// bf16 elements with the 128-byte swizzle (MMA operands), bytes with the 128-byte
// swizzle (e4m3 MMA operands), or raw quantised bytes with the 64- or 32-byte swizzle (the
// converters' input: a tile row is 64 bytes of e4m3 or 32 of 4-bit codes, and the swizzle
// spreads 32 consecutive rows' 16-byte chunks over all banks)
enum MapKind { kMapBf16Sw128, kMapBytesSw128, kMapBytesSw64, kMapBytesSw32 };

int encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
           const cuuint32_t* box, MapKind kind = kMapBf16Sw128) {
  EncodeTiledFn fn = get_encode();
  if (fn == nullptr) return PMOE_ECUDA;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};  // element strides, one per dimension (rank <= 5)
  const CUresult r = fn(m, kind == kMapBf16Sw128 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        rank, base, dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        kind == kMapBytesSw64   ? CU_TENSOR_MAP_SWIZZLE_64B
                        : kind == kMapBytesSw32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PMOE_OK : PMOE_ECUDA;
}

template <bool GATEUP>
cudaError_t launch_f8_n(const CUtensorMap& mw, const CUtensorMap& mb, const CUtensorMap& mbb, const int32_t* plan, int E,
                        int wave, int sub,
                        const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                        int32_t* err, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(tc_fp8_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               F8Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc_fp8_kernel<GATEUP><<<num_sms, F8Cfg::kThreads, F8Cfg::kSmemBytes, s>>>(
      mw, mb, mbb, plan, E, wave, sub, ws, I, H, arena, stride, expert_layout(PMOE_FP8_BLOCK128, H, I), err);
  return cudaGetLastError();
}

// block-FP8 with the small pair cap (tc_fp8_planes)
template <bool GATEUP>
cudaError_t launch_f8(const CUtensorMap& mw, const CUtensorMap& mb, const CUtensorMap& mbb, const int32_t* plan, int E,
                      int wave, int sub,
                      const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                      int32_t* err, int tile_n, cudaStream_t s) {
  if (tile_n > F8Cfg::kN) return cudaErrorInvalidValue;
  return launch_f8_n<GATEUP>(mw, mb, mbb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, s);
}

template <bool GATEUP, int FMT, int NMAX>
cudaError_t launch_tc_n(const CUtensorMap& mw, const CUtensorMap& mb, const CUtensorMap& mbb, const int32_t* plan, int E,
                        int wave, int sub,
                        const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                        int32_t* err, cudaStream_t s) {
  using C = TcCfg<FMT, NMAX>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(tc_grouped_kernel<GATEUP, FMT, NMAX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc_grouped_kernel<GATEUP, FMT, NMAX><<<num_sms, C::kThreads, C::kSmemBytes, s>>>(
      mw, mb, mbb, plan, E, wave, sub, ws, I, H, arena, stride, expert_layout(FMT, H, I), err);
  return cudaGetLastError();
}

// tile_n: the pair cap the grouping used for this forward's tiles (kTcSmallN or kTcMaxN)
template <bool GATEUP, int FMT>
cudaError_t launch_tc(const CUtensorMap& mw, const CUtensorMap& mb, const CUtensorMap& mbb, const int32_t* plan, int E,
                      int wave, int sub,
                      const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                      int32_t* err, int tile_n, cudaStream_t s) {
  if (tile_n <= kTcSmallN)
    return launch_tc_n<GATEUP, FMT, kTcSmallN>(mw, mb, mbb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err,
                                               s);
  return launch_tc_n<GATEUP, FMT, kTcMaxN>(mw, mb, mbb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, s);
}

}  // namespace

bool tc_supported(int H, int I) {
  return H % 128 == 0 && I % 128 == 0 && H >= 128 && I >= 128 && get_encode() != nullptr;
}

int tc_make_weight_maps(uint8_t* arena, size_t stride, int K, int H, int I, int fmt, TcMaps* out) {
  if (stride % 16 != 0) return PMOE_EUNSUPPORTED;
  const ExpertLayout lay = expert_layout(fmt, H, I);
  if (fmt == PMOE_BF16) {
    {
      const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)(2 * I), (cuuint64_t)K};
      const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)stride};
      const cuuint32_t box[3] = {(cuuint32_t)kBK, 64, 1};  // 64 gate or 64 up rows
      if (encode(&out->gu, arena, 3, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
    }
    {
      const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)K};
      const cuuint64_t strides[3] = {(cuuint64_t)H * 2, (cuuint64_t)I * H * 2, (cuuint64_t)stride};
      const cuuint32_t box[4] = {(cuuint32_t)kBK, 64, 2, 1};  // 64 gate rows and the matching 64 up rows
      if (encode(&out->gu4, arena, 4, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
    }
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)K};
    const cuuint64_t strides[2] = {(cuuint64_t)I * 2, (cuuint64_t)stride};
    const cuuint32_t box[3] = {(cuuint32_t)kBK, 128, 1};
    return encode(&out->d, arena + lay.d_w, 3, dims, strides, box) == PMOE_OK ? PMOE_OK : PMOE_ECUDA;
  }
  if (fmt != PMOE_FP8_BLOCK128 && fmt != PMOE_INT4_GPTQ_G128 && fmt != PMOE_MXFP4 && fmt != PMOE_NVFP4)
    return PMOE_EUNSUPPORTED;
  if (fmt == PMOE_FP8_BLOCK128) {
    // e4m3 rows as MMA operands: 128-byte boxes (128 K), 128-byte swizzle
    {
      // {H, I, 2 (gate, up), K}: one box holds a tile's 64 gate rows and the matching 64 up rows
      const cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)K};
      const cuuint64_t strides[3] = {(cuuint64_t)H, (cuuint64_t)I * H, (cuuint64_t)stride};
      const cuuint32_t box[4] = {128, 64, 2, 1};
      if (encode(&out->gu8, arena + lay.gu_w, 4, dims, strides, box, kMapBytesSw128) != PMOE_OK) return PMOE_ECUDA;
    }
    const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)K};
    const cuuint64_t strides[2] = {(cuuint64_t)I, (cuuint64_t)stride};
    const cuuint32_t box[3] = {128, 128, 1};
    if (encode(&out->d8, arena + lay.d_w, 3, dims, strides, box, kMapBytesSw128) != PMOE_OK) return PMOE_ECUDA;
  }
  // quantised weights are loaded as bytes (one e4m3, or two int4 / E2M1 codes, per byte), rows of
  // 64 or 32 bytes with the swizzle of that width (NVFP4's codes are laid out as MXFP4's)
  const MapKind qkind = fmt == PMOE_FP8_BLOCK128 ? kMapBytesSw64 : kMapBytesSw32;
  const cuuint64_t hb = fmt == PMOE_FP8_BLOCK128 ? (cuuint64_t)H : (cuuint64_t)H / 2;
  const cuuint64_t ib = fmt == PMOE_FP8_BLOCK128 ? (cuuint64_t)I : (cuuint64_t)I / 2;
  const cuuint32_t kbb = fmt == PMOE_FP8_BLOCK128 ? (cuuint32_t)kBK : (cuuint32_t)kBK / 2;
  {
    const cuuint64_t dims[3] = {hb, (cuuint64_t)(2 * I), (cuuint64_t)K};
    const cuuint64_t strides[2] = {hb, (cuuint64_t)stride};
    const cuuint32_t box[3] = {kbb, 64, 1};
    if (encode(&out->gu, arena + lay.gu_w, 3, dims, strides, box, qkind) != PMOE_OK) return PMOE_ECUDA;
  }
  const cuuint64_t dims[3] = {ib, (cuuint64_t)H, (cuuint64_t)K};
  const cuuint64_t strides[2] = {ib, (cuuint64_t)stride};
  const cuuint32_t box[3] = {kbb, 128, 1};
  return encode(&out->d, arena + lay.d_w, 3, dims, strides, box, qkind) == PMOE_OK ? PMOE_OK : PMOE_ECUDA;
}

int tc_make_act_maps(int fmt, __nv_bfloat16* x_perm, __nv_bfloat16* h, size_t P, int H, int I, TcMaps* out) {
  if (fmt == PMOE_FP8_BLOCK128) {
    // the two e4m3 planes of x and of h, [2][P][cols] bytes in the bf16 buffers' place; a box
    // spans both planes (32 or 64 rows of each)
    for (int big = 0; big < 2; ++big) {
      const cuuint32_t rows = big ? 64 : 32;
      {
        const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)P, 2};
        const cuuint64_t strides[2] = {(cuuint64_t)H, (cuuint64_t)H * P};
        const cuuint32_t box[3] = {128, rows, 2};
        if (encode(big ? &out->x8b : &out->x8, x_perm, 3, dims, strides, box, kMapBytesSw128) != PMOE_OK)
          return PMOE_ECUDA;
      }
      const cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)P, 2};
      const cuuint64_t strides[2] = {(cuuint64_t)I, (cuuint64_t)I * P};
      const cuuint32_t box[3] = {128, rows, 2};
      if (encode(big ? &out->h8b : &out->h8, h, 3, dims, strides, box, kMapBytesSw128) != PMOE_OK) return PMOE_ECUDA;
    }
  }
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
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)P};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBigRowsB};
    if (encode(&out->xb, x_perm, 2, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)P};
    const cuuint64_t strides[1] = {(cuuint64_t)I * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBigRowsB};
    if (encode(&out->hb, h, 2, dims, strides, box) != PMOE_OK) return PMOE_ECUDA;
  }
  return PMOE_OK;
}

cudaError_t tc_gateup(int fmt, const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, int sub,
                      const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                      int32_t* err, int tile_n, cudaStream_t s) {
  if (tc_fp8_planes(fmt, tile_n))
    return launch_f8<true>(wm.gu8, am.x8, am.x8b, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_FP8_BLOCK128)
    return launch_tc<true, PMOE_FP8_BLOCK128>(wm.gu, am.x, am.xb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_INT4_GPTQ_G128)
    return launch_tc<true, PMOE_INT4_GPTQ_G128>(wm.gu, am.x, am.xb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n,
                                                s);
  if (fmt == PMOE_NVFP4)
    return launch_tc<true, PMOE_NVFP4>(wm.gu, am.x, am.xb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_MXFP4)
    return launch_tc<true, PMOE_MXFP4>(wm.gu, am.x, am.xb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  return launch_tc<true, PMOE_BF16>(wm.gu4, am.x, am.xb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
}

cudaError_t tc_down(int fmt, const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, int sub,
                    const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms, int32_t* err,
                    int tile_n, cudaStream_t s) {
  if (tc_fp8_planes(fmt, tile_n))
    return launch_f8<false>(wm.d8, am.h8, am.h8b, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_FP8_BLOCK128)
    return launch_tc<false, PMOE_FP8_BLOCK128>(wm.d, am.h, am.hb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_INT4_GPTQ_G128)
    return launch_tc<false, PMOE_INT4_GPTQ_G128>(wm.d, am.h, am.hb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n,
                                                 s);
  if (fmt == PMOE_NVFP4)
    return launch_tc<false, PMOE_NVFP4>(wm.d, am.h, am.hb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  if (fmt == PMOE_MXFP4)
    return launch_tc<false, PMOE_MXFP4>(wm.d, am.h, am.hb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
  return launch_tc<false, PMOE_BF16>(wm.d, am.h, am.hb, plan, E, wave, sub, ws, I, H, arena, stride, num_sms, err, tile_n, s);
}

}  // namespace pmoe
