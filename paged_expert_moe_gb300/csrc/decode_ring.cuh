// Shared pieces of the decode kernels that stream expert weights through a shared-memory
// byte ring (the fused single-layer decode kernel and the persistent multi-layer one):
// the block's warp roles and limits, mbarrier and bulk-copy wrappers, the page-in copy
// loops, the per-CTA chunk schedule, ring placement and the scale rows that travel with a
// quantised chunk. Every wait is bounded: after kDfWaitLimit cycles it raises the abort
// flag and the error bit kErrDecodeTimeout.
#pragma once

#include "decode_common.cuh"

namespace pmoe {
namespace {

using namespace dec;

// 16 warps, four per SM sub-partition (whose register file then allows 128 per thread)
constexpr int kDfConsumerWarps = 11;  // warps 0-10 consume, 11 produces, 12 fetches h, 13-15 page in
constexpr int kDfPagerWarps = 3;
constexpr int kDfThreads = (kDfConsumerWarps + 2 + kDfPagerWarps) * 32;
constexpr int kDfSlots = 16;                // chunks in flight at most (one mbarrier pair each)
constexpr int kDfMaxChunkBytes = 32 * 1024;  // weight bytes of one chunk
constexpr int kDfMaxPairs = kDecodeMaxPairs;
constexpr int kDfMaxRows = 32;              // down-projection output rows per CTA (ceil(H / grid))
constexpr int kDfMaxChunks = 256;           // chunks per CTA
static_assert(kDfMaxChunks <= 2 * kDfThreads, "the chunk-list scan covers two entries per thread");
constexpr int kDfLag = 3;                   // down of expert e follows gate/up of expert e + kDfLag
constexpr int kDfMaxTokens = kGemvMaxTokens;
constexpr size_t kDfSmemBudget = 223 * 1024;  // dynamic shared memory; the static arrays fit in the rest
constexpr long long kDfWaitLimit = 4000000000LL;
constexpr int32_t kErrDecodeTimeout = 32;
constexpr unsigned long long kTagMask = (1ull << 48) - 1;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
// non-blocking probe (try_wait may suspend the thread until the phase completes)
__device__ __forceinline__ bool mb_test(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t par, volatile int* abort_flag, int32_t* err) {
  if (mb_try(b, par)) return true;
  const long long t0 = clock64();
  while (!mb_try(b, par)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kDfWaitLimit) {
      *abort_flag = 1;
      atomicOr(err, kErrDecodeTimeout);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_relaxed_u64x2(const unsigned long long* p) {
  ulonglong2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
  return v;
}
// Gate and up partial dot products of one 16-byte chunk (8 bf16 weights of each row)
// against the same 8 bf16 activations. The two chains advance together in packed
// fp32 FMAs; each lane of the pair is an ordinary fused multiply-add, so the sums are
// bit-identical to two separate fmaf chains.
__device__ __forceinline__ float2 gu_dot_bf16(uint4 wg, uint4 wu, uint4 xa) {
  unsigned long long acc = 0ull;  // (+0.f, +0.f)
  const uint32_t g4[4] = {wg.x, wg.y, wg.z, wg.w}, u4[4] = {wu.x, wu.y, wu.z, wu.w}, x4[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    unsigned long long wlo, whi, xlo, xhi;
    asm("mov.b64 %0, {%1, %2};" : "=l"(wlo) : "r"(g4[i] << 16), "r"(u4[i] << 16));
    asm("mov.b64 %0, {%1, %2};" : "=l"(whi) : "r"(g4[i] & 0xffff0000u), "r"(u4[i] & 0xffff0000u));
    asm("mov.b64 %0, {%1, %1};" : "=l"(xlo) : "r"(x4[i] << 16));
    asm("mov.b64 %0, {%1, %1};" : "=l"(xhi) : "r"(x4[i] & 0xffff0000u));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(wlo), "l"(xlo));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(whi), "l"(xhi));
  }
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(acc));
  return r;
}

// Copy of two byte ranges (sizes multiples of 16) from src + off_i to dst + off_i by `nl`
// cooperating lanes (this thread is lane vl of them), as one sequence with 16 16-byte
// loads in flight per lane: the source is host memory across the link, so the bytes in
// flight set the rate, and a whole chunk goes in one round trip.
__device__ __forceinline__ void lanes_copy16x2(const uint8_t* src, uint8_t* dst, size_t off1, size_t bytes1,
                                               size_t off2, size_t bytes2, int vl, int nl) {
  constexpr int U = 10;
  const size_t n1 = bytes1 / 16, n = n1 + bytes2 / 16;
  for (size_t base = (size_t)vl; base < n; base += (size_t)nl * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + (size_t)u * nl;
      if (i < n) v[u] = ld_stream(src + (i < n1 ? off1 + i * 16 : off2 + (i - n1) * 16));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + (size_t)u * nl;
      if (i < n) *reinterpret_cast<uint4*>(dst + (i < n1 ? off1 + i * 16 : off2 + (i - n1) * 16)) = v[u];
    }
  }
}
// The same for small ranges whose sizes and offsets are multiples of 4 (scale rows): 8
// loads in flight per lane (over the host link a load costs a round trip; one at a time,
// a few hundred bytes of scale rows took several round trips per chunk).
// (not inlined: its registers would otherwise count against the whole decode kernel)
__device__ __noinline__ void lanes_copy4x2(const uint8_t* src, uint8_t* dst, size_t off1, size_t bytes1,
                                           size_t off2, size_t bytes2, int vl, int nl) {
  constexpr int U = 8;
  const size_t n1 = bytes1 / 4, n = n1 + bytes2 / 4;
  for (size_t base = (size_t)vl; base < n; base += (size_t)nl * U) {
    uint32_t v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + (size_t)u * nl;
      if (i < n) v[u] = *reinterpret_cast<const uint32_t*>(src + (i < n1 ? off1 + i * 4 : off2 + (i - n1) * 4));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + (size_t)u * nl;
      if (i < n) *reinterpret_cast<uint32_t*>(dst + (i < n1 ? off1 + i * 4 : off2 + (i - n1) * 4)) = v[u];
    }
  }
}
// One load in flight per lane (inlined; the persistent stack kernel keeps this form for
// the formats whose scale rows are short).
__device__ __forceinline__ void lanes_copy4(const uint8_t* src, uint8_t* dst, size_t off, size_t bytes, int vl,
                                            int nl) {
  for (size_t i = (size_t)vl * 4; i < bytes; i += (size_t)nl * 4)
    *reinterpret_cast<uint32_t*>(dst + off + i) = *reinterpret_cast<const uint32_t*>(src + off + i);
}
__device__ __forceinline__ void pagers_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kDfPagerWarps * 32) : "memory");
}
// Barrier among the pager warps that ORs a predicate over them.
__device__ __forceinline__ int pagers_any(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred), "n"(kDfPagerWarps * 32)
      : "memory");
  return r;
}

// Reads n16 * 8 tagged h words starting at src (waiting until each carries `tag`) and
// packs their bf16 values into n16 16-byte vectors. Used only for an expert that one
// token routes to more than once.
__device__ bool fetch_h_direct(const unsigned long long* src, unsigned long long tag, uint4* out, int n16,
                               volatile int* abort_flag, int32_t* err) {
  for (int q = 0; q < n16; ++q) {
    uint32_t w[4];
    for (int h = 0; h < 4; ++h) {
      const long long t0 = clock64();
      ulonglong2 v = ld_relaxed_u64x2(src + q * 8 + h * 2);
      while ((v.x >> 16) != tag || (v.y >> 16) != tag) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kDfWaitLimit) {
          *abort_flag = 1;
          atomicOr(err, kErrDecodeTimeout);
          return false;
        }
        __nanosleep(64);
        v = ld_relaxed_u64x2(src + q * 8 + h * 2);
      }
      w[h] = (uint32_t)(v.x & 0xffffu) | ((uint32_t)(v.y & 0xffffu) << 16);
    }
    out[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return true;
}
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(su32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDfConsumerWarps * 32) : "memory");
}
// A CTA's schedule. With D experts in the wave and lag L = min(kDfLag, D):
//   GU(0) .. GU(L-1), then for e = L .. D-1: GU(e) D(e-L), then D(D-L) .. D(D-1),
// where GU(e) is the CTA's gate/up part of expert e in cg chunks and D(e) its down
// rows of expert e in cd chunks. Entry q is (kind, expert index, first row, rows),
// computed from q alone so that the whole list is built in parallel.
struct DfSched {
  int D, G, b, I, H, cg, cd;
};

__device__ __forceinline__ int4 sched_entry(int q, const DfSched& s) {
  const int L = min(kDfLag, s.D), per = s.cg + s.cd;
  int kind, e, sub;
  if (q < L * s.cg) {
    kind = 1;
    e = q / s.cg;
    sub = q - e * s.cg;
  } else {
    const int q1 = q - L * s.cg;
    if (q1 < (s.D - L) * per) {
      const int st = q1 / per, r = q1 - st * per;
      if (r < s.cg) {
        kind = 1;
        e = L + st;
        sub = r;
      } else {
        kind = 2;
        e = st;
        sub = r - s.cg;
      }
    } else {
      const int q2 = q1 - (s.D - L) * per;
      kind = 2;
      e = s.D - L + q2 / s.cd;
      sub = q2 - (q2 / s.cd) * s.cd;
    }
  }
  // (32-bit arithmetic: I, H < 2^20 and G <= 1024 are checked on the host)
  const unsigned G = (unsigned)s.G;
  if (kind == 1) {
    const unsigned part = ((unsigned)s.b + (unsigned)e) % G;
    const int j0 = (int)((unsigned)s.I * part / G);
    const int n = (int)((unsigned)s.I * (part + 1) / G) - j0;
    const int a0 = n * sub / s.cg, a1 = n * (sub + 1) / s.cg;
    return make_int4(1, e, j0 + a0, a1 - a0);
  }
  const int r0 = (int)((unsigned)s.H * (unsigned)s.b / G);
  const int n = (int)((unsigned)s.H * (unsigned)(s.b + 1) / G) - r0;
  const int a0 = n * sub / s.cd, a1 = n * (sub + 1) / s.cd;
  return make_int4(2, e, r0 + a0, a1 - a0);
}

// Ring placement: the live chunks occupy [lo, head) or, wrapped, [lo, R) + [0, head).
// Returns the offset for `need` bytes, or -1 if they do not fit until older chunks go.
__device__ __forceinline__ int ring_place(unsigned head, unsigned lo, bool empty, unsigned need, unsigned R) {
  if (empty) return (int)(head + need <= R ? head : 0u);
  if (lo < head) {
    if (head + need <= R) return (int)head;
    if (need <= lo) return 0;
    return -1;
  }
  return head + need <= lo ? (int)head : -1;
}

// Scales of a quantised chunk travel in the ring with its weight rows, so that the
// consumers read them from shared memory instead of waiting on global loads per row.
// A scale row covers one weight row (int4: the row's (s, z) per group of 128) or one
// block row of 128 weight rows (FP8: the fp32 scale per 128x128 block). For rows
// [r0, r0 + n) of a region whose scale rows are RS bytes apart, the copy spans the scale
// rows they need, widened to 16-byte boundaries (the host requires the scale regions to
// start and end on such boundaries); `first` is the byte offset of row r0's scale row in
// the copy.
struct ScaleSpan {
  uint32_t src, bytes, first;  // src: byte offset in the expert
};
// Bytes of one scale row of a matrix with n inputs per row: an fp32 per 128x128 block
// (FP8, per block row), an (s, z) fp16 pair per 128 (int4), an E8M0 byte per 32 (MXFP4),
// an e4m3 byte per 16 (NVFP4).
__host__ __device__ __forceinline__ int row_scale_bytes(int fmt, int n) {
  return fmt == PMOE_NVFP4 ? n / 16 : (n / 128) * 4;
}
template <int FMT>
__device__ __forceinline__ int scale_row(int r) {
  return FMT == PMOE_FP8_BLOCK128 ? (r >> 7) : r;
}
template <int FMT>
__device__ __forceinline__ ScaleSpan scale_span(size_t region, int RS, int r0, int n) {
  const uint32_t b0 = (uint32_t)(region + (size_t)scale_row<FMT>(r0) * RS);
  const uint32_t b1 = (uint32_t)(region + (size_t)(scale_row<FMT>(r0 + n - 1) + 1) * RS);
  const uint32_t a0 = b0 & ~15u, a1 = (b1 + 15u) & ~15u;
  return ScaleSpan{a0, a1 - a0, b0 - a0};
}
// t: NVFP4's tensor scale of the row's matrix (unused by the other formats)
template <int FMT>
__device__ __forceinline__ ChunkQ chunk_q_ring(const uint8_t* row_scales, int c, float t = 1.f) {
  ChunkQ q{1.f, 0.f};
  if constexpr (FMT == PMOE_NVFP4) {
    const uint32_t b = reinterpret_cast<const uint16_t*>(row_scales)[c];  // blocks 2c and 2c + 1
    q.s = e4m3_f32(b & 0xffu) * t;
    q.z = e4m3_f32(b >> 8) * t;
  } else if constexpr (FMT == PMOE_FP8_BLOCK128) {
    q.s = reinterpret_cast<const float*>(row_scales)[(c * 16) >> 7];
  } else if constexpr (FMT == PMOE_MXFP4) {
    q.s = e8m0_f32(row_scales[c]);  // one byte per block of 32 inputs: chunk c is block c
  } else if constexpr (FMT == PMOE_INT4_GPTQ_G128) {
    const uint32_t raw = reinterpret_cast<const uint32_t*>(row_scales)[(c * 32) >> 7];
    const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    q.s = sz.x;
    q.z = sz.y;
  }
  return q;
}

}  // namespace
}  // namespace pmoe
