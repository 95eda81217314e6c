// Device helpers shared by the decode kernels: streaming loads, bf16 unpacking, the
// per-format dequantisation of one 16-byte weight chunk (bf16 / block-FP8 e4m3 with
// fp32 128x128 scales / GPTQ int4 g128 with fp16 scale and zero / MXFP4: E2M1 codes with
// an E8M0 scale per 32 inputs), warp reductions.
#pragma once

#include "pmoe_internal.h"

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

namespace pmoe {
namespace dec {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load from shared memory (an explicit shared-window access)
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float dot_bf16x8(uint32_t w, uint32_t x, float acc) {
  acc = fmaf(bf_lo(w), bf_lo(x), acc);
  return fmaf(bf_hi(w), bf_hi(x), acc);
}

// Format traits: elements per 16-byte weight chunk, weight bytes per element (x2).
template <int FMT> struct Fmt;
template <> struct Fmt<PMOE_BF16> { static constexpr int EPC = 8; static constexpr int BPE2 = 4; };
template <> struct Fmt<PMOE_FP8_BLOCK128> { static constexpr int EPC = 16; static constexpr int BPE2 = 2; };
template <> struct Fmt<PMOE_INT4_GPTQ_G128> { static constexpr int EPC = 32; static constexpr int BPE2 = 1; };
template <> struct Fmt<PMOE_MXFP4> { static constexpr int EPC = 32; static constexpr int BPE2 = 1; };
template <> struct Fmt<PMOE_NVFP4> { static constexpr int EPC = 32; static constexpr int BPE2 = 1; };

// E8M0 scale byte -> 2^(b - 127) as fp32 (b = 0 is the subnormal 2^-127)
__device__ __forceinline__ float e8m0_f32(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Per-chunk dequantisation parameters of row `row` (of a [rows][cols] matrix), chunk `c`:
// the scale s and the zero point z (int4), or, for NVFP4, the scales of the chunk's two
// blocks of 16 (s, then z), each times the matrix's tensor scale.
struct ChunkQ {
  float s, z;
};

// e4m3 code -> fp32 (exact)
__device__ __forceinline__ float e4m3_f32(uint32_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

// COHERENT: the scales may have been written earlier in the same launch (an expert the
// launch pages in itself), so they are read through L2 rather than the read-only path.
template <int FMT, bool COHERENT = false>
__device__ __forceinline__ ChunkQ chunk_q(const uint8_t* scales, int row, int c, int cols) {
  ChunkQ q{1.f, 0.f};
  if constexpr (FMT == PMOE_FP8_BLOCK128) {
    const float* S = reinterpret_cast<const float*>(scales) + (size_t)(row >> 7) * (cols >> 7) + ((c * 16) >> 7);
    if constexpr (COHERENT) {
      asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(q.s) : "l"(S));
    } else {
      q.s = __ldg(S);
    }
  } else if constexpr (FMT == PMOE_MXFP4) {
    // one scale byte per row and block of 32 inputs: chunk c is exactly block c
    const uint8_t* X = scales + (size_t)row * (cols >> 5) + c;
    uint32_t b;
    if constexpr (COHERENT) {
      asm volatile("ld.global.cg.u8 %0, [%1];" : "=r"(b) : "l"(X));
    } else {
      b = __ldg(X);
    }
    q.s = e8m0_f32(b);
  } else if constexpr (FMT == PMOE_NVFP4) {
    // the matrix's scale section: fp32 tensor scale, 12 bytes of padding, then one e4m3
    // byte per row and block of 16 inputs (chunk c holds blocks 2c and 2c + 1)
    const uint16_t* B = reinterpret_cast<const uint16_t*>(scales + 16 + (size_t)row * (cols >> 4)) + c;
    uint32_t b;
    float t;
    if constexpr (COHERENT) {
      asm volatile("ld.global.cg.u16 %0, [%1];" : "=r"(b) : "l"(B));
      asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(t) : "l"(scales));
    } else {
      b = __ldg(B);
      t = __ldg(reinterpret_cast<const float*>(scales));
    }
    q.s = e4m3_f32(b & 0xffu) * t;
    q.z = e4m3_f32(b >> 8) * t;
  } else if constexpr (FMT == PMOE_INT4_GPTQ_G128) {
    const __half2* SZ = reinterpret_cast<const __half2*>(scales) + (size_t)row * (cols >> 7) + ((c * 32) >> 7);
    uint32_t raw;
    if constexpr (COHERENT) {
      asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(raw) : "l"(SZ));
    } else {
      raw = *reinterpret_cast<const uint32_t*>(SZ);
    }
    const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&raw));
    q.s = sz.x;
    q.z = sz.y;
  }
  return q;
}

// Where chunk_dot reads its activations from.
enum : int { kSrcGlobal = 0, kSrcShared = 1, kSrcRegs = 2 };

template <int FMT, int SRC>
__device__ __forceinline__ uint4 load_act(const uint4* p) {
  if constexpr (SRC == kSrcShared) return lds128(p);
  else if constexpr (SRC == kSrcGlobal) return __ldg(p);
  else return *p;
}

template <int FMT, int SRC>
__device__ __forceinline__ float chunk_dot(uint4 w, const uint4* av, ChunkQ q) {
  if constexpr (FMT == PMOE_BF16) {
    const uint4 a = load_act<FMT, SRC>(av);
    float acc = 0.f;
    acc = dot_bf16x8(w.x, a.x, acc);
    acc = dot_bf16x8(w.y, a.y, acc);
    acc = dot_bf16x8(w.z, a.z, acc);
    acc = dot_bf16x8(w.w, a.w, acc);
    return acc;
  } else if constexpr (FMT == PMOE_FP8_BLOCK128) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 a = load_act<FMT, SRC>(av + h);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t word = wv[2 * h + k];
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(word & 0xffffu), __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(word >> 16), __NV_E4M3);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        const uint32_t a0 = aw[2 * k], a1 = aw[2 * k + 1];
        acc = fmaf(f0.x, bf_lo(a0), acc);
        acc = fmaf(f0.y, bf_hi(a0), acc);
        acc = fmaf(f1.x, bf_lo(a1), acc);
        acc = fmaf(f1.y, bf_hi(a1), acc);
      }
    }
    return acc * q.s;
  } else if constexpr (FMT == PMOE_MXFP4) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 a = load_act<FMT, SRC>(av + h);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t word = wv[h];  // 8 codes = elements 8h .. 8h+7, low nibble first
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // one byte = two E2M1 codes -> two fp16 values (exact), low nibble first
        const __half2_raw pr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * k)) & 0xffu), __NV_E2M1);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pr));
        acc = fmaf(f.x, bf_lo(aw[k]), acc);
        acc = fmaf(f.y, bf_hi(aw[k]), acc);
      }
    }
    return acc * q.s;
  } else if constexpr (FMT == PMOE_NVFP4) {
    // E2M1 codes as MXFP4, two blocks of 16: words 0-1 (scale s) and 2-3 (scale z)
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float acc[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 a = load_act<FMT, SRC>(av + h);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t word = wv[h];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2_raw pr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((word >> (8 * k)) & 0xffu), __NV_E2M1);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pr));
        acc[h >> 1] = fmaf(f.x, bf_lo(aw[k]), acc[h >> 1]);
        acc[h >> 1] = fmaf(f.y, bf_hi(aw[k]), acc[h >> 1]);
      }
    }
    return acc[0] * q.s + acc[1] * q.z;
  } else {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 a = load_act<FMT, SRC>(av + h);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t word = wv[h];  // 8 nibbles = elements 8h .. 8h+7
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float q0 = (float)((word >> (8 * k)) & 0xFu) - q.z;
        const float q1 = (float)((word >> (8 * k + 4)) & 0xFu) - q.z;
        acc = fmaf(q0, bf_lo(aw[k]), acc);
        acc = fmaf(q1, bf_hi(aw[k]), acc);
      }
    }
    return acc * q.s;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

}  // namespace dec
}  // namespace pmoe
