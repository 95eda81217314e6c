// Activations for the FP8 tensor path: a value v is carried as two e4m3 codes on one
// power-of-two scale s, v ~= s * (hi + lo), hi = e4m3(v / s), lo = e4m3(v / s - hi).
// Two planes keep ~8 significant bits (about bf16's), one plane only 4; both planes go
// through the same weight tile, so the pair costs two FP8 MMAs, the price of one bf16 MMA.
//
// The scale is 2^(E - 8) for the block's largest magnitude amax = m * 2^E, m in [0.5, 1):
// every |v / s| < 256 stays below e4m3's 448, and dividing by a power of two is exact.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace pmoe {

// s and 1/s for a block whose largest magnitude is amax (s = 1 for an all-zero or
// vanishing block, whose codes then round to zero).
__device__ __forceinline__ void plane_scale(float amax, float* s, float* inv) {
  const int be = (int)((__float_as_uint(amax) >> 23) & 0xffu);  // biased exponent: amax in [2^(be-127), 2^(be-126))
  if (be < 8 || be > 254) {
    *s = 1.f;
    *inv = 1.f;
    return;
  }
  *s = __uint_as_float((uint32_t)(be - 7) << 23);     // 2^(be - 134)
  *inv = __uint_as_float((uint32_t)(261 - be) << 23);  // 2^(134 - be)
}

// Two values already divided by the scale -> (hi codes, lo codes), first value in the low byte.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint16_t* hi, uint16_t* lo) {
  const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(make_float2(a - hf.x, b - hf.y), __NV_SATFINITE, __NV_E4M3);
  *hi = (uint16_t)h;
  *lo = (uint16_t)l;
}

}  // namespace pmoe
