// Tensor-core (tcgen05 / TMEM / TMA) grouped GEMMs of the prefill path.
#pragma once

#include <cuda.h>

#include "pmoe_internal.h"

namespace pmoe {

constexpr int kTcMaxN = 256;   // pairs per tile (MMA N)
constexpr int kTcSmallN = 64;  // the cap for forwards with few tokens per expert (deeper TMA pipeline)

struct TcMaps {
  CUtensorMap gu;  // gate/up rows of every slot: dims {H (bytes if quantised), 2I, K}
  CUtensorMap d;   // down rows of every slot: dims {I (bytes if quantised), H, K}
  CUtensorMap x;   // gathered activations x_perm: dims {H, P} bf16, 32-row boxes
  CUtensorMap h;   // intermediate h: dims {I, P} bf16, 32-row boxes
  // the same with 128-row boxes, for a tile's whole 128-pair chunks: each TMA instruction
  // costs time of its own, so fewer and larger boxes stream a stage faster
  CUtensorMap xb, hb;
  // block-FP8 on the e4m3 MMAs: weight rows in 128-byte swizzled boxes, and the two
  // e4m3 planes of x and h ({H or I, P, 2} bytes, in the bf16 buffers' place; one box holds
  // 32 (x8, h8) or 64 (x8b, h8b) rows of both planes, the lo rows after the hi rows)
  CUtensorMap gu8, d8, x8, h8, x8b, h8b;
  // bf16 gate/up rows as {H, I, 2 (gate, up), K}: one box holds a tile's 64 gate rows and
  // the matching 64 up rows
  CUtensorMap gu4;
};

bool tc_supported(int H, int I);
// Weight tensor maps over one layer's slot arena: bf16 rows (128-byte swizzle) or the raw
// quantised bytes (dequantised in shared memory); block-FP8 also as 128-byte swizzled
// e4m3 operand boxes.
int tc_make_weight_maps(uint8_t* arena, size_t stride, int K, int H, int I, int fmt, TcMaps* out);
int tc_make_act_maps(int fmt, __nv_bfloat16* x_perm, __nv_bfloat16* h, size_t P, int H, int I, TcMaps* out);
// sub: 0 = the whole wave, 1 = its experts that were resident before the step,
// 2 = its experts paged in for this wave (tiles of the two parts are contiguous).
cudaError_t tc_gateup(int fmt, const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, int sub,
                      const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms,
                      int32_t* err, int tile_n, cudaStream_t s);
cudaError_t tc_down(int fmt, const TcMaps& wm, const TcMaps& am, const int32_t* plan, int E, int wave, int sub,
                    const Workspace& ws, int I, int H, const uint8_t* arena, size_t stride, int num_sms, int32_t* err,
                    int tile_n, cudaStream_t s);
// The pair cap of a forward's tiles: small tiles (and a deeper pipeline) when the mean
// pairs per expert is at most half of kTcSmallN; any cap is correct (an expert with more
// pairs takes several tiles, which re-streams its weights).
inline int tc_tile_n(int T, int top_k, int E) {
  return (long long)T * top_k <= (long long)(kTcSmallN / 2) * E ? kTcSmallN : kTcMaxN;
}
// Block-FP8 forwards with small tiles run e4m3 MMAs on two-plane activations (x gathered
// by launch_gather_rows_fp8x2); with large tiles the weights are dequantised to bf16.
inline bool tc_fp8_planes(int fmt, int tile_n) { return fmt == PMOE_FP8_BLOCK128 && tile_n <= kTcSmallN; }
// Whether the down GEMM writes o_part as bf16 rows (else fp32): the bf16 kernel and the
// e4m3 kernel do; the kernels with converter warps do not.
inline bool tc_o_part_bf16(int fmt, int tile_n) { return fmt == PMOE_BF16 || tc_fp8_planes(fmt, tile_n); }

}  // namespace pmoe
