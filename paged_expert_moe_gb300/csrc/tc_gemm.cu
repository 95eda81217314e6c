#include "tc_gemm.h"

namespace pmoe {
bool tc_supported(int, int) { return false; }
int tc_make_weight_maps(uint8_t*, size_t, int, int, int, TcMaps*) { return PMOE_EUNSUPPORTED; }
int tc_make_act_maps(__nv_bfloat16*, __nv_bfloat16*, size_t, int, int, TcMaps*) { return PMOE_EUNSUPPORTED; }
cudaError_t tc_gateup(const TcMaps&, const TcMaps&, const int32_t*, int, int, const Workspace&, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t tc_down(const TcMaps&, const TcMaps&, const int32_t*, int, int, const Workspace&, int, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pmoe
