// Decode-attention instantiation for FP8 E5M2 with per-tensor scales.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_fp8_e5m2(const DecodeParams& p, int smem, cudaStream_t s) {
  return launch_decode_t<17, 1>(p, smem, s);
}

cudaError_t occupancy_decode_fp8_e5m2(int ngv, int g, int multi, int smem, int* n) {
  (void)ngv;
  return occupancy_t<17, 1>(g, multi, smem, n);
}

}  // namespace kvq
