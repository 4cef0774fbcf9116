// Decode-attention instantiation for FP8 E4M3 with per-tensor scales.
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_fp8(const DecodeParams& p, int smem, cudaStream_t s) {
  return launch_decode_t<16, 1>(p, smem, s);
}

cudaError_t occupancy_decode_fp8(int ngv, int g, int multi, int smem, int* n) {
  (void)ngv;
  return occupancy_t<16, 1>(g, multi, smem, n);
}

}  // namespace kvq
