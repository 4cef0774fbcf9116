// Decode-attention instantiations for the 4-bit affine format, one per
// number of Value groups per token (d / Gv).
#include "kvq_decode.cuh"

namespace kvq {

cudaError_t launch_decode_int4(const DecodeParams& p, int smem, cudaStream_t s) {
  switch (p.L.ngv) {
    case 1: return launch_decode_t<4, 1>(p, smem, s);
    case 2: return launch_decode_t<4, 2>(p, smem, s);
    case 4: return launch_decode_t<4, 4>(p, smem, s);
    case 8: return launch_decode_t<4, 8>(p, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t occupancy_decode_int4(int ngv, int g, int multi, int smem, int* n) {
  switch (ngv) {
    case 1: return occupancy_t<4, 1>(g, multi, smem, n);
    case 2: return occupancy_t<4, 2>(g, multi, smem, n);
    case 4: return occupancy_t<4, 4>(g, multi, smem, n);
    case 8: return occupancy_t<4, 8>(g, multi, smem, n);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
