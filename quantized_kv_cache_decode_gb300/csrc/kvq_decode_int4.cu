// Decode-attention dispatch for the 4-bit affine format over the number of Value
// groups per token (d / Gv), and its instantiations for 1 and 2 groups.
#include "kvq_decode.cuh"

namespace kvq {

// d/Gv = 4 and 8 are instantiated in kvq_decode_int4_wide.cu (a second translation
// unit, so that the build compiles the two halves in parallel)
extern template cudaError_t launch_decode_t<4, 4>(const DecodeParams&, int, cudaStream_t);
extern template cudaError_t launch_decode_t<4, 8>(const DecodeParams&, int, cudaStream_t);
extern template cudaError_t occupancy_t<4, 4>(int, int, int, int*);
extern template cudaError_t occupancy_t<4, 8>(int, int, int, int*);

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
