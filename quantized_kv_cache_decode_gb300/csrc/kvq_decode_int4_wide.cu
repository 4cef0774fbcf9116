// Decode-attention instantiations for the 4-bit affine format with 4 and 8
// Value groups per token (d / Gv); kvq_decode_int4.cu dispatches to them.
#include "kvq_decode.cuh"

namespace kvq {

template cudaError_t launch_decode_t<4, 4>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode_t<4, 8>(const DecodeParams&, int, cudaStream_t);
template cudaError_t occupancy_t<4, 4>(int, int, int, int*);
template cudaError_t occupancy_t<4, 8>(int, int, int, int*);

}  // namespace kvq
