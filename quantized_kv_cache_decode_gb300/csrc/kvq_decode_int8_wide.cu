// Decode-attention instantiations for the 8-bit affine format with 4 and 8
// Value groups per token (d / Gv); kvq_decode_int8.cu dispatches to them.
#include "kvq_decode.cuh"

namespace kvq {

template cudaError_t launch_decode_t<8, 4>(const DecodeParams&, int, cudaStream_t);
template cudaError_t launch_decode_t<8, 8>(const DecodeParams&, int, cudaStream_t);
template cudaError_t occupancy_t<8, 4>(int, int, int, int*);
template cudaError_t occupancy_t<8, 8>(int, int, int, int*);

}  // namespace kvq
