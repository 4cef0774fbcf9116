// Merge of attention results computed over disjoint parts of a sequence's tokens
// (sequence-split decode: one part per device, each run through the decode
// kernel with its log-sum-exp).  Softmax over the union of the parts:
//   lse = log sum_i exp(lse_i),  out = sum_i exp(lse_i - lse) o_i,
// each o_i normalised by its own part's softmax sum.  Natural-log lse values,
// shifted by their maximum before exponentiation; a part with lse = -inf holds
// no tokens and gets weight 0.
#include "kvq_common.cuh"

namespace kvq {

constexpr int kMergeRowsPerBlock = 8;  // one warp per row

__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
    lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n_parts,
                     long long rows, void* out, int out_bf16, float* lse_out) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kMergeRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  float M = -INFINITY;
  for (int i = 0; i < n_parts; ++i) M = fmaxf(M, lse_parts[(long long)i * rows + row]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int i = 0; i < n_parts; ++i) {
      const float f = expf(lse_parts[(long long)i * rows + row] - M);
      const float4 o = reinterpret_cast<const float4*>(o_parts + ((long long)i * rows + row) * 128)[lane];
      L += f;
      acc.x = fmaf(f, o.x, acc.x);
      acc.y = fmaf(f, o.y, acc.y);
      acc.z = fmaf(f, o.z, acc.z);
      acc.w = fmaf(f, o.w, acc.w);
    }
  }
  const bool empty = !(L > 0.f);
  const float inv = empty ? 0.f : 1.f / L;
  const float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (out_bf16) {
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(out) + row * 128 + 4 * lane;
    ob[0] = __float2bfloat16_rn(r.x);
    ob[1] = __float2bfloat16_rn(r.y);
    ob[2] = __float2bfloat16_rn(r.z);
    ob[3] = __float2bfloat16_rn(r.w);
  } else {
    reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * 128)[lane] = r;
  }
  if (lse_out && lane == 0) lse_out[row] = empty ? -INFINITY : M + logf(L);
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n_parts, long long rows, void* out,
                             int out_bf16, float* lse_out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock;
  lse_merge_kernel<<<(unsigned)blocks, 32 * kMergeRowsPerBlock, 0, stream>>>(o_parts, lse_parts, n_parts, rows, out,
                                                                              out_bf16, lse_out);
  return cudaGetLastError();
}

}  // namespace kvq
