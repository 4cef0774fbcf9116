// Log-sum-exp merge of the decode kernel's per-CTA partials.
//
// Pair (b, h) was covered by the CTAs c_lo..c_hi of the decode grid; CTA c
// wrote its partial for the pair into slot c + b*H + h: the output normalised
// by its own softmax sum, and its log2-domain log-sum-exp.  The merged result
// is out = sum_i 2^(lse_i - LSE) o_i with LSE = log2 sum_i 2^lse_i, and the
// natural-log lse = LSE * ln 2.
#include "kvq_common.cuh"

namespace kvq {

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  pdl_wait();  // the previous kernel of the stream has finished (programmatic launch)
  pdl_trigger();
  const int bq = blockIdx.x;
  const int b = bq / p.Hq, hq = bq % p.Hq;
  const int h = hq / p.g, r = hq % p.g;
  const int c = threadIdx.x;
  const long long U = p.ws_prefix[p.batch];
  const int units = (p.ws_prefix[b + 1] - p.ws_prefix[b]) / p.H;
  const long long outi = ((long long)b * p.Hq + hq) * 128 + c;
  if (units == 0 || U == 0) {
    if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[outi] = __float2bfloat16_rn(0.f);
    else reinterpret_cast<float*>(p.out)[outi] = 0.f;
    if (p.lse && c == 0) p.lse[(long long)b * p.Hq + hq] = -INFINITY;
    return;
  }
  const long long C = p.ws_prefix[p.batch + 1];  // the split pass's choice (range_ctas)
  const long long P0 = p.ws_prefix[b] + (long long)h * units;
  const long long P1 = P0 + units;
  const long long c_lo = ((P0 + 1) * C - 1) / U;
  const long long c_hi = (P1 * C - 1) / U;
  const long long pair = (long long)b * p.H + h;
  // the CTAs whose unit range overlaps the pair and is not empty, listed once per block
  __shared__ int act[64];
  __shared__ int n_act;
  if (c == 0) {
    const long long qd = U / C, rd = U % C;
    long long qv = (c_lo * U) / C, rv = (c_lo * U) % C;
    int n = 0;
    for (long long cc = c_lo; cc <= c_hi; ++cc) {
      long long qn = qv + qd, rn = rv + rd;
      if (rn >= C) {
        rn -= C;
        ++qn;
      }
      if (qn != qv) {
        if (n < 64) act[n] = (int)cc;
        ++n;
      }
      qv = qn;
      rv = rn;
    }
    n_act = n;
  }
  __syncthreads();
  const int na = n_act;
  float M = -INFINITY, Lsum = 0.f, O = 0.f;
  if (na <= 64) {
    for (int k = 0; k < na; ++k) M = fmaxf(M, p.ws_lse[((long long)act[k] + pair) * p.g + r]);
    if (M != -INFINITY) {
      for (int k = 0; k < na; ++k) {
        const long long slot = (long long)act[k] + pair;
        const float f = exp2f(p.ws_lse[slot * p.g + r] - M);
        Lsum += f;
        O = fmaf(f, p.ws_o[(slot * p.g + r) * 128 + c], O);
      }
    }
  } else {
    auto active = [&](long long cc) { return (cc * U) / C != ((cc + 1) * U) / C; };
    for (long long cc = c_lo; cc <= c_hi; ++cc)
      if (active(cc)) M = fmaxf(M, p.ws_lse[(cc + pair) * p.g + r]);
    if (M != -INFINITY) {
      for (long long cc = c_lo; cc <= c_hi; ++cc) {
        if (!active(cc)) continue;
        const long long slot = cc + pair;
        const float f = exp2f(p.ws_lse[slot * p.g + r] - M);
        Lsum += f;
        O = fmaf(f, p.ws_o[(slot * p.g + r) * 128 + c], O);
      }
    }
  }
  const bool empty = !(Lsum > 0.f);
  const float o = empty ? 0.f : O / Lsum;
  if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[outi] = __float2bfloat16_rn(o);
  else reinterpret_cast<float*>(p.out)[outi] = o;
  if (p.lse && c == 0) p.lse[(long long)b * p.Hq + hq] = empty ? -INFINITY : (M + log2f(Lsum)) * 0.69314718055994531f;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.batch * p.Hq == 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(p.batch * p.Hq), dim3(128), 0, stream, p);
}

}  // namespace kvq
