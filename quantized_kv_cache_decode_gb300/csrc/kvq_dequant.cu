// Export of the dequantized cache as fp32 (sm_103a).
//
// "KV Cache Quantization Analysis", section 2: x_hat = s (q - z); section 4:
// an FP8 value times its fp32 scale.  Evaluated as two IEEE fp32 operations
// (q - z, then times s), or one (s times the exact E4M3 / E5M2 value), so the
// result is reproducible bit for bit.  Sink and residual tokens (every token of
// a bf16 layer) are their bf16 values.
#include "kvq_common.cuh"

namespace kvq {

__device__ __forceinline__ float e4m3_value(uint8_t c) {
  const uint32_t h = e4m3x2_to_f16x2((uint32_t)c);
  return unpack_f16(h).x;
}
// an E5M2 code is the high byte of the binary16 of the same value
__device__ __forceinline__ float e5m2_value(uint8_t c) { return unpack_f16((uint32_t)c << 8).x; }

// grid: (batch * H, ceil(max_tokens / 16)); block: 128 threads (one channel each)
__global__ void __launch_bounds__(128) dequant_kernel(const DequantParams p) {
  const LayerDesc& L = p.L;
  const int b = blockIdx.x / L.H, h = blockIdx.x % L.H;
  const int c = threadIdx.x;
  const long long pair = (long long)b * L.H + h;
  long long T = p.seq_lens[b];
  const long long cap = max_tokens(L) < p.max_tokens ? max_tokens(L) : p.max_tokens;
  if (T > cap) {
    if (blockIdx.y == 0 && c == 0) report(p.status, KVQ_DEV_CAPACITY);
    T = cap;
  }
  if (T < 0) T = 0;
  const TokenSplit ts = split_tokens((int)T, L);
  const __nv_bfloat16* sink_k = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_k);
  const __nv_bfloat16* sink_v = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_v);
  const __nv_bfloat16* ring_k = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_k);
  const __nv_bfloat16* ring_v = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_v);
  const uint32_t cmask = (1u << L.bits) - 1u;
  for (int tt = 0; tt < 16; ++tt) {
    const long long t = (long long)blockIdx.y * 16 + tt;
    if (t >= p.max_tokens) break;
    float kx = 0.f, vx = 0.f;
    if (t < ts.n_sink) {
      kx = __bfloat162float(sink_k[(pair * L.S + t) * L.d + c]);
      vx = __bfloat162float(sink_v[(pair * L.S + t) * L.d + c]);
    } else if (t < ts.n_sink + ts.qn) {
      const long long x = t - L.S;
      const long long i = x / 16;
      const uint8_t* rec = record_addr(L, p.C, b, h, i / L.tpg, c == 0 ? p.status : nullptr);
      if (rec) {
        const uint8_t* tile = tile_in_record(L, rec, i);
        const int row = (int)(x % 16);
        int kbyte, kbit, byte, bit;
        ktile_pos(L.bits, L.fp8 != 0, row, c, kbyte, kbit);
        vtile_pos(L.bits, L.fp8 != 0, row, c, byte, bit);
        if (L.fp8) {
          const uint8_t kc = tile[kbyte], vc = tile[16 * L.rb + byte];
          kx = __fmul_rn(*p.C.k_tscale, L.e5m2 ? e5m2_value(kc) : e4m3_value(kc));
          vx = __fmul_rn(*p.C.v_tscale, L.e5m2 ? e5m2_value(vc) : e4m3_value(vc));
        } else {
          const float* ks = reinterpret_cast<const float*>(rec);
          const float* kz = ks + 128;
          const float* vs = reinterpret_cast<const float*>(tile + 32 * L.rb);
          const float* vz = vs + 16 * L.ngv;
          const uint32_t kcode = (tile[kbyte] >> kbit) & cmask;
          const uint32_t vcode = (tile[16 * L.rb + byte] >> bit) & cmask;
          const int j = c / L.Gv;
          kx = __fmul_rn(ks[c], __fsub_rn((float)kcode, kz[c]));
          vx = __fmul_rn(vs[row * L.ngv + j], __fsub_rn((float)vcode, vz[row * L.ngv + j]));
          // dense-and-sparse: a kept entry adds its exact value (one more fp32 add)
          const uint32_t* ksp = reinterpret_cast<const uint32_t*>(tile + L.sp_off) + row * L.k_out;
          const uint32_t* vsp = reinterpret_cast<const uint32_t*>(tile + L.sp_off + 64 * L.k_out) + row * L.v_out;
          for (int e = 0; e < L.k_out; ++e)
            if ((int)(ksp[e] & 127u) == c) kx = __fadd_rn(kx, __uint_as_float(ksp[e] & 0xFFFF0000u));
          for (int e = 0; e < L.v_out; ++e)
            if ((int)(vsp[e] & 127u) == c) vx = __fadd_rn(vx, __uint_as_float(vsp[e] & 0xFFFF0000u));
        }
      }
    } else if (t < T) {
      const long long slot = (t - L.S) % L.W;
      kx = __bfloat162float(ring_k[(pair * L.W + slot) * L.d + c]);
      vx = __bfloat162float(ring_v[(pair * L.W + slot) * L.d + c]);
    }
    const long long o = (pair * p.max_tokens + t) * L.d + c;
    p.k_out[o] = kx;
    p.v_out[o] = vx;
  }
}

cudaError_t launch_dequantize(const DequantParams& p, cudaStream_t stream) {
  if (p.batch * p.L.H == 0 || p.max_tokens == 0) return cudaSuccess;
  dim3 grid(p.batch * p.L.H, (p.max_tokens + 15) / 16);
  dequant_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
