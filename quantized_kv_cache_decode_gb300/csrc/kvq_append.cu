// Quantize-on-append and FP8 calibration kernels (sm_103a).
//
// "KV Cache Quantization Analysis", section 5: the new token's K and V are
// quantized right after they are computed and stored.  Section 2: uniform
// affine quantization q = round(x/s + z), x_hat = s(q - z), asymmetric.
// Section 3: Keys per channel (over a group of G tokens), Values per token
// (over groups of Gv channels), recent tokens kept in full precision.
// Section 4: FP8 E4M3 with an fp32 scale.  "W4A16 + KV cache quantization
// combined accuracy": the first (sink) token kept in 16-bit precision.
//
// Every arithmetic step of the quantizer is one IEEE fp32 operation with
// round-to-nearest-even and no contraction (explicit __f*_rn intrinsics), so
// codes, scales and zero-points are reproducible bit for bit.
#include <mutex>

#include "kvq_common.cuh"

namespace kvq {

constexpr int kAppendThreads = 128;

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  uint16_t v;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(0.f), "f"(x));
  return (uint8_t)(v & 0xFFu);
}
__device__ __forceinline__ uint8_t f32_to_e5m2(float x) {
  uint16_t v;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(v) : "f"(0.f), "f"(x));
  return (uint8_t)(v & 0xFFu);
}

// s, z of one group from its min and max; returns s (z by reference)
__device__ __forceinline__ float affine_params(float mn, float mx, float levels, float& z) {
  float s = __fdiv_rn(__fsub_rn(mx, mn), levels);
  if (!(s >= 1.17549435e-38f)) s = 1.0f;  // constant group (or s not a normal float)
  z = -__fdiv_rn(mn, s);
  return s;
}
__device__ __forceinline__ uint32_t affine_code(float x, float s, float z, int levels) {
  const float t = __fadd_rn(__fdiv_rn(x, s), z);
  int qv = __float2int_rn(t);
  qv = qv < 0 ? 0 : (qv > levels ? levels : qv);
  return (uint32_t)qv;
}

// Writable record r of (b, h); nullptr (reported) for a bad block.
__device__ __forceinline__ uint8_t* record_w(const LayerDesc& L, const CachePtrs& C, int b, int h, long long r,
                                             uint32_t* status) {
  return const_cast<uint8_t*>(record_addr(L, C, b, h, r, status));
}

// One CTA per (sequence, kv head).  Dynamic smem: K and V of one group as fp32
// [G][128] each, their codes [G][128] bytes each, and one V tile staging buffer.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const LayerDesc& L = p.L;
  const int b = blockIdx.x / L.H, h = blockIdx.x % L.H;
  const int tid = threadIdx.x;
  const long long pair = (long long)b * L.H + h;
  const long long T0 = p.seq_lens[b];
  const long long T1 = T0 + p.n_new;
  if (T0 < 0 || T1 > max_tokens(L)) {
    if (tid == 0) report(p.status, KVQ_DEV_CAPACITY);
    return;
  }
  const __nv_bfloat16* knew = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + pair * p.n_new * L.d;
  const __nv_bfloat16* vnew = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + pair * p.n_new * L.d;
  __nv_bfloat16* ring_k = reinterpret_cast<__nv_bfloat16*>(p.C.resid_k);
  __nv_bfloat16* ring_v = reinterpret_cast<__nv_bfloat16*>(p.C.resid_v);
  __nv_bfloat16* sink_k = reinterpret_cast<__nv_bfloat16*>(p.C.sink_k);
  __nv_bfloat16* sink_v = reinterpret_cast<__nv_bfloat16*>(p.C.sink_v);
  const TokenSplit t0s = split_tokens((int)T0, L);
  const TokenSplit t1s = split_tokens((int)T1, L);

  if (L.fp8) {
    const float sk = *p.C.k_tscale, sv = *p.C.v_tscale;
    const long long first = T0 > L.S ? T0 : (long long)L.S;
    for (long long t = first; t < T1; ++t) {
      const long long x = t - L.S;
      const long long i = x / 16;
      uint8_t* rec = record_w(L, p.C, b, h, i / L.tpg, tid == 0 ? p.status : nullptr);
      if (!rec) continue;
      uint8_t* tile = rec + L.hdr_bytes + (long long)(i % L.tpg) * L.tile_bytes;
      if (x % 16 == 0) {
        // a new tile: clear it, so the codes of tokens not yet written read as 0
        for (int w = tid; w < 2 * 16 * L.rb / 16; w += kAppendThreads)
          reinterpret_cast<uint4*>(tile)[w] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
      }
      const int c = tid;
      const int tt = (int)(x % 16);
      const float kx = __bfloat162float(knew[(t - T0) * L.d + c]);
      const float vx = __bfloat162float(vnew[(t - T0) * L.d + c]);
      int byte, bit;
      const float kd = __fdiv_rn(kx, sk), vd = __fdiv_rn(vx, sv);
      ktile_pos(8, true, tt, c, byte, bit);
      tile[byte] = L.e5m2 ? f32_to_e5m2(kd) : f32_to_e4m3(kd);
      vtile_pos(8, true, tt, c, byte, bit);
      tile[16 * L.rb + byte] = L.e5m2 ? f32_to_e5m2(vd) : f32_to_e4m3(vd);
    }
  } else {
    const int G = L.G, levels = (1 << L.bits) - 1;
    const float flev = (float)levels;
    float* kf = reinterpret_cast<float*>(smem);         // [G][128]
    float* vf = kf + G * 128;                           // [G][128]
    uint8_t* kq = reinterpret_cast<uint8_t*>(vf + G * 128);  // [G][128]
    uint8_t* vq = kq + G * 128;                          // [G][128]
    uint32_t* tile = reinterpret_cast<uint32_t*>(vq + G * 128);  // one tile's K and V codes (2 * 16 * rb bytes)
    for (int grp = t0s.qn / G; grp < t1s.qn / G; ++grp) {
      const long long x0 = (long long)grp * G;  // first quantized index of the group
      // gather the group's tokens: old ones from the ring, new ones from the input
      for (int i = tid; i < G * 128; i += kAppendThreads) {
        const int tt = i >> 7, c = i & 127;
        const long long t = L.S + x0 + tt;
        float kx, vx;
        if (t < T0) {
          const long long slot = (t - L.S) % L.W;
          kx = __bfloat162float(ring_k[(pair * L.W + slot) * L.d + c]);
          vx = __bfloat162float(ring_v[(pair * L.W + slot) * L.d + c]);
        } else {
          kx = __bfloat162float(knew[(t - T0) * L.d + c]);
          vx = __bfloat162float(vnew[(t - T0) * L.d + c]);
        }
        kf[i] = kx;
        vf[i] = vx;
      }
      __syncthreads();
      // the group is record grp (G = 16 * tpg tokens): header = K scale, K zero; then G/16 tiles
      uint8_t* rec = record_w(L, p.C, b, h, grp, tid == 0 ? p.status : nullptr);
      if (rec) {
        float* ks = reinterpret_cast<float*>(rec);
        float* kz = ks + 128;
        // Keys: per channel over the G tokens (thread = channel)
        {
          const int c = tid;
          float mn = kf[c], mx = kf[c];
          for (int tt = 1; tt < G; ++tt) {
            mn = fminf(mn, kf[tt * 128 + c]);
            mx = fmaxf(mx, kf[tt * 128 + c]);
          }
          float z;
          const float s = affine_params(mn, mx, flev, z);
          for (int tt = 0; tt < G; ++tt) kq[tt * 128 + c] = (uint8_t)affine_code(kf[tt * 128 + c], s, z, levels);
          ks[c] = s;
          kz[c] = z;
        }
        // Values: per token over Gv channels
        for (int item = tid; item < G * L.ngv; item += kAppendThreads) {
          const int tt = item / L.ngv, j = item % L.ngv;
          const float* row = vf + tt * 128 + j * L.Gv;
          float mn = row[0], mx = row[0];
          for (int c = 1; c < L.Gv; ++c) {
            mn = fminf(mn, row[c]);
            mx = fmaxf(mx, row[c]);
          }
          float z;
          const float s = affine_params(mn, mx, flev, z);
          uint8_t* qrow = vq + tt * 128 + j * L.Gv;
          for (int c = 0; c < L.Gv; ++c) qrow[c] = (uint8_t)affine_code(row[c], s, z, levels);
          float* tvs = reinterpret_cast<float*>(rec + L.hdr_bytes + (long long)(tt / 16) * L.tile_bytes + 32 * L.rb);
          tvs[(tt % 16) * L.ngv + j] = s;
          tvs[16 * L.ngv + (tt % 16) * L.ngv + j] = z;
        }
        __syncthreads();
        // K and V codes of each 16-token tile, in fragment order
        const int tile_words = 2 * 16 * L.rb / 4;  // K part, then V part
        uint32_t* vtile = tile + 16 * L.rb / 4;
        for (int t16 = 0; t16 < G / 16; ++t16) {
          for (int i = tid; i < tile_words; i += kAppendThreads) tile[i] = 0u;
          __syncthreads();
          for (int i = tid; i < 16 * 128; i += kAppendThreads) {
            const int tt = i >> 7, c = i & 127;
            int byte, bit;
            ktile_pos(L.bits, false, tt, c, byte, bit);
            atomicOr(&tile[byte >> 2], (uint32_t)kq[(t16 * 16 + tt) * 128 + c] << ((byte & 3) * 8 + bit));
            vtile_pos(L.bits, false, tt, c, byte, bit);
            atomicOr(&vtile[byte >> 2], (uint32_t)vq[(t16 * 16 + tt) * 128 + c] << ((byte & 3) * 8 + bit));
          }
          __syncthreads();
          uint32_t* dst = reinterpret_cast<uint32_t*>(rec + L.hdr_bytes + (long long)t16 * L.tile_bytes);
          for (int i = tid; i < tile_words; i += kAppendThreads) dst[i] = tile[i];
          __syncthreads();
        }
      }
      __syncthreads();
    }
    // new tokens that stay in the bf16 residual window
    const long long rfirst = (T0 > L.S + t1s.qn) ? T0 : (long long)L.S + t1s.qn;
    for (long long t = rfirst; t < T1; ++t) {
      const long long slot = (t - L.S) % L.W;
      const int c = tid;
      ring_k[(pair * L.W + slot) * L.d + c] = knew[(t - T0) * L.d + c];
      ring_v[(pair * L.W + slot) * L.d + c] = vnew[(t - T0) * L.d + c];
    }
  }
  // sink tokens
  for (long long t = T0; t < T1 && t < L.S; ++t) {
    const int c = tid;
    sink_k[(pair * L.S + t) * L.d + c] = knew[(t - T0) * L.d + c];
    sink_v[(pair * L.S + t) * L.d + c] = vnew[(t - T0) * L.d + c];
  }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int blocks = p.batch * p.L.H;
  if (blocks == 0 || p.n_new == 0) return cudaSuccess;
  size_t smem = 0;
  if (!p.L.fp8 && !p.L.bf16) smem = (size_t)p.L.G * 128 * (4 + 4 + 1 + 1) + 2 * 16 * (size_t)p.L.rb;
  {
    // the limit is a per-device attribute that persists: raise it once per size
    static std::mutex mu;
    static int set_for[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64 || set_for[dev] < (int)smem) {
      e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) set_for[dev] = (int)smem;
    }
  }
  append_kernel<<<blocks, kAppendThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// FP8 per-tensor scale: s = amax / 448 (fp32 division), 1 when amax == 0
// ---------------------------------------------------------------------------
__global__ void absmax_kernel(const __nv_bfloat16* __restrict__ x, size_t n, unsigned int* amax_bits) {
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(__bfloat162float(x[i])));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // m >= 0: bits order like values
}

__global__ void scale_from_absmax_kernel(float* scale, float fmax) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned int*>(scale));
  *scale = amax > 0.f ? __fdiv_rn(amax, fmax) : 1.0f;
}

cudaError_t launch_fp8_calibrate(const void* x, size_t n, float fmax, float* scale_out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(scale_out, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    size_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    absmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(x), n,
                                                        reinterpret_cast<unsigned int*>(scale_out));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  scale_from_absmax_kernel<<<1, 1, 0, stream>>>(scale_out, fmax);
  return cudaGetLastError();
}

}  // namespace kvq
