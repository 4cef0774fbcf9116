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
constexpr unsigned kFull32 = 0xffffffffu;

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

// One CTA per (sequence, kv head): FP8 tokens (encoded one by one), bf16 rows of
// the residual window (integer layers: only the tokens that stay there after the
// groups that spill, which spill_kernel quantizes) and sink rows.
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  pdl_wait();  // the previous kernel of the stream has finished (programmatic launch)
  pdl_trigger();
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
    // integer layers: the groups that spill are quantized by spill_kernel; here only the
    // new tokens that stay in the bf16 residual window (bf16 layers: every token after the sink)
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

// ---------------------------------------------------------------------------
// spill_kernel: the Key groups (and their G Value tokens) that leave the residual
// window in this append, quantized and written in fragment order.
// One CTA of NT threads per (sequence, kv head, spilled group): the group's G
// bf16 Key and Value rows are staged in shared memory (coalesced 16-byte loads,
// from the ring for tokens already cached, from the input for new ones); every
// channel's Key min/max is found by NT/128 threads over runs of the tokens, every
// (token, Gv-channel group) Value min/max by a segmented warp-shuffle reduction;
// then each 32-bit word of the tile's fragment-order code matrices is assembled
// in registers (the inverse of the layout formula: which (token, channel) each
// field of the word holds) and stored once, consecutive threads on consecutive
// words.  The arithmetic of each code is the same IEEE fp32 sequence as above.
// With `rest` the CTAs of group 0 also write the sink rows and the new rows that
// stay in the residual window (one-token appends: those rows are never read by
// the spill of the same call; longer appends write them in a second launch).
// ---------------------------------------------------------------------------
constexpr int kSRow = 136;  // staged row stride (bf16): rows 8 banks apart, so the code pass reads without conflicts

// (step, reg, half) of the b-bit field at bit bp of operand word w: the inverse
// of frag_pos for the integer formats
template <int BITS>
__device__ __forceinline__ void frag_field(int w, int bp, int& step, int& reg, int& h) {
  if constexpr (BITS == 4) {
    step = w;
    reg = (bp & 15) >> 2;
    h = bp >> 4;
  } else if constexpr (BITS == 2) {
    h = bp >> 4;
    const int rem = bp & 15;
    step = 2 * w + (rem >> 3);
    reg = (rem & 7) >> 1;
  } else {
    step = w >> 1;
    const int bi = bp >> 3;
    reg = 2 * (w & 1) + (bi & 1);
    h = bi >> 1;
  }
}

template <int BITS, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) spill_kernel(const AppendParams p, int rest) {
  pdl_wait();  // the previous kernel of the stream has finished (programmatic launch)
  pdl_trigger();
  constexpr int kKSegs = NT / 128;  // runs of tokens per Key channel in the min/max pass (G >= 16 >= 2 kKSegs)
  extern __shared__ __align__(16) uint8_t smem[];
  const LayerDesc& L = p.L;
  constexpr int kLevels = (1 << BITS) - 1;
  constexpr float kFLevels = (float)kLevels;
  constexpr int kRB = 128 * BITS / 8;        // bytes of one token row of codes
  constexpr int kWPart = 16 * kRB / 4;       // operand words of one code matrix
  constexpr int kFields = 32 / BITS;         // codes per word
  const int b = blockIdx.x / L.H, h = blockIdx.x % L.H;
  const int gi = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long pair = (long long)b * L.H + h;
  const long long T0 = p.seq_lens[b];
  const long long T1 = T0 + p.n_new;
  if (T0 < 0 || T1 > max_tokens(L)) {
    if (gi == 0 && tid == 0) report(p.status, KVQ_DEV_CAPACITY);
    return;
  }
  const __nv_bfloat16* knew = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + pair * p.n_new * L.d;
  const __nv_bfloat16* vnew = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + pair * p.n_new * L.d;
  __nv_bfloat16* ring_k = reinterpret_cast<__nv_bfloat16*>(p.C.resid_k);
  __nv_bfloat16* ring_v = reinterpret_cast<__nv_bfloat16*>(p.C.resid_v);
  const TokenSplit t0s = split_tokens((int)T0, L);
  const TokenSplit t1s = split_tokens((int)T1, L);
  const int G = L.G, ngv = L.ngv, Gv = L.Gv;
  const int ng = (t1s.qn - t0s.qn) / G;  // groups that spill in this call

  if (gi < ng) {
    const int grp = t0s.qn / G + gi;
    const long long x0 = (long long)grp * G;  // first quantized index of the group
    uint8_t* rec = record_w(L, p.C, b, h, grp, tid == 0 ? p.status : nullptr);
    if (rec) {  // (uniform over the CTA)
      __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem);  // [G][kSRow]
      __nv_bfloat16* Vs = Ks + G * kSRow;                           // [G][kSRow]
      float* ksz = reinterpret_cast<float*>(Vs + G * kSRow);        // K scale [128], K zero [128]
      float* red = ksz + 256;                                       // [kKSegs][min, max][128]
      float* vsz = red + kKSegs * 256;                              // V scale [G][ngv], V zero [G][ngv]
      // stage the group's rows: 16-byte chunk ch of row tt, K then V; each thread issues up to
      // four loads before their stores (one HBM round trip instead of four), and the ring slot of
      // row tt is the group's first slot plus tt, wrapped once (tt < G <= W)
      const int slot0 = (int)(x0 % L.W);
      constexpr int kBatch = 4;
      for (int base = tid; base < 2 * G * 16; base += kBatch * NT) {
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = base + u * NT;
          if (idx < 2 * G * 16) {
            const int which = idx >= G * 16, rem = idx - which * G * 16, tt = rem >> 4, ch = rem & 15;
            const long long t = L.S + x0 + tt;
            const __nv_bfloat16* src;
            if (t < T0) {
              int sl = slot0 + tt;
              if (sl >= L.W) sl -= L.W;
              src = (which ? ring_v : ring_k) + (pair * L.W + sl) * L.d;
            } else {
              src = (which ? vnew : knew) + (t - T0) * L.d;
            }
            v[u] = reinterpret_cast<const uint4*>(src)[ch];
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = base + u * NT;
          if (idx < 2 * G * 16) {
            const int which = idx >= G * 16, rem = idx - which * G * 16, tt = rem >> 4, ch = rem & 15;
            reinterpret_cast<uint4*>((which ? Vs : Ks) + tt * kSRow)[ch] = v[u];
          }
        }
      }
      __syncthreads();
      if (L.k_out | L.v_out) {
        // dense-and-sparse: in each Key and Value row, the n entries of largest magnitude (ties:
        // the lower channel) go to the tile's sparse list, in channel order, and are set to 0 in
        // the staged row, which the statistics and codes below then see (one warp per row;
        // lane l holds channels 4l .. 4l + 3; bf16 magnitude bits order like the magnitudes)
        for (int row = warp; row < 2 * G; row += NT / 32) {
          const int isv = row >= G, tt = row - isv * G, n = isv ? L.v_out : L.k_out;
          if (n == 0) continue;
          uint2* xr = reinterpret_cast<uint2*>((isv ? Vs : Ks) + tt * kSRow) + lane;
          const uint2 raw = *xr;
          uint32_t v4[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
          uint32_t chosen = 0;
          for (int j = 0; j < n; ++j) {
            uint32_t best = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (!((chosen >> e) & 1u)) best = max(best, ((v4[e] & 0x7FFFu) << 8) | (255u - (uint32_t)(4 * lane + e)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(kFull32, best, o));
            const int c = 255 - (int)(best & 0xFFu);
            if ((c >> 2) == lane) chosen |= 1u << (c & 3);
          }
          // rank of an entry in channel order: the entries of the lower lanes, then the lower bits
          const int cnt = __popc(chosen);
          int incl = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull32, incl, o);
            if (lane >= o) incl += v;
          }
          uint32_t* sp = reinterpret_cast<uint32_t*>(rec + L.hdr_bytes + (long long)(tt >> 4) * L.tile_bytes +
                                                     L.sp_off + (isv ? 64 * L.k_out : 0)) + (tt & 15) * n;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if ((chosen >> e) & 1u) {
              sp[incl - cnt + __popc(chosen & ((1u << e) - 1u))] = (v4[e] << 16) | (uint32_t)(4 * lane + e);
              v4[e] = 0u;
            }
          *xr = make_uint2(v4[0] | (v4[1] << 16), v4[2] | (v4[3] << 16));
        }
        __syncthreads();
      }
      // Keys, per channel over the G tokens: kKSegs equal runs of tokens, then the runs combined
      {
        const int c = tid & 127, sg = tid >> 7, h0 = sg * (G / kKSegs), h1 = h0 + G / kKSegs;
        float mn = __bfloat162float(Ks[h0 * kSRow + c]), mx = mn;
        for (int tt = h0 + 1; tt < h1; ++tt) {
          const float x = __bfloat162float(Ks[tt * kSRow + c]);
          mn = fminf(mn, x);
          mx = fmaxf(mx, x);
        }
        red[sg * 256 + c] = mn;
        red[sg * 256 + 128 + c] = mx;
      }
      // Values, per token and Gv-channel group: lane holds channels 4 lane .. 4 lane + 3
      {
        const int seg = Gv >> 2;  // lanes per Value group
        for (int tt = warp; tt < G; tt += NT / 32) {
          const uint2 raw = reinterpret_cast<const uint2*>(Vs + tt * kSRow)[lane];
          const float2 a = unpack_bf16(raw.x), c2 = unpack_bf16(raw.y);
          float mn = fminf(fminf(a.x, a.y), fminf(c2.x, c2.y)), mx = fmaxf(fmaxf(a.x, a.y), fmaxf(c2.x, c2.y));
          for (int o = 1; o < seg; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(kFull32, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(kFull32, mx, o));
          }
          if ((lane & (seg - 1)) == 0) {
            const int j = lane / seg;
            float z;
            const float sc = affine_params(mn, mx, kFLevels, z);
            vsz[tt * ngv + j] = sc;
            vsz[G * ngv + tt * ngv + j] = z;
            float* tv = reinterpret_cast<float*>(rec + L.hdr_bytes + (long long)(tt >> 4) * L.tile_bytes + 32 * kRB);
            tv[(tt & 15) * ngv + j] = sc;
            tv[16 * ngv + (tt & 15) * ngv + j] = z;
          }
        }
      }
      __syncthreads();
      if (tid < 128) {
        float mn = red[tid], mx = red[128 + tid];
#pragma unroll
        for (int sg = 1; sg < kKSegs; ++sg) {
          mn = fminf(mn, red[sg * 256 + tid]);
          mx = fmaxf(mx, red[sg * 256 + 128 + tid]);
        }
        float z;
        const float sc = affine_params(mn, mx, kFLevels, z);
        ksz[tid] = sc;
        ksz[128 + tid] = z;
        reinterpret_cast<float*>(rec)[tid] = sc;         // header: K scale [128]
        reinterpret_cast<float*>(rec)[128 + tid] = z;    //         K zero  [128]
      }
      __syncthreads();
      // the codes: word m of a tile's code matrices (K words, then V words; memory order: lane
      // (m >> 2) & 31, operand word ((m >> 7) << 2) | (m & 3)) is assembled in registers for
      // every 16-token tile of the group by the thread(s) that own position m; a Key word's
      // channels, with their scales and zero-points, are the same in every tile
      constexpr int W2 = 2 * kWPart;
      constexpr int kStride = NT >= W2 ? NT / W2 : 1;  // threads per word position (over the tiles)
      const int ntile = G >> 4;
      for (int m = NT >= W2 ? tid % W2 : tid; m < W2; m += NT) {
        const int part = m >= kWPart, mm = m - part * kWPart;
        const int l = (mm >> 2) & 31, w = ((mm >> 7) << 2) | (mm & 3);
        // field f of the word: its staged (row, channel) offset, its Value scale index, its Key channel
        auto field = [&](int f, int& off, int& vj, int& c) {
          int step, reg, hh;
          frag_field<BITS>(w, f * BITS, step, reg, hh);
          const int i = (l >> 2) + 8 * (reg & 1), k = 2 * (l & 3) + hh + 8 * (reg >> 1);
          if (!part) {  // Keys: rows = tokens, column k holds channel 16 step + 4 ((k & 7) >> 1) + (k & 1) + 2 (k >> 3)
            c = 16 * step + 4 * ((k & 7) >> 1) + (k & 1) + 2 * (k >> 3);
            off = i * kSRow + c;
            vj = 0;
          } else {      // Values: rows = channels 16 step + i, columns = tokens
            c = 16 * step + i;
            off = k * kSRow + c;
            vj = k * ngv + c / Gv;
          }
        };
        // 4- and 8-bit words (8 and 4 fields): the fields' offsets and Key scales are kept in
        // registers over the tiles; 2-bit words (16 fields) recompute them (register budget)
        constexpr bool kKeep = kFields <= 8;
        int off[kKeep ? kFields : 1], vj[kKeep ? kFields : 1];
        float ks[kKeep ? kFields : 1], kz[kKeep ? kFields : 1];
        if constexpr (kKeep) {
#pragma unroll
          for (int f = 0; f < kFields; ++f) {
            int c;
            field(f, off[f], vj[f], c);
            ks[f] = part ? 0.f : ksz[c];
            kz[f] = part ? 0.f : ksz[128 + c];
          }
        }
        for (int t16 = NT >= W2 ? tid / W2 : 0; t16 < ntile; t16 += kStride) {
          const __nv_bfloat16* rows = (part ? Vs : Ks) + t16 * 16 * kSRow;
          const float* vs = vsz + t16 * 16 * ngv;
          uint32_t word = 0;
#pragma unroll
          for (int f = 0; f < kFields; ++f) {
            int o, j, c = 0;
            float sk, zk;
            if constexpr (kKeep) {
              o = off[f];
              j = vj[f];
              sk = ks[f];
              zk = kz[f];
            } else {
              field(f, o, j, c);
              sk = part ? 0.f : ksz[c];
              zk = part ? 0.f : ksz[128 + c];
            }
            const float x = __bfloat162float(rows[o]);
            const uint32_t code = part ? affine_code(x, vs[j], vs[G * ngv + j], kLevels) : affine_code(x, sk, zk, kLevels);
            word |= code << (f * BITS);
          }
          reinterpret_cast<uint32_t*>(rec + L.hdr_bytes + (long long)t16 * L.tile_bytes)[m] = word;
        }
      }
    }
  }
  if (rest && gi == 0) {
    // sink rows, and the new rows that stay in the residual window (16-byte chunks)
    __nv_bfloat16* sink_k = reinterpret_cast<__nv_bfloat16*>(p.C.sink_k);
    __nv_bfloat16* sink_v = reinterpret_cast<__nv_bfloat16*>(p.C.sink_v);
    const long long rfirst = (T0 > L.S + t1s.qn) ? T0 : (long long)L.S + t1s.qn;
    const int n = (int)(T1 - T0);
    for (int idx = tid; idx < 2 * n * 16; idx += NT) {
      const int which = idx >= n * 16, rem = idx - which * n * 16, j = rem >> 4, ch = rem & 15;
      const long long t = T0 + j;
      const __nv_bfloat16* src = (which ? vnew : knew) + (long long)j * L.d;
      __nv_bfloat16* dst = nullptr;
      if (t < L.S) dst = (which ? sink_v : sink_k) + (pair * L.S + t) * L.d;
      else if (t >= rfirst) dst = (which ? ring_v : ring_k) + (pair * L.W + (t - L.S) % L.W) * L.d;
      if (dst) reinterpret_cast<uint4*>(dst)[ch] = reinterpret_cast<const uint4*>(src)[ch];
    }
  }
}

template <int BITS, int NT>
cudaError_t launch_spill_nt(const AppendParams& p, int groups, int rest, cudaStream_t stream) {
  const size_t smem =
      (size_t)p.L.G * kSRow * 2 * 2 + (256 + (NT / 128) * 256) * 4 + (size_t)p.L.G * p.L.ngv * 8;
  static std::mutex mu;
  static int set_for[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64 || set_for[dev] < (int)smem) {
      e = cudaFuncSetAttribute(spill_kernel<BITS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) set_for[dev] = (int)smem;
    }
  }
  return launch_pdl(spill_kernel<BITS, NT>, dim3(p.batch * p.L.H, groups), dim3(NT), smem, stream, p, rest);
}

// Threads per spill CTA: few CTAs (one group per sequence and head, few pairs) get
// 1024 threads each (2-bit codes: 512), many get 256, so that every SM has work and each CTA's serial
// passes are short.  Measured on GB300: the 70B INT4 layer's spill (128 CTAs of a
// 128-token group) 41 -> 26 us from 256 to 1024 threads, the INT2 MHA layer's
// (1024 CTAs of a 32-token group) 37 -> 76 us the other way.
template <int BITS>
cudaError_t launch_spill_t(const AppendParams& p, int groups, int rest, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const long long ctas = (long long)p.batch * p.L.H * groups;
  if constexpr (BITS != 2) {  // (2-bit words hold 16 codes: the 1024-thread form would spill registers)
    if (ctas <= 2LL * sms) return launch_spill_nt<BITS, 1024>(p, groups, rest, stream);
  }
  if (ctas <= 4LL * sms) return launch_spill_nt<BITS, 512>(p, groups, rest, stream);
  return launch_spill_nt<BITS, 256>(p, groups, rest, stream);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int blocks = p.batch * p.L.H;
  if (blocks == 0 || p.n_new == 0) return cudaSuccess;
  if (p.L.fp8 || p.L.bf16) {
    return launch_pdl(append_kernel, dim3(blocks), dim3(kAppendThreads), 0, stream, p);
  }
  // integer layers: at most ceil(n_new / G) groups spill per (sequence, head)
  const int groups = (int)(((long long)p.n_new + p.L.G - 1) / p.L.G);
  const int fused = p.n_new == 1;  // one new token: its row never aliases a ring row the spill reads
  cudaError_t e;
  switch (p.L.bits) {
    case 2: e = launch_spill_t<2>(p, groups, fused, stream); break;
    case 4: e = launch_spill_t<4>(p, groups, fused, stream); break;
    default: e = launch_spill_t<8>(p, groups, fused, stream); break;
  }
  if (e != cudaSuccess || fused) return e;
  return launch_pdl(append_kernel, dim3(blocks), dim3(kAppendThreads), 0, stream, p);  // window and sink rows after the spills
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
