// Fused decode attention over a quantized KV cache (sm_103a).
//
// softmax(q K^T / sqrt(d)) V for one new query per head, reading the compressed
// cache once ("W4A16 + KV cache quantization combined accuracy", section
// "오차가 어디서 만나는가"; dequantization fused with the matmuls as "KV Cache
// Quantization Analysis" section 5 asks, since decode is bound by reading the
// cache, section 1).
//
// Work decomposition.  Every (sequence, kv head) pair is a list of work units:
// 16-token bf16 tiles (sink + residual window, charged `bf_weight` units) and
// 16-token quantized tiles (1 unit).  The pairs' lists are concatenated and cut
// into num_ctas equal ranges, one per CTA (num_ctas = SMs x resident CTAs), so
// every CTA moves the same number of bytes whatever the sequence lengths.  A
// CTA writes one partial (normalised output + log-sum-exp) per pair it touches,
// into slot cta + pair; a second kernel merges the partials of each pair.
//
// Inside a CTA each of the 4 warps takes a contiguous sub-range and runs its
// own pipeline: its lane 0 streams 16-token tiles (codes, scales) into shared
// memory with bulk asynchronous copies (cp.async.bulk, TMA engine) completing
// on per-stage mbarriers, several stages ahead of the compute.
//
// Tensor-core mapping (mma.sync m16n8k16, fp32 accumulate).  The 16 MMA rows
// are the g <= 8 query heads of the kv head (row r) and, in rows r + 8, the
// low-order half of a two-term split of the same operand, so operands that are
// not exactly representable in 16 bits keep ~22 bits:
//   QK:  D[head][token] += A[head][channel] * B[channel][token]
//        A = q_c * s_c (Key scale of the channel, hi/lo split), B = centred Key
//        codes (exact in f16); the zero-point term sum_c q_c s_c (2^(b-1) - z_c)
//        is added per group in fp32.  FP8: A = q (exact in f16 after a power-of-
//        two rescale), B = E4M3 codes (exact in f16).  bf16 tiles: A = q, B = K.
//   PV:  D[head][channel] += A[head][token] * B[token][channel]
//        A = p_t * s_t (Value scale of the token, hi/lo split), B = centred Value
//        codes; zero-point term accumulated per Value group in fp32.
// The score tile of QK comes out of the MMA in exactly the register layout the
// PV A operand needs, so probabilities never leave registers.  Values are
// stored in "fragment order" so that each lane's 32-bit words unpack with one
// lop3 + one fma.f16x2 into B-operand registers.
#pragma once

#include <mutex>

#include "kvq_common.cuh"

namespace kvq {

constexpr int kNW = 4;                 // warps per CTA
constexpr int kThreads = kNW * 32;
constexpr int kMaxStages = 4;
constexpr float kPrescale = 64.f;      // w = p * (s / S_ref) * 64 < 2^14: f16 range is safe
constexpr float kTau = 6.f;            // score max may exceed its reference by 2^6 before a rescale
constexpr float kSTau = 4.f;           // a Value scale may exceed its reference 4x before a rescale
constexpr int kQStride = 36;           // floats per (head, lane-group) chunk of the query in smem
constexpr int kBfRow = 272;            // bytes per bf16 row in the warp scratch (256 + 16 pad)
constexpr int kWarpScratch = 16 * kBfRow;   // 4352 B: bf16 V tile, later the warp's merge record
                                            // (smaller when the layer has no bf16 tiles: p.warp_scratch)
constexpr int kMergeStride = 132;      // floats per head in the merge record: m, l, -, -, o[128]
constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ constexpr uint32_t f16_bits_of_int(int v) {
  // exact f16 encoding of an integer with |v| < 2048
  uint32_t s = v < 0 ? 0x8000u : 0u;
  uint32_t a = (uint32_t)(v < 0 ? -v : v);
  if (a == 0) return s;
  int e = 0;
  while ((a >> (e + 1)) != 0) ++e;
  return s | ((uint32_t)(e + 15) << 10) | ((a << (10 - e)) & 0x3FFu);
}
__host__ __device__ constexpr uint32_t f16_bits_pow2(int k) { return (uint32_t)(k + 15) << 10; }
__host__ __device__ constexpr uint32_t dup16(uint32_t h) { return h | (h << 16); }

constexpr uint32_t kMagic = 0x64006400u;  // f16 1024.0 in both halves: (1024 | field) = 1024 + field

template <int FMT>
struct FT {
  static constexpr bool kFp8 = FMT == 16;
  static constexpr bool kInt = !kFp8;
  static constexpr int kBits = kFp8 ? 8 : FMT;
  static constexpr int kRB = 128 * kBits / 8;   // bytes of one token row of codes
  static constexpr int kTile = 16 * kRB;        // bytes of 16 rows
  static constexpr int kKChunk = kRB / 4;       // bytes of a lane's 32 channels in a row
  static constexpr int kVChunk = kTile / 32;    // bytes of a lane's share of a V tile
  static constexpr int kHalf = kFp8 ? 0 : (1 << (kBits - 1));
};

// Channels (relative to the lane's 32-channel window) held in the low / high
// half of unpacked Key register j.
template <int FMT>
__host__ __device__ constexpr int kchan0(int j) {
  return FMT == 4 ? 8 * (j / 4) + (j % 4)
       : FMT == 2 ? 16 * (j / 8) + (j % 8)
       : FMT == 8 ? 4 * (j / 2) + (j % 2)
                  : 2 * j;  // FP8 and bf16: natural pairs
}
template <int FMT>
__host__ __device__ constexpr int kchan1(int j) {
  return FMT == 4 ? kchan0<FMT>(j) + 4 : FMT == 2 ? kchan0<FMT>(j) + 8 : FMT == 8 ? kchan0<FMT>(j) + 2
                                                                                  : kchan0<FMT>(j) + 1;
}

// --------------------------------------------------------------------------
// operand unpacking
// --------------------------------------------------------------------------
template <int P>  // 2-bit field at bit 2P of each half -> (n - 2)
__device__ __forceinline__ uint32_t int2_pair(uint32_t w) {
  constexpr uint32_t mask = (3u << (2 * P)) | (3u << (2 * P + 16));
  return hfma2(lop3_and_or(w, mask, kMagic), dup16(f16_bits_pow2(-2 * P)),
               dup16(f16_bits_of_int(-((1024 >> (2 * P)) + 2))));
}
__device__ __forceinline__ uint32_t int4_lo(uint32_t w) {  // nibbles at bits 0, 16 -> (n - 8)
  return hfma2(lop3_and_or(w, 0x000F000Fu, kMagic), dup16(f16_bits_of_int(1)), dup16(f16_bits_of_int(-1032)));
}
__device__ __forceinline__ uint32_t int4_hi(uint32_t w) {  // nibbles at bits 4, 20 -> (n - 8)
  return hfma2(lop3_and_or(w, 0x00F000F0u, kMagic), dup16(f16_bits_pow2(-4)), dup16(f16_bits_of_int(-72)));
}
__device__ __forceinline__ uint32_t int8_lo(uint32_t w) {  // bytes 0, 2 -> (n - 128)
  return hfma2(lop3_and_or(w, 0x00FF00FFu, kMagic), dup16(f16_bits_of_int(1)), dup16(f16_bits_of_int(-1152)));
}

// Key row: the lane's 32 channels -> 16 packed f16 pairs (channels kchan0/1(j)).
template <int FMT>
__device__ __forceinline__ void unpack_k(const uint8_t* p, uint32_t (&R)[16]) {
  if constexpr (FMT == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t s = w[i] >> 8;
      R[4 * i + 0] = int4_lo(w[i]);
      R[4 * i + 1] = int4_hi(w[i]);
      R[4 * i + 2] = int4_lo(s);
      R[4 * i + 3] = int4_hi(s);
    }
  } else if constexpr (FMT == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t s = w[i] >> 8;
      R[8 * i + 0] = int2_pair<0>(w[i]);
      R[8 * i + 1] = int2_pair<1>(w[i]);
      R[8 * i + 2] = int2_pair<2>(w[i]);
      R[8 * i + 3] = int2_pair<3>(w[i]);
      R[8 * i + 4] = int2_pair<0>(s);
      R[8 * i + 5] = int2_pair<1>(s);
      R[8 * i + 6] = int2_pair<2>(s);
      R[8 * i + 7] = int2_pair<3>(s);
    }
  } else if constexpr (FMT == 8) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(p);
    const uint4 v1 = *reinterpret_cast<const uint4*>(p + 16);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      R[2 * i + 0] = int8_lo(w[i]);
      R[2 * i + 1] = int8_lo(w[i] >> 8);
    }
  } else {  // FP8 E4M3
    const uint4 v0 = *reinterpret_cast<const uint4*>(p);
    const uint4 v1 = *reinterpret_cast<const uint4*>(p + 16);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      e4m3x4_to_f16x4(w[i], R[2 * i + 0], R[2 * i + 1]);
    }
  }
}

// Value tile: B-operand registers of n-tile jt from the lane's words W.
template <int FMT, int JT, int NWORDS>
__device__ __forceinline__ void unpack_v(const uint32_t (&W)[NWORDS], uint32_t& b01, uint32_t& b23) {
  if constexpr (FMT == 4) {
    const uint32_t src = (JT & 1) ? (W[JT / 2] >> 8) : W[JT / 2];
    b01 = int4_lo(src);
    b23 = int4_hi(src);
  } else if constexpr (FMT == 2) {
    constexpr int a = JT & 3;
    constexpr int p0 = 2 * a, p1 = 2 * a + 1;
    const uint32_t w = W[JT / 4];
    const uint32_t s = w >> 8;
    b01 = int2_pair<(p0 & 3)>(p0 < 4 ? w : s);
    b23 = int2_pair<(p1 & 3)>(p1 < 4 ? w : s);
  } else if constexpr (FMT == 8) {
    b01 = int8_lo(W[JT]);
    b23 = int8_lo(W[JT] >> 8);
  } else {
    e4m3x4_to_f16x4(W[JT], b01, b23);
  }
}

// --------------------------------------------------------------------------
// per-warp online-softmax state (thread (r, q) holds head r)
// --------------------------------------------------------------------------
template <int NGV>
struct WarpState {
  float o[16][4];    // PV accumulators: rows r (hi) in [0..1], rows r+8 (lo) in [2..3]
  float zacc[NGV];   // zero-point terms per Value group (thread-partial)
  float m;           // reference max (log2 domain)
  float l;           // sum of p (thread-partial)
  float S;           // reference Value scale
  float inv_S;       // 1 / S
};

template <int NGV>
__device__ __forceinline__ void state_init(WarpState<NGV>& st) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
#pragma unroll
  for (int j = 0; j < NGV; ++j) st.zacc[j] = 0.f;
  st.m = -INFINITY;
  st.l = 0.f;
  st.S = 0.f;
  st.inv_S = 0.f;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Update the running max / scale references for a stage with scores sig[N]
// (the lane's tokens of head r, 4 per 16-token tile; -inf when masked) and the
// lane's largest Value scale smax; return p[N] * kPrescale and 1 / S.  A token's
// PV weight is then (s_t / S) * (p_t * kPrescale) <= 4 * 2^6 * 64 = 2^14.
template <int NGV, int N>
__device__ __forceinline__ float softmax_step(WarpState<NGV>& st, const float (&sig)[N], float smax, float (&pr)[N]) {
  float tmax = sig[0];
#pragma unroll
  for (int e = 1; e < N; ++e) tmax = fmaxf(tmax, sig[e]);
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
  tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
  smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, 1));
  smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, 2));
  const bool bump_m = tmax > st.m + kTau;
  const bool bump_s = smax > st.S * kSTau;
  if (__any_sync(kFull, bump_m || bump_s)) {
    const float m_new = bump_m ? tmax : st.m;
    const float S_new = bump_s ? smax : st.S;
    const float a = (st.m == -INFINITY) ? 0.f : fast_exp2(st.m - m_new);
    const float ao = (S_new > 0.f) ? a * (st.S / S_new) : 0.f;
    st.l *= a;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[j][e] *= ao;
#pragma unroll
    for (int j = 0; j < NGV; ++j) st.zacc[j] *= ao;
    st.m = m_new;
    st.S = S_new;
    st.inv_S = 1.f / S_new;
  }
  float lsum = 0.f;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    pr[e] = (sig[e] == -INFINITY) ? 0.f : fast_exp2(sig[e] - st.m);
    lsum += pr[e];
    pr[e] *= kPrescale;
  }
  st.l += lsum;
  return st.inv_S;
}

// --------------------------------------------------------------------------
// A operands built from the query
// --------------------------------------------------------------------------
// INT: A = q_c * s_c (this group's Key scales) split hi/lo, plus the group's
// zero-point term and the score multiplier.  qv: the lane's 32 query values of
// head r; ks/kz: this group's Key scale / zero row (smem, 128 floats).
template <int FMT>
__device__ __forceinline__ void build_a_int(const float* qrow, const float* ks, const float* kz, int q,
                                            float scale_log2, uint32_t (&A)[8][4], float& kfac, float& cterm) {
  // pass 1: largest |q_c s_c| of the head (sets the f16 range) and the zero-point term
  constexpr float kH = (float)FT<FMT>::kHalf;
  const float* ksq = ks + 32 * q;
  const float* kzq = kz + 32 * q;
  float mx = 0.f, cz = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ci = 4 * ((i + q) & 7);  // rotated per lane group: the 4 groups hit different banks
    const float4 q4 = *reinterpret_cast<const float4*>(qrow + ci);
    const float4 s4 = *reinterpret_cast<const float4*>(ksq + ci);
    const float4 z4 = *reinterpret_cast<const float4*>(kzq + ci);
    const float x0 = q4.x * s4.x, x1 = q4.y * s4.y, x2 = q4.z * s4.z, x3 = q4.w * s4.w;
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))));
    cz = fmaf(x0, kH - z4.x, cz);
    cz = fmaf(x1, kH - z4.y, cz);
    cz = fmaf(x2, kH - z4.z, cz);
    cz = fmaf(x3, kH - z4.w, cz);
  }
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  cz += __shfl_xor_sync(kFull, cz, 1);
  cz += __shfl_xor_sync(kFull, cz, 2);
  const float kappa = mx > 0.f ? 16384.f / mx : 1.f;
  // pass 2: A = hi/lo split of q_c s_c kappa, in the channel order the Key unpacking produces
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int c0 = kchan0<FMT>(j), c1 = kchan1<FMT>(j);
    uint32_t hi, lo;
    split_f16(qrow[c0] * ksq[c0] * kappa, qrow[c1] * ksq[c1] * kappa, hi, lo);
    if ((j & 1) == 0) {
      A[j >> 1][0] = hi;
      A[j >> 1][1] = lo;
    } else {
      A[j >> 1][2] = hi;
      A[j >> 1][3] = lo;
    }
  }
  kfac = scale_log2 / kappa;
  cterm = scale_log2 * cz;
}

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
// final output of (sequence b, query head hq), channel c; l2 = log2-domain log-sum-exp
__device__ __forceinline__ void write_out(const DecodeParams& p, int b, int hq, int c, float o, float l2) {
  const long long oi = ((long long)b * p.Hq + hq) * 128 + c;
  if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  else reinterpret_cast<float*>(p.out)[oi] = o;
  if (p.lse && c == 0) p.lse[(long long)b * p.Hq + hq] = l2 * 0.69314718055994531f;
}

// CTAs c in [c_lo, c_hi] whose unit range [floor(cU/C), floor((c+1)U/C)) is not
// empty, written to list[0..n) (at most cap entries; returns the full count).
// Walks c with a running quotient/remainder: no division per step.
__device__ __forceinline__ int active_ctas(long long c_lo, long long c_hi, long long U, long long C, int* list,
                                           int cap) {
  const long long qd = U / C, rd = U % C;
  long long qv = (c_lo * U) / C, rv = (c_lo * U) % C;  // floor(c U / C), remainder
  int n = 0;
  for (long long c = c_lo; c <= c_hi; ++c) {
    long long qn = qv + qd, rn = rv + rd;
    if (rn >= C) {
      rn -= C;
      ++qn;
    }
    if (qn != qv) {
      if (n < cap) list[n] = (int)c;
      ++n;
    }
    qv = qn;
    rv = rn;
  }
  return n;
}
constexpr int kMaxParts = 64;  // partials of one pair merged from a shared-memory list

// One (sequence, kv head) pair's share of this CTA's unit range.
struct SegRec {
  long long pair_start;  // first unit of the pair in the flat unit list
  int b, h, ua, ue, units;
  int n_sink, qn, r, nbf, nq;
};
constexpr int kMaxSeg = 16;  // segments per table batch
constexpr int kChunk = 2;    // quantized tiles per softmax step

// Unit order inside a pair: the nbf bf16 tiles (wbf units each) are spread
// evenly among the nq quantized tiles (1 unit each): bf16 tile i sits right
// before quantized tile floor(i * nq / nbf).  Every warp's contiguous unit range
// then gets its share of the (slower) bf16 tiles.
__device__ __forceinline__ long long unit_of_bf(int i, int nbf, int nq, int wbf) {
  return (long long)i * nq / nbf + (long long)i * wbf;
}
__device__ __forceinline__ long long unit_of_q(int k, int nbf, int nq, int wbf) {
  const long long before = nbf == 0 ? 0 : min((long long)nbf, ((long long)(k + 1) * nbf + nq - 1) / nq);
  return k + wbf * before;
}

// This warp's part of a segment: bf16 tiles [bf0, bf0 + nbf_w), quantized tiles
// [q0, q0 + nq_w); stages: two per bf16 tile (its K rows, then its V rows), then
// ceil(nq_w / tps) quantized stages.
struct WarpPart {
  int bf0, nbf_w, q0, nq_w, nstage;
};

__device__ __forceinline__ WarpPart warp_part(const SegRec& sg, int warp, int wbf, int tps) {
  WarpPart w;
  const long long wa = sg.ua + (long long)(sg.ue - sg.ua) * warp / kNW;
  const long long we = sg.ua + (long long)(sg.ue - sg.ua) * (warp + 1) / kNW;
  // first bf16 tile / quantized tile whose unit is at or after x
  auto first_bf = [&](long long x) {
    int lo = 0, hi = sg.nbf;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (unit_of_bf(mid, sg.nbf, sg.nq, wbf) >= x) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  auto first_q = [&](long long x) {
    int lo = 0, hi = sg.nq;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (unit_of_q(mid, sg.nbf, sg.nq, wbf) >= x) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  w.bf0 = first_bf(wa);
  w.nbf_w = first_bf(we) - w.bf0;
  w.q0 = first_q(wa);
  w.nq_w = first_q(we) - w.q0;
  w.nstage = 2 * w.nbf_w + (w.nq_w + tps - 1) / tps;
  return w;
}

template <int FMT, int NGV>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeParams p) {
  using F = FT<FMT>;
  constexpr int kHdr = F::kInt ? 1024 : 0;  // every stage starts with a header slot (INT)
  extern __shared__ __align__(128) uint8_t smem[];
  const LayerDesc& L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, q = lane & 3;
  const int B = p.batch, H = L.H, g = p.g;
  const int tps = p.tps, nst = p.nst, wbf = p.bf_weight;

  // ---- shared memory carve-up ----
  uint8_t* stage_base = smem;
  size_t off = (size_t)kNW * nst * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off);
  off += kNW * kMaxStages * sizeof(uint64_t);
  float* q_s = reinterpret_cast<float*>(smem + off);
  off += 8 * 4 * kQStride * sizeof(float);
  uint8_t* scratch = smem + off;
  off += (size_t)kNW * p.warp_scratch;
  SegRec* segs = reinterpret_cast<SegRec*>(smem + off);
  off += kMaxSeg * sizeof(SegRec);
  int* prefix = reinterpret_cast<int*>(smem + off);  // [B + 1]
  __shared__ int seg_count;
  __shared__ long long batch_end;

  if (tid == 0) {
    for (int i = 0; i < kNW * kMaxStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_barrier_init();
  }

  // ---- per-sequence work units and their prefix (units of all H heads) ----
  const long long tmax_tok = max_tokens(L);
  auto seq_tokens = [&](int b) -> int {
    long long T = p.seq_lens[b];
    if (T < 0) T = 0;
    if (T > tmax_tok) T = tmax_tok;
    return (int)T;
  };
  auto seq_units = [&](int b) -> int {
    const TokenSplit ts = split_tokens(seq_tokens(b), L);
    const int nbf = (ts.n_sink + ts.r + 15) >> 4;
    const int nq = (ts.qn + 15) >> 4;
    return nbf * wbf + nq;
  };
  {
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = local;
      local += seq_units(b) * H;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_tot[kNW];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += warp_tot[w];
    const int excl = wbase + incl - local;
    for (int b = b0; b < b1; ++b) prefix[b] += excl;
    if (tid == kThreads - 1) prefix[B] = wbase + incl;
    if (blockIdx.x == 0) {
      for (int b = tid; b < B; b += kThreads)
        if (p.seq_lens[b] > tmax_tok) report(p.status, KVQ_DEV_CAPACITY);
    }
    __syncthreads();
    if (blockIdx.x == 0)
      for (int b = tid; b <= B; b += kThreads) p.ws_prefix[b] = prefix[b];
  }

  const long long U = prefix[B];
  const long long C = p.num_ctas;
  if (p.fuse) {
    // sequences without tokens belong to no CTA's range: out = 0, lse = -inf
    for (int b = blockIdx.x; b < B; b += gridDim.x)
      if (prefix[b + 1] == prefix[b])
        for (int i = tid; i < p.Hq * 128; i += kThreads) write_out(p, b, i >> 7, i & 127, 0.f, -INFINITY);
  }
  const long long st = (long long)blockIdx.x * U / C;
  const long long en = (long long)(blockIdx.x + 1) * U / C;

  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* sink_k = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_k);
  const __nv_bfloat16* sink_v = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_v);
  const __nv_bfloat16* ring_k = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_k);
  const __nv_bfloat16* ring_v = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_v);

  uint8_t* my_stages = stage_base + (size_t)warp * nst * p.stage_bytes;
  uint64_t* my_bars = bars + warp * kMaxStages;
  uint8_t* my_scratch = scratch + warp * p.warp_scratch;
  const float* qrow = q_s + (r * 4 + q) * kQStride;  // the lane's 32 query values of head r
  uint32_t phase_bits = 0;  // expected parity of each stage barrier of this warp
  uint32_t slot_valid = 0;  // lane 0: 8 bits per slot, the tiles its stage holds
  uint32_t pending = 0;     // slots with copies in flight
  bool alive = true;
  int n_issued = 0, n_consumed = 0;
  const float s_v8 = F::kFp8 ? __ldg(p.C.v_tscale) : 1.f;

  auto load_q = [&](const SegRec& sg) {
    for (int i = tid; i < 8 * 128; i += kThreads) {
      const int hr = i >> 7, c = i & 127;
      float v = 0.f;
      if (hr < g) v = __bfloat162float(qg[((long long)sg.b * p.Hq + sg.h * g + hr) * 128 + c]);
      q_s[(hr * 4 + (c >> 5)) * kQStride + (c & 31)] = v;
    }
  };

  long long pos = st;
  while (pos < en) {
    // ---- the next batch of segments of this CTA's range ----
    __syncthreads();
    if (tid == 0) {
      int ns = 0;
      long long pp = pos;
      while (pp < en && ns < kMaxSeg) {
        int lo = 0, hi = B;  // largest b with prefix[b] <= pp
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix[mid] <= pp) lo = mid; else hi = mid - 1;
        }
        SegRec sg;
        sg.b = lo;
        sg.units = (prefix[lo + 1] - prefix[lo]) / H;
        sg.h = (int)((pp - prefix[lo]) / sg.units);
        sg.pair_start = prefix[lo] + (long long)sg.h * sg.units;
        const long long se = min(en, sg.pair_start + sg.units);
        sg.ua = (int)(pp - sg.pair_start);
        sg.ue = (int)(se - sg.pair_start);
        const TokenSplit ts = split_tokens(seq_tokens(lo), L);
        sg.n_sink = ts.n_sink;
        sg.qn = ts.qn;
        sg.r = ts.r;
        sg.nbf = (ts.n_sink + ts.r + 15) >> 4;
        sg.nq = (ts.qn + 15) >> 4;
        segs[ns++] = sg;
        pp = se;
      }
      seg_count = ns;
      batch_end = pp;
    }
    __syncthreads();
    const int nseg = seg_count;

    // ---- producer (lane 0 copies; every lane keeps the same cursor) ----
    int ps = 0, pj = 0;
    WarpPart pw = warp_part(segs[0], warp, wbf, tps);
    while (ps < nseg && pw.nstage == 0) {
      ++ps;
      if (ps < nseg) pw = warp_part(segs[ps], warp, wbf, tps);
    }
    auto issue_next = [&]() {
      const int slot = n_issued % nst;
      uint32_t vm = 0;
      if (lane == 0) {
        const SegRec& sg = segs[ps];
        uint8_t* dst = my_stages + (size_t)slot * p.stage_bytes;
        const uint32_t bar = smem_addr(&my_bars[slot]);
        if (pj < 2 * pw.nbf_w) {
          // bf16 tile: its 16 K rows (even stage) or V rows (odd stage), one 256-byte copy per row
          const int bt = pw.bf0 + pj / 2;
          const int rows = min(16, sg.n_sink + sg.r - bt * 16);
          const TokenSplit ts = {sg.n_sink, sg.qn, sg.r};
          mbar_arrive_expect_tx(bar, 256u * rows);
          for (int rr = 0; rr < rows; ++rr) {
            const __nv_bfloat16* src = (pj & 1) ? bf16_row(L, sink_v, ring_v, sg.b, sg.h, bt * 16 + rr, ts)
                                                : bf16_row(L, sink_k, ring_k, sg.b, sg.h, bt * 16 + rr, ts);
            bulk_copy_g2s(smem_addr(dst + rr * kBfRow), src, 256, bar);
          }
          vm = 1;
        } else {
          // quantized tiles [i0, i0 + n): one contiguous range per record touched
          const int qs = pj - 2 * pw.nbf_w;
          const long long i0 = pw.q0 + (long long)qs * tps;
          const int n = (int)min((long long)tps, (long long)(pw.q0 + pw.nq_w) - i0);
          const long long last = i0 + n - 1;
          const bool hdr0 = F::kInt && qs == 0 && (i0 % L.tpg) != 0;
          if (!L.paged) {
            const uint8_t* base = reinterpret_cast<const uint8_t*>(p.C.qstore) +
                                  ((long long)sg.b * H + sg.h) * L.nrec * L.rec_bytes;
            const uint8_t* rec0 = base + (i0 / L.tpg) * L.rec_bytes;
            const uint8_t* start = (F::kInt && i0 % L.tpg == 0) ? rec0 : rec0 + L.hdr_bytes + (i0 % L.tpg) * L.tile_bytes;
            const uint8_t* end = base + (last / L.tpg) * L.rec_bytes + L.hdr_bytes + (last % L.tpg + 1) * L.tile_bytes;
            const uint32_t len = (uint32_t)(end - start);
            mbar_arrive_expect_tx(bar, len + (hdr0 ? 1024u : 0u));
            bulk_copy_g2s(smem_addr(dst + kHdr), start, len, bar);
            if (hdr0) bulk_copy_g2s(smem_addr(dst), rec0, 1024, bar);
            vm = (1u << n) - 1u;
          } else {
            uint32_t bytes = 0;
            for (long long rr = i0 / L.tpg; rr <= last / L.tpg; ++rr) {
              const uint8_t* rec = record_addr(L, p.C, sg.b, sg.h, rr, p.status);
              const long long a0 = max(i0, rr * L.tpg), a1 = min(last, rr * L.tpg + L.tpg - 1);
              if (!rec) continue;
              for (long long i = a0; i <= a1; ++i) vm |= 1u << (int)(i - i0);
              const bool with_hdr = F::kInt && (a0 % L.tpg) == 0;
              bytes += (uint32_t)((with_hdr ? L.hdr_bytes : 0) + (a1 - a0 + 1) * L.tile_bytes);
              if (hdr0 && rr == i0 / L.tpg) bytes += 1024;
            }
            if (vm) {
              mbar_arrive_expect_tx(bar, bytes);
              uint32_t so = kHdr;
              for (long long rr = i0 / L.tpg; rr <= last / L.tpg; ++rr) {
                const long long a0 = max(i0, rr * L.tpg), a1 = min(last, rr * L.tpg + L.tpg - 1);
                const bool with_hdr = F::kInt && (a0 % L.tpg) == 0;
                const uint32_t len = (uint32_t)((with_hdr ? L.hdr_bytes : 0) + (a1 - a0 + 1) * L.tile_bytes);
                const uint8_t* rec = record_addr(L, p.C, sg.b, sg.h, rr, nullptr);
                if (rec) {
                  const uint8_t* src = with_hdr ? rec : rec + L.hdr_bytes + (a0 % L.tpg) * L.tile_bytes;
                  bulk_copy_g2s(smem_addr(dst + so), src, len, bar);
                  if (hdr0 && rr == i0 / L.tpg) bulk_copy_g2s(smem_addr(dst), rec, 1024, bar);
                }
                so += len;
              }
            }
          }
        }
        slot_valid = (slot_valid & ~(0xFFu << (8 * slot))) | (vm << (8 * slot));
      }
      vm = __shfl_sync(kFull, vm, 0);
      if (vm) pending |= 1u << slot;
      ++n_issued;
      if (++pj == pw.nstage) {
        pj = 0;
        ++ps;
        while (ps < nseg) {
          pw = warp_part(segs[ps], warp, wbf, tps);
          if (pw.nstage) break;
          ++ps;
        }
      }
    };
    while (alive && n_issued - n_consumed < nst && ps < nseg) issue_next();
    // the query of the first segment, while the first copies are in flight
    load_q(segs[0]);
    __syncthreads();

    // ---- consumer ----
    for (int s = 0; s < nseg; ++s) {
      const SegRec sg = segs[s];
      const WarpPart wp = warp_part(sg, warp, wbf, tps);
      const int nbf_tok = sg.n_sink + sg.r;
      WarpState<NGV> stt;
      state_init(stt);
      uint32_t A[8][4];
      float kfac = 0.f, cterm = 0.f;
      if constexpr (F::kFp8) {
        // A = q * 2^E (exact in f16), E from the head's largest |q|
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(qrow[i]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        int ex = 0;
        if (mx > 0.f) (void)frexpf(mx, &ex);
        const float sc = mx > 0.f ? ldexpf(1.f, 15 - ex) : 1.f;  // max |q| * sc in [2^14, 2^15)
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          const float4 qq = *reinterpret_cast<const float4*>(qrow + 4 * s2);
          A[s2][0] = pack_f16(qq.x * sc, qq.y * sc);
          A[s2][1] = 0u;
          A[s2][2] = pack_f16(qq.z * sc, qq.w * sc);
          A[s2][3] = 0u;
        }
        kfac = p.scale_log2 * __ldg(p.C.k_tscale) / sc;
      }
      float sig_bf[4];  // scores of a bf16 tile between its K and V stages

      for (int j = 0; j < wp.nstage; ++j) {
        const int slot = n_consumed % nst;
        const uint32_t vmask = (__shfl_sync(kFull, slot_valid, 0) >> (8 * slot)) & 0xFFu;
        if (vmask) {
          bool ok = alive && mbar_wait_bounded(smem_addr(&my_bars[slot]), (phase_bits >> slot) & 1u, kWaitLimitCycles);
          ok = __all_sync(kFull, ok);
          if (ok) {
            phase_bits ^= 1u << slot;
            pending &= ~(1u << slot);
          } else if (alive) {
            alive = false;
            if (lane == 0) report(p.status, KVQ_DEV_TIMEOUT);
          }
        }
        const uint8_t* stg = my_stages + (size_t)slot * p.stage_bytes;
        if (vmask && alive && j < 2 * wp.nbf_w) {
          const int bt = wp.bf0 + j / 2;
          const int rows = min(16, nbf_tok - bt * 16);
          if ((j & 1) == 0) {
            // ---- bf16 tile, K rows: QK with A = q (bf16, exact) ----
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const int row = nt * 8 + r;
              uint32_t R[16];
              if (row < rows) {
                const uint4* r4 = reinterpret_cast<const uint4*>(stg + row * kBfRow + 64 * q);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint4 v = r4[i];
                  R[4 * i] = v.x; R[4 * i + 1] = v.y; R[4 * i + 2] = v.z; R[4 * i + 3] = v.w;
                }
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) R[i] = 0u;
              }
#pragma unroll
              for (int s2 = 0; s2 < 8; ++s2) {
                const float4 qq = *reinterpret_cast<const float4*>(qrow + 4 * s2);
                mma_bf16(acc[nt], pack_bf16(qq.x, qq.y), 0u, pack_bf16(qq.z, qq.w), 0u, R[2 * s2], R[2 * s2 + 1]);
              }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = (e >> 1) * 8 + 2 * q + (e & 1);
              sig_bf[e] = (t < rows) ? acc[e >> 1][e & 1] * p.scale_log2 : -INFINITY;
            }
          } else {
            // ---- bf16 tile, V rows: softmax, then PV through transposed loads ----
            uint8_t* stw = const_cast<uint8_t*>(stg);
            for (int idx = lane; idx < (16 - rows) * 16; idx += 32)
              *reinterpret_cast<uint4*>(stw + (rows + idx / 16) * kBfRow + (idx % 16) * 16) = make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
            float pr[4];
            const float inv_s = softmax_step<NGV, 4>(stt, sig_bf, 1.f, pr);
            uint32_t ah0, al0, ah1, al1;
            split_bf16(pr[0] * inv_s, pr[1] * inv_s, ah0, al0);
            split_bf16(pr[2] * inv_s, pr[3] * inv_s, ah1, al1);
            const uint32_t sbase = smem_addr(stg);
#pragma unroll
            for (int jp = 0; jp < 8; ++jp) {
              const int mi = lane >> 3, rr = lane & 7;
              const int tok = 8 * (mi & 1) + rr;
              const uint32_t addr = sbase + tok * kBfRow + (2 * jp + (mi >> 1)) * 16;
              uint32_t v0, v1, v2, v3;
              ldmatrix_x4_trans(addr, v0, v1, v2, v3);
              mma_bf16(stt.o[2 * jp], ah0, al0, ah1, al1, v0, v1);
              mma_bf16(stt.o[2 * jp + 1], ah0, al0, ah1, al1, v2, v3);
            }
          }
        } else if (vmask && alive) {
          // ---- quantized stage: tiles [i0, i0 + n), walked in smem ----
          const int qs = j - 2 * wp.nbf_w;
          const long long i0 = wp.q0 + (long long)qs * tps;
          const int n = (int)min((long long)tps, (long long)(wp.q0 + wp.nq_w) - i0);
          int walk = kHdr;  // smem offset of the next tile (headers inline at record starts)
          bool a_ready = false;
          for (int k = 0; k < n; k += kChunk) {
            float sig[kChunk * 4];
            int toff[kChunk];
            float smax = s_v8;
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
              const int kk = k + tt;
              const long long i = i0 + kk;
              int hoff = 0;
              toff[tt] = -1;
              if (kk < n) {
                if (F::kInt && (i % L.tpg) == 0) {
                  hoff = walk;
                  walk += L.hdr_bytes;
                }
                toff[tt] = walk;
                walk += L.tile_bytes;
              }
              const bool present = kk < n && ((vmask >> kk) & 1u);
              if (!present) toff[tt] = -1;
              if (present) {
                if constexpr (F::kInt) {
                  // the group's A operand (q * s, hi/lo) lives in the warp's shared scratch between chunks
                  uint4* afr = reinterpret_cast<uint4*>(my_scratch) + lane;  // word i of lane at [i][lane]
                  if ((i % L.tpg) == 0 || (qs == 0 && kk == 0)) {
                    build_a_int<FMT>(qrow, reinterpret_cast<const float*>(stg + hoff),
                                     reinterpret_cast<const float*>(stg + hoff + 512), q, p.scale_log2, A, kfac,
                                     cterm);
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) afr[32 * i2] = make_uint4(A[i2][0], A[i2][1], A[i2][2], A[i2][3]);
                    a_ready = true;
                  } else if (!a_ready || tt == 0) {
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) {
                      const uint4 v = afr[32 * i2];
                      A[i2][0] = v.x; A[i2][1] = v.y; A[i2][2] = v.z; A[i2][3] = v.w;
                    }
                    a_ready = true;
                  }
                }
                const uint8_t* tile = stg + toff[tt];
                float acc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                  for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
                  uint32_t R[16];
                  unpack_k<FMT>(tile + (nt * 8 + r) * F::kRB + q * F::kKChunk, R);
#pragma unroll
                  for (int s2 = 0; s2 < 8; ++s2)
                    mma_f16(acc[nt], A[s2][0], A[s2][1], A[s2][2], A[s2][3], R[2 * s2], R[2 * s2 + 1]);
                }
                const int tok_valid = (int)min(16LL, (long long)sg.qn - i * 16);  // < 16 only for a partial FP8 tile
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int nt = e >> 1, c = e & 1;
                  const float dot = acc[nt][c] + acc[nt][c + 2];
                  const int t = nt * 8 + 2 * q + c;
                  sig[tt * 4 + e] = (t < tok_valid) ? fmaf(dot, kfac, cterm) : -INFINITY;
                }
                if constexpr (F::kInt) {
                  const float* vsp = reinterpret_cast<const float*>(tile + 32 * F::kRB);
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int t = (e >> 1) * 8 + 2 * q + (e & 1);
#pragma unroll
                    for (int jg = 0; jg < NGV; ++jg) smax = fmaxf(smax, vsp[t * NGV + jg]);
                  }
                }
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) sig[tt * 4 + e] = -INFINITY;
              }
            }
            float pr[kChunk * 4];
            const float inv_s = softmax_step<NGV, kChunk * 4>(stt, sig, smax, pr);
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
              if (toff[tt] < 0) continue;
              const long long i = i0 + k + tt;
              const uint8_t* tile = stg + toff[tt];
              uint32_t W[F::kVChunk / 4];
              {
                const uint4* vp = reinterpret_cast<const uint4*>(tile + F::kTile + lane * F::kVChunk);
#pragma unroll
                for (int i2 = 0; i2 < F::kVChunk / 16; ++i2) {
                  const uint4 v = vp[i2];
                  W[4 * i2] = v.x; W[4 * i2 + 1] = v.y; W[4 * i2 + 2] = v.z; W[4 * i2 + 3] = v.w;
                }
              }
              if constexpr (F::kFp8) {
                const int tok_valid = (int)min(16LL, (long long)sg.qn - i * 16);
                if (tok_valid < 16) {
                  // partial tile: bytes past the end may be stale; zero the lane's invalid tokens (byte e = token e)
                  const bool v0 = 2 * q < tok_valid, v1 = 2 * q + 1 < tok_valid;
                  const bool v2 = 8 + 2 * q < tok_valid, v3 = 9 + 2 * q < tok_valid;
                  const uint32_t mk =
                      (v0 ? 0xFFu : 0u) | (v1 ? 0xFF00u : 0u) | (v2 ? 0xFF0000u : 0u) | (v3 ? 0xFF000000u : 0u);
#pragma unroll
                  for (int i2 = 0; i2 < F::kVChunk / 4; ++i2) W[i2] &= mk;
                }
                uint32_t ah0, al0, ah1, al1;
                const float f = s_v8 * inv_s;
                split_f16(pr[tt * 4 + 0] * f, pr[tt * 4 + 1] * f, ah0, al0);
                split_f16(pr[tt * 4 + 2] * f, pr[tt * 4 + 3] * f, ah1, al1);
#pragma unroll
                for (int jt = 0; jt < 16; ++jt) {
                  uint32_t b01, b23;
                  switch (jt) {
#define KVQ_V(J) case J: unpack_v<FMT, J>(W, b01, b23); break;
                    KVQ_V(0) KVQ_V(1) KVQ_V(2) KVQ_V(3) KVQ_V(4) KVQ_V(5) KVQ_V(6) KVQ_V(7)
                    KVQ_V(8) KVQ_V(9) KVQ_V(10) KVQ_V(11) KVQ_V(12) KVQ_V(13) KVQ_V(14) KVQ_V(15)
                  }
                  mma_f16(stt.o[jt], ah0, al0, ah1, al1, b01, b23);
                }
              } else {
                constexpr int kTilesPerGroup = 16 / NGV;  // n-tiles of 8 channels per Value group
                constexpr float kH = (float)F::kHalf;
                const float* vsp = reinterpret_cast<const float*>(tile + 32 * F::kRB);
                const float* vzp = vsp + 16 * NGV;
#pragma unroll
                for (int jg = 0; jg < NGV; ++jg) {
                  float w[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int t = (e >> 1) * 8 + 2 * q + (e & 1);
                    w[e] = (vsp[t * NGV + jg] * inv_s) * pr[tt * 4 + e];
                    stt.zacc[jg] = fmaf(w[e], kH - vzp[t * NGV + jg], stt.zacc[jg]);
                  }
                  uint32_t ah0, al0, ah1, al1;
                  split_f16(w[0], w[1], ah0, al0);
                  split_f16(w[2], w[3], ah1, al1);
#pragma unroll
                  for (int jj = 0; jj < kTilesPerGroup; ++jj) {
                    uint32_t b01, b23;
                    switch (jg * kTilesPerGroup + jj) {
                      KVQ_V(0) KVQ_V(1) KVQ_V(2) KVQ_V(3) KVQ_V(4) KVQ_V(5) KVQ_V(6) KVQ_V(7)
                      KVQ_V(8) KVQ_V(9) KVQ_V(10) KVQ_V(11) KVQ_V(12) KVQ_V(13) KVQ_V(14) KVQ_V(15)
#undef KVQ_V
                    }
                    mma_f16(stt.o[jg * kTilesPerGroup + jj], ah0, al0, ah1, al1, b01, b23);
                  }
                }
              }
            }
          }
        }
        __syncwarp();
        ++n_consumed;
        while (alive && n_issued - n_consumed < nst && ps < nseg) issue_next();
      }

      // ---- finalise the warp's state and publish it ----
      float l = stt.l;
      l += __shfl_xor_sync(kFull, l, 1);
      l += __shfl_xor_sync(kFull, l, 2);
      float zs[NGV];
#pragma unroll
      for (int jg = 0; jg < NGV; ++jg) {
        float z = stt.zacc[jg];
        z += __shfl_xor_sync(kFull, z, 1);
        z += __shfl_xor_sync(kFull, z, 2);
        zs[jg] = z;
      }
      __syncwarp();
      float* rec = reinterpret_cast<float*>(my_scratch);
      if (r < g) {
        const float unit = stt.S / kPrescale;
        float* rr = rec + r * kMergeStride;
        if (q == 0) {
          rr[0] = stt.m;
          rr[1] = l;
        }
#pragma unroll
        for (int jt = 0; jt < 16; ++jt) {
          const float z = F::kInt ? zs[jt / (16 / NGV)] : 0.f;
          float2 v;
          v.x = (stt.o[jt][0] + stt.o[jt][2] + z) * unit;
          v.y = (stt.o[jt][1] + stt.o[jt][3] + z) * unit;
          if (stt.m == -INFINITY) v.x = v.y = 0.f;
          *reinterpret_cast<float2*>(rr + 4 + jt * 8 + 2 * q) = v;
        }
      }
      __syncthreads();
      // ---- merge the warps; write the partial of (b, h), or the result when this CTA owns the pair ----
      {
        const int b = sg.b, h = sg.h;
        const long long pair = (long long)b * H + h;
        const long long slot = (long long)blockIdx.x + pair;
        const long long P0 = sg.pair_start, P1 = sg.pair_start + sg.units;
        const long long c_lo = ((P0 + 1) * C - 1) / U, c_hi = (P1 * C - 1) / U;
        const bool whole = p.fuse && c_lo == c_hi;  // no other CTA touches this pair
        const float* recs = reinterpret_cast<const float*>(scratch);
        for (int i = tid; i < g * 128; i += kThreads) {
          const int hr = i >> 7, c = i & 127;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kNW; ++w) M = fmaxf(M, recs[w * (p.warp_scratch / 4) + hr * kMergeStride]);
          float Lsum = 0.f, O = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
              const float* rw = recs + w * (p.warp_scratch / 4) + hr * kMergeStride;
              const float f = exp2f(rw[0] - M);  // 0 for an empty warp (m = -inf)
              Lsum = fmaf(rw[1], f, Lsum);
              O = fmaf(rw[4 + c], f, O);
            }
          }
          const bool empty = !(Lsum > 0.f);
          const float o = empty ? 0.f : O / Lsum;
          const float l2 = empty ? -INFINITY : M + log2f(Lsum);
          if (whole) {
            write_out(p, b, h * g + hr, c, o, l2);
          } else {
            p.ws_o[(slot * g + hr) * 128 + c] = o;
            if (c == 0) p.ws_lse[slot * g + hr] = l2;
          }
        }
        if (p.fuse && !whole) {
          // the last CTA to finish this pair merges every partial of it
          __shared__ int last_flag, n_act;
          __shared__ int act[kMaxParts];
          __threadfence();
          __syncthreads();
          if (tid == 0) {
            const int nparts = active_ctas(c_lo, c_hi, U, C, act, kMaxParts);
            const unsigned old = atomicAdd(&p.counters[pair], 1u);
            last_flag = (old + 1u == (unsigned)nparts);
            if (last_flag) p.counters[pair] = 0u;  // ready for the next call
            n_act = nparts;
          }
          __syncthreads();
          if (last_flag) {
            __threadfence();
            const int na = n_act;
            for (int i = tid; i < g * 128; i += kThreads) {
              const int hr = i >> 7, c = i & 127;
              float M = -INFINITY, Lsum = 0.f, O = 0.f;
              if (na <= kMaxParts) {
                for (int k2 = 0; k2 < na; ++k2) M = fmaxf(M, __ldcg(&p.ws_lse[((long long)act[k2] + pair) * g + hr]));
                if (M != -INFINITY) {
                  for (int k2 = 0; k2 < na; ++k2) {
                    const long long sl = (long long)act[k2] + pair;
                    const float f = exp2f(__ldcg(&p.ws_lse[sl * g + hr]) - M);
                    Lsum += f;
                    O = fmaf(f, __ldcg(&p.ws_o[(sl * g + hr) * 128 + c]), O);
                  }
                }
              } else {
                // more partials than the list holds (tiny per-CTA ranges): walk [c_lo, c_hi]
                for (long long cc = c_lo; cc <= c_hi; ++cc)
                  if ((cc * U) / C != ((cc + 1) * U) / C) M = fmaxf(M, __ldcg(&p.ws_lse[(cc + pair) * g + hr]));
                if (M != -INFINITY) {
                  for (long long cc = c_lo; cc <= c_hi; ++cc) {
                    if ((cc * U) / C == ((cc + 1) * U) / C) continue;
                    const float f = exp2f(__ldcg(&p.ws_lse[(cc + pair) * g + hr]) - M);
                    Lsum += f;
                    O = fmaf(f, __ldcg(&p.ws_o[((cc + pair) * g + hr) * 128 + c]), O);
                  }
                }
              }
              const bool empty = !(Lsum > 0.f);
              write_out(p, b, h * g + hr, c, empty ? 0.f : O / Lsum, empty ? -INFINITY : M + log2f(Lsum));
            }
          }
        }
        if (s + 1 < nseg) load_q(segs[s + 1]);
      }
      __syncthreads();
    }
    // drain copies still in flight after a timeout (bounded)
    if (pending) {
      for (int sl = 0; sl < nst; ++sl)
        if ((pending >> sl) & 1u) {
          mbar_wait_bounded(smem_addr(&my_bars[sl]), (phase_bits >> sl) & 1u, kWaitLimitCycles);
          phase_bits ^= 1u << sl;
        }
      pending = 0;
    }
    pos = batch_end;
  }
}

// Raise the kernel's dynamic shared-memory limit on the current device once per
// size (the attribute is per device and persists; repeated calls are skipped).
template <int FMT, int NGV>
cudaError_t ensure_smem_attr(int smem) {
  static std::mutex mu;
  static int set_for[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && set_for[dev] >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_kernel<FMT, NGV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) set_for[dev] = smem;
  return e;
}

template <int FMT, int NGV>
cudaError_t launch_decode_t(const DecodeParams& p, int smem, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr<FMT, NGV>(smem);
  if (e != cudaSuccess) return e;
  decode_kernel<FMT, NGV><<<p.num_ctas, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int FMT, int NGV>
cudaError_t occupancy_t(int smem, int* n) {
  cudaError_t e = ensure_smem_attr<FMT, NGV>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, decode_kernel<FMT, NGV>, kThreads, smem);
}

}  // namespace kvq
