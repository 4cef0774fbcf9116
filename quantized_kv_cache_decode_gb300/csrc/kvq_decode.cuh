// Fused decode attention over a quantized KV cache (sm_103a).
//
// softmax(q K^T / sqrt(d)) V for the new query (or queries) of each head, reading the compressed
// cache once ("W4A16 + KV cache quantization combined accuracy", section
// "오차가 어디서 만나는가"; dequantization fused with the matmuls as "KV Cache
// Quantization Analysis" section 5 asks, since decode is bound by reading the
// cache, section 1).
//
// Work decomposition.  Every (sequence, kv head) pair is a list of work units:
// its 16-token bf16 tiles (sink + residual window, charged `bf_weight` units
// each) followed by its 16-token quantized tiles (1 unit each).  The pairs'
// lists are concatenated and cut into equal ranges, one per working CTA, so every
// CTA moves the same number of bytes whatever the sequence lengths; when every
// sequence holds the same number of units, each working CTA takes whole pairs
// instead (range_ctas).  A CTA writes one partial (normalised output +
// log-sum-exp) per pair it shares with another CTA; the last CTA to finish such
// a pair merges them.
//
// Inside a CTA the warps (12; 8 for 8-bit codes) take a segment's work items (a
// bf16 tile, or whole records of quantized tiles) round robin, interleaved over
// the whole segment, and run their own two-stage pipelines: a warp streams
// stages (tiles with their scales and Key-group headers) into shared memory with
// bulk asynchronous copies (cp.async.bulk, TMA engine; in the paged one-tile
// case every lane copies one record) completing on per-stage mbarriers, a stage
// ahead of the compute.  Every lane keeps the same producer cursor, so the slots'
// tags live in registers.
//
// Tensor-core mapping (mma.sync m16n8k16, fp32 accumulate), query rows: the A
// operand is the query side -- row r (r < 8) the high f16 half, row r + 8 the
// low half of x_c = q_c s_c kappa of query column r (s_c the Key group's
// per-channel scale, kappa a power of two) -- and the B operand the Key codes
// themselves, in their stored fragment order, as f16 values (subnormal
// placement for 8-bit codes, centred values for 2- and 4-bit ones).  The scores
// of column r land in lane (r, q) for tokens 2q, 2q + 1, 2q + 8, 2q + 9: the
// layout of the PV B operand, so the online softmax needs no shuffles.  PV: A =
// the Value codes (V^T fragment order, subnormal placement), B = W = p s_V (one
// f16 term); the zero-point sums are kept in fp32 with the rounded weights.
// With at most four query columns (one query token) the Key tile is the A
// operand and the query the B operand instead (qk_tile_ka: half the MMAs);
// pre-RoPE Keys take that form too (qk_tile_rope).  bf16 tiles: the same
// layouts with ldmatrix loads.  The codes are stored in an A operand's register
// order (include/kvq.h, "fragment order"): each lane loads its words with
// conflict-free 16-byte loads and unpacks them in registers.
#pragma once

#include <mutex>

#include "kvq_common.cuh"

namespace kvq {

// Warps per CTA (one CTA per SM at most): 12 (168 registers a thread; with 16
// warps and 128 registers the integer variants spill), 8 for 8-bit codes;
// decode_warps() in kvq_internal.h states the same for the host.
template <int FMT>
struct DecodeWarps {
  // 8-bit codes: 8 warps of up to 255 registers (measured on GB300: the paged INT8 layers
  // 643 -> 600 us; the 2/4-bit and FP8 layers are faster with 12)
  static constexpr int kNW = FMT == 8 ? 8 : 12;
  static constexpr int kThreads = kNW * 32;
};
constexpr int kMaxStages = 2;
constexpr float kPrescale = 64.f;      // w = p * (s / S_ref) * 64 < 2^14: f16 range is safe
constexpr float kTau = 6.f;            // score max may exceed its reference by 2^6 before a rescale
constexpr float kSTau = 4.f;           // a Value scale may exceed its reference 4x before a rescale
// floats per query column in shared memory (128 + 16 pad): the 16-byte loads of the
// operand builds (column r, channels 16s + 4q ..) of the 8 lanes of a load phase
// (two columns) fall in different banks
constexpr int kQRow = 144;
// A bf16 half tile in a stage: 16 rows of 256 bytes, the 16-byte chunk c of row r
// stored at chunk c ^ (r & 7), so that the 8 rows an ldmatrix reads at one chunk
// fall in 8 different bank groups.
constexpr int kBfHalf = 16 * 256;
__host__ __device__ constexpr int bf_chunk_off(int row, int chunk) { return row * 256 + ((chunk ^ (row & 7)) << 4); }
constexpr int kMergeStride = 132;      // floats per head in a warp's merge record: m, l, -, -, o[128]
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
  static constexpr bool kFp8 = FMT == 16 || FMT == 17;  // E4M3, E5M2
  static constexpr bool kInt = !kFp8;
  static constexpr int kBits = kFp8 ? 8 : FMT;
  static constexpr int kRB = 128 * kBits / 8;   // bytes of one token row of codes
  static constexpr int kTile = 16 * kRB;        // bytes of the 16 x 128 code matrix
  static constexpr int kWords = kRB / 8;        // operand words of one lane per code matrix
  static constexpr int kHalf = kFp8 ? 0 : (1 << (kBits - 1));
  // Integer codes can enter the MMAs as f16 subnormals: a b-bit field placed in the
  // low mantissa bits is exactly field * 2^-24 (one logic operation per two codes,
  // no centring; the zero-points are applied in fp32 afterwards).  Fields above bit
  // 0 carry a power-of-two factor, compensated where it lands (Value codes):
  //   kVHi  the PV product of channels 16mb + 8 .. 15 (rows r + 8) relative to rows r
  //   kW1   multiplier of the PV weights of tokens 8-15 (INT2: registers 2, 3 carry 16x
  //         the factor of registers 0, 1)
  // kKRaw: the Key codes take the subnormal path (else centred normal f16 values,
  // code - 2^(b-1), with the zero-point term sum_c x_c (2^(b-1) - z_c)).  Measured on
  // GB300: with 2- and 4-bit codes as subnormal B operands the QK sums lose precision
  // (lse errors up to 2e-4 for INT2, 2e-5 for INT4, against 1e-6 with centred
  // values); 8-bit codes keep it (3e-6), so only they take the cheaper path.  The
  // Value codes (PV) take it for every width: the output error stays at its level.
  static constexpr bool kKRaw = FMT == 8;
  static constexpr float kVHi = FMT == 4 ? 16.f : FMT == 2 ? 4.f : 1.f;
  static constexpr float kW1 = FMT == 2 ? 0.0625f : 1.f;
};
constexpr float kCodeUnit = 16777216.f;  // 2^24: a subnormal-placed code n reads as n * 2^-24

// --------------------------------------------------------------------------
// operand unpacking: packed codes -> centred f16 pairs (exact)
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
// bytes 0, 2 (sel 0x7170) or 1, 3 (sel 0x7371) of w under the f16 exponent byte 0x64, minus 1152 -> (n - 128)
template <uint32_t SEL>
__device__ __forceinline__ uint32_t int8_pair(uint32_t w) {
  uint32_t t;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(w), "r"(0x64646464u), "n"(SEL));
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(dup16(f16_bits_of_int(1152))));
  return d;
}

// The lane's operand words of one code matrix (fragment order): kWords words,
// word w at byte ((w >> 2) * 32 + lane) * 16 + (w & 3) * 4.
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* base, int lane, uint32_t (&W)[N]) {
  const uint4* p = reinterpret_cast<const uint4*>(base) + lane;
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const uint4 v = p[32 * j];
    W[4 * j] = v.x;
    W[4 * j + 1] = v.y;
    W[4 * j + 2] = v.z;
    W[4 * j + 3] = v.w;
  }
}

// Fragment registers of step s (a compile-time constant after unrolling): reg 0 =
// (row r, columns 2q, 2q + 1), reg 1 = (row r + 8, ...), reg 2 = (row r, columns
// 2q + 8, 2q + 9), reg 3 = (row r + 8, ...) of the stored 16 x 16 code block.
template <int FMT, int N>
__device__ __forceinline__ void unpack_a(const uint32_t (&W)[N], int s, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                         uint32_t& a3) {
  if constexpr (FMT == 4) {
    const uint32_t w = W[s], w8 = w >> 8;
    a0 = int4_lo(w);
    a1 = int4_hi(w);
    a2 = int4_lo(w8);
    a3 = int4_hi(w8);
  } else if constexpr (FMT == 2) {
    const uint32_t w = (s & 1) ? (W[s >> 1] >> 8) : W[s >> 1];
    a0 = int2_pair<0>(w);
    a1 = int2_pair<1>(w);
    a2 = int2_pair<2>(w);
    a3 = int2_pair<3>(w);
  } else if constexpr (FMT == 8) {
    a0 = int8_pair<0x7270>(W[2 * s]);
    a1 = int8_pair<0x7371>(W[2 * s]);
    a2 = int8_pair<0x7270>(W[2 * s + 1]);
    a3 = int8_pair<0x7371>(W[2 * s + 1]);
  } else if constexpr (FMT == 17) {  // FP8 E5M2
    e5m2x4_to_f16x4(W[2 * s], a0, a1);
    e5m2x4_to_f16x4(W[2 * s + 1], a2, a3);
  } else {  // FP8 E4M3
    e4m3x4_to_f16x4(W[2 * s], a0, a1);
    e4m3x4_to_f16x4(W[2 * s + 1], a2, a3);
  }
}

// Integer codes of step s as f16 subnormals (fields in the low mantissa bits), in
// the same register order as unpack_a; the power-of-two factors of the fields
// above bit 0 are listed in FT.  FP8 codes: unpack_a.
template <int FMT, int N>
__device__ __forceinline__ void unpack_raw(const uint32_t (&W)[N], int s, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                           uint32_t& a3) {
  if constexpr (FMT == 4) {  // nibbles 0, 4 of each half (x1, x16); then the byte above them
    const uint32_t w = W[s], w8 = w >> 8;
    a0 = w & 0x000F000Fu;
    a1 = w & 0x00F000F0u;
    a2 = w8 & 0x000F000Fu;
    a3 = w8 & 0x00F000F0u;
  } else if constexpr (FMT == 2) {  // 2-bit fields at bits 0, 2, 4, 6 of each half (x1, x4, x16, x64)
    const uint32_t w = (s & 1) ? (W[s >> 1] >> 8) : W[s >> 1];
    a0 = w & 0x00030003u;
    a1 = w & 0x000C000Cu;
    a2 = w & 0x00300030u;
    a3 = w & 0x00C000C0u;
  } else if constexpr (FMT == 8) {  // bytes 0, 2 and bytes 1, 3 (moved down by a byte permute)
    const uint32_t w0 = W[2 * s], w1 = W[2 * s + 1];
    a0 = w0 & 0x00FF00FFu;
    asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(a1) : "r"(w0));
    a2 = w1 & 0x00FF00FFu;
    asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(a3) : "r"(w1));
  } else {
    unpack_a<FMT>(W, s, a0, a1, a2, a3);
  }
}

// 2^k with k chosen from the exponent of bound (> 0): bound * 2^k < 2^14 (at least
// 2^13 for a normal bound), so every |x| <= bound scaled by it fits f16 with room;
// inv = 2^-k.  No division: exponent arithmetic only (k within [-126, 102]).
__device__ __forceinline__ float pow2_fit_f16(float bound, float& inv) {
  const int eb = (__float_as_int(bound) >> 23) & 0xFF;  // biased exponent
  const int ek = max(25, min(253, 267 - eb));           // biased exponent of 2^k = 2^(13 - (eb - 127))
  inv = __int_as_float((254 - ek) << 23);
  return __int_as_float(ek << 23);
}

// NGV consecutive floats (a token's Value scales or zero-points of all groups)
template <int NGV>
__device__ __forceinline__ void load_row(const float* p, float (&v)[NGV]) {
  if constexpr (NGV == 1) {
    v[0] = p[0];
  } else if constexpr (NGV == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    v[0] = a.x;
    v[1] = a.y;
  } else {
#pragma unroll
    for (int j = 0; j < NGV / 4; ++j) {
      const float4 a = reinterpret_cast<const float4*>(p)[j];
      v[4 * j] = a.x;
      v[4 * j + 1] = a.y;
      v[4 * j + 2] = a.z;
      v[4 * j + 3] = a.w;
    }
  }
}

// --------------------------------------------------------------------------
// per-warp online-softmax state
// --------------------------------------------------------------------------
// Score layout: lane (r, q) holds query column r for tokens 2q, 2q + 1, 2q + 8,
// 2q + 9 of a tile -- which is also the B-operand (W) layout of the PV product.
// Output layout: lane (r, q) holds columns 2q and 2q + 1 of channels 16 mb + r and
// 16 mb + r + 8 (mb = 0..7).
template <int NGV>
struct WarpState {
  float o[8][4];     // PV accumulators (output layout): [mb][0/1] = channel 16mb+r, columns 2q / 2q+1;
                     // [mb][2/3] = channel 16mb+r+8
  float zacc[NGV];   // zero-point sums per Value group of column r, lane-partial
  float m;           // reference max of column r (log2 domain), the same in the row's four lanes
  float l;           // sum of p of column r, lane-partial
  float S;           // reference Value scale (warp-uniform: Value scales do not depend on the column)
  float inv_S;       // 1 / S
};

template <int NGV>
__device__ __forceinline__ void state_init(WarpState<NGV>& st) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
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

// One softmax step over a tile: sig[e] are the scores (log2 domain, -inf when
// masked) of the lane's four tokens for column r; smax is the largest Value scale
// among the lane's tokens (warp-uniform already when kVarS is false).  The
// references m (per column) and S move only when a score exceeds m by 2^kTau or a
// scale exceeds S by kSTau -- each lane checks its own values and the warp votes;
// only then are the maxima reduced over the lanes and every accumulator
// rescaled.  Returns p = 2^(sig - m).
template <int NGV, bool kVarS>
__device__ __forceinline__ void softmax_tile(WarpState<NGV>& st, const float (&sig)[4], float smax, int q,
                                             float (&pr)[4], float* sp_row = nullptr) {
  const float mx = fmaxf(fmaxf(sig[0], sig[1]), fmaxf(sig[2], sig[3]));
  const bool bump = (smax > st.S * kSTau) || (mx > st.m + kTau);
  if (__any_sync(kFull, bump)) {
    float t = mx;  // the column's largest score in the tile: reduce over the row's token lanes q
    t = fmaxf(t, __shfl_xor_sync(kFull, t, 1));
    t = fmaxf(t, __shfl_xor_sync(kFull, t, 2));
    const float mn = t > st.m + kTau ? t : st.m;
    const float alpha = (st.m == -INFINITY) ? 0.f : fast_exp2(st.m - mn);
    st.m = mn;
    st.l *= alpha;
    if constexpr (kVarS) {  // per-token Value scales: the tile's largest over the token lanes q
      smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, 1));
      smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, 2));
    }
    const float S_new = smax > st.S * kSTau ? smax : st.S;
    const float ratio = S_new > 0.f ? st.S / S_new : 0.f;
    // output layout: columns 2q, 2q + 1 live in the score lanes of rows 2q, 2q + 1
    const float a0 = __shfl_sync(kFull, alpha, 8 * q) * ratio, a1 = __shfl_sync(kFull, alpha, 8 * q + 4) * ratio;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      st.o[mb][0] *= a0;
      st.o[mb][2] *= a0;
      st.o[mb][1] *= a1;
      st.o[mb][3] *= a1;
    }
#pragma unroll
    for (int j = 0; j < NGV; ++j) st.zacc[j] *= alpha * ratio;
    st.S = S_new;
    st.inv_S = 1.f / S_new;
    if (sp_row) {  // dense-and-sparse: the column's sparse Value sums (lane q: channels 32q .. 32q + 31)
      float4* p4 = reinterpret_cast<float4*>(sp_row + 32 * q);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 v = p4[i];
        v.x *= alpha;
        v.y *= alpha;
        v.z *= alpha;
        v.w *= alpha;
        p4[i] = v;
      }
      __syncwarp();
    }
  }
  // ex2(-inf) = +0 for masked scores; the reference is -inf only while every score seen
  // so far (this tile's included) is -inf, then 0 stands in for it
  const float ms = st.m == -INFINITY ? 0.f : st.m;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    pr[e] = fast_exp2(sig[e] - ms);
    st.l += pr[e];
  }
}

// --------------------------------------------------------------------------
// the query-side A operand of the quantized tiles
// --------------------------------------------------------------------------
// Row r of the 16-row A operand is query column r (high f16 half), row r + 8 the
// same column's low half; its K index follows the Key codes' fragment order
// (channel 16s + 4q + e at K index 2q + (e & 1) + 8 (e >> 1)), so lane (r, q)
// holds, per step s, X[s][0] = hi(x_c) and X[s][1] = lo(x_c) of channels
// 16s + 4q, +1, and X[s][2], X[s][3] the same of channels 16s + 4q + 2, +3.  The
// lane computes each of its 32 products once and keeps both halves.
// qrow: the column's query row in shared memory (a zero row for absent columns).

// FP8 layers (one build per segment): x_c = q_c kappa, kappa the power of two that
// brings max_c |q_c| into [2^13, 2^14); kfac (the score multiplier) = kfac0 / kappa,
// kfac0 = log2(e) / sqrt(d) * the Key scale.
__device__ __forceinline__ void build_x_fp8(const float* qrow, int q, float kfac0, uint32_t (&X)[8][4],
                                            float& kfac) {
  float mx = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 16 * s + 4 * q);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
  }
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  float inv;
  const float kap = pow2_fit_f16(mx, inv);
  const float2 k2 = make_float2(kap, kap);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 16 * s + 4 * q);
    split_f16x2(mul_f32x2(make_float2(x.x, x.y), k2), X[s][0], X[s][1]);
    split_f16x2(mul_f32x2(make_float2(x.z, x.w), k2), X[s][2], X[s][3]);
  }
  kfac = kfac0 * inv;
}

// Max |q_c| of the lane's column (lane q reads channels 32q .. 32q + 31; the four lanes of a row combine).
__device__ __forceinline__ float column_qmax(const float* qrow, int q) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 32 * q + 4 * j);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
  }
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
  return fmaxf(m, __shfl_xor_sync(kFull, m, 2));
}

// A Key group of an INT layer: x_c = q_c s_c (s_c: the Key scale of channel c),
// with the zero-point term sum_c x_c z_c, in one pass over the channels: kappa,
// the power of two that brings max_c |q_c| * max_c s_c into [2^13, 2^14), bounds
// |x_c kappa| by 2^14 without first finding max_c |x_c| (qm: the column's max
// |q_c|, per segment).  A smaller kappa than the exact one only moves the hi/lo
// split: the two f16 terms still hold x_c kappa to about 22 bits, or to the f16
// subnormal step (2^-24, against elements up to 2^14 times the bound ratio) for
// tiny x_c.  The codes are read as subnormals (n * 2^-24), so the score of a
// token is (D * 2^24 / kappa - sum_c x_c z_c) * kfac0: kfac and cterm return those
// two factors (centred codes: D / kappa and z_c - 2^(b-1) in place of z_c).
template <int FMT, bool SCALE>
__device__ __forceinline__ void build_x_pass(const float* qrow, const float* ks, const float* kz, int q, float kap,
                                             uint32_t (&X)[8][4], float2& cz) {
  using F = FT<FMT>;
  constexpr float zh = F::kKRaw ? 0.f : (float)F::kHalf;
  const float2 k2 = make_float2(kap, kap);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 16 * s + 4 * q);
    const float4 s4 = *reinterpret_cast<const float4*>(ks + 16 * s + 4 * q);
    const float4 z4 = *reinterpret_cast<const float4*>(kz + 16 * s + 4 * q);
    float2 x01 = mul_f32x2(make_float2(x.x, x.y), make_float2(s4.x, s4.y));
    float2 x23 = mul_f32x2(make_float2(x.z, x.w), make_float2(s4.z, s4.w));
    cz = fma_f32x2(x01, make_float2(z4.x - zh, z4.y - zh), cz);
    cz = fma_f32x2(x23, make_float2(z4.z - zh, z4.w - zh), cz);
    if constexpr (SCALE) {
      x01 = mul_f32x2(x01, k2);
      x23 = mul_f32x2(x23, k2);
    }
    split_f16x2(x01, X[s][0], X[s][1]);
    split_f16x2(x23, X[s][2], X[s][3]);
    asm volatile("" ::: "memory");  // one step's loads at a time: keeps the build's registers few
  }
}

template <int FMT>
__device__ __forceinline__ void build_x_group(const float* qrow, const float* ks, const float* kz, int lane, int q,
                                              float kfac0, float qm, uint32_t (&X)[8][4], float& kfac,
                                              float& cterm) {
  using F = FT<FMT>;
  // the largest Key scale of the group (scales are positive)
  float sm;
  {
    const float4 a = *reinterpret_cast<const float4*>(ks + 4 * lane);
    sm = fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm = fmaxf(sm, __shfl_xor_sync(kFull, sm, o));
  }
  float2 cz = make_float2(0.f, 0.f);
  float inv;
  const float kap = pow2_fit_f16(qm * sm, inv);
  build_x_pass<FMT, true>(qrow, ks, kz, q, kap, X, cz);
  float c = cz.x + cz.y;
  c += __shfl_xor_sync(kFull, c, 1);
  c += __shfl_xor_sync(kFull, c, 2);
  kfac = kfac0 * (F::kKRaw ? inv * kCodeUnit : inv);
  cterm = -kfac0 * c;  // score = (D * kfac) + cterm
}

// Raw scores of one quantized tile for the lane's column: d[0..3] = tokens 2q, 2q + 1,
// 2q + 8, 2q + 9.  Two MMAs per step: tokens 0-7 (Key fragment registers 0, 2 as
// the B operand) and tokens 8-15 (registers 1, 3); D row r holds the high-half
// product of column r, row r + 8 the low-half one.  Even and odd steps accumulate
// apart (four independent MMA chains).  8-bit integer codes are the
// subnormal-placed ones (FT::kKRaw), narrower ones centred.
template <int FMT>
__device__ __forceinline__ void qk_tile(const uint32_t (&KW)[FT<FMT>::kWords], const uint32_t (&X)[8][4],
                                        float (&d)[4]) {
  float lo[2][4] = {}, hi[2][4] = {};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t k0, k1, k2, k3;
    if constexpr (FT<FMT>::kKRaw) unpack_raw<FMT>(KW, s, k0, k1, k2, k3);
    else unpack_a<FMT>(KW, s, k0, k1, k2, k3);
    mma_f16(lo[s & 1], X[s][0], X[s][1], X[s][2], X[s][3], k0, k2);
    mma_f16(hi[s & 1], X[s][0], X[s][1], X[s][2], X[s][3], k1, k3);
  }
  d[0] = (lo[0][0] + lo[0][2]) + (lo[1][0] + lo[1][2]);
  d[1] = (lo[0][1] + lo[0][3]) + (lo[1][1] + lo[1][3]);
  d[2] = (hi[0][0] + hi[0][2]) + (hi[1][0] + hi[1][2]);
  d[3] = (hi[0][1] + hi[0][3]) + (hi[1][1] + hi[1][3]);
}

// PV of one quantized tile: o[mb] += V^T(channels 16mb..) * W(group of mb).  Integer
// codes are the subnormal-placed ones: rows r (channels 16mb + r) accumulate
// n * 2^-24 * W, rows r + 8 FT::kVHi times that (INT2: the weights of tokens 8-15
// carry FT::kW1).
template <int FMT, int NGV>
__device__ __forceinline__ void pv_tile(const uint32_t (&VW)[FT<FMT>::kWords], const uint32_t (&B0)[NGV],
                                        const uint32_t (&B1)[NGV], float (&o)[8][4]) {
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
    uint32_t a0, a1, a2, a3;
    unpack_raw<FMT>(VW, mb, a0, a1, a2, a3);
    mma_f16(o[mb], a0, a1, a2, a3, B0[mb * NGV / 8], B1[mb * NGV / 8]);
  }
}

// Few query columns (KA: at most 4 heads, one query token): the Key tile is the A
// operand (rows = tokens r, r + 8 of the lane, K index in the codes' fragment
// order) and the query side the B operand, whose column n holds head n / 2's high
// (n even) or low (n odd) f16 half.  The B fragment of lane (r, q) is column r at
// K indices 2q, 2q + 1, 2q + 8, 2q + 9, i.e. channels 16s + 4q .. 16s + 4q + 3 of
// head r / 2: the query-rows operand of that head (built by the same builders from
// its query row), one half of it.  ka_operand keeps the lane's half and moves the
// per-head score factors (kfac, cterm; built per head r / 2) to the column layout
// of the scores (column r = head r, taken from lane 8r).
__device__ __forceinline__ void ka_operand(uint32_t (&X)[8][4], int r, float& kfac, float& cterm) {
  const bool lo = (r & 1) != 0;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t b0 = lo ? X[s][1] : X[s][0], b1 = lo ? X[s][3] : X[s][2];
    X[s][0] = b0;
    X[s][1] = b1;
  }
  const int src = 8 * (r & 3);
  kfac = __shfl_sync(kFull, kfac, src);
  cterm = __shfl_sync(kFull, cterm, src);
}

// Raw scores of one quantized tile with the Key tile as the A operand (KA): one
// MMA per step (8 per tile, two chains); D(token, column) of lane (r, q) holds
// tokens r, r + 8 of head q, high and low halves in columns 2q, 2q + 1.  Four
// shuffles bring them to the query-rows layout of qk_tile (column r, tokens 2q,
// 2q + 1, 2q + 8, 2q + 9): token 2q's score sits in lane 8q + r, token 2q + 1's
// in lane 8q + 4 + r (columns r >= 4 read some lane's value; they are masked).
template <int FMT>
__device__ __forceinline__ void qk_tile_ka(const uint32_t (&KW)[FT<FMT>::kWords], const uint32_t (&X)[8][4],
                                           int lane, float (&d)[4]) {
  float acc[2][4] = {};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t a0, a1, a2, a3;
    if constexpr (FT<FMT>::kKRaw) unpack_raw<FMT>(KW, s, a0, a1, a2, a3);
    else unpack_a<FMT>(KW, s, a0, a1, a2, a3);
    mma_f16(acc[s & 1], a0, a1, a2, a3, X[s][0], X[s][1]);
  }
  const float t0 = (acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]);  // token r
  const float t8 = (acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]);  // token r + 8
  const int src = 8 * (lane & 3) + ((lane >> 2) & 3);
  d[0] = __shfl_sync(kFull, t0, src);
  d[1] = __shfl_sync(kFull, t0, src + 4);
  d[2] = __shfl_sync(kFull, t8, src);
  d[3] = __shfl_sync(kFull, t8, src + 4);
}

// One-token append folded into the decode (FP8 layers without sink tokens): the
// new token of (sequence b, kv head h) is token tt of quantized tile i, which one
// warp of the launch reads, from its staged copy `stile`.  That warp encodes the
// token as the append does (code = FP8(fl32(x / s)) with the tensor's scale s, at
// the token's positions in the fragment-order K and V parts) and writes the codes
// into the cache record, for later steps, and into the staged copy it is about to
// read.  A token that starts a tile clears both copies of the tile first, so the
// codes of tokens not yet written read as 0.  (Lane l encodes channels 4l .. 4l + 3.)
__device__ __forceinline__ void fp8_append_token(const DecodeParams& p, uint8_t* stile, int b, int h, long long i,
                                                 int tt, int lane) {
  const LayerDesc& L = p.L;
  const uint8_t* rec = record_addr(L, p.C, b, h, i / L.tpg, nullptr);
  if (!rec) return;  // a bad block: its tile was not copied either (reported by the producer)
  uint8_t* gtile = const_cast<uint8_t*>(tile_in_record(L, rec, i));
  constexpr int kCodeBytes = 2 * 16 * 128;  // K and V codes of a 16-token FP8 tile
  if (tt == 0) {
#pragma unroll
    for (int w = lane; w < kCodeBytes / 16; w += 32) {
      reinterpret_cast<uint4*>(stile)[w] = make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(gtile)[w] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
  }
  const long long pair = (long long)b * L.H + h;
  const uint2 kr = reinterpret_cast<const uint2*>(p.k_new)[pair * 32 + lane];
  const uint2 vr = reinterpret_cast<const uint2*>(p.v_new)[pair * 32 + lane];
  const float sk = __ldg(p.C.k_tscale), sv = __ldg(p.C.v_tscale);
  const float2 k01 = unpack_bf16(kr.x), k23 = unpack_bf16(kr.y), v01 = unpack_bf16(vr.x), v23 = unpack_bf16(vr.y);
  const float kx[4] = {k01.x, k01.y, k23.x, k23.y}, vx[4] = {v01.x, v01.y, v23.x, v23.y};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = 4 * lane + e;
    const float kd = __fdiv_rn(kx[e], sk), vd = __fdiv_rn(vx[e], sv);
    const uint8_t kc = L.e5m2 ? f32_to_e5m2(kd) : f32_to_e4m3(kd);
    const uint8_t vc = L.e5m2 ? f32_to_e5m2(vd) : f32_to_e4m3(vd);
    int byte, bit;
    ktile_pos(8, true, tt, c, byte, bit);
    stile[byte] = kc;
    gtile[byte] = kc;
    vtile_pos(8, true, tt, c, byte, bit);
    stile[16 * 128 + byte] = vc;
    gtile[16 * 128 + byte] = vc;
  }
  __syncwarp();
}

// Scores of a bf16 tile from its K rows in shared memory (rows past `rows` masked):
// the query column (bf16, exact) in A rows 0-7, rows 8-15 zero; the K rows as the B
// operand through ldmatrix (natural channel order).
__device__ __forceinline__ void bf16_qk(const uint8_t* stg, const float* qrow, int lane, int q, bool hv, int rows,
                                        float scale_log2, float (&sig)[4]) {
  // lane's row (lane & 7) + 8 ((lane >> 3) & 1), chunk 2s + (lane >> 4), swizzled:
  // (2s + h) ^ x = 2 (s ^ (x >> 1)) + (h ^ (x & 1)) with x = lane & 7
  const int x = lane & 7;
  const uint32_t lbase =
      smem_addr(stg) + ((lane & 7) + 8 * ((lane >> 3) & 1)) * 256 + 16 * ((lane >> 4) ^ (x & 1));
  float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    uint32_t k0, k1, k2, k3;
    ldmatrix_x4(lbase + 32 * (s ^ (x >> 1)), k0, k1, k2, k3);
    const float2 x0 = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * q);
    const float2 x1 = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * q + 8);
    const uint32_t a0 = pack_bf16(x0.x, x0.y), a2 = pack_bf16(x1.x, x1.y);
    mma_bf16(lo, a0, 0u, a2, 0u, k0, k2);
    mma_bf16(hi, a0, 0u, a2, 0u, k1, k3);
  }
  const int t0 = 2 * q;
  sig[0] = (hv && t0 < rows) ? lo[0] * scale_log2 : -INFINITY;
  sig[1] = (hv && t0 + 1 < rows) ? lo[1] * scale_log2 : -INFINITY;
  sig[2] = (hv && t0 + 8 < rows) ? hi[0] * scale_log2 : -INFINITY;
  sig[3] = (hv && t0 + 9 < rows) ? hi[1] * scale_log2 : -INFINITY;
}

// PV of a bf16 tile from its V rows (rows past the end zeroed); W = pt * f split
// into two bf16 terms.  RH: factor of rows r + 8 (so that the accumulators keep
// the scale the quantized tiles of the layer give them; f carries the rest).
template <int RH>
__device__ __forceinline__ void bf16_pv(const uint8_t* stg, int lane, const float (&pt)[4], float f,
                                        float (&o)[8][4]) {
  const int mi = lane >> 3, x = lane & 7;  // row (lane & 7) + 8 (mi >> 1), chunk 2 mb + (mi & 1), swizzled
  const uint32_t lbase = smem_addr(stg) + ((lane & 7) + 8 * (mi >> 1)) * 256 + 16 * ((mi & 1) ^ (x & 1));
  uint32_t h01, l01, h23, l23;
  split_bf16(pt[0] * f, pt[1] * f, h01, l01);
  split_bf16(pt[2] * f, pt[3] * f, h23, l23);
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
    uint32_t a0, a1, a2, a3;
    ldmatrix_x4_trans(lbase + 32 * (mb ^ (x >> 1)), a0, a1, a2, a3);
    if constexpr (RH != 1) {  // exact: a power of two on bf16 values
      constexpr uint32_t kRh = dup16((uint32_t)(127 + (RH == 16 ? 4 : 2)) << 7);  // bf16 bits of 16 or 4
      asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(a1) : "r"(kRh));
      asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(a3) : "r"(kRh));
    }
    mma_bf16(o[mb], a0, a1, a2, a3, h01, h23);
    mma_bf16(o[mb], a0, a1, a2, a3, l01, l23);
  }
}

// --------------------------------------------------------------------------
// pre-RoPE Keys: rotation at the Key's position inside the decode
// --------------------------------------------------------------------------
// Keys of a layer with rope_base > 0 are stored before the rotary embedding
// ("KV Cache Quantization Analysis", section 3, the RoPE bullet: the rotation
// mixes channel pairs and smears the per-channel outliers, so KVQuant quantizes
// Keys before it; section 4, KVQuant item (ii)).  The decode dequantizes each Key
// to fp32, turns channel pair (i, i + 64) by t * theta_i (t: the Key's position),
// and multiplies the rotated Key, split in two f16 terms, with the query (already
// rotated by the caller) on the tensor cores.  In the fragment order of the Key
// codes channel c and c + 64 sit in the same lane (steps s and s + 4), so the
// rotation needs no data exchange.

// cos and sin of the angle of position t for a pair whose angle per position is
// `turn` (a turn fraction, 64-bit fixed point): the top 32 bits of t * turn
// (mod 2^64) are the angle modulo one turn, read as a signed fraction in [-1/2, 1/2)
__device__ __forceinline__ void rope_cs(unsigned long long turn, int t, float& c, float& s) {
  const uint32_t fl = (uint32_t)turn, fh = (uint32_t)(turn >> 32);
  const uint32_t top = __umulhi((uint32_t)t, fl) + (uint32_t)t * fh;
  const float a = (float)(int32_t)top * 1.46291807926715968e-09f;  // 2 pi / 2^32
  __sincosf(a, &s, &c);
}

// the power of two that keeps every rotated Key of a group below 2^14: the group's
// Keys are s_c (n - z_c) with n in [0, L], so |Key| <= s_c (|z_c| + L) and a
// rotation grows a component by at most sqrt(2) (lane l reads channels 4l .. 4l + 3)
template <int FMT>
__device__ __forceinline__ float rope_group_scale(const float* ks, const float* kz, int lane, float& inv) {
  constexpr float kL = (float)((1 << FT<FMT>::kBits) - 1);
  const float4 s4 = *reinterpret_cast<const float4*>(ks + 4 * lane);
  const float4 z4 = *reinterpret_cast<const float4*>(kz + 4 * lane);
  float m = fmaxf(fmaxf(s4.x * (fabsf(z4.x) + kL), s4.y * (fabsf(z4.y) + kL)),
                  fmaxf(s4.z * (fabsf(z4.z) + kL), s4.w * (fabsf(z4.w) + kL)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  return pow2_fit_f16(2.f * m, inv);
}

// Raw scores (d * kfac: the score in the log2 domain) of one quantized tile with the
// Keys rotated at positions t0 + token.  The rotated fp32 Keys, scaled by kapk and
// split in two f16 terms, are the A operand (the fragment order of the codes: rows =
// tokens r, r + 8 of the lane) and the query the B operand: column n holds query
// head n (exact in one f16 term: q is bf16), so one pair of MMAs per step covers the
// 16 tokens for up to 8 heads (16 MMAs per tile).  D(token, head) of lane (r, q) holds
// tokens r, r + 8 of heads 2q, 2q + 1; eight shuffles bring the scores to the
// query-rows layout of qk_tile (head r, tokens 2q, 2q + 1, 2q + 8, 2q + 9).
template <int FMT>
__device__ __forceinline__ void qk_tile_rope(const uint32_t (&KW)[FT<FMT>::kWords], const uint32_t (&X)[8][4],
                                             const float* ks, const float* kz, const unsigned long long* turn, int t0,
                                             int r, int q, float kapk, float (&d)[4]) {
  constexpr float kH = (float)FT<FMT>::kHalf;
  float acc[2][4] = {};
  const int tpos[2] = {t0 + r, t0 + r + 8};
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t a[4], b[4];
    unpack_a<FMT>(KW, s, a[0], a[1], a[2], a[3]);      // channels 16s + 4q + e (centred codes)
    unpack_a<FMT>(KW, s + 4, b[0], b[1], b[2], b[3]);  // channels 16s + 64 + 4q + e
    const int c0 = 16 * s + 4 * q;
    const float4 sl = *reinterpret_cast<const float4*>(ks + c0), zl = *reinterpret_cast<const float4*>(kz + c0);
    const float4 sh = *reinterpret_cast<const float4*>(ks + c0 + 64), zh = *reinterpret_cast<const float4*>(kz + c0 + 64);
    const float slo[4] = {sl.x, sl.y, sl.z, sl.w}, zlo[4] = {zl.x, zl.y, zl.z, zl.w};
    const float shi[4] = {sh.x, sh.y, sh.z, sh.w}, zhi[4] = {zh.x, zh.y, zh.z, zh.w};
    const ulonglong2 u01 = *reinterpret_cast<const ulonglong2*>(turn + c0);
    const ulonglong2 u23 = *reinterpret_cast<const ulonglong2*>(turn + c0 + 2);
    const unsigned long long tu[4] = {u01.x, u01.y, u23.x, u23.y};
    float cs[2][4], sn[2][4];  // [token r / r + 8][channel 4q + e]
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int e = 0; e < 4; ++e) rope_cs(tu[e], tpos[tt], cs[tt][e], sn[tt][e]);
    uint32_t kh[4][2], kl[4][2];  // register reg of steps s (0) and s + 4 (1), high / low f16 terms
#pragma unroll
    for (int reg = 0; reg < 4; ++reg) {
      const int tt = reg & 1, e0 = 2 * (reg >> 1);
      const float2 u = unpack_f16(a[reg]), w = unpack_f16(b[reg]);
      // Keys s (n - z) in fp32 (n - 2^(b-1) is exact in the f16 operand)
      const float x0 = slo[e0] * ((u.x + kH) - zlo[e0]), x1 = slo[e0 + 1] * ((u.y + kH) - zlo[e0 + 1]);
      const float y0 = shi[e0] * ((w.x + kH) - zhi[e0]), y1 = shi[e0 + 1] * ((w.y + kH) - zhi[e0 + 1]);
      const float ca = cs[tt][e0], sa = sn[tt][e0], cb = cs[tt][e0 + 1], sb = sn[tt][e0 + 1];
      split_f16x2(make_float2((x0 * ca - y0 * sa) * kapk, (x1 * cb - y1 * sb) * kapk), kh[reg][0], kl[reg][0]);
      split_f16x2(make_float2((y0 * ca + x0 * sa) * kapk, (y1 * cb + x1 * sb) * kapk), kh[reg][1], kl[reg][1]);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int st = s + 4 * j;
      mma_f16(acc[j], kh[0][j], kh[1][j], kh[2][j], kh[3][j], X[st][0], X[st][1]);
      mma_f16(acc[j], kl[0][j], kl[1][j], kl[2][j], kl[3][j], X[st][0], X[st][1]);
    }
  }
  const float a0 = acc[0][0] + acc[1][0], a1 = acc[0][1] + acc[1][1];  // token r: heads 2q, 2q + 1
  const float a8 = acc[0][2] + acc[1][2], a9 = acc[0][3] + acc[1][3];  // token r + 8
  // head r, token 2q (2q + 8) sits in lane 8q + r / 2 as its head (r & 1) of row 2q; token
  // 2q + 1 (2q + 9) in lane 8q + 4 + r / 2
  const int src = 8 * q + (r >> 1);
  const bool odd = (r & 1) != 0;
  float v0 = __shfl_sync(kFull, a0, src), v1 = __shfl_sync(kFull, a1, src);
  d[0] = odd ? v1 : v0;
  v0 = __shfl_sync(kFull, a0, src + 4);
  v1 = __shfl_sync(kFull, a1, src + 4);
  d[1] = odd ? v1 : v0;
  v0 = __shfl_sync(kFull, a8, src);
  v1 = __shfl_sync(kFull, a9, src);
  d[2] = odd ? v1 : v0;
  v0 = __shfl_sync(kFull, a8, src + 4);
  v1 = __shfl_sync(kFull, a9, src + 4);
  d[3] = odd ? v1 : v0;
}

// Scores of a bf16 tile (sink / residual rows, stored before RoPE) with its Keys
// rotated at their positions (row r: pos_a, row r + 8: pos_b): K rows through ldmatrix
// (natural channel order: channel c and c + 64 in steps s and s + 4 of the same lane),
// rotated in fp32, scaled by a power of two from the tile's largest |Key| and split in
// two f16 terms; the query column (q * kapq, hi/lo) in A rows r, r + 8.  kfacq:
// the score multiplier of the query scale.  Rows past `rows` masked.
__device__ __forceinline__ void bf16_qk_rope(const uint8_t* stg, const float* qrow, int lane, int q, bool hv, int rows,
                                             float kapq, float kfacq, const unsigned long long* turn, int pos_a,
                                             int pos_b, float (&sig)[4]) {
  // the largest |Key| of the tile's rows (16-byte chunk lane + 32 j is in row (lane >> 4) + 2 j)
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if ((lane >> 4) + 2 * j >= rows) continue;
    const uint4 v = reinterpret_cast<const uint4*>(stg)[lane + 32 * j];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack_bf16(w4[k]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  float invk;
  const float kapk = pow2_fit_f16(2.f * m, invk);
  const int x = lane & 7;
  const uint32_t lbase =
      smem_addr(stg) + ((lane & 7) + 8 * ((lane >> 3) & 1)) * 256 + 16 * ((lane >> 4) ^ (x & 1));
  float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
  const int tpos[2] = {pos_a, pos_b};
  const float2 kq = make_float2(kapq, kapq);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t a[4], b[4];  // rows r / r + 8, channels 16s + 2q + {0, 1} (regs 0, 1) and 16s + 8 + 2q + {0, 1} (2, 3)
    ldmatrix_x4(lbase + 32 * (s ^ (x >> 1)), a[0], a[1], a[2], a[3]);
    ldmatrix_x4(lbase + 32 * ((s + 4) ^ (x >> 1)), b[0], b[1], b[2], b[3]);
    const int cbase[2] = {16 * s + 2 * q, 16 * s + 8 + 2 * q};
    float cs[2][4], sn[2][4];  // [row r / r + 8][pair 2h + j: channel cbase[h] + j]
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) rope_cs(turn[cbase[h] + j], tpos[tt], cs[tt][2 * h + j], sn[tt][2 * h + j]);
    uint32_t kh[4][2], kl[4][2];
#pragma unroll
    for (int reg = 0; reg < 4; ++reg) {
      const int tt = reg & 1, h = reg >> 1;
      const float2 u = unpack_bf16(a[reg]), w = unpack_bf16(b[reg]);
      const float ca = cs[tt][2 * h], sa = sn[tt][2 * h], cb = cs[tt][2 * h + 1], sb = sn[tt][2 * h + 1];
      split_f16x2(make_float2((u.x * ca - w.x * sa) * kapk, (u.y * cb - w.y * sb) * kapk), kh[reg][0], kl[reg][0]);
      split_f16x2(make_float2((w.x * ca + u.x * sa) * kapk, (w.y * cb + u.y * sb) * kapk), kh[reg][1], kl[reg][1]);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int st = s + 4 * j;
      uint32_t x0h, x0l, x2h, x2l;  // the query column, channels 16 st + 2q .. and 16 st + 8 + 2q ..
      const float2 q0 = *reinterpret_cast<const float2*>(qrow + 16 * st + 2 * q);
      const float2 q2 = *reinterpret_cast<const float2*>(qrow + 16 * st + 8 + 2 * q);
      split_f16x2(mul_f32x2(q0, kq), x0h, x0l);
      split_f16x2(mul_f32x2(q2, kq), x2h, x2l);
      mma_f16(lo, x0h, x0l, x2h, x2l, kh[0][j], kh[2][j]);
      mma_f16(lo, x0h, x0l, x2h, x2l, kl[0][j], kl[2][j]);
      mma_f16(hi, x0h, x0l, x2h, x2l, kh[1][j], kh[3][j]);
      mma_f16(hi, x0h, x0l, x2h, x2l, kl[1][j], kl[3][j]);
    }
  }
  const float f = kfacq * invk;
  const int t0 = 2 * q;
  sig[0] = (hv && t0 < rows) ? (lo[0] + lo[2]) * f : -INFINITY;
  sig[1] = (hv && t0 + 1 < rows) ? (lo[1] + lo[3]) * f : -INFINITY;
  sig[2] = (hv && t0 + 8 < rows) ? (hi[0] + hi[2]) * f : -INFINITY;
  sig[3] = (hv && t0 + 9 < rows) ? (hi[1] + hi[3]) * f : -INFINITY;
}

// The query-side operand of a pre-RoPE layer, once per segment: x_c = q_c kappa (kappa
// the power of two bringing max |q_c| into [2^13, 2^14)), hi/lo as in build_x_fp8.
// Query operand of pre-RoPE layers (qk_tile_rope's B operand, column = the lane's
// head r): channels 16s + 4q, +1 in X[s][0] and 16s + 4q + 2, +3 in X[s][1], the
// bf16 query times a power of two kap (one f16 term, exact: max |q| kap < 2^14).
__device__ __forceinline__ void build_x_rope(const float* qrow, int q, uint32_t (&X)[8][4], float& kap, float& inv) {
  float mx = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 16 * s + 4 * q);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
  }
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  kap = pow2_fit_f16(mx, inv);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(qrow + 16 * s + 4 * q);
    X[s][0] = pack_f16(x.x * kap, x.y * kap);
    X[s][1] = pack_f16(x.z * kap, x.w * kap);
    X[s][2] = X[s][3] = 0u;
  }
}

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
// Query columns of a kv head h: column j is query token j / gh (of n_query per
// sequence) of query head h * gh + j % gh.  Its row in q, out and lse
// ([B][n_query][Hq]) is b * n_query * Hq + (j / gh) * Hq + h * gh + j % gh.
__device__ __forceinline__ long long query_row(const DecodeParams& p, int b, int h, int j) {
  const int m = j / p.gh, hr = j - m * p.gh;
  return ((long long)b * p.n_query + m) * p.Hq + h * p.gh + hr;
}

// final output of row `row` of out / lse, channel c; l2 = log2-domain log-sum-exp
__device__ __forceinline__ void write_row(const DecodeParams& p, long long row, int c, float o, float l2) {
  const long long oi = row * 128 + c;
  if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  else reinterpret_cast<float*>(p.out)[oi] = o;
  if (p.lse && c == 0) p.lse[row] = l2 * 0.69314718055994531f;
}
__device__ __forceinline__ void write_out(const DecodeParams& p, int b, int h, int j, int c, float o, float l2) {
  write_row(p, query_row(p, b, h, j), c, o, l2);
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
static_assert(kMaxParts + 2 <= kMergeStride, "the merge weights live in a merge-record row");

// Work items of one segment, dealt to the CTA's warps round robin (item t to
// warp t mod NW: every warp's share is interleaved over the segment, so the
// warps finish together and each warp's sums run in a fixed order): its bf16
// tiles [bl, bl + nbf_items) (a pair's units are its nbf bf16 tiles, wbf units
// each, then its nq quantized tiles, 1 unit each; a bf16 tile belongs to the
// range holding its first unit), then its quantized tiles [ql, qh) in items of
// `it` tiles aligned at multiples of `it` (whole records for the integer
// formats, so an item starts at a record header except at ql).
struct SegItems {
  int bl, nbf_items, ql, qh, al, nq_items;
};

// One (sequence, kv head) pair's share of this CTA's unit range, with its work
// items and the address of its first record (contiguous store).
struct SegRec {
  long long pair_start;  // first unit of the pair in the flat unit list
  const uint8_t* rec0;   // contiguous store: record 0 of the pair
  int b, h, ua, ue, units;
  int n_sink, qn, r, nbf, nq;
  SegItems it;
};
constexpr int kMaxSeg = 16;  // segments per table batch


__device__ __forceinline__ SegItems seg_items(const SegRec& sg, int wbf, int it) {  // thread 0, once
  SegItems s;
  const int nbu = sg.nbf * wbf;
  s.bl = min(sg.nbf, (sg.ua + wbf - 1) / wbf);
  s.nbf_items = min(sg.nbf, (sg.ue + wbf - 1) / wbf) - s.bl;
  s.ql = min(sg.nq, max(0, sg.ua - nbu));
  s.qh = min(sg.nq, max(0, sg.ue - nbu));
  s.al = s.ql / it * it;
  s.nq_items = s.qh > s.ql ? (s.qh - s.al + it - 1) / it : 0;
  return s;
}

// Tag of a pipeline slot: what its stage holds.  seg: segment index; kind 1/2:
// K/V rows of bf16 tile `a`; kind 3: n quantized tiles from tile `a` (at
// position rpos of its record), `first` when the stage starts an item (the Key
// group's B operand is built there).
struct SlotTag {
  int seg, a, rpos;
  short kind, n;
  int first;
};
static_assert(sizeof(SegRec) == 80, "the host reserves 80 bytes per segment record");

// BF: the layer may have bf16 tiles (sink or residual tokens); the variant without
// them (FP8 layers with no sink tokens) carries no bf16-tile code at all.  MQ:
// several query tokens per sequence (causal limits per column); only that
// variant carries the limit checks.  ONE: one tile per record -- integer layers
// whose Key groups are one tile each (G = 16, the paged blocks: every tile rebuilds
// the query-side operand) and contiguous FP8 stores -- in straight-line code.  ROPE: pre-RoPE Keys (integer layers), rotated
// at their positions.  OUT: dense-and-sparse rows (integer layers): the kept Key
// entries add q_c x_c to the scores, the kept Value entries p x_c to the outputs
// (through a per-warp shared-memory sum of 8 columns x 128 channels).  KA: at most
// four query columns (one query token): the Key tile is the A operand of the QK
// MMAs and the query side the B operand (qk_tile_ka), half the MMAs of the
// query-rows form.
template <int FMT, int NGV, bool BF, bool MQ, bool ONE, bool ROPE, bool OUT, bool KA>
__global__ void __launch_bounds__(DecodeWarps<FMT>::kThreads, 1) decode_kernel(const DecodeParams p) {
  pdl_wait();  // the previous kernel of the stream has finished (programmatic launch)
  pdl_trigger();
  using F = FT<FMT>;
  static_assert(!KA || (!MQ && !ROPE && !OUT), "the Key-as-A form serves one query token, plain Keys");
  constexpr int NW = DecodeWarps<FMT>::kNW;
  constexpr int NT = NW * 32;
  constexpr int NR = NW / 2;  // merge records (warps fold pairwise into them)
  extern __shared__ __align__(128) uint8_t smem[];
  const LayerDesc& L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, q = lane & 3;
  const int B = p.batch, H = L.H, g = p.g;
  const int tps = p.tps, nst = p.nst, wbf = p.bf_weight;
  const bool bfj = p.bf_joint != 0;  // a bf16 tile's K and V rows share one stage
  const int it = p.item_tiles;

  // ---- shared memory carve-up ----
  uint8_t* stage_base = smem;
  size_t off = (size_t)NW * nst * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off);
  off += NW * kMaxStages * sizeof(uint64_t);
  int* tbl = reinterpret_cast<int*>(smem + off);  // per warp: a window of 32 block-table entries
  off += NW * 32 * sizeof(int);
  float* q_s = reinterpret_cast<float*>(smem + off);  // [g + 1 rows][kQRow]: the query heads, a zero row
  off += (size_t)(g + 1) * kQRow * sizeof(float);
  float* recs = reinterpret_cast<float*>(smem + off);  // NW/2 merge records [g heads][kMergeStride]
  off += (size_t)NR * p.merge_bytes;
  SegRec* segs = reinterpret_cast<SegRec*>(smem + off);
  off += kMaxSeg * sizeof(SegRec);
  int* prefix = reinterpret_cast<int*>(smem + off);  // [B + 1]
  off += ((size_t)(B + 1) * sizeof(int) + 15) / 16 * 16;
  int* toks = reinterpret_cast<int*>(smem + off);    // [B]: each sequence's token count (clamped)
  off += ((size_t)B * sizeof(int) + 15) / 16 * 16;
  // pre-RoPE Keys: per warp, the current Key group's header (K scale [128], K zero [128])
  float* rope_hdr = ROPE ? reinterpret_cast<float*>(smem + off) + warp * 256 : nullptr;
  // dense-and-sparse Values: per warp, the sparse part of the 8 columns' outputs [8][kSparseRow]
  float* sp_acc = (OUT && L.v_out) ? reinterpret_cast<float*>(smem + off) + warp * 8 * kSparseRow : nullptr;
  __shared__ int seg_count;
  __shared__ long long batch_end;

  if (tid == 0) {
    for (int i = 0; i < NW * kMaxStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_barrier_init();
  }
  unsigned long long* s_turn = nullptr;  // pre-RoPE Keys: the pairs' angle per position
  if constexpr (ROPE) {
    __shared__ unsigned long long turn_tab[64];
    if (tid < 64) turn_tab[tid] = p.rope_turn[tid];
    s_turn = turn_tab;
  }

  // ---- per-sequence work units and their prefix (units of all H heads) ----
  const long long tmax_tok = max_tokens(L);
  auto seq_tokens = [&](int b) -> int {
    long long T = (long long)p.seq_lens[b] + p.len_add;
    if (T < 0) T = 0;
    if (T > tmax_tok) T = tmax_tok;
    return (int)T;
  };
  {
    const int per = (B + NT - 1) / NT;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      const int T = seq_tokens(b);
      toks[b] = T;
      prefix[b] = local;
      const TokenSplit ts = split_tokens(T, L);
      local += (((ts.n_sink + ts.r + 15) >> 4) * wbf + ((ts.qn + 15) >> 4)) * H;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_tot[NW];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += warp_tot[w];
    const int excl = wbase + incl - local;
    for (int b = b0; b < b1; ++b) prefix[b] += excl;
    if (tid == NT - 1) prefix[B] = wbase + incl;
    if (blockIdx.x == 0) {
      for (int b = tid; b < B; b += NT)
        if ((long long)p.seq_lens[b] + p.len_add > tmax_tok) report(p.status, KVQ_DEV_CAPACITY);
    }
    __syncthreads();
    if (blockIdx.x == 0)
      for (int b = tid; b <= B; b += NT) p.ws_prefix[b] = prefix[b];
  }

  const long long U = prefix[B];
  bool same_len = true;  // every sequence holds the same number of units
  for (int b = tid; b < B; b += NT) same_len &= (prefix[b + 1] - prefix[b]) == (prefix[1] - prefix[0]);
  const long long C = range_ctas(p.num_ctas, U, (long long)B * H, __syncthreads_and(same_len) != 0);
  if (blockIdx.x == 0 && tid == 0) p.ws_prefix[B + 1] = (int)C;  // for the two-launch merge
  if (p.fuse) {
    // sequences without tokens belong to no CTA's range: out = 0, lse = -inf
    for (int b = blockIdx.x; b < B; b += gridDim.x)
      if (prefix[b + 1] == prefix[b])
        for (int i = tid; i < p.n_query * p.Hq * 128; i += NT)
          write_row(p, (long long)b * p.n_query * p.Hq + (i >> 7), i & 127, 0.f, -INFINITY);
  }
  // CTAs at or beyond C have nothing to do
  const long long st = blockIdx.x < C ? (long long)blockIdx.x * U / C : U;
  const long long en = blockIdx.x < C ? (long long)(blockIdx.x + 1) * U / C : U;

  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* sink_k = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_k);
  const __nv_bfloat16* sink_v = reinterpret_cast<const __nv_bfloat16*>(p.C.sink_v);
  const __nv_bfloat16* ring_k = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_k);
  const __nv_bfloat16* ring_v = reinterpret_cast<const __nv_bfloat16*>(p.C.resid_v);

  uint8_t* my_stages = stage_base + (size_t)warp * nst * p.stage_bytes;
  uint64_t* my_bars = bars + warp * kMaxStages;
  int* my_tbl = tbl + warp * 32;
  float* my_rec = recs + (size_t)(warp % NR) * (p.merge_bytes / 4);
  uint32_t phase_bits = 0;  // expected parity of each stage barrier of this warp
  uint32_t slot_valid = 0;  // 8 bits per slot: the tiles its stage holds (every lane keeps the same)
  // the two slots' tags, kept in registers by every lane (the producer's cursor is the same in all
  // lanes): the first tile (a), and seg | kind << 8 | n << 12 | rpos << 16 | first << 24
  uint32_t tga0 = 0, tgb0 = 0, tga1 = 0, tgb1 = 0;
  static_assert(kMaxStages == 2, "two slots per warp: two register sets of tags");
  uint32_t pending = 0;     // slots with copies in flight
  bool alive = true;
  int n_issued = 0, n_consumed = 0;
  int p_slot = 0, c_slot = 0;  // the slots of the next copy and of the next stage to consume
  const float s_v8 = F::kFp8 ? __ldg(p.C.v_tscale) : 1.f;

  // the g query heads of a pair into q_s (row g zero)
  auto load_q = [&](const SegRec& sg) {
    for (int i = tid; i < (g + 1) * 128; i += NT) {
      const int hr = i >> 7, c = i & 127;
      float v = 0.f;
      if (hr < g) v = __bfloat162float(qg[query_row(p, sg.b, sg.h, hr) * 128 + c]);
      q_s[hr * kQRow + c] = v;
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
        sg.h = (int)(pp - prefix[lo]) / sg.units;
        sg.pair_start = prefix[lo] + (long long)sg.h * sg.units;
        const long long se = min(en, sg.pair_start + sg.units);
        sg.ua = (int)(pp - sg.pair_start);
        sg.ue = (int)(se - sg.pair_start);
        const TokenSplit ts = split_tokens(toks[lo], L);
        sg.n_sink = ts.n_sink;
        sg.qn = ts.qn;
        sg.r = ts.r;
        sg.nbf = (ts.n_sink + ts.r + 15) >> 4;
        sg.nq = (ts.qn + 15) >> 4;
        sg.it = seg_items(sg, wbf, it);
        sg.rec0 = L.paged ? nullptr
                          : reinterpret_cast<const uint8_t*>(p.C.qstore) +
                                ((long long)sg.b * H + sg.h) * L.nrec * L.rec_bytes;
        segs[ns++] = sg;
        pp = se;
      }
      seg_count = ns;
      batch_end = pp;
    }
    __syncthreads();
    const int nseg = seg_count;

    // ---- producer: lane 0 copies; every lane keeps the same cursor ----
    int ps = 0;                  // segment of the producer
    int pk = 0;                  // kind of the current item: 0 none, 1 bf16, 3 quantized
    int p_a = 0, p_end = 0;      // bf16: tile and next half (0 K, 1 V, 2 done); quantized: next tile, end
    bool p_first = false;        // the item's first stage is next
    int q_rec = 0, q_pos = 0;    // record and position in it of the next quantized tile
    int tb_base = -1;            // paged: first record of the block-table window in my_tbl (-1: none)
    int tb_seg = -1;             // ... and its segment
    int p_claims = 0;            // items taken from segment ps
    // the next item with stages left, taken from the segments in order; false when none
    auto producer_ready = [&]() -> bool {
      while (ps < nseg) {
        if (pk == 1 && p_end < 2) return true;
        if (pk == 3 && p_a < p_end) return true;
        const int t = warp + NW * (p_claims++);  // items warp, warp + NW, ... of the segment
        const SegItems si = segs[ps].it;
        if (BF && t < si.nbf_items) {
          pk = 1;
          p_a = si.bl + t;
          p_end = 0;
        } else if (t - si.nbf_items < si.nq_items) {
          const int k = t - si.nbf_items;
          pk = 3;
          p_a = max(si.ql, si.al + k * it);
          p_end = min(si.qh, si.al + (k + 1) * it);
          p_first = true;
          if (L.tpg == 1) {
            q_rec = p_a;
            q_pos = 0;
          } else {
            q_rec = p_a / L.tpg;
            q_pos = p_a - q_rec * L.tpg;
          }
        } else {
          pk = 0;
          ++ps;
          p_claims = 0;
        }
      }
      return false;
    };
    auto issue_next = [&]() {
      const int slot = p_slot;
      const SegRec& sg = segs[ps];
      uint32_t vm = 0;
      SlotTag tg;
      tg.seg = ps;
      if (BF && pk == 1) {
        tg.kind = (short)(1 + p_end);
        tg.a = p_a;
        tg.rpos = 0;
        tg.n = 1;
        tg.first = 0;
        {
          // bf16 tile: its 16 K rows and 16 V rows in one stage (joint), or the K rows in
          // one stage and the V rows in the next.  Every lane copies 16-byte chunk
          // (lane & 15) of rows (lane >> 4) + 2i with cp.async (coalesced) as one commit
          // group; the consumer waits for the group (cp.async.wait_group), the slot's
          // barrier only keeps the phases in step.
          uint8_t* dst = my_stages + (size_t)slot * p.stage_bytes;
          const uint32_t bar = smem_addr(&my_bars[slot]);
          const int x0 = p_a * 16;  // bf16-list index of the first row (sinks, then residual)
          const int rows = min(16, sg.n_sink + sg.r - x0);
          const long long pair = (long long)sg.b * H + sg.h;
          const int ch = lane & 15, hi = lane >> 4;
          // ring slot of the tile's first residual row (one modulo per stage); rows
          // [nsk, rows) are residual rows, the first nsk (if any) sink rows
          const int nsk = max(0, min(rows, sg.n_sink - x0));
          int slot0 = 0;
          if (rows > nsk) slot0 = (sg.qn - sg.n_sink + x0 + nsk) % L.W;
          const int hv0 = bfj ? 0 : p_end, hv1 = bfj ? 1 : p_end;
          if (nsk == 0 && slot0 + rows <= L.W) {
            // common case: the 16 rows are consecutive ring rows
            const long long roff = (pair * L.W + slot0) * L.d + 8 * ch;
            for (int hv = hv0; hv <= hv1; ++hv) {
              const __nv_bfloat16* src = (hv ? ring_v : ring_k) + roff;
              const uint32_t half = smem_addr(dst + (bfj ? hv * kBfHalf : 0));
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int rr = hi + 2 * i;
                if (rr < rows) cp_async_16(half + bf_chunk_off(rr, ch), src + rr * 128);
              }
            }
          } else {
            // sink rows first, or a ring that wraps inside the tile: row by row
            for (int hv = hv0; hv <= hv1; ++hv) {
              const __nv_bfloat16* sink = hv ? sink_v : sink_k;
              const __nv_bfloat16* ring = hv ? ring_v : ring_k;
              const uint32_t half = smem_addr(dst + (bfj ? hv * kBfHalf : 0));
              for (int i = 0; i < 8; ++i) {
                const int rr = hi + 2 * i;
                if (rr < rows) {
                  const __nv_bfloat16* src;
                  if (rr < nsk) {
                    src = sink + (pair * L.S + x0 + rr) * L.d;
                  } else {
                    int sl = slot0 + (rr - nsk);
                    if (sl >= L.W) sl -= L.W;
                    src = ring + (pair * L.W + sl) * L.d;
                  }
                  cp_async_16(half + bf_chunk_off(rr, ch), src + 8 * ch);
                }
              }
            }
          }
          cp_async_commit();
          if (lane == 0) mbar_arrive(bar);
        }
        vm = 1;
        p_end = bfj ? 2 : p_end + 1;
      } else {
        // n quantized tiles from (q_rec, q_pos), one contiguous range per record touched
        const int n = min(tps, p_end - p_a);
        const bool hdr0 = F::kInt && p_first && q_pos != 0;  // the group's header, copied to slot offset 0
        int l_rec = q_rec, l_pos = q_pos + n - 1;              // the last tile's record and position
        if (L.tpg == 1) {
          l_rec = q_rec + n - 1;
          l_pos = 0;
        } else {
          while (l_pos >= L.tpg) {
            l_pos -= L.tpg;
            ++l_rec;
          }
        }
        tg.kind = 3;
        tg.a = p_a;
        tg.rpos = q_pos;
        tg.n = (short)n;
        tg.first = p_first ? 1 : 0;
        if (L.paged && (tb_seg != ps || tb_base < 0 || q_rec < tb_base || l_rec >= tb_base + 32)) {
          // the block-table entries of 32 records from q_rec, one per lane
          tb_base = q_rec;
          tb_seg = ps;
          const int x = q_rec + lane;
          my_tbl[lane] = x < L.mbps ? __ldg(&p.C.block_table[(long long)sg.b * L.mbps + x]) : -1;
          __syncwarp();
        }
        if (L.paged && L.tpg == 1) {
          // one tile per record (blocks of 16 tokens): lane j copies record q_rec + j whole
          // (header inline) to stage offset j * rec_bytes, all lanes at once; the stage
          // barrier expects the bytes of the records whose block is inside the pool
          uint8_t* dst = my_stages + (size_t)slot * p.stage_bytes;
          const uint32_t bar = smem_addr(&my_bars[slot]);
          int blk = -1;
          if (lane < n) blk = my_tbl[q_rec + lane - tb_base];
          const bool ok = lane < n && blk >= 0 && blk < L.num_blocks;
          const uint32_t okm = __ballot_sync(kFull, ok);
          if (lane < n && !ok) report(p.status, KVQ_DEV_BAD_BLOCK);
          if (lane == 0 && okm) mbar_arrive_expect_tx(bar, (uint32_t)__popc(okm) * (uint32_t)L.rec_bytes);
          __syncwarp();
          if (ok)
            bulk_copy_g2s(smem_addr(dst + lane * L.rec_bytes),
                          reinterpret_cast<const uint8_t*>(p.C.block_pool) + (long long)blk * L.block_bytes +
                              (long long)sg.h * L.rec_bytes,
                          (uint32_t)L.rec_bytes, bar);
          vm = okm;
        } else if (lane == 0) {
          uint8_t* dst = my_stages + (size_t)slot * p.stage_bytes;
          const uint32_t bar = smem_addr(&my_bars[slot]);
          if (!L.paged) {
            const uint8_t* base = sg.rec0;
            const uint8_t* rec0 = base + (long long)q_rec * L.rec_bytes;
            const uint8_t* start = (F::kInt && q_pos == 0) ? rec0 : rec0 + L.hdr_bytes + q_pos * L.tile_bytes;
            const uint8_t* end = base + (long long)l_rec * L.rec_bytes + L.hdr_bytes + (l_pos + 1) * L.tile_bytes;
            const uint32_t len = (uint32_t)(end - start);
            mbar_arrive_expect_tx(bar, len + (hdr0 ? 1024u : 0u));
            // (the self-test of the bounded waits withholds CTA 0 / warp 0's first copy)
            if (!(p.withhold_copy && blockIdx.x == 0 && warp == 0 && n_issued == 0)) {
              bulk_copy_g2s(smem_addr(dst + (hdr0 ? 1024 : 0)), start, len, bar);
              if (hdr0) bulk_copy_g2s(smem_addr(dst), rec0, 1024, bar);
            }
            vm = (1u << n) - 1u;
          } else {
            // records q_rec .. l_rec: present ones are copied, missing ones (bad block) leave holes
            const uint8_t* pool = reinterpret_cast<const uint8_t*>(p.C.block_pool);
            uint32_t bytes = 0;
            for (int pass = 0; pass < 2; ++pass) {
              uint32_t so = hdr0 ? 1024u : 0u;
              int t = 0;  // tiles of the stage before record rr
              for (int rr = q_rec; rr <= l_rec; ++rr) {
                const int a0 = rr == q_rec ? q_pos : 0;
                const int cnt = min(L.tpg - a0, n - t);
                const bool with_hdr = F::kInt && a0 == 0;
                const uint32_t len = (uint32_t)((with_hdr ? L.hdr_bytes : 0) + cnt * L.tile_bytes);
                const int blk = my_tbl[rr - tb_base];
                const bool ok = blk >= 0 && blk < L.num_blocks;
                if (pass == 0) {
                  if (ok) {
                    vm |= ((1u << cnt) - 1u) << t;
                    bytes += len + ((hdr0 && rr == q_rec) ? 1024u : 0u);
                  } else {
                    report(p.status, KVQ_DEV_BAD_BLOCK);
                  }
                } else if (ok) {
                  const uint8_t* rec = pool + (long long)blk * L.block_bytes + (long long)sg.h * L.rec_bytes;
                  bulk_copy_g2s(smem_addr(dst + so), with_hdr ? rec : rec + L.hdr_bytes + a0 * L.tile_bytes, len, bar);
                  if (hdr0 && rr == q_rec) bulk_copy_g2s(smem_addr(dst), rec, 1024, bar);
                }
                so += len;
                t += cnt;
              }
              if (pass == 0) {
                if (!vm) break;
                mbar_arrive_expect_tx(bar, bytes);
              }
            }
          }
        }
        // advance the cursor by n tiles
        p_a += n;
        p_first = false;
        q_rec = l_rec;
        q_pos = l_pos + 1;
        if (q_pos == L.tpg) {
          q_pos = 0;
          ++q_rec;
        }
      }
      {
        const uint32_t pk2 = (uint32_t)tg.seg | ((uint32_t)tg.kind << 8) | ((uint32_t)tg.n << 12) |
                             ((uint32_t)tg.rpos << 16) | ((uint32_t)tg.first << 24);
        if (slot) { tga1 = (uint32_t)tg.a; tgb1 = pk2; } else { tga0 = (uint32_t)tg.a; tgb0 = pk2; }
      }
      vm = __shfl_sync(kFull, vm, 0);
      slot_valid = (slot_valid & ~(0xFFu << (8 * slot))) | (vm << (8 * slot));
      if (vm) pending |= 1u << slot;
      ++n_issued;
      if (++p_slot == nst) p_slot = 0;
    };
    auto pump = [&]() {
      while (alive && n_issued - n_consumed < nst && producer_ready()) issue_next();
      __syncwarp();
    };

    // the query of the first segment: loads issued before the first copies, stored after them
    constexpr int kQPer = (8 * 128 + NT - 1) / NT;
    unsigned short qpre[kQPer];  // raw bf16: converted only after the copies are issued
    {
      const SegRec& s0 = segs[0];
      const unsigned short* qraw = reinterpret_cast<const unsigned short*>(qg);
#pragma unroll
      for (int k = 0; k < kQPer; ++k) {
        const int i = tid + k * NT, hr = i >> 7, c = i & 127;
        qpre[k] = (i < 8 * 128 && hr < g) ? qraw[query_row(p, s0.b, s0.h, hr) * 128 + c] : 0;
      }
    }
    pump();
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * NT, hr = i >> 7, c = i & 127;
      if (i < 8 * 128 && hr <= g) q_s[hr * kQRow + c] = __uint_as_float((unsigned)qpre[k] << 16);  // row g stays zero
    }
    __syncthreads();

    // ---- consumer ----
    for (int s = 0; s < nseg; ++s) {
      const SegRec sg = segs[s];
      const int nbf_tok = sg.n_sink + sg.r;
      WarpState<NGV> stt;
      state_init(stt);
      if (sp_acc) {
#pragma unroll
        for (int i = 0; i < 8; ++i) reinterpret_cast<float4*>(sp_acc + i * kSparseRow)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
      }
      float* sp_row = sp_acc ? sp_acc + r * kSparseRow : nullptr;  // the lane's column
      const float* qrow = q_s + min(r, g) * kQRow;  // the lane's query column (row g is zero)
      const float* qrow_op = KA ? q_s + min(r >> 1, g) * kQRow : qrow;  // the row the lane's operand is built from
      const bool hv = r < g;                         // the column exists
      uint32_t X[8][4];  // query-side A operand (hi/lo rows), rebuilt per Key group for INT layers
      float kfac = 0.f, cterm = 0.f;
      float qm = 0.f;    // INT: the column's max |q_c| (the Key groups' kappa bound)
      float kapq = 1.f, kfacq = 0.f;  // pre-RoPE Keys: the query operand's scale and score multiplier
      if constexpr (ROPE) {
        float invq;
        build_x_rope(qrow, q, X, kapq, invq);
        kfacq = p.scale_log2 * invq;
      } else if constexpr (F::kFp8) {
        build_x_fp8(qrow_op, q, p.scale_log2 * __ldg(p.C.k_tscale), X, kfac);
        if constexpr (KA) ka_operand(X, r, kfac, cterm);
      } else {
        qm = column_qmax(qrow_op, q);

#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) X[s2][0] = X[s2][1] = X[s2][2] = X[s2][3] = 0u;
      }
      float kapk = 1.f;  // pre-RoPE Keys: the current group's Key scale
      float sig_bf[4];  // scores of a bf16 tile between its K and V stages
      // the lane's four tokens of a tile (score and W layout)
      const int tk[4] = {2 * q, 2 * q + 1, 2 * q + 8, 2 * q + 9};
      // several query tokens per sequence: column r (query token r / gh) sees the tokens
      // t <= T - n_query + r / gh (causal: where that query token sits); computed once per
      // segment, only in the multi-query variant
      const int mq_lim = MQ ? toks[sg.b] - p.n_query + r / p.gh : 0;
      auto col_limit = [&]() { return mq_lim; };

      // this warp's stages of segment s, in the order its producer issued them
      while (true) {
        if (n_consumed == n_issued) {
          pump();
          if (n_consumed == n_issued) break;  // no work left for this warp in this batch
        }
        const int slot = c_slot;
        SlotTag tg;
        {
          const uint32_t w = slot ? tgb1 : tgb0;
          tg.a = (int)(slot ? tga1 : tga0);
          tg.seg = (int)(w & 0xFFu);
          tg.kind = (short)((w >> 8) & 0xFu);
          tg.n = (short)((w >> 12) & 0xFu);
          tg.rpos = (int)((w >> 16) & 0xFFu);
          tg.first = (int)(w >> 24);
        }
        if (tg.seg != s) break;  // the producer has moved on: segment s is done for this warp
        const uint32_t vmask = (slot_valid >> (8 * slot)) & 0xFFu;
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
        if (BF && vmask && alive && tg.kind != 3) {
          // this stage's cp.async group: complete once at most `newer` groups (the bf16
          // stages issued after it) are pending; then every lane's copies are visible
          int newer = 0;
          for (int j = 1; j < n_issued - n_consumed; ++j) {
            int sl = slot + j;
            if (sl >= nst) sl -= nst;
            newer += (((sl ? tgb1 : tgb0) >> 8) & 0xFu) != 3u;
          }
          if (newer == 0) cp_async_wait<0>();
          else if (newer == 1) cp_async_wait<1>();
          else if (newer == 2) cp_async_wait<2>();
          else cp_async_wait<3>();
          __syncwarp();
          const int rows = min(16, nbf_tok - tg.a * 16);
          // K rows: scores.  V rows (the same stage when joint, else the next one): rows past
          // the end zeroed (their p is 0, garbage could be NaN), the softmax step, then PV
          const uint8_t* vst = stg;
          bool vpart = tg.kind == 2;
          if (tg.kind == 1) {
            if constexpr (ROPE) {  // bf16 list index -> position: sinks first, then the window after Q_n
              const int xa = 16 * tg.a + r, xb = xa + 8;
              bf16_qk_rope(stg, qrow, lane, q, hv, rows, kapq, kfacq, s_turn, xa + (xa >= sg.n_sink ? sg.qn : 0),
                           xb + (xb >= sg.n_sink ? sg.qn : 0), sig_bf);
            } else {
              bf16_qk(stg, qrow, lane, q, hv, rows, p.scale_log2, sig_bf);
            }
            if (MQ && p.n_query > 1) {  // bf16 list index -> token: sinks first, then the residual window after Q_n
              const int lim = col_limit();
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = 16 * tg.a + tk[e];
                if (x + (x >= sg.n_sink ? sg.qn : 0) > lim) sig_bf[e] = -INFINITY;
              }
            }
            vpart = bfj;
            vst = stg + kBfHalf;
          }
          if (vpart) {
            uint8_t* stw = const_cast<uint8_t*>(vst);
            for (int idx = lane; idx < (16 - rows) * 16; idx += 32)
              *reinterpret_cast<uint4*>(stw + (rows + idx / 16) * 256 + (idx % 16) * 16) = make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
            float pr[4];
            softmax_tile<NGV, false>(stt, sig_bf, 1.f, q, pr, sp_row);
            // integer layers: the accumulators hold code units (2^-24, rows r + 8 FT::kVHi more)
            constexpr float kUnit = F::kInt ? 1.f / kCodeUnit : 1.f;
            bf16_pv<F::kInt ? (int)F::kVHi : 1>(vst, lane, pr, stt.inv_S * (kPrescale * kUnit), stt.o);
          }
        } else if (vmask && alive) {
          // ---- quantized stage: tiles [tg.a, tg.a + n), one softmax step each ----
          // tile i at `tile`; INT: `hdrp` the Key-group header, the query-side operand (q * s,
          // hi/lo) rebuilt from it when `build` (at each record, i.e. Key group, start)
          // a tile's step in two halves: tile_qk, the scores of the lane's column for its four tokens;
          // tile_sv, the online softmax step and PV
          auto tile_qk = [&](const int i, const uint8_t* tile, const uint8_t* hdrp, const bool build,
                             float (&sig)[4]) {
            if constexpr (ROPE) {
              // the group's header to the warp's copy (the tiles of a group may span stages)
              if (build) {
                __syncwarp();
                reinterpret_cast<uint4*>(rope_hdr)[lane] = reinterpret_cast<const uint4*>(hdrp)[lane];
                reinterpret_cast<uint4*>(rope_hdr)[lane + 32] = reinterpret_cast<const uint4*>(hdrp)[lane + 32];
                __syncwarp();
                float invk;
                kapk = rope_group_scale<FMT>(rope_hdr, rope_hdr + 128, lane, invk);
                kfac = kfacq * invk;
              }
            } else if constexpr (F::kInt) {
              if (build) {
                build_x_group<FMT>(qrow_op, reinterpret_cast<const float*>(hdrp),
                                   reinterpret_cast<const float*>(hdrp + 512), lane, q, p.scale_log2, qm, X, kfac,
                                   cterm);
                if constexpr (KA) ka_operand(X, r, kfac, cterm);
              }
            }
            // QK
            float d[4];
            {
              uint32_t KW[F::kWords];
              load_words(tile, lane, KW);
              if constexpr (ROPE)
                qk_tile_rope<FMT>(KW, X, rope_hdr, rope_hdr + 128, s_turn, L.S + 16 * i, r, q, kapk, d);
              else if constexpr (KA)
                qk_tile_ka<FMT>(KW, X, lane, d);
              else
                qk_tile<FMT>(KW, X, d);
            }
            const int tok_valid = min(16, sg.qn - i * 16);  // < 16 only for a partial FP8 tile
#pragma unroll
            for (int e = 0; e < 4; ++e)  // integer tiles are always full (Key groups of 16k tokens)
              sig[e] = (hv && (F::kInt || tk[e] < tok_valid)) ? fmaf(d[e], kfac, cterm) : -INFINITY;
            if constexpr (OUT) {  // the tokens' kept Key entries: q_c x_c (exact bf16 x_c)
              const uint32_t* ksp = reinterpret_cast<const uint32_t*>(tile + L.sp_off);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float a = 0.f;
                for (int j = 0; j < L.k_out; ++j) {
                  const uint32_t en = ksp[tk[e] * L.k_out + j];
                  a = fmaf(qrow[en & 127u], __uint_as_float(en & 0xFFFF0000u), a);
                }
                sig[e] = fmaf(a, p.scale_log2, sig[e]);
              }
            }
            if (MQ && p.n_query > 1) {
              const int lim = col_limit() - (L.S + 16 * i);  // in tile rows (quantized token x = t - S)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (tk[e] > lim) sig[e] = -INFINITY;
            }
          };
          auto tile_sv = [&](const uint8_t* tile, float (&sig)[4]) {
            const float* vsp = reinterpret_cast<const float*>(tile + 2 * F::kTile);  // INT: Value scales [16][NGV]
            const float* vzp = vsp + 16 * NGV;                                         // INT: Value zero-points
            float smax = s_v8;
            if constexpr (F::kInt) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float sv[NGV];
                load_row<NGV>(vsp + tk[e] * NGV, sv);
#pragma unroll
                for (int jg = 0; jg < NGV; ++jg) smax = fmaxf(smax, sv[jg]);
              }
            }
            float pt[4];
            softmax_tile<NGV, F::kInt>(stt, sig, smax, q, pt, sp_row);
            if constexpr (OUT) {  // the tokens' kept Value entries: p x_c into the column's sparse sums
              if (sp_row) {
                const uint32_t* vsp = reinterpret_cast<const uint32_t*>(tile + L.sp_off + 64 * L.k_out);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  for (int j = 0; j < L.v_out; ++j) {
                    const uint32_t en = vsp[tk[e] * L.v_out + j];
                    atomicAdd(sp_row + (en & 127u), pt[e] * __uint_as_float(en & 0xFFFF0000u));
                  }
              }
            }
            // PV: the lane's probabilities are already in the W layout (column r, its four tokens)
            uint32_t B0[NGV], B1[NGV];
            if constexpr (F::kFp8) {
              const float f = s_v8 * stt.inv_S * kPrescale;
              B0[0] = pack_f16(pt[0] * f, pt[1] * f);
              B1[0] = pack_f16(pt[2] * f, pt[3] * f);
            } else {
              const float f = stt.inv_S * kPrescale;
#pragma unroll
              for (int jg = 0; jg < NGV; ++jg) {  // one Value group at a time: few live registers
                float w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = pt[e] * (vsp[tk[e] * NGV + jg] * f);
                B0[jg] = pack_f16(w[0], w[1]);
                B1[jg] = pack_f16(w[2] * F::kW1, w[3] * F::kW1);
                // the zero-point sum with the weights the MMA multiplies (rounded to f16)
                const float2 r0 = unpack_f16(B0[jg]), r1 = unpack_f16(B1[jg]);
                float z = stt.zacc[jg];
                z = fmaf(r0.x, vzp[tk[0] * NGV + jg], z);
                z = fmaf(r0.y, vzp[tk[1] * NGV + jg], z);
                z = fmaf(r1.x * (1.f / F::kW1), vzp[tk[2] * NGV + jg], z);
                z = fmaf(r1.y * (1.f / F::kW1), vzp[tk[3] * NGV + jg], z);
                stt.zacc[jg] = z;
              }
            }
            {
              uint32_t VW[F::kWords];
              load_words(tile + F::kTile, lane, VW);
              pv_tile<FMT, NGV>(VW, B0, B1, stt.o);
            }
          };
          auto tile_step = [&](const int i, const uint8_t* tile, const uint8_t* hdrp, const bool build) {
            float sig[4];
            tile_qk(i, tile, hdrp, build, sig);
            tile_sv(tile, sig);
          };
          const int n = tg.n;
          if constexpr (ONE) {
            // one tile per record (16-token Key groups, or FP8 tiles): record k of the stage at
            // k * rec_bytes, every integer tile starts a group (straight-line code: the build
            // overlaps the rest)
            if constexpr (F::kFp8) {  // the step's token (one-token append folded into this launch)
              const int inew = (sg.qn - 1) >> 4;
              if (p.fp8_append && inew >= tg.a && inew < tg.a + n && ((vmask >> (inew - tg.a)) & 1u) &&
                  (long long)p.seq_lens[sg.b] + 1 <= tmax_tok)
                fp8_append_token(p, const_cast<uint8_t*>(stg + (inew - tg.a) * L.rec_bytes + L.hdr_bytes), sg.b,
                                 sg.h, inew, (sg.qn - 1) & 15, lane);
            }
            if (n == 2 && vmask == 3u) {
              // the common stage, two tiles as straight-line code: the second tile's operand build
              // and Key unpack fill the first tile's MMA latencies (paged INT4 layer 537 -> 525 us)
              if constexpr (FMT == 8) {
                // 8-bit codes (8 warps, registers to spare): both tiles' scores first, so the second
                // tile's QK MMAs are in flight during the first tile's softmax (INT8 599 -> 586 us)
                float s0[4], s1[4];
                tile_qk(tg.a, stg + L.hdr_bytes, stg, true, s0);
                tile_qk(tg.a + 1, stg + L.rec_bytes + L.hdr_bytes, stg + L.rec_bytes, true, s1);
                tile_sv(stg + L.hdr_bytes, s0);
                tile_sv(stg + L.rec_bytes + L.hdr_bytes, s1);
              } else {
                tile_step(tg.a, stg + L.hdr_bytes, stg, true);
                tile_step(tg.a + 1, stg + L.rec_bytes + L.hdr_bytes, stg + L.rec_bytes, true);
              }
            } else {
              for (int k = 0; k < n; ++k) {
                if (!((vmask >> k) & 1u)) continue;  // tile of a missing block
                const uint8_t* rec = stg + k * L.rec_bytes;
                tile_step(tg.a + k, rec + L.hdr_bytes, rec, true);
              }
            }
          } else {
            int walk = 0;        // smem offset of the next tile (headers inline)
            int rpos = tg.rpos;  // position of tile tg.a + k in its record
            for (int k = 0; k < n; ++k) {
              const bool hdr = F::kInt && (rpos == 0 || (tg.first && k == 0));
              const int hoff = walk;
              if (hdr) walk += L.hdr_bytes;
              const uint8_t* tile = stg + walk;
              walk += L.tile_bytes;
              if (++rpos == L.tpg) rpos = 0;
              if (!((vmask >> k) & 1u)) continue;  // tile of a missing block
              if constexpr (F::kFp8) {
                // the step's token (one-token append folded into this launch) lies in the last tile
                if (p.fp8_append && tg.a + k == ((sg.qn - 1) >> 4) &&
                    (long long)p.seq_lens[sg.b] + 1 <= tmax_tok)
                  fp8_append_token(p, const_cast<uint8_t*>(tile), sg.b, sg.h, tg.a + k, (sg.qn - 1) & 15, lane);
              }
              tile_step(tg.a + k, tile, stg + hoff, hdr);
            }
          }
        }
        // hand the slot back to the producer (shared-memory reads and writes of the slot
        // ordered before the bulk copies that will overwrite it)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        ++n_consumed;
        if (++c_slot == nst) c_slot = 0;
        pump();
      }

      // ---- finalise the warp's state (output layout: columns 2q, 2q + 1) into its merge record ----
      float lsum = stt.l;  // column r: summed over the row's token lanes q
      lsum += __shfl_xor_sync(kFull, lsum, 1);
      lsum += __shfl_xor_sync(kFull, lsum, 2);
      // m and l of columns 2q and 2q + 1 (held by the score lanes of rows 2q, 2q + 1)
      float mo[2], lo2[2];
      mo[0] = __shfl_sync(kFull, stt.m, 8 * q);
      mo[1] = __shfl_sync(kFull, stt.m, 8 * q + 4);
      lo2[0] = __shfl_sync(kFull, lsum, 8 * q);
      lo2[1] = __shfl_sync(kFull, lsum, 8 * q + 4);
      // zero-point sums: column r in the W layout, summed over the token lanes q; head 2q (+1) is at lane 8q (+4)
      float zo[2][NGV];
#pragma unroll
      for (int jg = 0; jg < NGV; ++jg) {
        float z = stt.zacc[jg];
        z += __shfl_xor_sync(kFull, z, 1);
        z += __shfl_xor_sync(kFull, z, 2);
        zo[0][jg] = __shfl_sync(kFull, z, 8 * q);
        zo[1][jg] = __shfl_sync(kFull, z, 8 * q + 4);
      }
      // o = sum of W * (Value operand) with W = p s kPrescale / S; integer layers: the
      // accumulators hold code units (2^-24 on rows r, FT::kVHi times that on rows r + 8)
      // and the zero-point sum sum W z is subtracted
      const float unit = stt.S / kPrescale;
      constexpr float kC0 = F::kInt ? kCodeUnit : 1.f, kC1 = F::kInt ? kCodeUnit / F::kVHi : 1.f;
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          const bool empty = mo[e] == -INFINITY;
          const float z = F::kInt ? zo[e][mb * NGV / 8] : 0.f;
          stt.o[mb][e] = empty ? 0.f : fmaf(stt.o[mb][e], kC0, -z) * unit;
          stt.o[mb][2 + e] = empty ? 0.f : fmaf(stt.o[mb][2 + e], kC1, -z) * unit;
        }
      if (sp_acc) {  // dense-and-sparse: the sparse Value sums of columns 2q, 2q + 1
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            const float* sr = sp_acc + (2 * q + e) * kSparseRow + 16 * mb + r;
            if (mo[e] != -INFINITY) {
              stt.o[mb][e] += sr[0];
              stt.o[mb][2 + e] += sr[8];
            }
          }
      }
      // ---- fold the warps pairwise into NW/2 merge records: warp w + NW/2 writes record w, then
      // warp w folds its own state into it ----
      if (warp >= NR) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 2 * q + e;
          if (hh < g) {
            float* rr = my_rec + hh * kMergeStride;
            if (r == 0) {
              rr[0] = mo[e];
              rr[1] = lo2[e];
            }
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
              rr[4 + 16 * mb + r] = stt.o[mb][e];
              rr[4 + 16 * mb + r + 8] = stt.o[mb][2 + e];
            }
          }
        }
      }
      __syncthreads();
      if (warp < NR) {
        float mr[2], lr[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = min(2 * q + e, g - 1);
          mr[e] = my_rec[hh * kMergeStride];
          lr[e] = my_rec[hh * kMergeStride + 1];
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 2 * q + e;
          if (hh < g) {
            float* rr = my_rec + hh * kMergeStride;
            const float M = fmaxf(mr[e], mo[e]);
            const float ar = mr[e] == -INFINITY ? 0.f : exp2f(mr[e] - M);
            const float aw = mo[e] == -INFINITY ? 0.f : exp2f(mo[e] - M);
            if (r == 0) {
              rr[0] = M;
              rr[1] = ar * lr[e] + aw * lo2[e];
            }
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
              const int c0 = 4 + 16 * mb + r, c1 = c0 + 8;
              rr[c0] = fmaf(ar, rr[c0], aw * stt.o[mb][e]);
              rr[c1] = fmaf(ar, rr[c1], aw * stt.o[mb][2 + e]);
            }
          }
        }
      }
      __syncthreads();
      // ---- merge the warps' records; write the partial of (b, h), or the result when this CTA owns the pair ----
      {
        const int b = sg.b, h = sg.h;
        const long long pair = (long long)b * H + h;
        const long long slot = (long long)blockIdx.x + pair;
        const long long P0 = sg.pair_start, P1 = sg.pair_start + sg.units;
        const long long c_lo = ((P0 + 1) * C - 1) / U, c_hi = (P1 * C - 1) / U;
        const bool whole = p.fuse && c_lo == c_hi;  // no other CTA touches this pair
        const int rstride = p.merge_bytes / 4;
        for (int i = tid; i < g * 128; i += NT) {
          const int hr = i >> 7, c = i & 127;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < NR; ++w) M = fmaxf(M, recs[w * rstride + hr * kMergeStride]);
          float Lsum = 0.f, O = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NR; ++w) {
              const float* rw = recs + w * rstride + hr * kMergeStride;
              const float f = exp2f(rw[0] - M);  // 0 for a warp without tiles (m = -inf)
              Lsum = fmaf(rw[1], f, Lsum);
              O = fmaf(rw[4 + c], f, O);
            }
          }
          const bool empty = !(Lsum > 0.f);
          const float o = empty ? 0.f : O / Lsum;
          const float l2 = empty ? -INFINITY : M + log2f(Lsum);
          if (whole) {
            write_out(p, b, h, hr, c, o, l2);
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
            float* wsc = recs;  // the warps' records are read: reuse the first one for the weights
            if (na <= 8) {
              // few partials: each output loads its head's lse values and its partial outputs in
              // one round trip, then sums in contributor order
              for (int i = tid; i < g * 128; i += NT) {
                const int hr = i >> 7, c = i & 127;
                float ls[8], v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const long long sl = j < na ? (long long)act[j] + pair : 0;
                  ls[j] = j < na ? __ldcg(&p.ws_lse[sl * g + hr]) : -INFINITY;
                  v[j] = j < na ? __ldcg(&p.ws_o[(sl * g + hr) * 128 + c]) : 0.f;
                }
                float M = -INFINITY, Lsum = 0.f, O = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (j < na) M = fmaxf(M, ls[j]);
                if (M != -INFINITY) {
#pragma unroll
                  for (int j = 0; j < 8; ++j)
                    if (j < na) {
                      const float f = exp2f(ls[j] - M);
                      Lsum += f;
                      O = fmaf(f, v[j], O);
                    }
                }
                const bool empty = !(Lsum > 0.f);
                write_out(p, b, h, hr, c, empty ? 0.f : O / Lsum, empty ? -INFINITY : M + log2f(Lsum));
              }
            } else if (na <= kMaxParts) {
              // every partial's lse at once: row hr, column k
              for (int i = tid; i < g * na; i += NT) {
                const int hr = i / na, k2 = i - hr * na;
                wsc[hr * kMergeStride + k2] = __ldcg(&p.ws_lse[((long long)act[k2] + pair) * g + hr]);
              }
              __syncthreads();
              if (tid < g) {  // per head: the largest lse, the weights 2^(lse - M) and their sum
                float* wr = wsc + tid * kMergeStride;
                float M = -INFINITY, Lsum = 0.f;
                for (int k2 = 0; k2 < na; ++k2) M = fmaxf(M, wr[k2]);
                if (M != -INFINITY)
                  for (int k2 = 0; k2 < na; ++k2) {
                    wr[k2] = exp2f(wr[k2] - M);
                    Lsum += wr[k2];
                  }
                wr[kMaxParts] = M;
                wr[kMaxParts + 1] = Lsum;
              }
              __syncthreads();
              for (int i = tid; i < g * 128; i += NT) {
                const int hr = i >> 7, c = i & 127;
                const float* wr = wsc + hr * kMergeStride;
                const float M = wr[kMaxParts], Lsum = wr[kMaxParts + 1];
                float O = 0.f;
                if (M != -INFINITY)
                  for (int k0 = 0; k0 < na; k0 += 8) {  // eight loads in flight, then the sums in order
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      v[j] = k0 + j < na ? __ldcg(&p.ws_o[(((long long)act[k0 + j] + pair) * g + hr) * 128 + c]) : 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      if (k0 + j < na) O = fmaf(wr[k0 + j], v[j], O);
                  }
                const bool empty = !(Lsum > 0.f);
                write_out(p, b, h, hr, c, empty ? 0.f : O / Lsum, empty ? -INFINITY : M + log2f(Lsum));
              }
            } else {
              // more partials than the list holds (tiny per-CTA ranges): walk [c_lo, c_hi]
              for (int i = tid; i < g * 128; i += NT) {
                const int hr = i >> 7, c = i & 127;
                float M = -INFINITY, Lsum = 0.f, O = 0.f;
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
                const bool empty = !(Lsum > 0.f);
                write_out(p, b, h, hr, c, empty ? 0.f : O / Lsum, empty ? -INFINITY : M + log2f(Lsum));
              }
            }
          }
        }
        if (s + 1 < nseg) load_q(segs[s + 1]);
      }
      __syncthreads();
    }
    if constexpr (BF) cp_async_wait<0>();  // no cp.async left in flight when the warp moves on or exits
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
template <int FMT, int NGV, bool BF, bool MQ, bool ONE, bool ROPE = false, bool OUT = false, bool KA = false>
cudaError_t ensure_smem_attr(int smem) {
  static std::mutex mu;
  static int set_for[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && set_for[dev] >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_kernel<FMT, NGV, BF, MQ, ONE, ROPE, OUT, KA>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) set_for[dev] = smem;
  return e;
}

template <int FMT, int NGV, bool BF, bool MQ, bool ONE, bool ROPE = false, bool OUT = false, bool KA = false>
cudaError_t launch_variant(const DecodeParams& p, int smem, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr<FMT, NGV, BF, MQ, ONE, ROPE, OUT, KA>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<FMT, NGV, BF, MQ, ONE, ROPE, OUT, KA>, dim3(p.num_ctas),
                    dim3(DecodeWarps<FMT>::kThreads), (size_t)smem, stream, p);
}

// FP8 layers without sink tokens (no bf16 tiles) take the variant without the bf16
// path; several query tokens per sequence take the multi-query variant; integer
// layers with one tile per Key group the straight-line variant.
template <int FMT, int NGV>
cudaError_t launch_decode_t(const DecodeParams& p, int smem, cudaStream_t stream) {
  const bool ka = p.n_query == 1 && p.g <= 4;  // few query columns: the Key tile as the A operand
  if constexpr (FT<FMT>::kFp8) {
    if (p.L.S == 0) {
      if (ka)  // one tile per record (contiguous store): the straight-line variant
        return p.L.tpg == 1 ? launch_variant<FMT, NGV, false, false, true, false, false, true>(p, smem, stream)
                            : launch_variant<FMT, NGV, false, false, false, false, false, true>(p, smem, stream);
      return p.n_query > 1 ? launch_variant<FMT, NGV, false, true, false>(p, smem, stream)
                           : launch_variant<FMT, NGV, false, false, false>(p, smem, stream);
    }
    if (ka) return launch_variant<FMT, NGV, true, false, false, false, false, true>(p, smem, stream);
    return p.n_query > 1 ? launch_variant<FMT, NGV, true, true, false>(p, smem, stream)
                         : launch_variant<FMT, NGV, true, false, false>(p, smem, stream);
  } else {
    if (p.L.k_out || p.L.v_out) {  // dense-and-sparse: Value groups of 64 or 128 channels, one query token
      if constexpr (NGV <= 2) {
        return p.L.tpg == 1 ? launch_variant<FMT, NGV, true, false, true, false, true>(p, smem, stream)
                            : launch_variant<FMT, NGV, true, false, false, false, true>(p, smem, stream);
      } else {
        return cudaErrorInvalidValue;
      }
    }
    if (p.L.rope) {  // pre-RoPE Keys: Value groups of 64 or 128 channels, one query token (host-checked)
      if constexpr (NGV <= 2) {
        return p.L.tpg == 1 ? launch_variant<FMT, NGV, true, false, true, true>(p, smem, stream)
                            : launch_variant<FMT, NGV, true, false, false, true>(p, smem, stream);
      } else {
        return cudaErrorInvalidValue;
      }
    }
    if (ka)
      return p.L.tpg == 1 ? launch_variant<FMT, NGV, true, false, true, false, false, true>(p, smem, stream)
                          : launch_variant<FMT, NGV, true, false, false, false, false, true>(p, smem, stream);
    if (p.L.tpg == 1)
      return p.n_query > 1 ? launch_variant<FMT, NGV, true, true, true>(p, smem, stream)
                           : launch_variant<FMT, NGV, true, false, true>(p, smem, stream);
    return p.n_query > 1 ? launch_variant<FMT, NGV, true, true, false>(p, smem, stream)
                         : launch_variant<FMT, NGV, true, false, false>(p, smem, stream);
  }
}

// Resident CTAs per SM (the variant with the bf16 path, the larger one; several
// query tokens: the multi-query variant).
template <int FMT, int NGV, bool MQ>
cudaError_t occupancy_variant(int smem, int* n) {
  cudaError_t e = ensure_smem_attr<FMT, NGV, true, MQ, false>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, decode_kernel<FMT, NGV, true, MQ, false, false, false, false>,
                                                       DecodeWarps<FMT>::kThreads, smem);
}
template <int FMT, int NGV>
cudaError_t occupancy_t(int g, int multi, int smem, int* n) {
  (void)g;
  return multi ? occupancy_variant<FMT, NGV, true>(smem, n) : occupancy_variant<FMT, NGV, false>(smem, n);
}

}  // namespace kvq
