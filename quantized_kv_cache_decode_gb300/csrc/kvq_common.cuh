// Device helpers shared by the libkvq kernels (sm_103a): inline PTX for the
// tensor-core MMA, bulk asynchronous copies (TMA engine), mbarriers, packed
// f16/bf16 conversions, and the layout arithmetic of the cache.
#pragma once

#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

// --------------------------------------------------------------------------
// small PTX wrappers
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// d = (a & b) | c
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// packed f16 fused multiply-add, one rounding
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// two E4M3FN bytes (low byte -> low half) to two f16 values, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t lo16) {
  uint32_t d;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(d) : "r"(lo16));
  return d;
}

// four E4M3FN bytes -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi), exact
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b; }"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Four E5M2 bytes -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi), exact: an
// E5M2 code is the high byte of the binary16 with the same value (both have a
// 5-bit exponent of bias 15), so each byte only moves to the top of its half.
__device__ __forceinline__ void e5m2x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, 0, 0x1404;" : "=r"(lo) : "r"(w));
  asm("prmt.b32 %0, %1, 0, 0x3424;" : "=r"(hi) : "r"(w));
}

// f32 pair -> packed f16 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float2 unpack_f16(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
  float2 r;
  r.x = __uint_as_float(v << 16);
  r.y = __uint_as_float(v & 0xFFFF0000u);
  return r;
}

// split two f32 values into hi + lo 16-bit pairs (hi = rn(x), lo = rn(x - hi))
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_f16(x0, x1);
  float2 h = unpack_f16(hi);
  lo = pack_f16(x0 - h.x, x1 - h.y);
}
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  float2 h = unpack_bf16(hi);
  lo = pack_bf16(x0 - h.x, x1 - h.y);
}

// Packed fp32 pairs (sm_100 and later): each half is one IEEE round-to-nearest
// operation, exactly as the scalar instruction would give it.
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mul.rn.f32x2 rd, ra, rb; "
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 sub_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; sub.rn.f32x2 rd, ra, rb; "
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mov.b64 rc, {%6, %7}; "
      "fma.rn.f32x2 rd, ra, rb, rc; mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// hi = rn_f16(x), lo = rn_f16(x - hi) of a pair: hi + lo holds x to about 22 bits
__device__ __forceinline__ void split_f16x2(float2 x, uint32_t& hi, uint32_t& lo) {
  hi = pack_f16(x.x, x.y);
  const float2 h = unpack_f16(hi);
  const float2 r = sub_f32x2(x, h);
  lo = pack_f16(r.x, r.y);
}

// D += A * B, m16n8k16, fp32 accumulate
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// --------------------------------------------------------------------------
// mbarrier + bulk copy (global -> shared through the TMA engine)
// --------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One test of the phase; a thread whose phase is not complete yet is suspended by
// the hardware until it completes or about kSuspendHintNs pass (a waiting warp
// does not spin through issue slots the other warps of the SM could use).
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of the barrier to complete, at most ~`limit` SM cycles.
// Returns false when the bound ran out (the caller records KVQ_DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}
// The cache is read once per decode: its lines are marked first to be evicted from
// L2, so the stream does not push out what the next kernels reuse (their code,
// the query, the partials of the merge).  Measured on GB300: a decode launched
// right after another kernel ran 10 us (15 %) faster with the hint.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// 16 bytes global -> shared by the calling thread (cp.async, L1 bypassed); the
// copies a thread issued are grouped by cp_async_commit and waited for with
// cp_async_wait<n> (all but the n most recent groups complete).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// CTAs that share the work units of a decode launch: the grid, or fewer when the
// units are so few that a CTA would get less than kMinCtaUnits of them (its
// fixed costs, and the merge of many tiny partials, would outweigh its share);
// the CTAs beyond that count have empty ranges (see range_ctas for the choice
// the decode kernel makes, which it records for the two-launch merge).
constexpr long long kMinCtaUnits = 16;
__host__ __device__ __forceinline__ long long working_ctas(long long grid, long long U) {
  const long long c = U / kMinCtaUnits;
  return c < 1 ? 1 : (c < grid ? c : grid);
}

// CTAs that take the units of a decode launch.  When every sequence holds the
// same number of units (equal lengths) and the B*H (sequence, kv head) pairs
// split evenly into k = ceil(pairs / grid) pairs per CTA over at least 80 % of
// the grid, each of those CTAs takes k whole pairs: no pair is cut across CTAs,
// so no partial is written, fenced and merged, and no warp waits on a pair's
// other part.  Measured on GB300: the 70B INT4 layer (128 pairs of 8192 tokens on
// 152 SMs) 76.0 -> 65.1 us; a larger k that leaves SMs idle did not pay (INT2 MHA
// layer, 1024 pairs on 128 instead of 152 CTAs: 1554 -> 1765 us).  Otherwise
// equal unit ranges over working_ctas.  The decode kernel records its choice for
// the two-launch merge.
__host__ __device__ __forceinline__ long long range_ctas(long long grid, long long U, long long pairs, bool equal) {
  if (equal && pairs > 0 && U > 0) {
    const long long k = (pairs + grid - 1) / grid;
    if (pairs % k == 0 && (pairs / k) * 5 >= grid * 4) return pairs / k;
  }
  return working_ctas(grid, U);
}

// about one second at GB300 clocks
constexpr long long kWaitLimitCycles = 2000000000LL;

// Programmatic dependent launch.  The kernels of a decode step (append, decode,
// combine) are launched with programmatic stream serialisation allowed: a kernel
// may be scheduled onto free SMs while the previous kernel of the stream is still
// finishing.  Each of them first waits (pdl_wait) until the previous kernel has
// completed and its memory writes are visible -- before touching any global
// memory -- and then lets the next kernel of the stream be scheduled
// (pdl_trigger).  The overlap hides the launch and CTA scheduling of a kernel
// behind the tail of the one before it; the order of memory effects is the plain
// stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl(void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

// FP8 encode of one fp32 value (round to nearest even, saturating to the largest finite code)
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

__device__ __forceinline__ void report(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// --------------------------------------------------------------------------
// token accounting of one (sequence, head)
// --------------------------------------------------------------------------
struct TokenSplit {
  int n_sink;  // bf16 sink tokens
  int qn;      // quantized tokens
  int r;       // bf16 residual tokens
};

__host__ __device__ __forceinline__ TokenSplit split_tokens(int T, const LayerDesc& L) {
  TokenSplit s;
  s.n_sink = T < L.S ? T : L.S;
  int n = T - s.n_sink;
  if (L.fp8) {
    s.qn = n;
    s.r = 0;
  } else if (L.bf16) {
    s.qn = 0;
    s.r = n;
  } else {
    int k = (n - L.R) >= 0 ? (n - L.R) / L.G : 0;
    s.qn = k * L.G;
    s.r = n - s.qn;
  }
  return s;
}

// Largest token count one (sequence, head) can hold.
__host__ __device__ __forceinline__ long long max_tokens(const LayerDesc& L) {
  long long qcap = L.paged ? (long long)L.mbps * L.P : (long long)L.cap;
  if (L.fp8) return L.S + qcap;
  if (L.bf16) return (long long)L.S + L.W;
  return L.S + qcap + L.R + L.G - 1;
}

// Record r of (sequence b, kv head h) in the quantized store, or nullptr (with
// KVQ_DEV_BAD_BLOCK reported) when its block-table entry is outside the pool.
// A record is [header (INT: K scale, K zero)][tpg tiles]; see include/kvq.h.
__device__ __forceinline__ const uint8_t* record_addr(const LayerDesc& L, const CachePtrs& C, int b, int h,
                                                     long long r, uint32_t* status) {
  if (L.paged) {
    const int blk = C.block_table[(long long)b * L.mbps + r];
    if (blk < 0 || blk >= L.num_blocks) {
      report(status, KVQ_DEV_BAD_BLOCK);
      return nullptr;
    }
    return reinterpret_cast<const uint8_t*>(C.block_pool) + (long long)blk * L.block_bytes +
           (long long)h * L.rec_bytes;
  }
  return reinterpret_cast<const uint8_t*>(C.qstore) + (((long long)b * L.H + h) * L.nrec + r) * L.rec_bytes;
}

// Tile i (quantized tokens 16i .. 16i+15) inside its record.
__device__ __forceinline__ const uint8_t* tile_in_record(const LayerDesc& L, const uint8_t* rec, long long i) {
  return rec + L.hdr_bytes + (long long)(i % L.tpg) * L.tile_bytes;
}

// bf16 row of bf16-list token index xb (sink tokens first, then residual tokens in order)
__device__ __forceinline__ const __nv_bfloat16* bf16_row(const LayerDesc& L, const __nv_bfloat16* sink,
                                                         const __nv_bfloat16* ring, int b, int h, int xb,
                                                         const TokenSplit& ts) {
  const long long pair = (long long)b * L.H + h;
  if (xb < ts.n_sink) return sink + (pair * L.S + xb) * L.d;
  const int slot = (ts.qn + (xb - ts.n_sink)) % L.W;
  return ring + (pair * L.W + slot) * L.d;
}

// --------------------------------------------------------------------------
// code tiles in fragment order
// --------------------------------------------------------------------------
// A 16-token tile stores its Key codes and its Value codes, each a 16 x 128
// matrix of codes, in the register order of the mma.sync m16n8k16 A operand,
// so that each lane fetches its own operand words with 16-byte shared-memory
// loads (consecutive lanes 16 bytes apart: no bank conflicts) and unpacks them
// in registers.  Step s of the A operand (s = 0..7) gives lane 4r+q four
// registers, each a pair (half 0, half 1):
//   reg 0: (row r, col 2q+h)    reg 1: (row r+8, col 2q+h)
//   reg 2: (row r, col 2q+8+h)  reg 3: (row r+8, col 2q+8+h)
// Keys:   rows = the 16 tokens, step s covers channels 16s..16s+15, column
//         2q + (e & 1) + 8 (e >> 1) of the step holding channel 16s + 4q + e.
// Values: rows = channels 16s + i (i = 0..15), columns = the 16 tokens.
// Word w of lane l sits at byte ((w >> 2) * 32 + l) * 16 + (w & 3) * 4; a
// lane owns rb / 8 words (rb = bytes of one token row of codes).
__host__ __device__ __forceinline__ void frag_pos(int bits, bool fp8, int lane, int step, int reg, int half,
                                                  int& byte, int& bit) {
  int w, bitpos;
  if (bits == 4) {  // one word per step: bits 4*reg + 16*half
    w = step;
    bitpos = 4 * reg + 16 * half;
  } else if (bits == 2) {  // one word per two steps: bits 8*(step&1) + 2*reg + 16*half
    w = step >> 1;
    bitpos = 8 * (step & 1) + 2 * reg + 16 * half;
  } else {  // 8-bit codes: two words per step (regs 0-1, regs 2-3)
    w = 2 * step + (reg >> 1);
    bitpos = 8 * (fp8 ? 2 * (reg & 1) + half : (reg & 1) + 2 * half);
  }
  byte = ((w >> 2) * 32 + lane) * 16 + (w & 3) * 4 + (bitpos >> 3);
  bit = bitpos & 7;
}

// Key code of (token t, channel c) inside the tile's Key part
__host__ __device__ __forceinline__ void ktile_pos(int bits, bool fp8, int t, int c, int& byte, int& bit) {
  const int e = c & 3;
  frag_pos(bits, fp8, 4 * (t & 7) + ((c >> 2) & 3), c >> 4, (t >> 3) + 2 * (e >> 1), e & 1, byte, bit);
}
// Value code of (token t, channel c) inside the tile's Value part
__host__ __device__ __forceinline__ void vtile_pos(int bits, bool fp8, int t, int c, int& byte, int& bit) {
  const int i = c & 15;
  frag_pos(bits, fp8, 4 * (i & 7) + ((t & 7) >> 1), c >> 4, (i >> 3) + 2 * (t >> 3), t & 1, byte, bit);
}

}  // namespace kvq
