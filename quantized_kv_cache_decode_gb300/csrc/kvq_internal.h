// Internal descriptors shared by the host API (kvq_api.cpp) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kMaxGqa = 8;
constexpr int kMaxBatch = 2048;
constexpr int kMaxGroupTokens = 256;  // Key group length the append kernel stages in shared memory
// dense-and-sparse decode: floats per query column of a warp's sparse Value sums in shared
// memory (128 channels + 4 pad, so that the 8 columns' rows start in different banks)
constexpr int kSparseRow = 132;

// Warps per decode CTA (one CTA per SM; the kernel's DecodeWarps states the same):
// 8 for 8-bit codes, else 12 (at most 168 registers a thread).
inline int decode_warps(int fmt) { return fmt == KVQ_FMT_INT8 ? 8 : 12; }

// The decode-kernel instantiation that serves a layer's format.  A bf16 layer
// has no quantized tiles, so any instantiation runs only its bf16-tile path;
// the 4-bit one (12 warps) is used.
inline int kernel_format(int fmt) { return fmt == KVQ_FMT_BF16 ? KVQ_FMT_INT4 : fmt; }

// Validated, derived form of kvq_layer_config.
struct LayerDesc {
  int H, d, fmt, bits, fp8;
  int e5m2;        // FP8 layer in E5M2 (else E4M3)
  int bf16;        // unquantized layer: every token after the sink in the bf16 buffers (W = their rows)
  int G, Gv, ngv, R, S, W;  // W = R + G ring slots (0 for FP8)
  int paged, P, cap, num_blocks, mbps;
  int rb;          // bytes of one token row of codes (d * bits / 8)
  int tile_bytes;  // one 16-token tile: K codes, V codes, (INT) V scales, V zeros
  int hdr_bytes;   // record header: K scale + K zero of the record's Key group (INT: 1024, FP8: 0)
  int tpg;         // tiles per record
  int rec_bytes;   // hdr_bytes + tpg * tile_bytes
  int nrec;        // contiguous: records per (seq, head)
  long long block_bytes;  // paged: H records
  int rope;               // Keys stored before RoPE, rotated at their position by the decode
  float rope_base;
  int k_out, v_out;       // dense-and-sparse: entries kept exactly per quantized Key / Value row
  int sp_off;             // byte offset of a tile's K sparse entries (the V ones follow, 64 * k_out later)
};

struct CachePtrs {
  void* qstore;
  void* block_pool;
  const int32_t* block_table;
  void* resid_k;
  void* resid_v;
  void* sink_k;
  void* sink_v;
  const float* k_tscale;
  const float* v_tscale;
};

struct DecodeParams {
  LayerDesc L;
  CachePtrs C;
  const void* q;  // bf16 [B][Hq][d]
  int Hq, g, batch;  // g: query columns per kv head = gh * n_query
  int gh;            // query heads per kv head
  int n_query;       // query tokens per sequence (1: plain decode)
  const int32_t* seq_lens;
  int len_add;       // tokens added to each seq_lens[b] (1: the call appended the step's token first)
  // FP8 layers without sink tokens, one-token append folded into the decode: the warp that
  // reads the new token's tile writes the token's codes (from k_new, v_new: bf16 [B][H][d])
  int fp8_append;
  const void* k_new;
  const void* v_new;
  float scale_log2;  // softmax_scale * log2(e)
  int num_ctas;      // CTAs of the decode grid (partial slot space = num_ctas + batch*H)
  int nst;           // pipeline stages per warp
  int stage_bytes;   // bytes of one stage
  int tps;           // quantized tiles per stage
  int item_tiles;    // quantized tiles per claimed work item (a multiple of the record size)
  int bf_weight;     // work units charged to a bf16 tile (quantized tiles cost 1)
  int bf_joint;      // 1: a bf16 tile's K and V rows (2 x 4 KB) share one stage; 0: one stage each
  float* ws_o;       // [slots][g][d] normalised partial outputs
  float* ws_lse;     // [slots][g] log2-domain log-sum-exp of each partial
  int* ws_prefix;    // [batch + 2]: per-sequence unit prefix, then the CTA count (written by CTA 0 for the combine)
  uint32_t* status;
  int merge_bytes;   // bytes of one warp's merge record in shared memory (g heads)
  int withhold_copy; // self-test only: CTA 0, warp 0 withholds its first bulk copy (its wait must run out)
  // fused combine: the last CTA to finish a (sequence, kv head) pair merges its partials
  int fuse;
  unsigned* counters;  // [batch * H] arrival counters, zero between calls
  void* out;
  int out_bf16;
  float* lse;
  // pre-RoPE Keys: per rotation pair i, frac(theta_i / 2 pi) * 2^64 (the angle of position t
  // in turns is t * rope_turn[i] mod 2^64, fixed point)
  unsigned long long rope_turn[64];
};

struct CombineParams {
  int H, g, Hq, batch, num_ctas;
  const int* ws_prefix;
  const float* ws_o;
  const float* ws_lse;
  void* out;
  int out_bf16;
  float* lse;
};

struct AppendParams {
  LayerDesc L;
  CachePtrs C;
  const void* k_new;  // bf16 [B][H][n_new][d]
  const void* v_new;
  int n_new, batch;
  const int32_t* seq_lens;
  uint32_t* status;
};

struct DequantParams {
  LayerDesc L;
  CachePtrs C;
  const int32_t* seq_lens;
  int batch, max_tokens;
  float* k_out;
  float* v_out;
  uint32_t* status;
};

// ---- launchers (defined in the .cu files) --------------------------------
// decode: one kernel instantiation per (format, Value groups per token)
cudaError_t decode_smem_and_occupancy(const LayerDesc& L, int batch, int* smem_bytes, int* nst, int* stage_bytes,
                                      int* ctas_per_sm);
cudaError_t launch_decode(const DecodeParams& p, int smem_bytes, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_decode_int2(const DecodeParams& p, int smem, cudaStream_t s);
cudaError_t launch_decode_int4(const DecodeParams& p, int smem, cudaStream_t s);
cudaError_t launch_decode_int8(const DecodeParams& p, int smem, cudaStream_t s);
cudaError_t launch_decode_fp8(const DecodeParams& p, int smem, cudaStream_t s);
cudaError_t launch_decode_fp8_e5m2(const DecodeParams& p, int smem, cudaStream_t s);
// multi: the multi-query variant (several query tokens per sequence)
cudaError_t occupancy_decode_int2(int ngv, int g, int multi, int smem, int* n);
cudaError_t occupancy_decode_int4(int ngv, int g, int multi, int smem, int* n);
cudaError_t occupancy_decode_int8(int ngv, int g, int multi, int smem, int* n);
cudaError_t occupancy_decode_fp8(int ngv, int g, int multi, int smem, int* n);
cudaError_t occupancy_decode_fp8_e5m2(int ngv, int g, int multi, int smem, int* n);

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n_parts, long long rows, void* out,
                             int out_bf16, float* lse_out, cudaStream_t stream);
// scale = amax / fmax (1 when amax == 0), fmax the format's largest finite value
cudaError_t launch_fp8_calibrate(const void* x, size_t n, float fmax, float* scale_out, cudaStream_t stream);
cudaError_t launch_dequantize(const DequantParams& p, cudaStream_t stream);

}  // namespace kvq
