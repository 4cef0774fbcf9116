// Host side of the libkvq C ABI: argument validation, cache layout, launch
// configuration and dispatch.  See include/kvq.h for the contract.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kMaxStages = 2;
constexpr int kStaticSmemMargin = 1024;           // the kernel's static __shared__ variables (384 B)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status make_desc(const kvq_layer_config* cfg, LayerDesc* L) {
  if (!cfg || !L) return KVQ_ERR_INVALID_ARG;
  memset(L, 0, sizeof(*L));
  if (cfg->num_kv_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (cfg->head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  const int f = cfg->format;
  if (f != KVQ_FMT_BF16 && f != KVQ_FMT_INT2 && f != KVQ_FMT_INT4 && f != KVQ_FMT_INT8 && f != KVQ_FMT_FP8_E4M3 &&
      f != KVQ_FMT_FP8_E5M2)
    return KVQ_ERR_INVALID_ARG;
  L->H = cfg->num_kv_heads;
  L->d = kHeadDim;
  L->fmt = f;
  L->fp8 = (f == KVQ_FMT_FP8_E4M3 || f == KVQ_FMT_FP8_E5M2);
  L->e5m2 = (f == KVQ_FMT_FP8_E5M2);
  L->bf16 = (f == KVQ_FMT_BF16);
  L->bits = (L->fp8 || L->bf16) ? 8 : f;  // bf16: nominal, no codes are stored
  L->rb = L->d * L->bits / 8;
  L->S = cfg->sink_tokens;
  if (L->S < 0) return KVQ_ERR_INVALID_ARG;
  L->rope_base = cfg->rope_base;
  L->rope = cfg->rope_base != 0.f;
  L->k_out = cfg->k_outliers;
  L->v_out = cfg->v_outliers;
  if (L->k_out < 0 || L->k_out > 8 || L->v_out < 0 || L->v_out > 8) return KVQ_ERR_INVALID_ARG;
  if (L->k_out || L->v_out) {
    if (f == KVQ_FMT_BF16 || f == KVQ_FMT_FP8_E4M3 || f == KVQ_FMT_FP8_E5M2 || L->rope) return KVQ_ERR_UNSUPPORTED;
    if (cfg->v_group_dims != 64 && cfg->v_group_dims != 128) return KVQ_ERR_UNSUPPORTED;
  }
  if (L->rope) {
    if (!(cfg->rope_base > 1.f) || !(cfg->rope_base < 3.0e38f)) return KVQ_ERR_INVALID_ARG;
    if (f == KVQ_FMT_BF16 || f == KVQ_FMT_FP8_E4M3 || f == KVQ_FMT_FP8_E5M2) return KVQ_ERR_UNSUPPORTED;
    if (cfg->v_group_dims != 64 && cfg->v_group_dims != 128) return KVQ_ERR_UNSUPPORTED;
  }
  if (L->bf16) {
    // every token after the sink lives in the bf16 buffers, row t - S; nothing is quantized
    if (cfg->paged) return KVQ_ERR_UNSUPPORTED;
    if (cfg->capacity_tokens < 1) return KVQ_ERR_INVALID_ARG;
    L->G = 16;
    L->Gv = kHeadDim;
    L->R = cfg->capacity_tokens;
    L->W = cfg->capacity_tokens;
    L->ngv = 1;
    L->tile_bytes = 32 * L->rb + 128;
    L->hdr_bytes = 2 * L->d * 4;
    L->tpg = 1;
    L->rec_bytes = L->hdr_bytes + L->tile_bytes;
    return KVQ_OK;  // cap = nrec = 0: no quantized store
  }
  if (L->fp8) {
    if (cfg->k_group_tokens != 1 || cfg->residual_tokens != 0) return KVQ_ERR_INVALID_ARG;
    L->G = 1;
    L->Gv = kHeadDim;
    L->R = 0;
    L->W = 0;
  } else {
    L->G = cfg->k_group_tokens;
    L->Gv = cfg->v_group_dims;
    L->R = cfg->residual_tokens;
    if (L->G < 16 || L->G % 16 != 0 || L->R < 0) return KVQ_ERR_INVALID_ARG;
    if (L->G > kMaxGroupTokens) return KVQ_ERR_UNSUPPORTED;
    if (L->Gv != 16 && L->Gv != 32 && L->Gv != 64 && L->Gv != 128) return KVQ_ERR_INVALID_ARG;
    L->W = L->R + L->G;
  }
  L->ngv = L->d / L->Gv;
  L->paged = cfg->paged ? 1 : 0;
  L->tile_bytes = 32 * L->rb + (L->fp8 ? 0 : 128 * L->ngv);
  L->sp_off = L->tile_bytes;  // dense-and-sparse entries after the Value scales and zero-points
  L->tile_bytes += 64 * (L->k_out + L->v_out);
  L->hdr_bytes = L->fp8 ? 0 : 2 * L->d * 4;
  if (L->paged) {
    L->P = cfg->block_tokens;
    L->num_blocks = cfg->num_blocks;
    L->mbps = cfg->max_blocks_per_seq;
    if (L->P < 16 || L->P % 16 != 0 || L->num_blocks < 1 || L->mbps < 1) return KVQ_ERR_INVALID_ARG;
    if (!L->fp8 && L->P != L->G) return KVQ_ERR_INVALID_ARG;
    L->tpg = L->P / 16;
  } else {
    L->cap = cfg->capacity_tokens;
    if (L->cap < 0 || L->cap % 16 != 0 || (!L->fp8 && L->cap % L->G != 0)) return KVQ_ERR_INVALID_ARG;
    L->tpg = L->fp8 ? 1 : L->G / 16;
  }
  L->rec_bytes = L->hdr_bytes + L->tpg * L->tile_bytes;
  L->nrec = L->paged ? 0 : L->cap / (16 * L->tpg);
  L->block_bytes = (long long)L->rec_bytes * L->H;
  return KVQ_OK;
}

CachePtrs make_ptrs(const kvq_layer_cache* c) {
  CachePtrs p;
  p.qstore = c->qstore;
  p.block_pool = c->block_pool;
  p.block_table = c->block_table;
  p.resid_k = c->resid_k;
  p.resid_v = c->resid_v;
  p.sink_k = c->sink_k;
  p.sink_v = c->sink_v;
  p.k_tscale = c->k_tensor_scale;
  p.v_tscale = c->v_tensor_scale;
  return p;
}

// The buffers a config uses must be present and 16-byte aligned (bulk copies).
kvq_status check_cache(const LayerDesc& L, const kvq_layer_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  auto need = [](const void* p) { return p != nullptr && aligned16(p); };
  if (L.paged) {
    if (!need(c->block_pool) || !c->block_table) return KVQ_ERR_INVALID_ARG;
  } else if (L.cap > 0) {
    if (!need(c->qstore)) return KVQ_ERR_INVALID_ARG;
  }
  if (!L.fp8 && (!need(c->resid_k) || !need(c->resid_v))) return KVQ_ERR_INVALID_ARG;
  if (L.S > 0 && (!need(c->sink_k) || !need(c->sink_v))) return KVQ_ERR_INVALID_ARG;
  if (L.fp8 && (!c->k_tensor_scale || !c->v_tensor_scale)) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// Quantized tiles per pipeline stage: about `target` bytes of cache per stage.
int tiles_per_stage(const LayerDesc& L, int target) {
  const int per = L.tile_bytes + (L.hdr_bytes + L.tpg - 1) / L.tpg;
  return std::max(1, std::min(8, (target + per / 2) / per));
}

constexpr int kBfHalfBytes = 16 * 256;  // the K (or V) rows of a 16-token bf16 tile

// A stage holds a header slot, tps tiles and the record headers between them,
// or (layers with bf16 tokens) the K or V rows of a 16-token bf16 tile (both
// when the stage has room for them: see bf16_joint).  A bf16 layer has only
// bf16 tiles: its stages hold both halves.
int stage_bytes_of(const LayerDesc& L, int tps) {
  if (L.bf16) return 2 * kBfHalfBytes;
  // headers a stage can hold: with one tile per record, every tile's own; with a
  // stage no longer than a record, one (work items are then whole records, so a
  // stage never crosses a record boundary: it holds either the inline header of
  // the record it starts, or the header copied ahead of a mid-record start);
  // otherwise the header copied ahead plus one per record started inside it
  int hdrs;
  if (L.tpg == 1) hdrs = tps;
  else if (tps <= L.tpg) hdrs = 1;
  else hdrs = 1 + (tps + L.tpg - 1) / L.tpg;
  const int q = tps * L.tile_bytes + (L.hdr_bytes ? hdrs * L.hdr_bytes : 0);
  const bool bf16_tiles = L.S > 0 || !L.fp8;
  const int bf = bf16_tiles ? kBfHalfBytes : 0;
  return (std::max(q, bf) + 127) / 128 * 128;
}
bool bf16_joint(int stage_bytes) { return stage_bytes >= 2 * kBfHalfBytes; }

constexpr int kMergeFloats = 132;        // floats per query head of a merge record (kvq_decode.cuh)
constexpr int kQRowFloats = 144;         // floats per query column row in shared memory (kvq_decode.cuh)

// A warp's merge record in shared memory: m, l, -, - and 128 outputs per query head.
int merge_bytes_of(const LayerDesc& L, int g) {
  (void)L;
  return g * kMergeFloats * 4;
}

constexpr int kSegTableBytes = 16 * 80;  // kMaxSeg segment records of 80 bytes (kvq_decode.cuh)

int fixed_smem(int batch, int merge_bytes, int nw) {
  int prefix = ((batch + 1) * 4 + 15) / 16 * 16 + (batch * 4 + 15) / 16 * 16;  // unit prefix, token counts
  // per warp: barriers, block-table window; nw/2 merge records; the query rows (g + 1)
  const int g = merge_bytes / (kMergeFloats * 4);
  const int per_warp = kMaxStages * 8 + 32 * 4;
  return nw * per_warp + nw / 2 * merge_bytes + (g + 1) * kQRowFloats * 4 + kSegTableBytes + prefix;
}

cudaError_t occupancy_query(const LayerDesc& L, int g, int multi, int smem, int* n) {
  switch (kernel_format(L.fmt)) {
    case KVQ_FMT_INT2: return occupancy_decode_int2(L.ngv, g, multi, smem, n);
    case KVQ_FMT_INT4: return occupancy_decode_int4(L.ngv, g, multi, smem, n);
    case KVQ_FMT_INT8: return occupancy_decode_int8(L.ngv, g, multi, smem, n);
    case KVQ_FMT_FP8_E5M2: return occupancy_decode_fp8_e5m2(L.ngv, g, multi, smem, n);
    default: return occupancy_decode_fp8(L.ngv, g, multi, smem, n);
  }
}

// Resident CTAs per SM of the decode kernel for (device, format, Value groups,
// single- or multi-query variant, shared memory), cached: the answer never changes for a
// given device.
cudaError_t occupancy(const LayerDesc& L, int g, int multi, int smem, int* n) {
  struct Entry {
    int dev, fmt, ngv, multi, smem, n;
  };
  const int mq = multi ? 1 : 0;  // the multi-query variant is a kernel of its own
  static std::mutex mu;
  static Entry cache[256];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].dev == dev && cache[i].fmt == L.fmt && cache[i].ngv == L.ngv && cache[i].multi == mq &&
          cache[i].smem == smem) {
        *n = cache[i].n;
        return cudaSuccess;
      }
  }
  e = occupancy_query(L, g, multi, smem, n);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (used < 256) cache[used++] = Entry{dev, L.fmt, L.ngv, mq, smem, *n};
  return cudaSuccess;
}

// CTAs of the decode grid.  One per SM, except for layers whose decode is bound by
// HBM bandwidth alone (FP8 and bf16: a fraction of the SMs already saturates it)
// when the batch x kv-head pairs split evenly into k pairs per CTA over at least
// 80 % of the SMs: then every CTA's range is k whole pairs (for equal sequence
// lengths), so no pair is split and no partial is written, fenced and merged
// across CTAs.  Measured on GB300 with 128 pairs (B = 16, 8 kv heads, T = 8192):
// FP8 decode 61.0 -> 52.6 us, bf16 121.2 -> 108.4 us.  The 2/4/8-bit layers are
// bound by their warps' dependency chains and keep every SM: the kernel itself
// gives whole pairs to the CTAs when the lengths turn out equal (range_ctas), and
// a ragged batch uses them all.
int grid_ctas(const LayerDesc& L, int batch, int sms) {
  const long long pairs = (long long)batch * L.H;
  if (!(L.fp8 || L.bf16) || pairs < 1) return sms;
  const long long k = (pairs + sms - 1) / sms;  // pairs per CTA
  if (pairs % k == 0 && (pairs / k) * 5 >= (long long)sms * 4) return (int)(pairs / k);
  return sms;
}

struct DecodeGeom {
  int smem, nst, stage_bytes, tps, num_ctas, merge_bytes;
  size_t ws_bytes, off_lse, off_prefix, off_counters;
};

// Launch shape: one CTA per SM (see grid_ctas), two stages per warp (one being
// computed on, one in flight) of the largest size among about 8, 6, 4 and 2 KB
// that fits the shared memory.
kvq_status decode_geometry(const LayerDesc& L, int batch, int g, DecodeGeom* G, int multi = 0) {
  const int wsc = merge_bytes_of(L, g);
  const int nw = decode_warps(kernel_format(L.fmt));
  // pre-RoPE Keys: each warp keeps a copy of its current Key group's header (1 KB);
  // dense-and-sparse Values: each warp accumulates the sparse part of its outputs (8 x kSparseRow floats)
  const int fixed = fixed_smem(batch, wsc, nw) + (L.rope ? nw * 1024 : 0) +
                    (L.v_out ? nw * 8 * kSparseRow * (int)sizeof(float) : 0);
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVQ_ERR_CUDA;
  const int n = kMaxStages;  // stages per warp (the kernel sizes its barriers and tags for kMaxStages)
  const int budget = 227 * 1024 - kStaticSmemMargin;
  int smem = 0, nst = 0, sb = 0, tps = 0;
  bool found = false;
  for (int target : {8192, 6144, 4096, 2048}) {
    const int t = tiles_per_stage(L, target);
    const int b = stage_bytes_of(L, t);
    if (fixed + nw * n * b > budget) continue;
    smem = fixed + nw * n * b;
    nst = n;
    sb = b;
    tps = t;
    found = true;
    break;
  }
  if (!found) return KVQ_ERR_UNSUPPORTED;
  if (occupancy(L, g, multi, smem, &per_sm) != cudaSuccess) return KVQ_ERR_CUDA;
  if (per_sm < 1) return KVQ_ERR_UNSUPPORTED;
  G->smem = smem;
  G->merge_bytes = wsc;
  G->nst = nst;
  G->stage_bytes = sb;
  G->tps = tps;
  G->num_ctas = grid_ctas(L, batch, sms);
  const size_t slots = (size_t)G->num_ctas + (size_t)batch * L.H;
  const size_t o_bytes = slots * g * kHeadDim * sizeof(float);
  const size_t l_bytes = slots * g * sizeof(float);
  G->off_lse = (o_bytes + 255) / 256 * 256;
  G->off_prefix = G->off_lse + (l_bytes + 255) / 256 * 256;
  // unit prefix [batch + 1] and the split pass's CTA count
  G->off_counters = G->off_prefix + ((size_t)(batch + 2) * sizeof(int) + 255) / 256 * 256;
  G->ws_bytes = G->off_counters + (size_t)batch * L.H * sizeof(unsigned);
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" {

kvq_status kvq_cache_layout(const kvq_layer_config* cfg, int32_t num_seqs, size_t bytes[KVQ_FIELD_COUNT]) {
  LayerDesc L;
  kvq_status st = make_desc(cfg, &L);
  if (st != KVQ_OK) return st;
  if (num_seqs < 0 || !bytes) return KVQ_ERR_INVALID_ARG;
  for (int i = 0; i < KVQ_FIELD_COUNT; ++i) bytes[i] = 0;
  const size_t pairs = (size_t)num_seqs * L.H;
  if (L.paged) {
    bytes[KVQ_FIELD_BLOCK_POOL] = (size_t)L.num_blocks * L.block_bytes;
  } else {
    bytes[KVQ_FIELD_QSTORE] = pairs * L.nrec * L.rec_bytes;
  }
  if (!L.fp8) {
    bytes[KVQ_FIELD_RESID_K] = pairs * L.W * L.d * 2;
    bytes[KVQ_FIELD_RESID_V] = bytes[KVQ_FIELD_RESID_K];
  }
  bytes[KVQ_FIELD_SINK_K] = pairs * L.S * L.d * 2;
  bytes[KVQ_FIELD_SINK_V] = bytes[KVQ_FIELD_SINK_K];
  return KVQ_OK;
}

kvq_status kvq_fp8_calibrate_format(const void* x, size_t n, int32_t format, float* scale_out, void* stream) {
  if (!scale_out || (n > 0 && !x)) return KVQ_ERR_INVALID_ARG;
  float fmax;
  if (format == KVQ_FMT_FP8_E4M3)
    fmax = 448.0f;  // largest finite E4M3FN value
  else if (format == KVQ_FMT_FP8_E5M2)
    fmax = 57344.0f;  // largest finite E5M2 value
  else
    return KVQ_ERR_INVALID_ARG;
  if (launch_fp8_calibrate(x, n, fmax, scale_out, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_fp8_calibrate(const void* x, size_t n, float* scale_out, void* stream) {
  return kvq_fp8_calibrate_format(x, n, KVQ_FMT_FP8_E4M3, scale_out, stream);
}

kvq_status kvq_quantize_append(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* k_new,
                               const void* v_new, int32_t n_new, const int32_t* seq_lens, int32_t batch,
                               uint32_t* dev_status, void* stream) {
  LayerDesc L;
  kvq_status st = make_desc(cfg, &L);
  if (st != KVQ_OK) return st;
  if ((st = check_cache(L, cache)) != KVQ_OK) return st;
  if (batch < 0 || batch > kMaxBatch || n_new < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0 || n_new == 0) return KVQ_OK;
  if (!k_new || !v_new || !seq_lens || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  if (!L.fp8 && !L.bf16 && ((long long)n_new + L.G - 1) / L.G > 65535) return KVQ_ERR_UNSUPPORTED;
  AppendParams p;
  p.L = L;
  p.C = make_ptrs(cache);
  p.k_new = k_new;
  p.v_new = v_new;
  p.n_new = n_new;
  p.batch = batch;
  p.seq_lens = seq_lens;
  p.status = dev_status;
  if (launch_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_layer_config* cfg, int32_t batch, int32_t num_q_heads,
                                     size_t* bytes) {
  LayerDesc L;
  kvq_status st = make_desc(cfg, &L);
  if (st != KVQ_OK) return st;
  if (!bytes || batch < 0 || batch > kMaxBatch || num_q_heads < L.H || num_q_heads % L.H != 0 ||
      num_q_heads / L.H > kMaxGqa)
    return KVQ_ERR_INVALID_ARG;
  DecodeGeom G;
  if ((st = decode_geometry(L, batch, num_q_heads / L.H, &G)) != KVQ_OK) return st;
  *bytes = G.ws_bytes;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size_multi(const kvq_layer_config* cfg, int32_t batch, int32_t n_query,
                                           int32_t num_q_heads, size_t* bytes) {
  LayerDesc L;
  kvq_status st = make_desc(cfg, &L);
  if (st != KVQ_OK) return st;
  if (!bytes || batch < 0 || batch > kMaxBatch || n_query < 1 || num_q_heads < L.H || num_q_heads % L.H != 0 ||
      num_q_heads / L.H * n_query > kMaxGqa)
    return KVQ_ERR_INVALID_ARG;
  DecodeGeom G;
  if ((st = decode_geometry(L, batch, num_q_heads / L.H * n_query, &G, n_query > 1)) != KVQ_OK) return st;
  *bytes = G.ws_bytes;
  return KVQ_OK;
}

}  // extern "C"

namespace kvq {
namespace {

kvq_status check_decode_args(const kvq_layer_config* cfg, int32_t num_q_heads, int32_t batch, LayerDesc* L) {
  kvq_status st = make_desc(cfg, L);
  if (st != KVQ_OK) return st;
  if (batch < 0 || batch > kMaxBatch || num_q_heads < L->H || num_q_heads % L->H != 0 ||
      num_q_heads / L->H > kMaxGqa)
    return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

kvq_status decode_partials_impl(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                int32_t num_q_heads, const int32_t* seq_lens, int32_t batch, float softmax_scale,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status, cudaStream_t s,
                                void* out = nullptr, int32_t out_bf16 = 0, float* lse = nullptr,
                                int32_t n_query = 1, int32_t withhold_copy = 0, const void* k_new = nullptr,
                                const void* v_new = nullptr, bool check_only = false) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (n_query < 1 || num_q_heads / L.H * n_query > kMaxGqa) return KVQ_ERR_INVALID_ARG;
  if ((L.rope || L.k_out || L.v_out) && n_query > 1) return KVQ_ERR_UNSUPPORTED;
  if ((st = check_cache(L, cache)) != KVQ_OK) return st;
  if (batch == 0) return KVQ_OK;
  if (!q || !seq_lens || !workspace || !aligned16(workspace) || !(softmax_scale == softmax_scale))
    return KVQ_ERR_INVALID_ARG;
  const int g = num_q_heads / L.H * n_query;  // query columns per kv head
  DecodeGeom G;
  if ((st = decode_geometry(L, batch, g, &G, n_query > 1)) != KVQ_OK) return st;
  if (workspace_bytes < G.ws_bytes) return KVQ_ERR_WORKSPACE;
  if (check_only) return KVQ_OK;
  DecodeParams p;
  p.L = L;
  p.C = make_ptrs(cache);
  p.q = q;
  p.Hq = num_q_heads;
  p.g = g;
  p.gh = num_q_heads / L.H;
  p.n_query = n_query;
  p.batch = batch;
  p.seq_lens = seq_lens;
  // a one-token append before the decode (k_new given): the decode sees seq_lens + 1 tokens; FP8
  // layers without sink tokens write the token's codes inside this launch (fp8_append_token)
  p.len_add = k_new ? 1 : 0;
  p.fp8_append = (k_new && L.fp8 && L.S == 0) ? 1 : 0;
  p.k_new = k_new;
  p.v_new = v_new;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.num_ctas = G.num_ctas;
  p.nst = G.nst;
  p.stage_bytes = G.stage_bytes;
  p.tps = G.tps;
  // a claimed work item: whole records, at least a stage's worth of tiles
  p.item_tiles = (std::max(G.tps, L.tpg) + L.tpg - 1) / L.tpg * L.tpg;
  // integer layers whose stages hold more than a record (their stage sizes budget a header for
  // every record a stage touches, see stage_bytes_of): items of at least two stages, whole records
  // (half the claims; measured on GB300: INT2 MHA layer 1555 -> 1498 us).  A stage no longer than a
  // record must not cross one, so there items stay single records.
  if (!L.fp8 && !L.bf16 && (L.tpg == 1 || G.tps > L.tpg))
    p.item_tiles = (std::max(2 * G.tps, L.tpg) + L.tpg - 1) / L.tpg * L.tpg;
  // a 16-token bf16 tile reads 8 KB; charge it in units of a quantized tile's bytes
  p.bf_weight = std::max(1, (8192 + L.tile_bytes / 2) / L.tile_bytes);
  p.bf_joint = bf16_joint(G.stage_bytes) ? 1 : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_o = reinterpret_cast<float*>(ws);
  p.ws_lse = reinterpret_cast<float*>(ws + G.off_lse);
  p.ws_prefix = reinterpret_cast<int*>(ws + G.off_prefix);
  p.status = dev_status;
  p.merge_bytes = G.merge_bytes;
  p.withhold_copy = withhold_copy;
  p.fuse = out != nullptr;
  p.counters = reinterpret_cast<unsigned*>(ws + G.off_counters);
  p.out = out;
  p.out_bf16 = out_bf16;
  p.lse = lse;
  if (L.rope) {
    // pair i turns by theta_i = base^(-2i/128) per position: its angle in turns, as a 64-bit
    // fraction, so that t * rope_turn[i] (mod 2^64) is the angle of position t reduced exactly
    for (int i = 0; i < 64; ++i) {
      const double theta = std::pow((double)L.rope_base, -2.0 * i / 128.0);
      double turn = theta / (2.0 * 3.14159265358979323846);
      turn -= std::floor(turn);
      p.rope_turn[i] = (unsigned long long)(turn * 18446744073709551616.0);
    }
  }
  cudaError_t e;
  switch (kernel_format(L.fmt)) {
    case KVQ_FMT_INT2: e = launch_decode_int2(p, G.smem, s); break;
    case KVQ_FMT_INT4: e = launch_decode_int4(p, G.smem, s); break;
    case KVQ_FMT_INT8: e = launch_decode_int8(p, G.smem, s); break;
    case KVQ_FMT_FP8_E5M2: e = launch_decode_fp8_e5m2(p, G.smem, s); break;
    default: e = launch_decode_fp8(p, G.smem, s); break;
  }
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status decode_combine_impl(const kvq_layer_config* cfg, int32_t num_q_heads, int32_t batch, void* out,
                               int32_t out_bf16, float* lse, const void* workspace, size_t workspace_bytes,
                               cudaStream_t s) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (out_bf16 != 0 && out_bf16 != 1) return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  if (!out || !workspace || !aligned16(workspace)) return KVQ_ERR_INVALID_ARG;
  const int g = num_q_heads / L.H;
  DecodeGeom G;
  if ((st = decode_geometry(L, batch, g, &G)) != KVQ_OK) return st;
  if (workspace_bytes < G.ws_bytes) return KVQ_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  CombineParams c;
  c.H = L.H;
  c.g = g;
  c.Hq = num_q_heads;
  c.batch = batch;
  c.num_ctas = G.num_ctas;
  c.ws_prefix = reinterpret_cast<const int*>(ws + G.off_prefix);
  c.ws_o = reinterpret_cast<const float*>(ws);
  c.ws_lse = reinterpret_cast<const float*>(ws + G.off_lse);
  c.out = out;
  c.out_bf16 = out_bf16;
  c.lse = lse;
  return launch_combine(c, s) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace
}  // namespace kvq

extern "C" {

kvq_status kvq_decode_partials(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                               int32_t num_q_heads, const int32_t* seq_lens, int32_t batch, float softmax_scale,
                               void* workspace, size_t workspace_bytes, uint32_t* dev_status, void* stream) {
  return decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                              workspace_bytes, dev_status, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_combine(const kvq_layer_config* cfg, int32_t num_q_heads, int32_t batch, void* out,
                              int32_t out_bf16, float* lse, const void* workspace, size_t workspace_bytes,
                              void* stream) {
  return decode_combine_impl(cfg, num_q_heads, batch, out, out_bf16, lse, workspace, workspace_bytes,
                             static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_attention(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                int32_t num_q_heads, const int32_t* seq_lens, int32_t batch, float softmax_scale,
                                void* out, int32_t out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, void* stream) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (out_bf16 != 0 && out_bf16 != 1) return KVQ_ERR_INVALID_ARG;
  if (batch > 0 && !out) return KVQ_ERR_INVALID_ARG;
  // one launch: the last CTA to finish each (sequence, kv head) merges its partials
  return decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                              workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), out, out_bf16, lse);
}

kvq_status kvq_append_decode_attention(const kvq_layer_config* cfg, const kvq_layer_cache* cache,
                                       const void* k_new, const void* v_new, const int32_t* seq_lens, int32_t batch,
                                       const void* q, int32_t num_q_heads, float softmax_scale, void* out,
                                       int32_t out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                       uint32_t* dev_status, void* stream) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (out_bf16 != 0 && out_bf16 != 1) return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  if (!out || !k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every host check of the decode before anything is enqueued
  if ((st = decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                                 workspace_bytes, dev_status, s, out, out_bf16, lse, 1, 0, k_new, v_new, true)) !=
      KVQ_OK)
    return st;
  if (!(L.fp8 && L.S == 0)) {  // the append as its own launch(es) first (see kvq_quantize_append)
    if ((st = kvq_quantize_append(cfg, cache, k_new, v_new, 1, seq_lens, batch, dev_status, stream)) != KVQ_OK)
      return st;
  }
  return decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                              workspace_bytes, dev_status, s, out, out_bf16, lse, 1, 0, k_new, v_new);
}

kvq_status kvq_selftest_bounded_wait(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                     int32_t num_q_heads, const int32_t* seq_lens, int32_t batch,
                                     float softmax_scale, void* out, int32_t out_bf16, float* lse, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_status, void* stream) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (L.paged || L.bf16) return KVQ_ERR_UNSUPPORTED;
  if ((out_bf16 != 0 && out_bf16 != 1) || !dev_status) return KVQ_ERR_INVALID_ARG;
  if (batch > 0 && !out) return KVQ_ERR_INVALID_ARG;
  return decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                              workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), out, out_bf16, lse, 1,
                              1);
}

kvq_status kvq_decode_attention_multi(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                      int32_t n_query, int32_t num_q_heads, const int32_t* seq_lens, int32_t batch,
                                      float softmax_scale, void* out, int32_t out_bf16, float* lse, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_status, void* stream) {
  LayerDesc L;
  kvq_status st = check_decode_args(cfg, num_q_heads, batch, &L);
  if (st != KVQ_OK) return st;
  if (out_bf16 != 0 && out_bf16 != 1) return KVQ_ERR_INVALID_ARG;
  if (batch > 0 && !out) return KVQ_ERR_INVALID_ARG;
  return decode_partials_impl(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, workspace,
                              workspace_bytes, dev_status, static_cast<cudaStream_t>(stream), out, out_bf16, lse,
                              n_query);
}

kvq_status kvq_dequantize(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const int32_t* seq_lens,
                          int32_t batch, int32_t max_tokens, float* k_out, float* v_out, uint32_t* dev_status,
                          void* stream) {
  LayerDesc L;
  kvq_status st = make_desc(cfg, &L);
  if (st != KVQ_OK) return st;
  if ((st = check_cache(L, cache)) != KVQ_OK) return st;
  if (batch < 0 || batch > kMaxBatch || max_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0 || max_tokens == 0) return KVQ_OK;
  if (!seq_lens || !k_out || !v_out) return KVQ_ERR_INVALID_ARG;
  if ((max_tokens + 15) / 16 > 65535) return KVQ_ERR_UNSUPPORTED;
  DequantParams p;
  p.L = L;
  p.C = make_ptrs(cache);
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.max_tokens = max_tokens;
  p.k_out = k_out;
  p.v_out = v_out;
  p.status = dev_status;
  if (launch_dequantize(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_lse_merge(const float* o_parts, const float* lse_parts, int32_t n_parts, int64_t rows, void* out,
                         int32_t out_bf16, float* lse_out, void* stream) {
  if (n_parts < 1 || rows < 0 || (out_bf16 != 0 && out_bf16 != 1)) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (rows > ((long long)1 << 40) || !o_parts || !lse_parts || !out || !aligned16(o_parts) || !aligned16(out))
    return KVQ_ERR_INVALID_ARG;
  if (launch_lse_merge(o_parts, lse_parts, n_parts, rows, out, out_bf16, lse_out, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG: an argument is outside its documented range";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: valid but unsupported combination";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace smaller than kvq_decode_workspace_size()";
    default: return "unknown kvq_status";
  }
}

}  // extern "C"
