/*
 * kvq.h -- C ABI of the GB300 (sm_103a) quantized KV-cache decode library (libkvq.so).
 *
 * The library implements attention decode over a KV cache stored with
 * asymmetric affine quantization (Keys per channel over groups of tokens,
 * Values per token over groups of channels) at 2, 4 or 8 bits, or as FP8 (E4M3
 * or E5M2) with a per-tensor fp32 scale; a bf16 residual window of recent
 * tokens and bf16 attention-sink tokens; per-layer formats, including bf16
 * "skip" layers left unquantized; contiguous or paged storage.
 *
 * Sources (web pages; cited by title and section):
 *   [KVQA] "KV Cache Quantization Analysis" (ryotta.opik.net, KV 캐시 양자화 심층 분석)
 *          s2 "양자화 기초 / 핵심 개념"       q = round(x/s + z), x_hat = s(q - z); asymmetric z
 *          s3 "Key=per-channel, Value=per-token" Key per channel, Value per token, residual window
 *          s4 "FP8 / INT8"                    E4M3 and E5M2 with an fp32 scale; INT8 needs scale storage
 *          s5 "구현·시스템 고려사항"          quantize the new K,V at write; dequantize right before
 *                                             attention, fused with the matmul; paging is orthogonal
 *          box "메모리 크기 감각"             KV bytes = 2 L H_kv d T B bytes
 *   [W4KV] "W4A16 + KV cache quantization combined accuracy" (hrletsgo.me)
 *          "오차가 어디서 만나는가"           softmax(Q K^T / sqrt(d))
 *          "어떤 레이어가 더 민감한가"        sink token K/V kept 16-bit; FP8/INT8 early/late, INT4 middle
 *          vLLM flags section                 fp8_e5m2 KV dtype; layers skipped from KV quantization
 *   [AIQK] "양자화와 KV 캐시" (ai-trend.me)    PagedAttention: fixed-size blocks and a per-request table
 *
 * Conventions for every entry point
 *   - All buffers are owned by the caller.  The library allocates no memory
 *     (kvq_decode_attention_static_scratch excepted, see there) and keeps no
 *     state between calls other than per-device caches of launch settings
 *     (kernel occupancy, shared-memory limits).  Pointers marked "device" are
 *     CUDA device pointers.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL =
 *     the legacy default stream).  They return once the work is enqueued.
 *   - A host-detectable error (bad sizes, unsupported combination, null pointer,
 *     workspace too small) returns a negative kvq_status and enqueues nothing.
 *     A failed launch returns KVQ_ERR_CUDA.
 *   - Data-dependent errors found on the device (a block id outside the pool, a
 *     length beyond the capacity, a bounded wait that gave up) are OR-ed as
 *     KVQ_DEV_* bits into *dev_status (device uint32; may be NULL to drop them).
 *     The offending load or store is skipped; kernels never trap and never wait
 *     without a bound.  The caller clears *dev_status.
 *   - head_dim must be 128; 1 <= num_q_heads / num_kv_heads <= 8.
 *
 * Token accounting of one (sequence, kv head) holding T tokens (S sink tokens,
 * R residual tokens, K group G):  the first min(T, S) tokens are the sink (bf16);
 * Q_n = max(0, floor((T - S - R) / G)) * G tokens are quantized; the last
 * r = T - S - Q_n tokens are the residual window (bf16).  FP8 layers use G = 1
 * and R = 0 (every token after the sink is quantized at once).  bf16 layers
 * quantize nothing: Q_n = 0 and every token after the sink is a "residual"
 * token, so the window holds the whole sequence.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = -1, /* argument outside its documented range, null pointer */
  KVQ_ERR_UNSUPPORTED = -2, /* valid but not implemented combination (e.g. head_dim != 128) */
  KVQ_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  KVQ_ERR_WORKSPACE = -4    /* workspace smaller than kvq_decode_workspace_size() */
} kvq_status;

typedef enum {
  KVQ_FMT_BF16 = 1,      /* no quantization ("skip layer"): every token kept in bf16 */
  KVQ_FMT_INT2 = 2,      /* 2-bit affine codes, fp32 scale + fp32 zero-point per group */
  KVQ_FMT_INT4 = 4,      /* 4-bit affine codes */
  KVQ_FMT_INT8 = 8,      /* 8-bit affine codes */
  KVQ_FMT_FP8_E4M3 = 16, /* OCP E4M3FN codes, one fp32 scale per tensor (K and V each) */
  KVQ_FMT_FP8_E5M2 = 17  /* OCP E5M2 codes, one fp32 scale per tensor (K and V each) */
} kvq_format;

/* bits OR-ed into *dev_status */
#define KVQ_DEV_BAD_BLOCK 0x1u  /* a block-table entry outside [0, num_blocks) */
#define KVQ_DEV_CAPACITY 0x2u   /* a sequence longer than the store can hold */
#define KVQ_DEV_TIMEOUT 0x4u    /* a bounded wait for an asynchronous copy gave up */

/* Per-layer configuration (host struct, read during the call only). */
typedef struct {
  int32_t num_kv_heads;       /* H_kv >= 1 */
  int32_t head_dim;           /* d, must be 128 */
  int32_t format;             /* kvq_format */
  int32_t k_group_tokens;     /* G: tokens per Key group (per-channel scale); multiple of 16, at most 256
                                 (KVQ_ERR_UNSUPPORTED above); 1 for FP8; ignored for bf16 */
  int32_t v_group_dims;       /* Gv: channels per Value group (per-token scale); 16,32,64,128; FP8: 128;
                                 ignored for bf16 */
  int32_t residual_tokens;    /* R >= 0 bf16 recent tokens kept (0 for FP8; ignored for bf16) */
  int32_t sink_tokens;        /* S >= 0 bf16 first tokens kept */
  int32_t paged;              /* 0: contiguous store, 1: paged store (not for bf16) */
  int32_t block_tokens;       /* paged: tokens per block P (INT: P == G; FP8: multiple of 16) */
  int32_t capacity_tokens;    /* contiguous: quantized tokens per (seq, head); multiple of 16 and of G.
                                 bf16: tokens after the sink per (seq, head), >= 1 */
  int32_t num_blocks;         /* paged: blocks in the pool */
  int32_t max_blocks_per_seq; /* paged: row length of the block table */
  float rope_base;            /* 0: Keys are used as stored.  > 1: pre-RoPE Keys -- the layer's Keys are
                                 appended (and quantized) before the rotary position embedding, and the
                                 decode rotates each dequantized Key at its position t: channel pair
                                 (i, i + 64) turned by t * rope_base^(-2i/128) (rotate-half pairing;
                                 the query is passed already rotated).  Integer formats with Gv of 64 or
                                 128, one query token (KVQ_ERR_UNSUPPORTED otherwise). */
  int32_t k_outliers;         /* 0..8 dense-and-sparse Keys: per quantized Key row, the k_outliers entries
                                 of largest magnitude (ties: the lower channel) are kept exactly (bf16)
                                 in a sparse list and the rest, those entries set to 0, is quantized */
  int32_t v_outliers;         /* 0..8 the same for the Value rows.  Integer formats with Gv of 64 or
                                 128, no pre-RoPE Keys, one query token (KVQ_ERR_UNSUPPORTED otherwise) */
} kvq_layer_config;

/*
 * Device buffers of one layer's cache.  Which fields are used depends on the
 * config; unused fields may be NULL.  With B = sequences, H = num_kv_heads,
 * d = 128, b = bits (8 for FP8), rb = d*b/8 bytes per token row, W = R + G,
 * ngv = d / Gv.  Only quantized tokens x = t - S live in the quantized store.
 *
 * A 16-token tile (quantized tokens 16i .. 16i+15) is, in this order:
 *   K codes  [16*rb]      in "fragment order" (below)
 *   V codes  [16*rb]      in "fragment order" (below)
 *   V scale  [16][ngv] f32, V zero [16][ngv] f32   (INT only: per token, per Gv channels)
 *   K sparse [16][k_outliers] u32, V sparse [16][v_outliers] u32   (dense-and-sparse layers:
 *            each token's kept entries in ascending channel order, entry = bf16 bits << 16 | channel)
 * tile_bytes = 32*rb (+ 128*ngv + 64*(k_outliers + v_outliers) for INT).
 * A record is a header followed by tpg consecutive tiles:
 *   INT: header = K scale [d] f32, K zero [d] f32 (the per-channel Key group of
 *        G = 16*tpg tokens, 1024 bytes); tpg = G/16
 *   FP8: no header; tpg = 1 (contiguous) or P/16 (paged)
 * record_bytes = header + tpg * tile_bytes.  A run of consecutive tiles is one
 * contiguous byte range, so the decode kernel fetches it with one bulk copy.
 *
 * Contiguous store (paged == 0): qstore holds, for each (seq, head) in [B][H]
 * order, cap/(16*tpg) records (cap = capacity_tokens).
 * Paged store (paged == 1), P = block_tokens: block_pool holds num_blocks
 * blocks; a block is H records, one per head (INT: P == G, so one Key group per
 * block).  Quantized token x of sequence b lives in block
 * block_table[b*max_blocks_per_seq + x/P].
 * bf16 parts (both stores):
 *   resid_k, resid_v  bf16 [B][H][W][d]  residual token t in slot (t - S) mod W
 *   sink_k,  sink_v   bf16 [B][H][S][d]
 * FP8: k_tensor_scale, v_tensor_scale point to one device float each (amax/448
 * for E4M3, amax/57344 for E5M2, see kvq_fp8_calibrate_format); they stay
 * fixed for later appends.
 * bf16 layers: no quantized store (qstore, block_pool unused); resid_k and
 * resid_v are bf16 [B][H][W][d] with W = capacity_tokens, token t >= S in row
 * t - S (the ring never wraps: a sequence holds at most S + W tokens).
 *
 * Fragment order.  The K codes and the V codes of a tile are each a 16 x 128
 * code matrix stored as the register file of a tensor-core A operand
 * (mma m16n8k16): element (row i, column k) of step s (s in [0,8)) goes to
 * lane 4(i mod 8) + (k mod 8)/2, register reg = (i / 8) + 2(k / 8), half
 * h = k mod 2.  For the K codes of token t, channel c: s = c/16, i = t, and
 * with e = c mod 4, k = 2((c/4) mod 4) + (e mod 2) + 8(e/2).  For the V codes
 * of token t, channel c: s = c/16, i = c mod 16, k = t.
 * Lane l owns rb/8 32-bit words; word w of lane l is at byte
 * ((w/4)*32 + l)*16 + (w mod 4)*4, and (lane, s, reg, h) is placed at
 *   INT4: word s,               bit 4 reg + 16 h
 *   INT2: word s/2,             bit 8(s mod 2) + 2 reg + 16 h
 *   INT8: word 2s + reg/2,      bit 8((reg mod 2) + 2h)
 *   FP8:  word 2s + reg/2,      bit 8(2(reg mod 2) + h)     (E4M3 and E5M2)
 * so that every lane of a decode warp fetches its words with conflict-free
 * 16-byte loads and unpacks them in registers.
 */
typedef struct {
  void* qstore;               /* contiguous quantized store (paged == 0) */
  void* block_pool;           /* paged quantized store (paged == 1) */
  const int32_t* block_table; /* paged: int32 [B][max_blocks_per_seq] */
  void* resid_k;
  void* resid_v;
  void* sink_k;
  void* sink_v;
  const float* k_tensor_scale;
  const float* v_tensor_scale;
} kvq_layer_cache;

/* Indices of kvq_cache_layout()'s output array. */
enum {
  KVQ_FIELD_QSTORE = 0,
  KVQ_FIELD_BLOCK_POOL,
  KVQ_FIELD_RESID_K,
  KVQ_FIELD_RESID_V,
  KVQ_FIELD_SINK_K,
  KVQ_FIELD_SINK_V,
  KVQ_FIELD_COUNT
};

/*
 * kvq_cache_layout -- bytes of each cache buffer for `num_seqs` sequences.
 * Validates `cfg` (same rules as the other calls).  bytes[i] is 0 for a field
 * the config does not use.  Host only; no CUDA call.
 * Layout: see kvq_layer_cache.  Source: [KVQA] box "메모리 크기 감각" (sizes),
 * s3 (per-channel K / per-token V groups), [AIQK] (blocks and block table).
 */
kvq_status kvq_cache_layout(const kvq_layer_config* cfg, int32_t num_seqs, size_t bytes[KVQ_FIELD_COUNT]);

/*
 * kvq_fp8_calibrate -- per-tensor FP8 scale s = amax/448 (fp32 division; s = 1
 * when amax == 0) of `n` bf16 values at device pointer x; written to the device
 * float *scale_out.  Source: [KVQA] s4 (E4M3 needs an fp32 scale) and s5
 * (calibrated scales).  448 is the largest finite OCP E4M3FN value.
 */
kvq_status kvq_fp8_calibrate(const void* x, size_t n, float* scale_out, void* stream);

/*
 * kvq_fp8_calibrate_format -- the same for a given FP8 format: s = amax/448
 * (KVQ_FMT_FP8_E4M3) or amax/57344 (KVQ_FMT_FP8_E5M2; 57344 is the largest
 * finite OCP E5M2 value).  Source: [KVQA] s4 (both formats take an fp32
 * scale).  Any other format returns KVQ_ERR_INVALID_ARG.
 */
kvq_status kvq_fp8_calibrate_format(const void* x, size_t n, int32_t format, float* scale_out, void* stream);

/*
 * kvq_quantize_append -- write `n_new` new tokens per (sequence, kv head).
 * Source: [KVQA] s5 (quantize the new K,V right after they are computed and
 * store them), s2 (affine formula), s3 (Key per channel over G tokens, Value
 * per token over Gv channels, full-precision residual window), s4 (FP8);
 * [W4KV] (sink tokens kept 16-bit).
 *   k_new, v_new  device bf16 [batch][H][n_new][d], 16-byte aligned
 *   seq_lens      device int32 [batch]: tokens already in the cache (before)
 * Tokens t < S go to the sink; otherwise to the residual ring; every time the
 * ring reaches R + G tokens its oldest G are quantized as one Key group (per
 * channel: s = (max - min)/(2^b - 1), z = -(min/s), q = clamp(rne(x/s + z))
 * in IEEE fp32, s = 1 for a constant group) and G Value tokens (per token and
 * Gv-channel group, same formula).  FP8: code = E4M3 (or E5M2) RNE satfinite
 * of fp32(x / s_tensor).  bf16 layers: the token is copied to row t - S of the
 * residual buffers, never quantized.  Result identical to n_new single-token
 * appends (integer layers: at most 65535 * G tokens per call).
 * The caller advances seq_lens by n_new afterwards, and for a paged store has
 * the blocks of every group that spills already in the block table.
 * Device errors: KVQ_DEV_CAPACITY (store full: nothing written for that
 * sequence), KVQ_DEV_BAD_BLOCK (that group skipped).
 */
kvq_status kvq_quantize_append(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* k_new,
                               const void* v_new, int32_t n_new, const int32_t* seq_lens, int32_t batch,
                               uint32_t* dev_status, void* stream);

/*
 * kvq_decode_workspace_size -- device workspace bytes kvq_decode_attention
 * needs for this config, batch and query-head count on the current device.
 */
kvq_status kvq_decode_workspace_size(const kvq_layer_config* cfg, int32_t batch, int32_t num_q_heads,
                                     size_t* bytes);

/*
 * kvq_decode_attention -- one decode step of attention over the quantized cache.
 * Source: [W4KV] "오차가 어디서 만나는가" (softmax(q K^T / sqrt(d)) V);
 * [KVQA] s5 (dequantize right before attention, fused with the matmul, else
 * the bandwidth saving is lost) and s1 (decode is bound by reading the cache).
 *   q         device bf16 [batch][num_q_heads][d]; query head h reads kv head
 *             h / (num_q_heads / H) (grouped-query attention)
 *   seq_lens  device int32 [batch]: tokens in the cache (after this step's append)
 *   softmax_scale  multiplies q.k (1/sqrt(d) for the plain formula)
 *   out       device [batch][num_q_heads][d], fp32 (out_bf16 == 0) or bf16
 *             (out_bf16 == 1: the round-to-nearest-even of the fp32 result)
 *   lse       device f32 [batch][num_q_heads] natural-log log-sum-exp of the
 *             scaled scores, or NULL
 *   workspace device, at least kvq_decode_workspace_size() bytes, 16-byte
 *             aligned.  Zero-fill it once before its first use: its last
 *             batch*H 32-bit words are arrival counters (the last CTA to finish
 *             a (sequence, kv head) merges that pair's partials, in the same
 *             launch) and every call leaves them at zero again.  After a call
 *             that reported KVQ_DEV_TIMEOUT, zero it again.  Calls that share a
 *             workspace must not overlap on the GPU.
 * A sequence with 0 tokens gets out = 0, lse = -inf.  Device errors:
 * KVQ_DEV_BAD_BLOCK (tile skipped), KVQ_DEV_CAPACITY (length clamped to the
 * capacity), KVQ_DEV_TIMEOUT.
 */
kvq_status kvq_decode_attention(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                int32_t num_q_heads, const int32_t* seq_lens, int32_t batch, float softmax_scale,
                                void* out, int32_t out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, void* stream);

/*
 * kvq_append_decode_attention -- one whole decode step of a layer: the step's
 * token is appended to every sequence, then attention runs over all tokens
 * including it.  Source: [KVQA] s5 (quantize the new K, V when they are
 * written, dequantize right before attention).  The result equals
 * kvq_quantize_append(..., n_new = 1, seq_lens, ...) followed by
 * kvq_decode_attention over seq_lens + 1 tokens (same cache contents, same out
 * and lse bits).  FP8 layers without sink tokens do it in ONE launch: the warp
 * that reads the new token's tile encodes the token and writes its codes both
 * into the cache and into the copy it reads (no other CTA reads that tile), so
 * the step pays no second launch and no launch gap; other layers run the append
 * launch(es), then the decode launch.
 *   k_new, v_new  device bf16 [batch][H][d], 16-byte aligned: the step's token
 *   seq_lens  device int32 [batch]: tokens in the cache BEFORE this step
 *   q, num_q_heads, softmax_scale, out, out_bf16, lse, workspace  as for
 *             kvq_decode_attention (workspace: kvq_decode_workspace_size)
 * Every host-detectable error is returned before anything is enqueued.  The
 * caller advances seq_lens by 1 afterwards.  Device errors: those of the two
 * calls it stands for (KVQ_DEV_CAPACITY: the token is not stored and the
 * sequence's length is clamped to the capacity).
 */
kvq_status kvq_append_decode_attention(const kvq_layer_config* cfg, const kvq_layer_cache* cache,
                                       const void* k_new, const void* v_new, const int32_t* seq_lens, int32_t batch,
                                       const void* q, int32_t num_q_heads, float softmax_scale, void* out,
                                       int32_t out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                       uint32_t* dev_status, void* stream);

/*
 * kvq_decode_attention_multi -- attention of n_query new tokens per sequence
 * (speculative-decoding verification, chunked prefill) over the quantized
 * cache in one launch.  Source: [W4KV] "오차가 어디서 만나는가" (the score
 * formula) applied causally to several query positions; the cache and its
 * formats as for kvq_decode_attention.
 *   q         device bf16 [batch][n_query][num_q_heads][d]: query token i of
 *             sequence b sits at position seq_lens[b] - n_query + i
 *   seq_lens  device int32 [batch]: tokens in the cache, the n_query new tokens
 *             included (append them with kvq_quantize_append first)
 *   out       device [batch][n_query][num_q_heads][d] (fp32 or bf16 as above)
 *   lse       device f32 [batch][n_query][num_q_heads] or NULL
 *   workspace at least kvq_decode_workspace_size_multi() bytes, zero-filled
 *             once before first use (the same arrival counters as above)
 * Query token i attends to tokens 0 .. seq_lens[b] - n_query + i (causal
 * among the new tokens); a query with no visible token (seq_lens[b] <
 * n_query - i) gets out = 0, lse = -inf.  Requires 1 <= n_query and
 * (num_q_heads / H) * n_query <= 8: the kernel runs the n_query query tokens
 * of a kv head's query heads as that many tensor-core columns.  n_query = 1 is
 * kvq_decode_attention.  Errors as for kvq_decode_attention.
 */
kvq_status kvq_decode_attention_multi(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                      int32_t n_query, int32_t num_q_heads, const int32_t* seq_lens, int32_t batch,
                                      float softmax_scale, void* out, int32_t out_bf16, float* lse, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_status, void* stream);

/* Workspace bytes kvq_decode_attention_multi needs (same rules as kvq_decode_workspace_size). */
kvq_status kvq_decode_workspace_size_multi(const kvq_layer_config* cfg, int32_t batch, int32_t n_query,
                                           int32_t num_q_heads, size_t* bytes);

/*
 * kvq_decode_partials / kvq_decode_combine -- kvq_decode_attention as two
 * launches (same arguments, same workspace; the counters are not used).
 * kvq_decode_partials runs the split pass: every CTA of the grid reads an equal
 * share of the cache and writes, into the workspace, one partial per (sequence,
 * kv head) it touches: the output normalised by its own softmax sum and its
 * log-sum-exp.  kvq_decode_combine merges the partials of each (sequence, query
 * head) by their log-sum-exp weights into out and lse.  Call them on the same
 * device and stream, with the same config, batch and query-head count, and
 * combine before the workspace is reused.  A caller that splits one sequence
 * over several devices can merge the per-device results with the same
 * log-sum-exp rule.  Errors as for kvq_decode_attention.
 */
kvq_status kvq_decode_partials(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                               int32_t num_q_heads, const int32_t* seq_lens, int32_t batch, float softmax_scale,
                               void* workspace, size_t workspace_bytes, uint32_t* dev_status, void* stream);
kvq_status kvq_decode_combine(const kvq_layer_config* cfg, int32_t num_q_heads, int32_t batch, void* out,
                              int32_t out_bf16, float* lse, const void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * kvq_decode_attention_static_scratch -- kvq_decode_attention for callers that
 * cannot allocate device memory.  (The pages have no counterpart to this call:
 * it exists for integration, not for the method.)
 * Who needs it: code hosted in an application that owns all device memory
 * through its own pool and forbids direct cudaMalloc, loops that cannot accept
 * the device-wide synchronisation an allocation may cause, or plug-ins with no
 * allocator at hand.  Instead of a caller workspace it uses one fixed array of
 * 8 MiB in device global memory inside libkvq, reserved on every GPU that
 * loads the library until the process exits.  Inputs and outputs are the
 * caller's, as for kvq_decode_attention (same arguments minus the workspace).
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library call.
 *   - Returns KVQ_ERR_WORKSPACE when kvq_decode_workspace_size() for this
 *     config, batch and query-head count exceeds 8 MiB (large batch x heads).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on the device.  The address is kept with the
 *     id of the device's context: after a device reset (cudaDeviceReset) the
 *     next call looks it up again, and that call too belongs outside capture.
 *   - Host-detectable errors (out == NULL with batch > 0, out_bf16 not 0 or 1,
 *     the checks of kvq_decode_attention) return before anything is enqueued.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero.  Calls that overlap on the
 *     GPU (other streams, other threads) race on it: serialise them.
 *   - Runs as two launches (split pass, then merge).
 */
kvq_status kvq_decode_attention_static_scratch(const kvq_layer_config* cfg, const kvq_layer_cache* cache,
                                               const void* q, int32_t num_q_heads, const int32_t* seq_lens,
                                               int32_t batch, float softmax_scale, void* out, int32_t out_bf16,
                                               float* lse, uint32_t* dev_status, void* stream);

/*
 * kvq_dequantize -- export the dequantized cache as fp32.
 * Source: [KVQA] s2 (x_hat = s(q - z)), s4 (FP8 value times its scale).
 *   k_out, v_out  device f32 [batch][H][max_tokens][d]; token t < seq_lens[b]
 *   gets x_hat (sink / residual: the bf16 value; INT: s*(q - z) as two fp32
 *   operations; FP8: s * E4M3 / E5M2 value in fp32), tokens t >= seq_lens[b]
 *   get 0.
 *   seq_lens      device int32 [batch]; a length above max_tokens is an error
 *   (KVQ_DEV_CAPACITY) and is clamped.
 */
kvq_status kvq_dequantize(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const int32_t* seq_lens,
                          int32_t batch, int32_t max_tokens, float* k_out, float* v_out, uint32_t* dev_status,
                          void* stream);

/*
 * kvq_lse_merge -- merge attention results computed over disjoint parts of the
 * same sequences' tokens: the split a sequence-parallel decode makes when one
 * long sequence's cache is spread over several devices (each part decoded with
 * kvq_decode_attention and its lse, the results gathered to one device).
 * Source: [W4KV] "오차가 어디서 만나는가" -- softmax over the union of the
 * parts, regrouped exactly as lse = log sum_i exp(lse_i) and
 * out = sum_i exp(lse_i - lse) * o_i.
 *   o_parts    device f32 [n_parts][rows][128], 16-byte aligned: each part's
 *              output, normalised by that part's own softmax sum (as
 *              kvq_decode_attention writes it in fp32)
 *   lse_parts  device f32 [n_parts][rows], natural log; -inf for a part with no
 *              tokens (weight 0)
 *   out        device [rows][128], 16-byte aligned: fp32 (out_bf16 == 0) or
 *              bf16 (RNE of the fp32 result); lse_out device f32 [rows] or NULL
 * A row whose parts are all empty gets out = 0, lse = -inf.
 */
kvq_status kvq_lse_merge(const float* o_parts, const float* lse_parts, int32_t n_parts, int64_t rows, void* out,
                         int32_t out_bf16, float* lse_out, void* stream);

/*
 * kvq_selftest_bounded_wait -- self-test of the device error path (no
 * counterpart in the pages: it exists to show the failure handling works).
 * Runs kvq_decode_attention (same arguments) with the first bulk copy of one
 * warp (CTA 0, warp 0) withheld while its stage barrier still expects the bytes,
 * so that warp's bounded wait (about one second of SM clocks) runs out.  The
 * launch must then report KVQ_DEV_TIMEOUT in *dev_status (required, not NULL)
 * and finish (the warp stops issuing copies and drains its own, each wait
 * bounded); the outputs of the affected pair are not valid.  Zero the workspace
 * again afterwards, as after any call that reported KVQ_DEV_TIMEOUT.
 * Contiguous INT and FP8 layers only (KVQ_ERR_UNSUPPORTED otherwise).
 */
kvq_status kvq_selftest_bounded_wait(const kvq_layer_config* cfg, const kvq_layer_cache* cache, const void* q,
                                     int32_t num_q_heads, const int32_t* seq_lens, int32_t batch,
                                     float softmax_scale, void* out, int32_t out_bf16, float* lse, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_status, void* stream);

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
