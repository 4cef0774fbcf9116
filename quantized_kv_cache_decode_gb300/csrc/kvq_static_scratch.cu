// Decode attention without a caller-provided workspace.
//
// kvq_decode_attention needs device scratch memory for its per-CTA partial
// results, which the caller normally allocates.  Some callers cannot do that:
// code that runs inside a host application owning every byte of device memory
// through its own pool (and forbids direct cudaMalloc), latency-critical loops
// where an allocation's implicit device synchronisation is not acceptable, or
// plug-ins with no access to an allocator at all.  For them this file keeps one
// fixed scratch array in device global memory, sized at compile time; every
// GPU that loads the library reserves it until the process exits.
//
// The entry point reuses the two-launch form of the decode (partials, then
// merge), which needs no scratch contents to start at zero: every word it reads
// in a call was written earlier in the same call.
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name only stands for the symbol; the runtime translates it once per
// device, with that device current.
kvq_status scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attention_static_scratch(const kvq_layer_config* cfg, const kvq_layer_cache* cache,
                                               const void* q, int32_t num_q_heads, const int32_t* seq_lens,
                                               int32_t batch, float softmax_scale, void* out, int32_t out_bf16,
                                               float* lse, uint32_t* dev_status, void* stream) {
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_size(cfg, batch, num_q_heads, &need);
  if (st != KVQ_OK) return st;
  if (need > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;  // batch * heads too large for the fixed array
  void* ws = nullptr;
  if ((st = scratch_address(&ws)) != KVQ_OK) return st;
  st = kvq_decode_partials(cfg, cache, q, num_q_heads, seq_lens, batch, softmax_scale, ws, need, dev_status, stream);
  if (st != KVQ_OK) return st;
  return kvq_decode_combine(cfg, num_q_heads, batch, out, out_bf16, lse, ws, need, stream);
}

}  // extern "C"
