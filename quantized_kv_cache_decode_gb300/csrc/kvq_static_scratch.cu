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
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// The array's device address on each device, with the id of the context it was
// looked up in: a device reset (cudaDeviceReset) gives the device a new primary
// context, in which the old address is not valid, so the lookup is repeated.
struct ScratchSlot {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_scratch_mutex;
ScratchSlot g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (0: none yet).  The two
// driver calls are fetched through the runtime, so the library does not link
// the driver library itself.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  if (!get_current || !get_id) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 4000, cudaEnableDefault, &q0) != cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess || !f0)
      return false;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f1)
      return false;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f0);
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f1);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  if (!ctx) {
    *id = 0;
    return true;
  }
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device.  In host code the
// array's name only stands for the symbol; the runtime translates it, with the
// device current, once per device (and again after a reset of the device).
kvq_status scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = 0;
  if (!current_context_id(&id)) return KVQ_ERR_CUDA;
  ScratchSlot& s = g_scratch[dev];
  if (id == 0 || !s.addr || s.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    if (!current_context_id(&id) || id == 0) return KVQ_ERR_CUDA;  // the lookup made the context current
    s.addr = p;
    s.ctx_id = id;
  }
  *addr = s.addr;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attention_static_scratch(const kvq_layer_config* cfg, const kvq_layer_cache* cache,
                                               const void* q, int32_t num_q_heads, const int32_t* seq_lens,
                                               int32_t batch, float softmax_scale, void* out, int32_t out_bf16,
                                               float* lse, uint32_t* dev_status, void* stream) {
  // every argument the merge launch takes is checked before the split pass is enqueued, so a
  // host-detectable error enqueues nothing (the split pass checks the rest itself)
  if (out_bf16 != 0 && out_bf16 != 1) return KVQ_ERR_INVALID_ARG;
  if (batch > 0 && !out) return KVQ_ERR_INVALID_ARG;
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
