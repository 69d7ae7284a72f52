// kvq_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// Some callers never get to call cudaMalloc.  A plugin inside a host engine
// that already owns every byte of HBM through its own pool is one.  So is code
// on a latency-critical path where an allocation (and the device-wide
// synchronization it can imply) is not allowed.  This entry point keeps the
// split-K workspace in a fixed array compiled into the library.  The caller
// passes only inputs and outputs.
//
// The scratch array lives in device memory on every GPU that loads the
// library, until the process exits.  In host code, the symbol g_kvq_scratch
// is only a host-side stand-in: it is not a device address and must never
// reach a kernel.  The device address is looked up with cudaGetSymbolAddress,
// on that device, the first time this entry point runs in a CUDA context of
// that device, and kept with the context's unique id.  A device reset (or any
// new primary context) loads the module again, possibly at another address,
// so a call in a context other than the remembered one looks the address up
// again.  The first call in each context should therefore come before any
// stream capture.
// Every call shares the one array, so calls whose kernels overlap on the GPU
// (for example on two streams at once) race on it.  Its arrival counters
// start at zero (static device memory is zero-initialised), and every
// completed call leaves them zero again, so nothing has to be cleared between
// calls.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

__device__ __align__(256) unsigned char g_kvq_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id;   // unique id of the context the address belongs to
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Unique id of the calling thread's current CUDA context, through the driver
// entry points the runtime hands out (no link against the driver library).
kvq_status current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (!get_current || !get_id) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult r0 = cudaDriverEntryPointSymbolNotFound, r1 = r0;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &r0);
    if (e == cudaSuccess)
      e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &r1);
    if (e != cudaSuccess || r0 != cudaDriverEntryPointSuccess || r1 != cudaDriverEntryPointSuccess || !f0 || !f1)
      return kvq::fail(KVQ_ERR_CUDA, "driver entry points cuCtxGetCurrent / cuCtxGetId not available");
    get_current = reinterpret_cast<GetCurrent>(f0);
    get_id = reinterpret_cast<GetId>(f1);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
    return kvq::fail(KVQ_ERR_CUDA, "no current CUDA context");
  return KVQ_OK;
}

// Device address of the scratch array in the current device's context.
kvq_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::fail(KVQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return kvq::fail(KVQ_ERR_UNSUPPORTED, "device index %d", dev);
  // Before the first runtime call on this thread there may be no current
  // context yet: then the cached entry is not used, and the context id is
  // read again after cudaGetSymbolAddress has made the primary context current.
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  kvq_status st = current_context_id(&id);
  if (st == KVQ_OK && g_scratch[dev].ptr && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return KVQ_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_kvq_scratch);
  if (e != cudaSuccess || !p)
    return kvq::fail(KVQ_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  st = current_context_id(&id);   // the lookup above made the context current if it was not
  if (st != KVQ_OK) return st;
  g_scratch[dev] = ScratchAddr{id, p};
  *out = p;
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, int32_t batch, const void* q,
                                                   const void* k_pool, const void* v_pool,
                                                   int32_t n_pool_pages, const int32_t* block_table,
                                                   int32_t max_pages_per_seq, const int32_t* seq_lens,
                                                   const float* rope_tab, int32_t rope_max_pos, void* out,
                                                   int32_t chunk_tokens, int32_t* dev_status,
                                                   kvq_stream_t stream) {
  kvq::clear_error();
  if (batch == 0)   // nothing to do; argument checks only
    return kvq_decode_attention(cfg, 0, q, k_pool, v_pool, n_pool_pages, block_table, max_pages_per_seq,
                                seq_lens, rope_tab, rope_max_pos, out, nullptr, 0, chunk_tokens, dev_status,
                                stream);
  const size_t need = kvq_decode_workspace_bytes(cfg, batch, max_pages_per_seq, chunk_tokens);
  if (need == 0) {
    const kvq_status v = kvq_validate_config(cfg);
    return v != KVQ_OK ? v
                       : kvq::fail(KVQ_ERR_INVALID_ARG, "bad batch, max_pages_per_seq or chunk_tokens");
  }
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES)
    return kvq::fail(KVQ_ERR_WORKSPACE_TOO_SMALL,
                     "this decode needs %zu bytes of workspace; the built-in scratch holds %zu. "
                     "Use kvq_decode_attention with a caller workspace, a larger chunk_tokens, "
                     "or a smaller batch", need, (size_t)KVQ_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  kvq_status st = scratch_address(&ws);
  if (st != KVQ_OK) return st;
  return kvq_decode_attention(cfg, batch, q, k_pool, v_pool, n_pool_pages, block_table, max_pages_per_seq,
                              seq_lens, rope_tab, rope_max_pos, out, ws, (size_t)KVQ_NOALLOC_SCRATCH_BYTES,
                              chunk_tokens, dev_status, stream);
}
