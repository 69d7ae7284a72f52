// Quantize-on-append: rotate K (RoPE, fp32), quantize K and V rows group-wise
// and write codes and scales into their pages.
//
// Method: [airllm] §4.2 group_quantize (scale = amax / (2^(bits-1) - 1),
// clamp_min, round, clamp, two codes per byte with the even element low);
// [Shimmy] §3.2 (one quantized vector per kv head with its scale);
// [Fieldfare] "量化和精度" (affine 4-bit with bf16 scale and bias) and
// "KV Cache 的双布局设计" (K rotated before caching, V not; ring rows
// overwritten in place); [airllm] §2.3 (fixed-size pages from a shared pool).
//
// One warp handles one (row, kv head) and both its K and V vectors; the row
// arithmetic (kvq_quant.cuh) is the one the fused append + decode path uses.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {

struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int32_t* seq_ids;
  const int32_t* pos;
  const int32_t* block_table;
  const float* rope_tab;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int32_t* status;
  int32_t n_rows, n_kv_heads, n_seqs, max_pages, ring_rows, rope_max_pos, n_pool_pages;
  int32_t act, rope;
  PoolLayout kl, vl;
};

template <int HD>
__global__ void __launch_bounds__(128) append_kernel(const AppendArgs a) {
  constexpr int DPL = HD / 32;
  constexpr int P = 16;
  const int lane = threadIdx.x & 31;
  // Programmatic dependent launch: the new rows may come from the kernel
  // before this one; the kernel after it may start launching at once (it
  // waits for this grid before reading the pools: a decode with early reads
  // is not to follow an append to its own pools).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (item >= (int64_t)a.n_rows * a.n_kv_heads) return;
  const int row = (int)(item / a.n_kv_heads);
  const int head = (int)(item % a.n_kv_heads);

  const int seq = a.seq_ids ? a.seq_ids[row] : row;
  const int pos = a.pos[row];
  if (seq < 0 || seq >= a.n_seqs) {
    if (lane == 0 && head == 0) report(a.status, KVQ_DEV_BAD_SEQ);
    return;
  }
  const int r = a.ring_rows > 0 ? (pos >= 0 ? pos % a.ring_rows : -1) : pos;
  if (pos < 0 || r / P >= a.max_pages || (a.rope != KVQ_ROPE_NONE && pos >= a.rope_max_pos)) {
    if (lane == 0 && head == 0) report(a.status, KVQ_DEV_BAD_POS);
    return;
  }
  const int page = a.block_table[(int64_t)seq * a.max_pages + r / P];
  if (page < 0 || page >= a.n_pool_pages) {
    if (lane == 0 && head == 0) report(a.status, KVQ_DEV_BAD_PAGE);
    return;
  }
  const int slot = r % P;
  const int64_t base = ((int64_t)row * a.n_kv_heads + head) * HD + lane * DPL;

  // K: load, rotate at `pos` in fp32 with one rounding per operation.
  float x[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) x[j] = load_act(a.k_new, a.act, base + j);
  if (a.rope != KVQ_ROPE_NONE)
    rope_rotate_row<DPL>(x, reinterpret_cast<const float2*>(a.rope_tab) + (int64_t)pos * (HD / 2), a.rope, lane);
  store_row(quantize_row<DPL>(x, a.kl, lane), a.kl,
            a.k_pool + (int64_t)page * a.kl.page_bytes + (int64_t)head * a.kl.sub_bytes, slot, lane);

  // V: no rotation.
#pragma unroll
  for (int j = 0; j < DPL; ++j) x[j] = load_act(a.v_new, a.act, base + j);
  store_row(quantize_row<DPL>(x, a.vl, lane), a.vl,
            a.v_pool + (int64_t)page * a.vl.page_bytes + (int64_t)head * a.vl.sub_bytes, slot, lane);
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_append(const kvq_config* cfg, int32_t n_rows, const void* k_new,
                                 const void* v_new, const int32_t* seq_ids, const int32_t* pos,
                                 const int32_t* block_table, int32_t n_seqs,
                                 int32_t max_pages_per_seq, int32_t ring_rows,
                                 const float* rope_tab, int32_t rope_max_pos, void* k_pool,
                                 void* v_pool, int32_t n_pool_pages, int32_t* dev_status,
                                 kvq_stream_t stream) {
  clear_error();
  kvq_status st = check_kernel_config(cfg);
  if (st != KVQ_OK) return st;
  if (n_rows < 0) return fail(KVQ_ERR_INVALID_ARG, "n_rows (%d) < 0", n_rows);
  if (n_rows == 0) return KVQ_OK;
  if (!k_new || !v_new || !pos || !block_table || !k_pool || !v_pool || !dev_status)
    return fail(KVQ_ERR_INVALID_ARG, "a required device pointer is NULL");
  if (n_seqs < 1 || max_pages_per_seq < 1 || n_pool_pages < 1)
    return fail(KVQ_ERR_INVALID_ARG, "n_seqs, max_pages_per_seq and n_pool_pages must be >= 1");
  if (!seq_ids && n_rows > n_seqs)
    return fail(KVQ_ERR_INVALID_ARG, "without seq_ids, n_rows (%d) must be <= n_seqs (%d)", n_rows, n_seqs);
  if (ring_rows < 0 || ring_rows % cfg->page_size != 0 || ring_rows / cfg->page_size > max_pages_per_seq)
    return fail(KVQ_ERR_INVALID_ARG, "ring_rows %d must be a multiple of page_size that fits the table",
                ring_rows);
  if (cfg->rope != KVQ_ROPE_NONE && (!rope_tab || rope_max_pos < 1))
    return fail(KVQ_ERR_INVALID_ARG, "RoPE config needs rope_tab and rope_max_pos >= 1");
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15)
    return fail(KVQ_ERR_INVALID_ARG, "pools must be 16-byte aligned");

  AppendArgs a;
  a.k_new = k_new; a.v_new = v_new; a.seq_ids = seq_ids; a.pos = pos;
  a.block_table = block_table; a.rope_tab = rope_tab;
  a.k_pool = static_cast<uint8_t*>(k_pool); a.v_pool = static_cast<uint8_t*>(v_pool);
  a.status = dev_status;
  a.n_rows = n_rows; a.n_kv_heads = cfg->n_kv_heads; a.n_seqs = n_seqs;
  a.max_pages = max_pages_per_seq; a.ring_rows = ring_rows; a.rope_max_pos = rope_max_pos;
  a.n_pool_pages = n_pool_pages; a.act = cfg->act_dtype; a.rope = cfg->rope;
  a.kl = pool_layout(*cfg, 0);
  a.vl = pool_layout(*cfg, 1);

  const int64_t warps = (int64_t)n_rows * cfg->n_kv_heads;
  const int64_t blocks = (warps + 3) / 4;
  if (blocks > 0x7fffffffLL) return fail(KVQ_ERR_INVALID_ARG, "too many rows");
  if (blocks == 0) return KVQ_OK;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)blocks);
  lc.blockDim = dim3(128);
  lc.stream = (cudaStream_t)stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e;
  switch (cfg->head_dim) {
    case 64: e = cudaLaunchKernelEx(&lc, append_kernel<64>, a); break;
    case 128: e = cudaLaunchKernelEx(&lc, append_kernel<128>, a); break;
    case 256: e = cudaLaunchKernelEx(&lc, append_kernel<256>, a); break;
    default: return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d", cfg->head_dim);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}
