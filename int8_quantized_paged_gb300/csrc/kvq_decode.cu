// Decode entry points: argument checks, workspace layout, the split-K launch
// and the log-sum-exp combine of the chunks.
//
// Combine: for chunks c with partial state (m_c, l_c, acc_c) in base 2,
//   M = max_c m_c ;  out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c,
// which equals the softmax over the whole context (the chunks partition it).
#include <cuda_runtime.h>

#include "kvq_decode_impl.cuh"

namespace kvq {

static constexpr int kMaxChunks = 8192;

struct WsLayout {
  int chunk_tokens, n_chunks;
  size_t acc_bytes, ml_offset, total;
};

static WsLayout ws_layout(const kvq_config& c, int32_t batch, int64_t max_tokens, int32_t requested) {
  WsLayout w{};
  w.chunk_tokens = chunk_tokens_for(c, batch, max_tokens, requested);
  w.n_chunks = (int)((max_tokens + w.chunk_tokens - 1) / w.chunk_tokens);
  if (w.n_chunks < 1) w.n_chunks = 1;
  const size_t units = (size_t)batch * c.n_kv_heads * w.n_chunks * (c.n_heads / c.n_kv_heads);
  w.acc_bytes = units * c.head_dim * sizeof(float);
  w.ml_offset = (w.acc_bytes + 255) / 256 * 256;
  w.total = w.ml_offset + units * 2 * sizeof(float);
  return w;
}

__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a, void* out, int G, int HD) {
  extern __shared__ float wgt[];          // n_chunks weights
  __shared__ float red[4];
  __shared__ float bcast;
  const int h = blockIdx.x, b = blockIdx.y;
  const int kvh = h / G, hh = h % G;
  const int L = a.seq_lens[b];
  const int64_t obase = ((int64_t)b * a.n_heads + h) * HD;
  int lo = 0, bad = 0;
  const int n_att = attended(a, L, &lo, &bad);
  const int nch = n_att > 0 ? (n_att + a.chunk_tokens - 1) / a.chunk_tokens : 0;
  if (nch == 0) {
    for (int d = threadIdx.x; d < HD; d += blockDim.x) store_act(out, a.act, obase + d, 0.f);
    return;
  }
  const int64_t cbase = ((int64_t)b * a.n_kv_heads + kvh) * a.n_chunks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float mx = -INFINITY;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) mx = fmaxf(mx, a.ws_ml[((cbase + c) * G + hh) * 2]);
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) bcast = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  const float M = bcast;

  float den = 0.f;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    const float mc = a.ws_ml[((cbase + c) * G + hh) * 2];
    const float w = (M == -INFINITY || mc == -INFINITY) ? 0.f : exp2f(mc - M);
    wgt[c] = w;
    den = fmaf(w, a.ws_ml[((cbase + c) * G + hh) * 2 + 1], den);
  }
  for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  __syncthreads();
  if (lane == 0) red[warp] = den;
  __syncthreads();
  if (threadIdx.x == 0) bcast = red[0] + red[1] + red[2] + red[3];
  __syncthreads();
  const float total = bcast;
  const float inv = total > 0.f ? 1.f / total : 0.f;

  for (int d = threadIdx.x; d < HD; d += blockDim.x) {
    float o = 0.f;
    for (int c = 0; c < nch; ++c) o = fmaf(wgt[c], a.ws_acc[((cbase + c) * G + hh) * HD + d], o);
    store_act(out, a.act, obase + d, o * inv);
  }
}

static kvq_status run_decode(const kvq_config* cfg, int32_t batch, const void* q, const void* k_pool,
                             const void* v_pool, int32_t n_pool_pages, const int32_t* block_table,
                             int32_t max_pages, const int32_t* seq_lens, const float* rope_tab,
                             int32_t rope_max_pos, void* out, void* workspace, size_t ws_bytes,
                             int32_t chunk_tokens, int32_t* dev_status, cudaStream_t stream,
                             int32_t ring_rows, int32_t window, int64_t max_tokens) {
  WsLayout w = ws_layout(*cfg, batch, max_tokens, chunk_tokens);
  if (w.n_chunks > kMaxChunks)
    return fail(KVQ_ERR_INVALID_ARG, "%d chunks of %d tokens exceed the limit %d; use larger chunks",
                w.n_chunks, w.chunk_tokens, kMaxChunks);
  if (ws_bytes < w.total)
    return fail(KVQ_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, w.total);
  if (batch == 0) return KVQ_OK;

  DecodeArgs a;
  a.q = q;
  a.k_pool = static_cast<const uint8_t*>(k_pool);
  a.v_pool = static_cast<const uint8_t*>(v_pool);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.rope_tab = rope_tab;
  a.ws_acc = static_cast<float*>(workspace);
  a.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.ml_offset);
  a.status = dev_status;
  a.batch = batch;
  a.n_heads = cfg->n_heads;
  a.n_kv_heads = cfg->n_kv_heads;
  a.n_pool_pages = n_pool_pages;
  a.max_pages = max_pages;
  a.rope_max_pos = rope_max_pos;
  a.ring_rows = ring_rows;
  a.window = window;
  a.chunk_tokens = w.chunk_tokens;
  a.n_chunks = w.n_chunks;
  a.act = cfg->act_dtype;
  a.rope = cfg->rope;
  a.score_scale = score_scale_log2(*cfg);
  a.kl = pool_layout(*cfg, 0);
  a.vl = pool_layout(*cfg, 1);

  const int G = cfg->n_heads / cfg->n_kv_heads;
  const dim3 grid(w.n_chunks, cfg->n_kv_heads, batch);
  kvq_status st;
  const int k = cfg->k_dtype, v = cfg->v_dtype;
  if (k == KVQ_SYM_INT4 && v == KVQ_SYM_INT4) st = launch_decode_s4s4(a, cfg->head_dim, G, grid, stream);
  else if (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT8) st = launch_decode_s8s8(a, cfg->head_dim, G, grid, stream);
  else if (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT4) st = launch_decode_s8s4(a, cfg->head_dim, G, grid, stream);
  else st = launch_decode_a4a4(a, cfg->head_dim, G, grid, stream);
  if (st != KVQ_OK) return st;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));

  combine_kernel<<<dim3(cfg->n_heads, batch), 128, w.n_chunks * sizeof(float), stream>>>(
      a, out, G, cfg->head_dim);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

static kvq_status check_decode_args(const kvq_config* cfg, int32_t batch, const void* q, const void* k_pool,
                                    const void* v_pool, int32_t n_pool_pages, const int32_t* table,
                                    const int32_t* seq_lens, const float* rope_tab, int32_t rope_max_pos,
                                    void* out, void* workspace, int32_t chunk_tokens, int32_t* dev_status) {
  kvq_status st = check_kernel_config(cfg);
  if (st != KVQ_OK) return st;
  if (batch < 0) return fail(KVQ_ERR_INVALID_ARG, "batch (%d) < 0", batch);
  if (batch == 0) return KVQ_OK;
  if (!q || !k_pool || !v_pool || !table || !seq_lens || !out || !workspace || !dev_status)
    return fail(KVQ_ERR_INVALID_ARG, "a required device pointer is NULL");
  if (n_pool_pages < 1) return fail(KVQ_ERR_INVALID_ARG, "n_pool_pages must be >= 1");
  if (chunk_tokens < 0 || chunk_tokens % cfg->page_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "chunk_tokens %d must be 0 or a multiple of page_size", chunk_tokens);
  if (cfg->rope != KVQ_ROPE_NONE && (!rope_tab || rope_max_pos < 1))
    return fail(KVQ_ERR_INVALID_ARG, "RoPE config needs rope_tab and rope_max_pos >= 1");
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15)
    return fail(KVQ_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(KVQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t max_pages_per_seq,
                                             int32_t chunk_tokens) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  if (batch < 0 || max_pages_per_seq < 1 || chunk_tokens < 0 || chunk_tokens % cfg->page_size) {
    set_error("bad batch, max_pages_per_seq or chunk_tokens");
    return 0;
  }
  return ws_layout(*cfg, batch, (int64_t)max_pages_per_seq * cfg->page_size, chunk_tokens).total;
}

extern "C" size_t kvq_window_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t window,
                                             int32_t chunk_tokens) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  if (batch < 0 || window < 1 || chunk_tokens < 0 || chunk_tokens % cfg->page_size) {
    set_error("bad batch, window or chunk_tokens");
    return 0;
  }
  return ws_layout(*cfg, batch, window, chunk_tokens).total;
}

extern "C" kvq_status kvq_decode_attention(const kvq_config* cfg, int32_t batch, const void* q,
                                           const void* k_pool, const void* v_pool, int32_t n_pool_pages,
                                           const int32_t* block_table, int32_t max_pages_per_seq,
                                           const int32_t* seq_lens, const float* rope_tab,
                                           int32_t rope_max_pos, void* out, void* workspace,
                                           size_t workspace_bytes, int32_t chunk_tokens,
                                           int32_t* dev_status, kvq_stream_t stream) {
  clear_error();
  kvq_status st = check_decode_args(cfg, batch, q, k_pool, v_pool, n_pool_pages, block_table, seq_lens,
                                    rope_tab, rope_max_pos, out, workspace, chunk_tokens, dev_status);
  if (st != KVQ_OK || batch == 0) return st;
  if (max_pages_per_seq < 1) return fail(KVQ_ERR_INVALID_ARG, "max_pages_per_seq must be >= 1");
  return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, block_table, max_pages_per_seq, seq_lens,
                    rope_tab, rope_max_pos, out, workspace, workspace_bytes, chunk_tokens, dev_status,
                    (cudaStream_t)stream, 0, 0, (int64_t)max_pages_per_seq * cfg->page_size);
}

extern "C" kvq_status kvq_window_decode(const kvq_config* cfg, int32_t batch, const void* q,
                                        const void* k_pool, const void* v_pool, int32_t n_pool_pages,
                                        const int32_t* ring_table, int32_t ring_rows, int32_t window,
                                        const int32_t* seq_lens, const float* rope_tab, int32_t rope_max_pos,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        int32_t chunk_tokens, int32_t* dev_status, kvq_stream_t stream) {
  clear_error();
  kvq_status st = check_decode_args(cfg, batch, q, k_pool, v_pool, n_pool_pages, ring_table, seq_lens,
                                    rope_tab, rope_max_pos, out, workspace, chunk_tokens, dev_status);
  if (st != KVQ_OK || batch == 0) return st;
  if (ring_rows < cfg->page_size || ring_rows % cfg->page_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "ring_rows %d must be a positive multiple of page_size", ring_rows);
  if (window < 1 || window > ring_rows)
    return fail(KVQ_ERR_INVALID_ARG, "window %d must be in [1, ring_rows=%d]", window, ring_rows);
  return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, ring_table, ring_rows / cfg->page_size,
                    seq_lens, rope_tab, rope_max_pos, out, workspace, workspace_bytes, chunk_tokens,
                    dev_status, (cudaStream_t)stream, ring_rows, window, window);
}
