// Decode entry points: argument checks, the chunk plan and workspace layout,
// and the launches.
//
// Two kernels compute the same decode.  The tensor-core kernel
// (kvq_decode_tc.cuh) is the default.  It fuses the log-sum-exp combine into
// the same launch, so a call is one launch: for a few long sequences the
// chunks of each (sequence, kv head) form one thread-block cluster and
// combine through distributed shared memory; otherwise the last CTA of each
// (sequence, kv head) combines the partials the others left in the
// workspace.  KVQ_DECODE_CLUSTER=0 in the environment turns the cluster mode
// off.  The
// CUDA-core kernel (kvq_decode_impl.cuh) covers shapes the tensor-core kernel
// does not take: groups that are not a multiple of 32, and 8-bit rows longer
// than 128 bytes.  It is followed by a separate combine kernel.  Setting
// KVQ_DECODE_IMPL=simt in the environment selects it for every shape, so the
// two can be compared side by side.
//
// Combine: for chunks c with partial state (m_c, l_c, acc_c) in base 2,
//   M = max_c m_c ;  out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c,
// which equals the softmax over the whole context (the chunks partition it).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvq_decode_impl.cuh"
#include "kvq_decode_tc.cuh"

namespace kvq {

static constexpr int kMaxChunks = 8192;

// Whether the tensor-core kernel takes this config (and is not switched off):
// power-of-two groups of at least 32 elements, a head_dim/G shape with an
// instantiation, and one stored type for the K and V scales.
// Scale groups per head of the tensor-core kernel (1 for unquantised f16).
static int tc_ng(const kvq_config& c) { return c.k_dtype == KVQ_F16_KV ? 1 : c.head_dim / c.k_group; }

// f16 K/V have only the tensor-core kernel (head_dim 64 and 128).
static bool tc_enabled(const kvq_config& c) {
  static int forced = -1;
  if (forced < 0) {
    const char* e = std::getenv("KVQ_DECODE_IMPL");
    forced = (e && std::strcmp(e, "simt") == 0) ? 0 : 1;
  }
  if (c.k_dtype == KVQ_F16_KV) {
    const int G = c.n_heads / c.n_kv_heads;
    return c.head_dim <= 128 && tc_has_shape(c.head_dim, G > 4 ? 2 : 1, 1);
  }
  if (!forced) return false;
  const bool pow2 = (c.k_group & (c.k_group - 1)) == 0 && (c.v_group & (c.v_group - 1)) == 0;
  if (!pow2 || c.k_param_dtype != c.v_param_dtype || c.k_group < 32 || c.v_group < 32) return false;
  const int G = c.n_heads / c.n_kv_heads;
  return c.k_group == c.v_group && tc_has_shape(c.head_dim, G > 4 ? 2 : 1, c.head_dim / c.k_group);
}

static bool cluster_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("KVQ_DECODE_CLUSTER");
    return !(e && std::strcmp(e, "0") == 0);
  }();
  return on;
}

// How many clusters of a launch configuration can be resident at once,
// cached per (launcher, shape, cluster size, shared memory, device).
static int max_active_clusters(TcLaunch fn, const TcArgs& t, int hd, int nt, int ng, const TcLaunchCfg& lc) {
  struct Entry {
    TcLaunch fn;
    int hd, nt, ng, cluster, dev;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> g(mu);
    for (const Entry& e : cache)
      if (e.fn == fn && e.hd == hd && e.nt == nt && e.ng == ng && e.cluster == lc.cluster && e.dev == dev &&
          e.smem == lc.smem)
        return e.n;
  }
  int n = 0;
  TcLaunchCfg q = lc;
  q.max_active = &n;
  if (fn(t, hd, nt, ng, q) != KVQ_OK) n = 0;
  std::lock_guard<std::mutex> g(mu);
  cache.push_back(Entry{fn, hd, nt, ng, lc.cluster, dev, lc.smem, n});
  return n;
}

// The tensor-core launcher of a config's K/V kinds and scale type.
static TcLaunch tc_launcher(const kvq_config& c) {
  if (c.k_dtype == KVQ_F16_KV) return launch_tc_h16;   // no scales: one instantiation
  if (c.k_dtype == KVQ_SHIMMY_INT4) return launch_tc_o4o4_f32;   // f32 scales only
  static const TcLaunch table[4][3] = {
      {launch_tc_s4s4_f32, launch_tc_s4s4_f16, launch_tc_s4s4_bf16},
      {launch_tc_s8s8_f32, launch_tc_s8s8_f16, launch_tc_s8s8_bf16},
      {launch_tc_s8s4_f32, launch_tc_s8s4_f16, launch_tc_s8s4_bf16},
      {launch_tc_a4a4_f32, launch_tc_a4a4_f16, launch_tc_a4a4_bf16}};
  const int k = c.k_dtype, v = c.v_dtype;
  const int kind = (k == KVQ_SYM_INT4 && v == KVQ_SYM_INT4) ? 0
                   : (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT8) ? 1
                   : (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT4) ? 2
                                                              : 3;
  return table[kind][c.k_param_dtype];
}

// Bytes of one warp's ring of page slots (the cluster mode keeps more pages in flight).
static size_t tc_ring_bytes(const kvq_config& c, bool cluster) {
  const int G = c.n_heads / c.n_kv_heads;
  return (size_t)tc_depth(c.head_dim, G > 4 ? 2 : 1, c.k_dtype, cluster) *
         tc_slot_bytes(c.k_dtype, c.v_dtype, c.head_dim, tc_ng(c), c.k_param_dtype);
}

// The cluster mode: a few sequences, each short enough that one cluster of
// up to kMaxCluster CTAs of kClusterWarps warps (one CTA per SM) covers it
// with at most eight pages per warp, and all the clusters resident at once.
// The cluster is as large as that allows, down to one page per warp: the
// pages of a short context spread over as many SMs as possible.  On success fills the launch
// configuration (grid, shared memory, warps, cluster size) and the 16-token
// blocks per CTA.
static bool pick_cluster(const kvq_config& c, int32_t batch, int64_t max_tokens, int32_t window, TcLaunch fn,
                         size_t ring, size_t pre, TcLaunchCfg* lc, int* cb_out, int* recv_out) {
  const int G = c.n_heads / c.n_kv_heads;
  const int hd = c.head_dim;
  const int nt = G > 4 ? 2 : 1;
  if (!cluster_enabled() || batch < 1 || !tc_cluster_shape(hd, nt)) return false;
  // blocks of the longest context (a window may start mid-page)
  const int64_t blocks = (max_tokens + c.page_size - 1) / c.page_size + (window > 0 ? 1 : 0);
  // pages per warp at most: 8, or 12 at head_dim 256, where a 16K-token global
  // layer in 12-CTA clusters (10.7 pages per warp) beat the workspace mode
  // (bench step of the sliding+global mix 669 -> 691 GB/s)
  const int64_t max_ppw = hd == 256 ? 12 : 8;
  if (blocks > (int64_t)kMaxCluster * kClusterWarps * max_ppw || (int64_t)batch * c.n_kv_heads > 4 * num_sms())
    return false;
  // The page rings and the query's staging, or the warps' merge that reuses
  // them; then the receive buffers of the combine, which peers write while
  // this CTA may still be in its loop.
  size_t base = (size_t)kClusterWarps * ring + pre;
  const size_t merge = ((size_t)kClusterWarps * G * (hd + 2) + G) * sizeof(float);
  if (base < merge) base = merge;
  base = (base + 15) & ~(size_t)15;
  if (base + tc_recv_bytes(G, hd, kMaxCluster) > 200 * 1024) return false;
  int64_t hi = (blocks + kClusterWarps - 1) / kClusterWarps;   // one page per warp
  if (hi > kMaxCluster) hi = kMaxCluster;
  const int64_t lo = (blocks + kClusterWarps * max_ppw - 1) / (kClusterWarps * max_ppw);
  TcArgs none{};
  for (int64_t want = hi; want >= lo && want >= 1; --want) {
    const int64_t cb = (blocks + want - 1) / want;
    const int64_t nc = (blocks + cb - 1) / cb;
    if (nc != want) continue;   // the same split as a smaller cluster
    // One CTA per SM: with two, some SMs hold two CTAs of a cluster while
    // others idle, and those CTAs finish last (measured: a smaller cluster at
    // one CTA per SM is faster than 16 CTAs placed two to an SM).
    size_t smem = base + tc_recv_bytes(G, hd, (int)nc);
    if (smem < smem_per_sm() / 2 + 1) smem = smem_per_sm() / 2 + 1;
    smem = (smem + 15) & ~(size_t)15;
    TcLaunchCfg q = *lc;
    q.grid = dim3((unsigned)nc, c.n_kv_heads, batch);
    q.smem = smem;
    q.warps = kClusterWarps;
    q.cluster = (int)nc;
    if (max_active_clusters(fn, none, hd, nt, tc_ng(c), q) >= batch * c.n_kv_heads) {
      *lc = q;
      *cb_out = (int)cb;
      *recv_out = (int)base;
      return true;
    }
  }
  return false;
}

// CTAs of the tensor-core kernel resident per SM (its launch bounds).
static int tc_resident(const kvq_config& c) {
  const int G = c.n_heads / c.n_kv_heads;
  return tc_min_blocks(c.head_dim, G > 4 ? 2 : 1, c.k_dtype);
}

// Chunking and workspace layout of one decode call.  The workspace holds, in
// order: arrival counters [batch][n_kv_heads] (int32, zero between calls),
// partial sums acc [batch][n_kv_heads][n_chunks][G][head_dim] and partial
// (max, sum) [batch][n_kv_heads][n_chunks][G][2], all fp32.  It is sized for
// whichever kernel would run.
struct Plan {
  bool tc;
  int chunk_tokens;          // CUDA-core kernel: tokens per chunk
  int blocks_per_chunk;      // tensor-core kernel: 16-token blocks per chunk
  int n_chunks;              // chunks per (sequence, kv head) the workspace holds
  int tc_chunks;             // chunks the tensor-core kernel uses (grid x)
  size_t acc_offset, ml_offset, total;
};

static Plan make_plan(const kvq_config& c, int32_t batch, int64_t max_tokens, bool window, int32_t requested) {
  Plan p{};
  p.tc = tc_enabled(c);
  const int P = c.page_size;
  // CUDA-core kernel: token chunks starting at the first attended token
  p.chunk_tokens = chunk_tokens_for(c, batch, max_tokens, requested);
  const int64_t n_simt = (max_tokens + p.chunk_tokens - 1) / p.chunk_tokens;
  // tensor-core kernel: page-aligned chunks; a window may start mid-page
  const int64_t max_blocks = (max_tokens + P - 1) / P + (window ? 1 : 0);
  if (requested > 0) {
    p.blocks_per_chunk = requested / P;
  } else {
    // About whole waves of resident CTAs, assuming every sequence is as long
    // as the longest, with 16 to 128 blocks per chunk: at least four pages
    // per warp, so a short context does not split into many small partials.
    const int64_t total = (int64_t)batch * c.n_kv_heads * max_blocks;
    const int64_t wave = (int64_t)num_sms() * tc_resident(c);
    const int64_t waves = (total + wave * 128 - 1) / (wave * 128);
    int64_t cb = (total + waves * wave - 1) / (waves * wave);
    cb = (cb + kWarps - 1) / kWarps * kWarps;
    p.blocks_per_chunk = (int)(cb < 4 * kWarps ? 4 * kWarps : (cb > 128 ? 128 : cb));
  }
  const int64_t n_tc = (max_blocks + p.blocks_per_chunk - 1) / p.blocks_per_chunk;
  p.tc_chunks = (int)(n_tc < 1 ? 1 : (n_tc > (1 << 30) ? (1 << 30) : n_tc));
  const int64_t n = n_simt > n_tc ? n_simt : n_tc;
  p.n_chunks = (int)(n < 1 ? 1 : (n > (1 << 30) ? (1 << 30) : n));
  const size_t units = (size_t)batch * c.n_kv_heads * p.n_chunks * (c.n_heads / c.n_kv_heads);
  const size_t counters = ((size_t)batch * c.n_kv_heads * sizeof(int32_t) + 255) / 256 * 256;
  p.acc_offset = counters;
  p.ml_offset = p.acc_offset + (units * c.head_dim * sizeof(float) + 255) / 256 * 256;
  p.total = p.ml_offset + units * 2 * sizeof(float);
  return p;
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
                             int32_t ring_rows, int32_t window, int64_t max_tokens,
                             const void* app_k = nullptr, const void* app_v = nullptr,
                             const int32_t* app_pos = nullptr) {
  const Plan w = make_plan(*cfg, batch, max_tokens, window > 0, chunk_tokens);
  if (w.n_chunks > kMaxChunks)
    return fail(KVQ_ERR_INVALID_ARG, "%d chunks exceed the limit %d; use larger chunks", w.n_chunks, kMaxChunks);
  if (ws_bytes < w.total)
    return fail(KVQ_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, w.total);
  if (batch == 0) return KVQ_OK;
  if (batch > 65535 || cfg->n_kv_heads > 65535) return fail(KVQ_ERR_INVALID_ARG, "batch or n_kv_heads too large");

  DecodeArgs a;
  a.q = q;
  a.app_k = app_k;
  a.app_v = app_v;
  a.app_pos = app_pos;
  a.k_pool = static_cast<const uint8_t*>(k_pool);
  a.v_pool = static_cast<const uint8_t*>(v_pool);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.rope_tab = rope_tab;
  a.ws_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.acc_offset);
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
  const int k = cfg->k_dtype, v = cfg->v_dtype;
  if (w.tc) {
    TcArgs t;
    t.d = a;
    t.out = out;
    t.counters = static_cast<int32_t*>(workspace);
    t.G = G;
    t.blocks_per_chunk = w.blocks_per_chunk;
    t.kc_bytes = cfg->page_size * a.kl.code_bytes;
    t.vc_bytes = cfg->page_size * a.vl.code_bytes;
    t.kp_bytes = cfg->page_size * a.kl.param_row_bytes;
    t.vp_bytes = cfg->page_size * a.vl.param_row_bytes;
    t.cluster = 0;
    t.recv_off = 0;
    t.early = (cfg->flags & KVQ_FLAG_EARLY_READS) != 0;
    const int nt = G > 4 ? 2 : 1;
    const int hd = cfg->head_dim;
    const int ng = tc_ng(*cfg);   // scale groups per head (K and V alike)
    const int pt = cfg->k_param_dtype;
    if (t.kp_bytes != tc_scale_bytes(k, ng, pt) || t.vp_bytes != tc_scale_bytes(v, ng, pt))
      return fail(KVQ_ERR_UNSUPPORTED, "scale rows do not match the tensor-core kernel's slots");
    const TcLaunch fn = tc_launcher(*cfg);
    // Shared memory: a ring of tc_depth pages per warp and the query's
    // fragments, reused at the end for the warps' merge and then either the
    // cluster's partial or the combine's weights.
    const size_t ring_cl = tc_ring_bytes(*cfg, true), ring = tc_ring_bytes(*cfg, false);
    const size_t pre_cl = tc_pre_bytes(hd, nt, ng, true), pre = tc_pre_bytes(hd, nt, ng, false);
    auto merge_bytes = [&](int warps) { return ((size_t)warps * G * (hd + 2) + G) * sizeof(float); };
    TcLaunchCfg lc{};
    lc.stream = stream;
    lc.pdl = pdl_enabled();

    int cb = 0, recv = 0;
    if (chunk_tokens == 0 && pick_cluster(*cfg, batch, max_tokens, window, fn, ring_cl, pre_cl, &lc, &cb, &recv)) {
      t.cluster = lc.cluster;
      t.blocks_per_chunk = cb;
      t.recv_off = recv;
      return fn(t, hd, nt, ng, lc);
    }

    size_t smem = (size_t)kWarps * ring + pre;
    const size_t need_merge = merge_bytes(kWarps);
    // combine: (m, l) of every chunk, then the per-group column sums
    const size_t need_comb = (size_t)w.n_chunks * G * 2 * sizeof(float) + 16 +
                             (size_t)kTcThreads * 4 * sizeof(float);
    if (smem < need_merge) smem = need_merge;
    if (smem < need_comb) smem = need_comb;
    if (smem > 200 * 1024)
      return fail(KVQ_ERR_UNSUPPORTED, "decode needs %zu bytes of shared memory; use larger chunks", smem);
    lc.grid = dim3(w.tc_chunks, cfg->n_kv_heads, batch);
    lc.smem = smem;
    lc.warps = kWarps;
    lc.cluster = 0;
    return fn(t, hd, nt, ng, lc);
  }

  if (k == KVQ_F16_KV || k == KVQ_SHIMMY_INT4)
    return fail(KVQ_ERR_UNSUPPORTED, "K/V kind %d: only the tensor-core kernel, which does not take head_dim %d, G %d",
                k, cfg->head_dim, G);
  const dim3 grid(w.n_chunks, cfg->n_kv_heads, batch);
  kvq_status st;
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
  if (reinterpret_cast<uintptr_t>(q) & 15) return fail(KVQ_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (cfg->rope != KVQ_ROPE_NONE && (reinterpret_cast<uintptr_t>(rope_tab) & 15))
    return fail(KVQ_ERR_INVALID_ARG, "rope_tab must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(KVQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

extern "C" int32_t kvq_decode_cluster_ctas(const kvq_config* cfg, int32_t batch, int32_t max_pages_per_seq,
                                           int32_t window, int32_t chunk_tokens) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return -1;
  if (batch < 1 || max_pages_per_seq < 1 || window < 0 || chunk_tokens < 0) {
    set_error("bad batch, max_pages_per_seq, window or chunk_tokens");
    return -1;
  }
  if (!tc_enabled(*cfg) || chunk_tokens != 0) return 0;
  const int G = cfg->n_heads / cfg->n_kv_heads;
  const int64_t max_tokens = window > 0 ? window : (int64_t)max_pages_per_seq * cfg->page_size;
  TcLaunchCfg lc{};
  int cb = 0, recv = 0;
  const bool on = pick_cluster(*cfg, batch, max_tokens, window, tc_launcher(*cfg), tc_ring_bytes(*cfg, true),
                               tc_pre_bytes(cfg->head_dim, G > 4 ? 2 : 1, tc_ng(*cfg), true), &lc, &cb, &recv);
  return on ? lc.cluster : 0;
}

extern "C" int32_t kvq_decode_launches(const kvq_config* cfg) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  return tc_enabled(*cfg) ? 1 : 2;
}

extern "C" size_t kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t max_pages_per_seq,
                                             int32_t chunk_tokens) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  if (batch < 0 || max_pages_per_seq < 1 || chunk_tokens < 0 || chunk_tokens % cfg->page_size) {
    set_error("bad batch, max_pages_per_seq or chunk_tokens");
    return 0;
  }
  return make_plan(*cfg, batch, (int64_t)max_pages_per_seq * cfg->page_size, false, chunk_tokens).total;
}

extern "C" size_t kvq_window_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t window,
                                             int32_t chunk_tokens) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  if (batch < 0 || window < 1 || chunk_tokens < 0 || chunk_tokens % cfg->page_size) {
    set_error("bad batch, window or chunk_tokens");
    return 0;
  }
  return make_plan(*cfg, batch, window, true, chunk_tokens).total;
}

extern "C" int32_t kvq_append_decode_launches(const kvq_config* cfg) {
  clear_error();
  if (check_kernel_config(cfg) != KVQ_OK) return 0;
  return tc_enabled(*cfg) ? 1 : 3;
}

extern "C" kvq_status kvq_append_decode_attention(const kvq_config* cfg, int32_t batch, const void* q,
                                                  const void* k_new, const void* v_new, const int32_t* pos,
                                                  void* k_pool, void* v_pool, int32_t n_pool_pages,
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
  if (!k_new || !v_new || !pos) return fail(KVQ_ERR_INVALID_ARG, "k_new, v_new and pos must not be NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return fail(KVQ_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  if (!tc_enabled(*cfg)) {
    // The CUDA-core decode has no fused append: the append kernel, then the decode.
    st = kvq_append(cfg, batch, k_new, v_new, nullptr, pos, block_table, batch, max_pages_per_seq, 0, rope_tab,
                    rope_max_pos, k_pool, v_pool, n_pool_pages, dev_status, stream);
    if (st != KVQ_OK) return st;
    return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, block_table, max_pages_per_seq, seq_lens,
                      rope_tab, rope_max_pos, out, workspace, workspace_bytes, chunk_tokens, dev_status,
                      (cudaStream_t)stream, 0, 0, (int64_t)max_pages_per_seq * cfg->page_size);
  }
  return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, block_table, max_pages_per_seq, seq_lens,
                    rope_tab, rope_max_pos, out, workspace, workspace_bytes, chunk_tokens, dev_status,
                    (cudaStream_t)stream, 0, 0, (int64_t)max_pages_per_seq * cfg->page_size, k_new, v_new, pos);
}

extern "C" kvq_status kvq_append_window_decode(const kvq_config* cfg, int32_t batch, const void* q,
                                               const void* k_new, const void* v_new, const int32_t* pos,
                                               void* k_pool, void* v_pool, int32_t n_pool_pages,
                                               const int32_t* ring_table, int32_t ring_rows, int32_t window,
                                               const int32_t* seq_lens, const float* rope_tab,
                                               int32_t rope_max_pos, void* out, void* workspace,
                                               size_t workspace_bytes, int32_t chunk_tokens,
                                               int32_t* dev_status, kvq_stream_t stream) {
  clear_error();
  kvq_status st = check_decode_args(cfg, batch, q, k_pool, v_pool, n_pool_pages, ring_table, seq_lens,
                                    rope_tab, rope_max_pos, out, workspace, chunk_tokens, dev_status);
  if (st != KVQ_OK || batch == 0) return st;
  if (ring_rows < cfg->page_size || ring_rows % cfg->page_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "ring_rows %d must be a positive multiple of page_size", ring_rows);
  if (window < 1 || window > ring_rows)
    return fail(KVQ_ERR_INVALID_ARG, "window %d must be in [1, ring_rows=%d]", window, ring_rows);
  if (!k_new || !v_new || !pos) return fail(KVQ_ERR_INVALID_ARG, "k_new, v_new and pos must not be NULL");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return fail(KVQ_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  const int32_t max_pages = ring_rows / cfg->page_size;
  if (!tc_enabled(*cfg)) {
    // The CUDA-core decode has no fused append: the append kernel, then the decode.
    st = kvq_append(cfg, batch, k_new, v_new, nullptr, pos, ring_table, batch, max_pages, ring_rows, rope_tab,
                    rope_max_pos, k_pool, v_pool, n_pool_pages, dev_status, stream);
    if (st != KVQ_OK) return st;
    return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, ring_table, max_pages, seq_lens, rope_tab,
                      rope_max_pos, out, workspace, workspace_bytes, chunk_tokens, dev_status, (cudaStream_t)stream,
                      ring_rows, window, window);
  }
  return run_decode(cfg, batch, q, k_pool, v_pool, n_pool_pages, ring_table, max_pages, seq_lens, rope_tab,
                    rope_max_pos, out, workspace, workspace_bytes, chunk_tokens, dev_status, (cudaStream_t)stream,
                    ring_rows, window, window, k_new, v_new, pos);
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
