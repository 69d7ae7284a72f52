// Host runtime of libkvq: errors, config checks, cache sizing, the page pool,
// block tables, the RoPE table and the device status word.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "kvq_internal.h"

namespace kvq {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

void clear_error() { g_err[0] = '\0'; }

kvq_status fail(kvq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

static bool valid_float(int32_t f) { return f == KVQ_F32 || f == KVQ_F16 || f == KVQ_BF16; }

// Checks shared by sizing and kernels.  Sizing accepts the unquantized kinds.
static kvq_status check_common(const kvq_config* c) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "config is NULL");
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "n_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                c->n_heads, c->n_kv_heads);
  if (c->head_dim < 2 || c->head_dim % 2 != 0)
    return fail(KVQ_ERR_INVALID_ARG, "head_dim (%d) must be a positive even number", c->head_dim);
  if (c->page_size < 1) return fail(KVQ_ERR_INVALID_ARG, "page_size (%d) must be >= 1", c->page_size);
  if (c->flags & ~KVQ_FLAG_EARLY_READS) return fail(KVQ_ERR_INVALID_ARG, "unknown flags 0x%x", c->flags);
  const int32_t kinds[2] = {c->k_dtype, c->v_dtype};
  const int32_t groups[2] = {c->k_group, c->v_group};
  const int32_t params[2] = {c->k_param_dtype, c->v_param_dtype};
  for (int i = 0; i < 2; ++i) {
    const char* kv = i ? "v" : "k";
    if (kinds[i] < KVQ_SYM_INT4 || kinds[i] > KVQ_SHIMMY_INT4)
      return fail(KVQ_ERR_INVALID_ARG, "%s_dtype %d is not a kvq_kv_dtype", kv, kinds[i]);
    if (!is_quant_kind(kinds[i])) continue;
    if (groups[i] < 2 || c->head_dim % groups[i] != 0 || groups[i] % 2 != 0)
      return fail(KVQ_ERR_INVALID_ARG, "%s_group %d must be even and divide head_dim %d", kv,
                  groups[i], c->head_dim);
    if (!valid_float(params[i]))
      return fail(KVQ_ERR_INVALID_ARG, "%s_param_dtype %d is not a kvq_float", kv, params[i]);
  }
  if (!valid_float(c->act_dtype)) return fail(KVQ_ERR_INVALID_ARG, "act_dtype %d invalid", c->act_dtype);
  if (c->rope < KVQ_ROPE_NONE || c->rope > KVQ_ROPE_NEOX)
    return fail(KVQ_ERR_INVALID_ARG, "rope %d invalid", c->rope);
  if (c->rope != KVQ_ROPE_NONE && !(c->rope_base > 0.0 && std::isfinite(c->rope_base)))
    return fail(KVQ_ERR_INVALID_ARG, "rope_base must be a positive finite number");
  if (!std::isfinite(c->attn_scale)) return fail(KVQ_ERR_INVALID_ARG, "attn_scale must be finite");
  return KVQ_OK;
}

kvq_status check_kernel_config(const kvq_config* c) {
  kvq_status st = check_common(c);
  if (st != KVQ_OK) return st;
  const int G = c->n_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(KVQ_ERR_UNSUPPORTED, "n_heads/n_kv_heads = %d; kernels exist for 1, 2, 4, 8", G);
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
    return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d; kernels exist for 64, 128, 256", c->head_dim);
  if (c->page_size != 16)
    return fail(KVQ_ERR_UNSUPPORTED, "page_size %d; kernels exist for 16", c->page_size);
  const int k = c->k_dtype, v = c->v_dtype;
  const bool pair_ok = (k == KVQ_SYM_INT4 && v == KVQ_SYM_INT4) ||
                       (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT8) ||
                       (k == KVQ_SYM_INT8 && v == KVQ_SYM_INT4) ||
                       (k == KVQ_AFFINE_INT4 && v == KVQ_AFFINE_INT4) ||
                       (k == KVQ_F16_KV && v == KVQ_F16_KV) ||
                       (k == KVQ_SHIMMY_INT4 && v == KVQ_SHIMMY_INT4);
  if (!pair_ok)
    return fail(KVQ_ERR_UNSUPPORTED,
                "K/V dtype pair (%d, %d); kernels exist for sym4/sym4, sym8/sym8, sym8/sym4, "
                "affine4/affine4, f16/f16, shimmy4/shimmy4", k, v);
  if (k == KVQ_SHIMMY_INT4) {   // the tensor-core kernel only: f32 scales, groups of 2^n >= 32
    if (c->k_param_dtype != KVQ_F32 || c->v_param_dtype != KVQ_F32 || c->k_group != c->v_group ||
        c->k_group < 32 || (c->k_group & (c->k_group - 1)) != 0)
      return fail(KVQ_ERR_UNSUPPORTED, "shimmy4 K/V: kernels exist for f32 scales and equal power-of-two groups >= 32");
  }
  if (k == KVQ_F16_KV) {   // unquantised: no groups; the tensor-core kernel only
    if (c->head_dim == 256)
      return fail(KVQ_ERR_UNSUPPORTED, "f16 K/V: kernels exist for head_dim 64 and 128");
    return KVQ_OK;
  }
  if (c->k_group % 16 != 0 || c->v_group % 16 != 0)
    return fail(KVQ_ERR_UNSUPPORTED, "groups (%d, %d) must be multiples of 16", c->k_group,
                c->v_group);
  return KVQ_OK;
}

PoolLayout pool_layout(const kvq_config& c, int which) {
  PoolLayout L{};
  L.kind = which ? c.v_dtype : c.k_dtype;
  L.group = which ? c.v_group : c.k_group;
  L.param = which ? c.v_param_dtype : c.k_param_dtype;
  if (L.kind == KVQ_F16_KV) {   // unquantised: fp16 rows, no parameters
    L.group = c.head_dim;
    L.n_groups = 1;
    L.n_params = 0;
    L.code_bytes = 2 * c.head_dim;
  } else {
    L.n_groups = c.head_dim / L.group;
    L.n_params = L.kind == KVQ_AFFINE_INT4 ? 2 : 1;
    L.code_bytes = L.kind == KVQ_SYM_INT8 ? c.head_dim : c.head_dim / 2;
  }
  L.param_row_bytes = L.n_groups * L.n_params * param_bytes(L.param);
  L.sub_bytes = c.page_size * (L.code_bytes + L.param_row_bytes);
  L.page_bytes = (int64_t)c.n_kv_heads * L.sub_bytes;
  return L;
}

float score_scale_log2(const kvq_config& c) {
  const double alpha = c.attn_scale > 0.f ? (double)c.attn_scale : 1.0 / std::sqrt((double)c.head_dim);
  return (float)(alpha * 1.4426950408889634);  // log2(e)
}

size_t smem_per_sm() {
  static size_t cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 228 * 1024;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || n <= 0)
      n = 228 * 1024;
    cache[dev] = (size_t)n;
  }
  return cache[dev];
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = std::getenv("KVQ_PDL");
    on = (e && std::strcmp(e, "0") == 0) ? 0 : 1;
  }
  return on != 0;
}

int chunk_tokens_for(const kvq_config& c, int32_t batch, int64_t max_tokens, int32_t requested) {
  if (requested > 0) return requested;
  const int64_t pairs = (int64_t)batch * c.n_kv_heads;
  const int64_t target = 4LL * num_sms();
  int64_t per_seq = (target + pairs - 1) / pairs;
  if (per_seq < 1) per_seq = 1;
  int64_t tc = (max_tokens + per_seq - 1) / per_seq;
  tc = (tc + 63) / 64 * 64;
  if (tc < 64) tc = 64;
  if (tc > (1 << 20)) tc = 1 << 20;
  return (int)tc;
}

}  // namespace kvq

using namespace kvq;

// ------------------------------------------------------------------ misc

extern "C" int32_t kvq_abi_version(void) { return KVQ_ABI_VERSION; }

extern "C" const char* kvq_last_error(void) { return g_err; }

extern "C" kvq_status kvq_validate_config(const kvq_config* cfg) {
  clear_error();
  return check_kernel_config(cfg);
}

// ---------------------------------------------------------------- sizing

static int64_t bytes_per_token_head(int kind, int hd, int group, int param) {
  if (kind == KVQ_F16_KV) return 2LL * hd;
  if (kind == KVQ_F32_KV) return 4LL * hd;
  const int64_t code = kind == KVQ_SYM_INT8 ? hd : hd / 2;
  const int64_t n_params = kind == KVQ_AFFINE_INT4 ? 2 : 1;
  return code + (int64_t)(hd / group) * n_params * param_bytes(param);
}

extern "C" size_t kvq_cache_bytes(const kvq_config* cfg, int32_t n_layers, int64_t ctx) {
  clear_error();
  if (check_common(cfg) != KVQ_OK) return 0;
  if (n_layers < 0 || ctx < 0) {
    set_error("n_layers and ctx must be >= 0");
    return 0;
  }
  const int64_t P = cfg->page_size;
  const int64_t ctx_pad = (ctx + P - 1) / P * P;
  const int64_t per = bytes_per_token_head(cfg->k_dtype, cfg->head_dim, cfg->k_group, cfg->k_param_dtype) +
                      bytes_per_token_head(cfg->v_dtype, cfg->head_dim, cfg->v_group, cfg->v_param_dtype);
  return (size_t)((int64_t)n_layers * cfg->n_kv_heads * ctx_pad * per);
}

extern "C" size_t kvq_page_bytes(const kvq_config* cfg, int32_t which) {
  clear_error();
  if (check_common(cfg) != KVQ_OK) return 0;
  if (which != 0 && which != 1) {
    set_error("which must be 0 (K) or 1 (V)");
    return 0;
  }
  const int kind = which ? cfg->v_dtype : cfg->k_dtype;
  if (!is_quant_kind(kind)) {
    return (size_t)cfg->n_kv_heads * cfg->page_size * bytes_per_token_head(kind, cfg->head_dim, 0, 0);
  }
  return (size_t)pool_layout(*cfg, which).page_bytes;
}

// ------------------------------------------------------------- page pool

struct kvq_pool {
  std::vector<int32_t> stack;  // free ids; back() is handed out next
  std::vector<uint8_t> is_free;
};

extern "C" kvq_status kvq_pool_create(int32_t n_pages, kvq_pool** out) {
  clear_error();
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n_pages < 1) return fail(KVQ_ERR_INVALID_ARG, "n_pages (%d) must be >= 1", n_pages);
  kvq_pool* p = new (std::nothrow) kvq_pool;
  if (!p) return fail(KVQ_ERR_OUT_OF_PAGES, "host allocation failed");
  p->stack.resize(n_pages);
  for (int32_t i = 0; i < n_pages; ++i) p->stack[i] = n_pages - 1 - i;
  p->is_free.assign(n_pages, 1);
  *out = p;
  return KVQ_OK;
}

extern "C" void kvq_pool_destroy(kvq_pool* pool) { delete pool; }

extern "C" kvq_status kvq_pool_alloc(kvq_pool* pool, int32_t n, int32_t* ids_out) {
  clear_error();
  if (!pool) return fail(KVQ_ERR_INVALID_ARG, "pool is NULL");
  if (n < 0 || (n > 0 && !ids_out)) return fail(KVQ_ERR_INVALID_ARG, "bad n or ids_out");
  if ((size_t)n > pool->stack.size())
    return fail(KVQ_ERR_OUT_OF_PAGES, "asked for %d pages, %zu free", n, pool->stack.size());
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = pool->stack.back();
    pool->stack.pop_back();
    pool->is_free[id] = 0;
    ids_out[i] = id;
  }
  return KVQ_OK;
}

extern "C" kvq_status kvq_pool_free(kvq_pool* pool, int32_t n, const int32_t* ids) {
  clear_error();
  if (!pool) return fail(KVQ_ERR_INVALID_ARG, "pool is NULL");
  if (n < 0 || (n > 0 && !ids)) return fail(KVQ_ERR_INVALID_ARG, "bad n or ids");
  const int32_t n_pages = (int32_t)pool->is_free.size();
  std::vector<uint8_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= n_pages) return fail(KVQ_ERR_INVALID_ARG, "page id %d is not in the pool", id);
    if (pool->is_free[id]) return fail(KVQ_ERR_INVALID_ARG, "page id %d is already free", id);
    if (seen.empty()) seen.assign(n_pages, 0);
    if (seen[id]) return fail(KVQ_ERR_INVALID_ARG, "page id %d is repeated", id);
    seen[id] = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    pool->is_free[ids[i]] = 1;
    pool->stack.push_back(ids[i]);
  }
  return KVQ_OK;
}

extern "C" int32_t kvq_pool_num_free(const kvq_pool* pool) {
  return pool ? (int32_t)pool->stack.size() : -1;
}

extern "C" int32_t kvq_pool_num_pages(const kvq_pool* pool) {
  return pool ? (int32_t)pool->is_free.size() : -1;
}

// ----------------------------------------------------------- block tables

struct kvq_table {
  kvq_pool* pool;
  int32_t n_seqs, max_pages, page_size;
  std::vector<int32_t> data;    // [n_seqs][max_pages]
  std::vector<int32_t> count;   // pages held per sequence
};

extern "C" kvq_status kvq_table_create(kvq_pool* pool, int32_t n_seqs, int32_t max_pages_per_seq,
                                       int32_t page_size, kvq_table** out) {
  clear_error();
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!pool || n_seqs < 1 || max_pages_per_seq < 1 || page_size < 1)
    return fail(KVQ_ERR_INVALID_ARG, "bad pool, n_seqs, max_pages_per_seq or page_size");
  kvq_table* t = new (std::nothrow) kvq_table;
  if (!t) return fail(KVQ_ERR_OUT_OF_PAGES, "host allocation failed");
  t->pool = pool;
  t->n_seqs = n_seqs;
  t->max_pages = max_pages_per_seq;
  t->page_size = page_size;
  t->data.assign((size_t)n_seqs * max_pages_per_seq, -1);
  t->count.assign(n_seqs, 0);
  *out = t;
  return KVQ_OK;
}

extern "C" kvq_status kvq_table_release(kvq_table* t, int32_t seq) {
  clear_error();
  if (!t || seq < 0 || seq >= t->n_seqs) return fail(KVQ_ERR_INVALID_ARG, "bad table or seq");
  int32_t* row = t->data.data() + (size_t)seq * t->max_pages;
  kvq_status st = kvq_pool_free(t->pool, t->count[seq], row);
  if (st != KVQ_OK) return st;
  for (int32_t i = 0; i < t->count[seq]; ++i) row[i] = -1;
  t->count[seq] = 0;
  return KVQ_OK;
}

extern "C" void kvq_table_destroy(kvq_table* t) {
  if (!t) return;
  for (int32_t s = 0; s < t->n_seqs; ++s) kvq_table_release(t, s);
  delete t;
}

extern "C" kvq_status kvq_table_reserve(kvq_table* t, int32_t seq, int64_t n_rows) {
  clear_error();
  if (!t || seq < 0 || seq >= t->n_seqs || n_rows < 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad table, seq or n_rows");
  const int64_t need = (n_rows + t->page_size - 1) / t->page_size;
  if (need > t->max_pages)
    return fail(KVQ_ERR_INVALID_ARG, "%lld rows need %lld pages; the table holds %d per sequence",
                (long long)n_rows, (long long)need, t->max_pages);
  const int32_t have = t->count[seq];
  if (need <= have) return KVQ_OK;
  int32_t* row = t->data.data() + (size_t)seq * t->max_pages;
  kvq_status st = kvq_pool_alloc(t->pool, (int32_t)(need - have), row + have);
  if (st != KVQ_OK) return st;
  t->count[seq] = (int32_t)need;
  return KVQ_OK;
}

extern "C" const int32_t* kvq_table_data(const kvq_table* t) { return t ? t->data.data() : nullptr; }

extern "C" int32_t kvq_table_num_pages(const kvq_table* t, int32_t seq) {
  if (!t || seq < 0 || seq >= t->n_seqs) return -1;
  return t->count[seq];
}

// ------------------------------------------------------------------ RoPE

extern "C" kvq_status kvq_rope_table(const kvq_config* cfg, int32_t max_pos, float* host_out) {
  clear_error();
  kvq_status st = check_common(cfg);
  if (st != KVQ_OK) return st;
  if (max_pos < 0 || (max_pos > 0 && !host_out)) return fail(KVQ_ERR_INVALID_ARG, "bad max_pos or host_out");
  if (cfg->rope == KVQ_ROPE_NONE) return fail(KVQ_ERR_INVALID_ARG, "config has no RoPE");
  const int hd = cfg->head_dim, half = hd / 2;
  std::vector<double> theta(half);
  for (int i = 0; i < half; ++i) theta[i] = std::pow(cfg->rope_base, -2.0 * i / hd);
  for (int64_t p = 0; p < max_pos; ++p) {
    float* row = host_out + p * (int64_t)half * 2;
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * theta[i];
      row[2 * i] = (float)std::cos(ang);
      row[2 * i + 1] = (float)std::sin(ang);
    }
  }
  return KVQ_OK;
}

// --------------------------------------------------------- device status

extern "C" kvq_status kvq_clear_device_status(int32_t* dev_status, kvq_stream_t stream) {
  clear_error();
  if (!dev_status) return fail(KVQ_ERR_INVALID_ARG, "dev_status is NULL");
  cudaError_t e = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

extern "C" kvq_status kvq_get_device_status(const int32_t* dev_status, kvq_stream_t stream,
                                            int32_t* bits_out) {
  clear_error();
  if (!dev_status) return fail(KVQ_ERR_INVALID_ARG, "dev_status is NULL");
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (bits_out) *bits_out = h;
  if (h != 0) return fail(KVQ_ERR_BAD_BLOCK_TABLE, "device status bits 0x%x", h);
  return KVQ_OK;
}
