// Internal declarations shared by the host runtime and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/kvq.h"

#if defined(__CUDACC__)
#define KVQ_HD __host__ __device__
#else
#define KVQ_HD
#endif

namespace kvq {

// Thread-local error text behind kvq_last_error().
void set_error(const char* fmt, ...);
void clear_error();
kvq_status fail(kvq_status st, const char* fmt, ...);

// Stored parameter type (same numbering as kvq_float).
KVQ_HD inline int param_bytes(int f) { return f == KVQ_F32 ? 4 : 2; }
KVQ_HD inline bool is_quant_kind(int k) {
  return k == KVQ_SYM_INT4 || k == KVQ_SYM_INT8 || k == KVQ_AFFINE_INT4 || k == KVQ_SHIMMY_INT4;
}

// Byte layout of one pool (see the storage format in kvq.h).
struct PoolLayout {
  int32_t kind;             // kvq_kv_dtype (quantized kinds only)
  int32_t group;            // elements per scale group
  int32_t param;            // kvq_float of scale (and bias)
  int32_t n_groups;         // head_dim / group
  int32_t n_params;         // 1 (symmetric) or 2 (affine)
  int32_t code_bytes;       // per token per kv head
  int32_t param_row_bytes;  // per token per kv head
  int32_t sub_bytes;        // per (page, kv head)
  int64_t page_bytes;       // per page, all kv heads
};

PoolLayout pool_layout(const kvq_config& c, int which);

// Validates a config for the quantized kernels (not just sizing).
kvq_status check_kernel_config(const kvq_config* c);

// Score scale used in the kernels: alpha * log2(e) (softmax runs in base 2).
float score_scale_log2(const kvq_config& c);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();
size_t smem_per_sm();   // shared memory of one SM of the current device (bytes)

// Whether kernels are launched with programmatic dependent launch (set
// KVQ_PDL=0 in the environment to turn it off).
bool pdl_enabled();

// Number of chunks a sequence of up to max_tokens attended tokens is split into.
int chunk_tokens_for(const kvq_config& c, int32_t batch, int64_t max_tokens,
                     int32_t requested);

}  // namespace kvq
