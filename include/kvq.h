/*
 * kvq -- quantized, paged KV-cache decode attention for one GB300 (sm_103a).
 *
 * C ABI of libkvq.so.  Plain pointers and sizes only.  Every device buffer
 * (pools, block tables, q, out, workspace, status word) is allocated and owned
 * by the caller.  The library never calls a device allocator.  Its only device
 * memory of its own is the fixed scratch array behind
 * kvq_decode_attention_noalloc.  The host-side page pool and block-table
 * objects are the only allocations it makes, and they live in host memory.
 *
 * The method restated here comes from four web pages:
 *   [Shimmy]    "Shimmy 深度解剖：Airframe 引擎与 TurboShimmy INT4 KV"
 *   [Fieldfare] the TurboFieldfare post ("KV Cache 的双布局设计", "量化和精度")
 *   [airllm]    the airllm light-weight inference post (§2.1-§2.3, §4.2, §5.4)
 *   [Kaiwu]     "我做了个工具让 8GB 显卡跑 30B 模型从 3 tok/s 提到 21 tok/s"
 *
 * Calls that take a stream are asynchronous.  The host checks the arguments and
 * returns an error at once when one is bad; nothing is enqueued in that case.
 * A launch failure returns KVQ_ERR_CUDA.  A device-side problem, such as a
 * block-table entry outside the pool, sets a bit in the caller's 32-bit status
 * word.  The kernel then skips that piece of work, and kvq_get_device_status()
 * reports the bit.  No kernel traps, asserts, or waits without a bound.  The
 * text of the last host-side error is kept per thread in kvq_last_error().
 *
 * ---------------------------------------------------------------------------
 * Storage format of one pool (K and V have separate pools that share the same
 * block table)
 *
 *   pool      = n_pool_pages pages, in page-id order
 *   page      = n_kv_heads sub-blocks, in kv-head order
 *   sub-block = codes [page_size][code_bytes], then params [page_size][param_row]
 *   code_bytes: head_dim/2 for 4-bit kinds, head_dim for 8-bit
 *   4-bit     : byte j holds element 2j in the low nibble and 2j+1 in the high
 *               nibble ([airllm] §4.2 packing); symmetric codes are
 *               two's-complement nibbles in [-7, 7], affine codes unsigned [0, 15]
 *   8-bit     : one int8 per element, in [-127, 127]
 *   param_row : for each group g = 0 .. head_dim/group-1, in order:
 *               symmetric: scale_g ; affine: scale_g, bias_g
 *               each a little-endian f32, f16 or bf16 (kvq_config.*_param_dtype)
 *
 * Every sub-block size is a multiple of 16 bytes.  Token t of a sequence (row r
 * = t, or t mod ring_rows for a ring) lives in page block_table[seq][r /
 * page_size], slot r % page_size ([airllm] §2.3: fixed-size blocks from a free
 * pool, an offset index inside each block).
 *
 * Codec.  All of it is IEEE fp32 with one rounding per operation and no
 * fused multiply-add.  Rounding is to nearest, ties to even, except where a
 * kind says otherwise.  The resulting codes are bit-exact across
 * implementations.
 *   symmetric ([airllm] §4.2 group_quantize; [Shimmy] §3.2):
 *     s  = stored(max(amax / Qmax, floor)),  Qmax = 7 (4-bit) or 127 (8-bit),
 *     floor = 2^-14 for f16 scales, else 1e-8;  code = clamp(rne(x / s), +-Qmax)
 *   affine ([Fieldfare] "量化和精度": 4-bit, group 64, bf16 scale + bias):
 *     s = stored((max - min) / 15),  b = stored(min),
 *     code = s == 0 ? 0 : clamp(rne((x - b) / s), 0, 15);   x^ = s*code + b
 *   offset-8 4-bit ([Shimmy] §3.2 quantize_head_vector; KVQ_SHIMMY_INT4):
 *     s = stored(amax / 7.5),  code = s == 0 ? 0 : clamp(round(x / s), -8, 7)
 *     with round half away from zero, nibble = code + 8;  x^ = (nibble - 8)*s
 *   f16 ([Kaiwu] finding 2, "f16+f16"; KVQ_F16_KV): each element rounded
 *     once to fp16, no scale.
 *   K is rotated (RoPE, fp32) at its own position before it is quantized; V
 *   is not ([Fieldfare] "KV Cache 的双布局设计").
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 1: the first release.  2: kvq_config.flags (formerly a reserved field
 * that had to be 0) accepts KVQ_FLAG_EARLY_READS; a caller that sets it can
 * check kvq_abi_version() >= 2 first, as a version-1 library refuses any
 * nonzero value with KVQ_ERR_INVALID_ARG.  The layout of every struct is
 * unchanged. */
#define KVQ_ABI_VERSION 2

/* A cudaStream_t.  NULL means the legacy default stream. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,        /* a null pointer, bad size or bad enum value */
  KVQ_ERR_UNSUPPORTED = 2,        /* a valid shape or dtype this build has no kernel for */
  KVQ_ERR_OUT_OF_PAGES = 3,       /* the page pool cannot satisfy an allocation */
  KVQ_ERR_BAD_BLOCK_TABLE = 4,    /* the device flagged a page id, position or length */
  KVQ_ERR_WORKSPACE_TOO_SMALL = 5,
  KVQ_ERR_CUDA = 6                /* a CUDA runtime call or kernel launch failed */
} kvq_status;

/* Bits a kernel ORs into the caller's device status word. */
#define KVQ_DEV_BAD_PAGE 1        /* a block-table entry outside [0, n_pool_pages) */
#define KVQ_DEV_BAD_POS 2         /* a position past the block table or the RoPE table */
#define KVQ_DEV_BAD_SEQ 4         /* a sequence id outside [0, n_seqs) */
#define KVQ_DEV_BAD_LEN 8         /* a seq_len < 0 or past the block table's capacity */

typedef enum kvq_float { KVQ_F32 = 0, KVQ_F16 = 1, KVQ_BF16 = 2 } kvq_float;

typedef enum kvq_kv_dtype {
  KVQ_SYM_INT4 = 0,       /* [airllm] §4.2, [Shimmy] §3.2: symmetric 4-bit */
  KVQ_SYM_INT8 = 1,       /* [Kaiwu] finding 2 "q8_0" K cache: symmetric 8-bit */
  KVQ_AFFINE_INT4 = 2,    /* [Fieldfare] "量化和精度": 4-bit with scale + bias */
  KVQ_F16_KV = 3,         /* unquantized f16 ([Kaiwu] "f16+f16"): fp16 rows, no scale;
                             decode with head_dim 64 or 128 */
  KVQ_F32_KV = 4,         /* unquantized f32 ([Shimmy] §3.1); sizing only */
  KVQ_SHIMMY_INT4 = 5     /* [Shimmy] §3.2 as written: scale = max|x| / 7.5,
                             code = clamp(round(x / scale), -8, 7) rounding half away
                             from zero, stored as code + 8; f32 scales */
} kvq_kv_dtype;

typedef enum kvq_rope {
  KVQ_ROPE_NONE = 0,
  KVQ_ROPE_NORMAL = 1,    /* pairs (2i, 2i+1) */
  KVQ_ROPE_NEOX = 2       /* pairs (i, i + head_dim/2) ([Fieldfare] "量化和精度") */
} kvq_rope;

/* One attention layer's cache description.  The fields follow the pages'
 * problem statement ([Shimmy] §2.2 ModelSpec: n_heads, n_kv_heads, head_dim,
 * rope_freq_base; [airllm] §2.1 group size; [Kaiwu] KV cache types). */
typedef struct kvq_config {
  int32_t n_heads;        /* query heads Hq */
  int32_t n_kv_heads;     /* K/V heads Hkv; Hq % Hkv == 0 and G = Hq/Hkv in {1,2,4,8} */
  int32_t head_dim;       /* 64, 128 or 256 */
  int32_t page_size;      /* tokens per page; 16 */
  int32_t k_dtype;        /* kvq_kv_dtype of the K pool */
  int32_t v_dtype;        /* kvq_kv_dtype of the V pool */
  int32_t k_group;        /* K elements per scale group: divides head_dim, multiple of 16 */
  int32_t v_group;        /* same for V */
  int32_t k_param_dtype;  /* kvq_float of K's stored scale (and bias) */
  int32_t v_param_dtype;  /* same for V */
  int32_t act_dtype;      /* kvq_float of q, k_new, v_new and out */
  int32_t rope;           /* kvq_rope */
  float attn_scale;       /* > 0: the score scale; <= 0: 1/sqrt(head_dim) */
  int32_t flags;          /* 0, or KVQ_FLAG_EARLY_READS; other bits are INVALID_ARG */
  double rope_base;       /* theta_i = rope_base^(-2i/head_dim) */
} kvq_config;

/* kvq_config.flags.
 *
 * KVQ_FLAG_EARLY_READS: a decode call (kvq_decode_attention, its no-alloc and
 * window forms, and the two fused append + decode calls) may read seq_lens,
 * pos, the block table, the RoPE table and the pool pages before the kernel
 * launched just before it on the same stream has finished.  The library
 * launches its kernels with programmatic dependent launch, so a call can start
 * while that kernel still runs; with the flag it streams its first pages in
 * that time.  q, k_new and v_new are read only after that kernel has
 * finished, and the output, the workspace and the new rows are written only
 * after it; a bad input found earlier is flagged in dev_status, an atomic OR.
 * The flag is a permission: a call may also read everything after the wait.
 *
 * Set it only when the kernel launched just before each call writes none of
 * the inputs read early.  That holds in a multi-layer decode loop, where the
 * kernel before a layer's call is the previous layer's call (other pools) or
 * the projection that makes q, k_new and v_new.  It does not hold for
 * back-to-back calls on the same pools, such as a single-layer model's
 * consecutive steps, or a kvq_decode_attention right after the kvq_append that
 * wrote its new row.  A copy (cudaMemcpyAsync) is not a kernel: the call
 * starts after it completes.  Only the kernel immediately before can overlap:
 * a call triggers the launch of the next one only after its own wait. */
#define KVQ_FLAG_EARLY_READS 1

/* ABI version of the loaded library (KVQ_ABI_VERSION). */
int32_t kvq_abi_version(void);

/* Text of the last error raised on this thread ("" if none).  The pointer is
 * valid until this thread's next kvq call. */
const char* kvq_last_error(void);

/* KVQ_OK when this build has kernels for cfg, else the reason
 * (INVALID_ARG / UNSUPPORTED) and a message. */
kvq_status kvq_validate_config(const kvq_config* cfg);

/* Kernel launches one kvq_decode_attention / kvq_window_decode call makes for
 * cfg: 1 on the tensor-core path (split-K decode with the log-sum-exp combine
 * fused in), 2 on the CUDA-core path (decode, then a combine kernel); 0 for an
 * invalid config.  Not part of the method; it lets a caller count launches. */
int32_t kvq_decode_launches(const kvq_config* cfg);

/* CTAs per thread-block cluster that a decode call with these arguments uses
 * on the current device: >= 1 when the chunks of every (sequence, kv head)
 * form one cluster and combine in distributed shared memory (few sequences of
 * up to 16K tokens, chunk_tokens 0), 0 when the partials go through the
 * workspace instead, -1 for invalid arguments.  window is 0 for
 * kvq_decode_attention and the window of kvq_window_decode otherwise.  Not
 * part of the method; it lets a caller see which combine runs.  Needs a
 * current CUDA device for an answer other than -1 or 0. */
int32_t kvq_decode_cluster_ctas(const kvq_config* cfg, int32_t batch, int32_t max_pages_per_seq,
                                int32_t window, int32_t chunk_tokens);

/* ---------------------------------------------------------------- sizing --
 * Bytes of the K and V caches for n_layers layers holding ctx tokens each, with
 * ctx rounded up to whole pages.  This is the closed form 2 x layers x kv_heads
 * x ctx x bytes_per_element of [Kaiwu] finding 2 (KV_MB, with kv_heads and not
 * heads, per its "GQA 架构识别" note).  It is generalised to
 * code bytes plus the scale and bias bytes of each group ([Shimmy] §3.2: 0.5 B
 * per INT4 element plus one 4-byte scale per head vector).  K and V are added
 * separately when their dtypes differ.  The f16/f32 kinds are accepted here
 * only.  Returns 0 on an invalid config, n_layers < 0 or ctx < 0. */
size_t kvq_cache_bytes(const kvq_config* cfg, int32_t n_layers, int64_t ctx);

/* Bytes of one page of the K pool (which == 0) or V pool (which == 1), all kv
 * heads.  Returns 0 on an invalid config or which. */
size_t kvq_page_bytes(const kvq_config* cfg, int32_t which);

/* ------------------------------------------------------- host page pool --
 * A LIFO free list of page ids over one pool of n_pages pages ([airllm] §2.3:
 * a free-block pool that grows caches one block at a time and that several
 * requests share).  A fresh pool hands out 0, 1, 2, ... in order.  A freed page
 * is handed out first.  Host memory only.  A pool is not thread-safe. */
typedef struct kvq_pool kvq_pool;

kvq_status kvq_pool_create(int32_t n_pages, kvq_pool** out);   /* n_pages >= 1 */
void kvq_pool_destroy(kvq_pool* pool);                          /* NULL is a no-op */
/* Take n pages (all or nothing): OUT_OF_PAGES if fewer are free. */
kvq_status kvq_pool_alloc(kvq_pool* pool, int32_t n, int32_t* ids_out);
/* Return n pages.  An id that is outside the pool, already free or repeated in
 * ids is INVALID_ARG, and then nothing is freed. */
kvq_status kvq_pool_free(kvq_pool* pool, int32_t n, const int32_t* ids);
int32_t kvq_pool_num_free(const kvq_pool* pool);                /* -1 for NULL */
int32_t kvq_pool_num_pages(const kvq_pool* pool);               /* -1 for NULL */

/* ---------------------------------------------------------- block tables --
 * Per-sequence page lists over a pool, mirrored as a dense host int32 matrix
 * [n_seqs][max_pages_per_seq] (unused entries -1).  Each sequence owns its
 * pages ([airllm] §5.4: sequences must not share cache rows, and a finished
 * sequence's rows must be freed).  The caller copies kvq_table_data() to the
 * device when it changes.  The table does not own the pool, and the pool must
 * outlive it. */
typedef struct kvq_table kvq_table;

kvq_status kvq_table_create(kvq_pool* pool, int32_t n_seqs, int32_t max_pages_per_seq,
                            int32_t page_size, kvq_table** out);
/* Frees every page the table still holds back to the pool.  NULL is a no-op. */
void kvq_table_destroy(kvq_table* table);
/* Grow sequence seq so that rows [0, n_rows) have pages, allocating whole pages
 * from the pool (a no-op if it already has them).  A ring of R rows reserves R
 * once.  OUT_OF_PAGES leaves the sequence unchanged; INVALID_ARG if n_rows
 * needs more than max_pages_per_seq pages. */
kvq_status kvq_table_reserve(kvq_table* table, int32_t seq, int64_t n_rows);
/* Return all of seq's pages to the pool (the sequence finished). */
kvq_status kvq_table_release(kvq_table* table, int32_t seq);
const int32_t* kvq_table_data(const kvq_table* table);          /* NULL for NULL */
int32_t kvq_table_num_pages(const kvq_table* table, int32_t seq); /* -1 if invalid */

/* ------------------------------------------------------------------ RoPE --
 * Host table of (cos, sin) of pos * theta_i for pos in [0, max_pos), i in
 * [0, head_dim/2): host_out is float[max_pos][head_dim/2][2].  theta_i =
 * rope_base^(-2i/head_dim).  pow, cos and sin are taken in double and each is
 * rounded once to float ([Shimmy] §2.2 rope_freq_base; §2.3 rotation of q and
 * k).  The kernels take a device copy of this table. */
kvq_status kvq_rope_table(const kvq_config* cfg, int32_t max_pos, float* host_out);

/* --------------------------------------------------- quantize-on-append --
 * Quantize n_rows new K and V rows and write them into their pages
 * ([airllm] §4.2 group quantization; §2.3 paged pool; [Fieldfare] "KV Cache
 * 的双布局设计": ring rows overwritten in place, K rotated and V not).
 *   k_new, v_new  device [n_rows][n_kv_heads][head_dim] of act_dtype
 *   seq_ids       device int32 [n_rows]: block-table row of each new row, or
 *                 NULL (row i belongs to sequence i)
 *   pos           device int32 [n_rows]: absolute token position (>= 0)
 *   block_table   device int32 [n_seqs][max_pages_per_seq]
 *   ring_rows     0: append-only (row = pos).  > 0: ring of ring_rows rows
 *                 (row = pos mod ring_rows); a multiple of page_size
 *   rope_tab      device float[rope_max_pos][head_dim/2][2] (kvq_rope_table);
 *                 may be NULL when cfg->rope == KVQ_ROPE_NONE
 *   k_pool, v_pool device pools of n_pool_pages pages (kvq_page_bytes each)
 *   dev_status    device int32 the kernels OR KVQ_DEV_* bits into
 * Rows that share one (page, slot) within a call race.  The caller must not
 * pass two rows for the same position of one sequence.  A row with a bad
 * sequence, position or page sets its bit and is skipped. */
kvq_status kvq_append(const kvq_config* cfg, int32_t n_rows,
                      const void* k_new, const void* v_new,
                      const int32_t* seq_ids, const int32_t* pos,
                      const int32_t* block_table, int32_t n_seqs,
                      int32_t max_pages_per_seq, int32_t ring_rows,
                      const float* rope_tab, int32_t rope_max_pos,
                      void* k_pool, void* v_pool, int32_t n_pool_pages,
                      int32_t* dev_status, kvq_stream_t stream);

/* ------------------------------------------------------- decode attention --
 * One decode step of GQA attention for a batch of sequences, read straight
 * from the packed codes through the block table ([airllm] §2.2: dequantize
 * inside the kernel, in registers; §2.3: a query may span blocks).  For every
 * sequence b (L = seq_lens[b]) and query head h, with kv head h / G:
 *   q~  = RoPE(q[b][h]) at position L-1
 *   s_t = alpha * <q~, K^_t>  for t in [0, L)
 *   out[b][h] = sum_t softmax(s)_t V^_t      (L = 0 gives zeros)
 * The context is split into chunks of chunk_tokens tokens.  Each chunk keeps an
 * fp32 online softmax (m, l, acc), and the last chunk of each (sequence, kv
 * head) to finish merges the chunks with log-sum-exp weights.  fp32 softmax:
 * [airllm] §3.4.
 *   q, out        device [batch][n_heads][head_dim] of act_dtype; q 16-byte
 *                 aligned (KVQ_ERR_INVALID_ARG otherwise)
 *   rope_tab      as for kvq_append, 16-byte aligned (KVQ_ERR_INVALID_ARG
 *                 otherwise); unused when cfg->rope is KVQ_ROPE_NONE
 *   seq_lens      device int32 [batch], 0 <= L <= max_pages_per_seq*page_size
 *   chunk_tokens  0: the library chooses; else a multiple of page_size
 *   workspace     device scratch of at least kvq_decode_workspace_bytes()
 *                 with the same batch, max_pages_per_seq and chunk_tokens;
 *                 256-byte aligned.  Zero it once before its first use: its
 *                 first bytes are per-(sequence, kv head) arrival counters,
 *                 and every completed call leaves them zero again.  Zero it
 *                 again before using it for a larger batch.
 * A sequence whose length is bad sets KVQ_DEV_BAD_LEN and gets a zero row.  A
 * bad page id sets KVQ_DEV_BAD_PAGE and its tokens are left out. */
size_t kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t batch,
                                  int32_t max_pages_per_seq, int32_t chunk_tokens);
kvq_status kvq_decode_attention(const kvq_config* cfg, int32_t batch, const void* q,
                                const void* k_pool, const void* v_pool, int32_t n_pool_pages,
                                const int32_t* block_table, int32_t max_pages_per_seq,
                                const int32_t* seq_lens,
                                const float* rope_tab, int32_t rope_max_pos,
                                void* out, void* workspace, size_t workspace_bytes,
                                int32_t chunk_tokens, int32_t* dev_status, kvq_stream_t stream);

/* -------------------------------------------------- sliding-window decode --
 * Decode attention over the last `window` tokens of each sequence, kept in a
 * ring of ring_rows rows ([Fieldfare] "KV Cache 的双布局设计": 1152 rows for a
 * 1024-token window; the extra 128 rows are the chunked-prefill write buffer,
 * and rows that left the window are overwritten with no explicit eviction).
 * Keys t in [max(0, L-window), L) are read from row t mod ring_rows.
 *   ring_table    device int32 [batch][ring_rows/page_size]
 *   window        1 <= window <= ring_rows; ring_rows a multiple of page_size
 *   workspace     at least kvq_window_workspace_bytes(cfg, batch, window, chunk_tokens)
 * All other arguments as in kvq_decode_attention. */
size_t kvq_window_workspace_bytes(const kvq_config* cfg, int32_t batch, int32_t window,
                                  int32_t chunk_tokens);
kvq_status kvq_window_decode(const kvq_config* cfg, int32_t batch, const void* q,
                             const void* k_pool, const void* v_pool, int32_t n_pool_pages,
                             const int32_t* ring_table, int32_t ring_rows, int32_t window,
                             const int32_t* seq_lens,
                             const float* rope_tab, int32_t rope_max_pos,
                             void* out, void* workspace, size_t workspace_bytes,
                             int32_t chunk_tokens, int32_t* dev_status, kvq_stream_t stream);

/* ------------------------------------------ fused append + decode step --
 * One decode step of every sequence in one call: kvq_append of the step's new
 * row of each sequence b (k_new[b], v_new[b] at position pos[b]: K rotated,
 * both quantized into their page) followed by kvq_decode_attention with
 * seq_lens, the caller's usual pos[b] = seq_lens[b] - 1 making the new row the
 * last key.  The pool bytes written and the output are those of the two calls
 * made one after the other.  On the tensor-core path it is one launch: the
 * CTA that reads the new row's page quantizes the row (the append kernel's
 * arithmetic), writes it to the pool and uses it straight from shared memory;
 * elsewhere it is the append kernel and then the decode.
 *   k_new, v_new  device [batch][n_kv_heads][head_dim] of act_dtype, 16-byte
 *                 aligned (KVQ_ERR_INVALID_ARG otherwise)
 *   pos           device int32 [batch]; row b goes to sequence b.  A bad
 *                 position sets KVQ_DEV_BAD_POS, a bad page id KVQ_DEV_BAD_PAGE,
 *                 and that row is not written
 *   k_pool, v_pool  written (the new rows) and read
 * All other arguments as in kvq_decode_attention (the same workspace size).
 * Its launches per call: kvq_append_decode_launches(cfg). */
kvq_status kvq_append_decode_attention(const kvq_config* cfg, int32_t batch, const void* q,
                                       const void* k_new, const void* v_new, const int32_t* pos,
                                       void* k_pool, void* v_pool, int32_t n_pool_pages,
                                       const int32_t* block_table, int32_t max_pages_per_seq,
                                       const int32_t* seq_lens,
                                       const float* rope_tab, int32_t rope_max_pos,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       int32_t chunk_tokens, int32_t* dev_status, kvq_stream_t stream);
/* Kernel launches of one kvq_append_decode_attention (or
 * kvq_append_window_decode) call for cfg: 1 on the tensor-core path, 3 on the
 * CUDA-core path; 0 for an invalid config. */
int32_t kvq_append_decode_launches(const kvq_config* cfg);

/* The same fused step for a sliding-window layer: kvq_append of row b at
 * pos[b] into ring row pos[b] mod ring_rows, then kvq_window_decode.  With
 * window <= ring_rows no attended key shares the new row's ring row.
 * Arguments as in kvq_window_decode plus k_new, v_new and pos as in
 * kvq_append_decode_attention. */
kvq_status kvq_append_window_decode(const kvq_config* cfg, int32_t batch, const void* q,
                                    const void* k_new, const void* v_new, const int32_t* pos,
                                    void* k_pool, void* v_pool, int32_t n_pool_pages,
                                    const int32_t* ring_table, int32_t ring_rows, int32_t window,
                                    const int32_t* seq_lens,
                                    const float* rope_tab, int32_t rope_max_pos,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    int32_t chunk_tokens, int32_t* dev_status, kvq_stream_t stream);

/* ------------------------------------------- decode without allocation --
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot allocate device memory, such as a plugin whose host engine owns
 * all of HBM through its own pool, or a hot path where an allocation and the
 * synchronization it may cause are not allowed.
 * It computes exactly what kvq_decode_attention computes, with the same
 * arguments minus the workspace.  The split-K workspace is a fixed
 * KVQ_NOALLOC_SCRATCH_BYTES array compiled into the library.  Every GPU that
 * loads the library holds that array until the process exits.  A decode whose
 * workspace (kvq_decode_workspace_bytes) is larger returns
 * KVQ_ERR_WORKSPACE_TOO_SMALL and launches nothing.  The first call in a CUDA
 * context of a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and the address is kept
 * for that context.  A device reset gives the device a new context, where the
 * array may sit elsewhere, so the next call looks it up again.  Make the first
 * call in each context before any stream capture.  All calls share
 * the one array: calls whose kernels overlap on the GPU (for example on two
 * streams at once) race.  The library neither allocates nor frees memory here.
 * The array starts zeroed when the library loads, and every completed call
 * leaves its arrival counters zero again, so nothing needs clearing. */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)   /* 8 MiB */
kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, int32_t batch, const void* q,
                                        const void* k_pool, const void* v_pool, int32_t n_pool_pages,
                                        const int32_t* block_table, int32_t max_pages_per_seq,
                                        const int32_t* seq_lens,
                                        const float* rope_tab, int32_t rope_max_pos,
                                        void* out, int32_t chunk_tokens, int32_t* dev_status,
                                        kvq_stream_t stream);

/* ---------------------------------------------------------- device status --
 * Clear the status word (an async memset on stream). */
kvq_status kvq_clear_device_status(int32_t* dev_status, kvq_stream_t stream);
/* Synchronize stream, read the status word into *bits_out (may be NULL) and
 * return KVQ_ERR_BAD_BLOCK_TABLE if any bit is set, else KVQ_OK. */
kvq_status kvq_get_device_status(const int32_t* dev_status, kvq_stream_t stream,
                                 int32_t* bits_out);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
