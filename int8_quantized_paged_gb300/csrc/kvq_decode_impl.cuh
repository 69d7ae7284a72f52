// Split-K GQA decode attention over a paged, group-quantized KV cache.
//
// Method: softmax(q K^T * s) V read straight from packed codes through a block
// table ([airllm] §2.2: dequantize inside the kernel after the load, no
// temporary tensor; §2.3: queries span fixed-size blocks; §3.4: fp32 softmax).
// [Shimmy] §2.3 gives the q/k rotation and the 1/sqrt(d) score scale.
// [Fieldfare] "KV Cache 的双布局设计" gives the ring-buffer window.
//
// One CTA (4 warps) owns one (sequence, kv head, chunk of the context).  The
// warps take 16-token blocks of the chunk in turn, and each warp keeps its own
// online-softmax state for the G query heads that share the kv head.  Scores
// run in base 2: q is pre-scaled by alpha*log2(e) and exp2f is used.
//
//  Q.K  : TPT lanes per token, each holding DPT consecutive elements of the
//         G rotated queries in registers.  Codes are turned into exact floats
//         with a mantissa trick, and the G partial dots are scaled per group
//         and summed with a butterfly over the TPT lanes.
//  P.V  : VT lanes per token, each owning DPV output elements of the G heads.
//         A token's weight p*scale multiplies its codes; the affine bias adds
//         p*bias per group.
// The 4 warp states are merged through shared memory, and the chunk's
// (m, l, acc[G][HD]) goes to the workspace for the log-sum-exp combine.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

struct DecodeArgs {
  const void* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* rope_tab;
  // Fused append (tensor-core decode only; NULL otherwise): the new K/V rows
  // [batch][n_kv_heads][HD] of act type and their positions, quantized into
  // the pools (for a ring, into row pos mod ring_rows) before the decode reads
  // them.
  const void* app_k;
  const void* app_v;
  const int32_t* app_pos;
  float* ws_acc;   // [batch][n_kv_heads][n_chunks][G][HD]
  float* ws_ml;    // [batch][n_kv_heads][n_chunks][G][2]
  int32_t* status;
  int32_t batch, n_heads, n_kv_heads, n_pool_pages, max_pages, rope_max_pos;
  int32_t ring_rows;      // 0: append-only
  int32_t window;         // 0: whole context
  int32_t chunk_tokens, n_chunks;
  int32_t act, rope;
  float score_scale;      // alpha * log2(e)
  PoolLayout kl, vl;
};

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

// Length checks shared by the decode and combine kernels.  Returns the number
// of attended tokens, or -1 (with the bit to report) for a bad length.
__device__ __forceinline__ int attended(const DecodeArgs& a, int L, int* lo, int* bad) {
  *bad = 0;
  const int64_t cap = a.ring_rows > 0 ? (int64_t)INT_MAX : (int64_t)a.max_pages * 16;
  if (L < 0 || L > cap) { *bad = KVQ_DEV_BAD_LEN; return -1; }
  if (L > 0 && a.rope != KVQ_ROPE_NONE && L - 1 >= a.rope_max_pos) { *bad = KVQ_DEV_BAD_POS; return -1; }
  *lo = a.window > 0 ? max(0, L - a.window) : 0;
  return L - *lo;
}

template <int KK, int VK, int HD, int G>
__global__ void __launch_bounds__(128) decode_chunk_kernel(const DecodeArgs a) {
  constexpr int P = 16;
  constexpr int NW = 4;
  constexpr int TPT = cmin(cmax(HD * G / 64, 8), 32);   // lanes per token (Q.K)
  constexpr int DPT = HD / TPT;                         // elements per lane (Q.K)
  constexpr int TPW = 32 / TPT;                         // tokens per pass (Q.K)
  constexpr int SUB = cmin(DPT, 16);                    // a run of elements inside one group
  constexpr int NSUB = DPT / SUB;
  constexpr int VT = cmin(cmax(HD * G / 64, 16), 32);   // lanes per token (P.V)
  constexpr int DPV = HD / VT;                          // elements per lane (P.V)
  constexpr int VTW = 32 / VT;                          // tokens per step (P.V)
  constexpr int KNB = DPT * (KK == KVQ_SYM_INT8 ? 8 : 4) / 8;
  constexpr int VNB = DPV * (VK == KVQ_SYM_INT8 ? 8 : 4) / 8;
  constexpr bool KAFF = KK == KVQ_AFFINE_INT4;
  constexpr bool VAFF = VK == KVQ_AFFINE_INT4;

  __shared__ float q_s[G][HD];
  __shared__ float s_s[NW][P][G];
  __shared__ float p_s[NW][P][G];
  __shared__ float wm_s[NW][G];
  __shared__ float wl_s[NW][G];
  __shared__ float acc_s[NW][G][HD];

  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int L = a.seq_lens[b];
  int lo = 0, bad = 0;
  const int n_att = attended(a, L, &lo, &bad);
  if (n_att < 0) {
    if (threadIdx.x == 0 && chunk == 0 && kvh == 0) report(a.status, bad);
    return;
  }
  const int t0 = lo + chunk * a.chunk_tokens;
  if (chunk * a.chunk_tokens >= n_att) return;        // empty chunk: never combined
  const int t1 = min(L, t0 + a.chunk_tokens);

  // Rotate the G queries at position L-1 (fp32) and fold in the score scale.
  {
    const int64_t qbase = ((int64_t)b * a.n_heads + (int64_t)kvh * G) * HD;
    const float2* cs = reinterpret_cast<const float2*>(a.rope_tab) + (int64_t)(L - 1) * (HD / 2);
    for (int i = threadIdx.x; i < G * (HD / 2); i += blockDim.x) {
      const int h = i / (HD / 2), pi = i % (HD / 2);
      const int d0 = a.rope == KVQ_ROPE_NEOX ? pi : 2 * pi;
      const int d1 = a.rope == KVQ_ROPE_NEOX ? pi + HD / 2 : 2 * pi + 1;
      float x0 = load_act(a.q, a.act, qbase + h * HD + d0);
      float x1 = load_act(a.q, a.act, qbase + h * HD + d1);
      if (a.rope != KVQ_ROPE_NONE) {
        const float2 t = cs[pi];
        const float r0 = x0 * t.x - x1 * t.y;
        const float r1 = x0 * t.y + x1 * t.x;
        x0 = r0;
        x1 = r1;
      }
      q_s[h][d0] = x0 * a.score_scale;
      q_s[h][d1] = x1 * a.score_scale;
    }
  }
  __syncthreads();

  const int kpart = lane % TPT;
  const int vpart = lane % VT;
  float qr[G][DPT];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPT; ++j) qr[h][j] = q_s[h][kpart * DPT + j];
  float qsum[G][NSUB];
  if constexpr (KAFF) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int r = 0; r < NSUB; ++r) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < SUB; ++j) s += qr[h][r * SUB + j];
        qsum[h][r] = s;
      }
  }

  const int kpb = param_bytes(a.kl.param), vpb = param_bytes(a.vl.param);
  const uint8_t* kbase = a.k_pool + (int64_t)kvh * a.kl.sub_bytes;
  const uint8_t* vbase = a.v_pool + (int64_t)kvh * a.vl.sub_bytes;
  const int32_t* bt = a.block_table + (int64_t)b * a.max_pages;
  const int vgroup_idx = vpart * DPV / a.vl.group;

  float m[G], l[G], acc[G][DPV], accb[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
    accb[h] = 0.f;
#pragma unroll
    for (int j = 0; j < DPV; ++j) acc[h][j] = 0.f;
  }

  const int n_blk = (t1 - t0 + P - 1) / P;
  for (int blk = warp; blk < n_blk; blk += NW) {
    const int tb = t0 + blk * P;
    // ---- scores
#pragma unroll
    for (int ps = 0; ps < P / TPW; ++ps) {
      const int tt = ps * TPW + lane / TPT;
      const int t = tb + tt;
      bool valid = t < t1;
      float sc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h] = 0.f;
      if (valid) {
        const int row = a.ring_rows > 0 ? t % a.ring_rows : t;
        const int page = bt[row / P];
        const int slot = row % P;
        if (page < 0 || page >= a.n_pool_pages) {
          valid = false;
          if (kpart == 0) report(a.status, KVQ_DEV_BAD_PAGE);
        } else {
          const uint8_t* sub = kbase + (int64_t)page * a.kl.page_bytes;
          uint32_t w[(KNB + 3) / 4];
          load_words<KNB>(sub + slot * a.kl.code_bytes + kpart * KNB, w);
          const uint8_t* prow = sub + P * a.kl.code_bytes + slot * a.kl.param_row_bytes;
#pragma unroll
          for (int r = 0; r < NSUB; ++r) {
            const int g = (kpart * DPT + r * SUB) / a.kl.group;
            const float ks = load_param(prow + g * a.kl.n_params * kpb, a.kl.param);
            float dot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] = 0.f;
#pragma unroll
            for (int j = 0; j < SUB; ++j) {
              const float c = code_at<KK>(w, r * SUB + j);
#pragma unroll
              for (int h = 0; h < G; ++h) dot[h] = fmaf(qr[h][r * SUB + j], c, dot[h]);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) sc[h] = fmaf(ks, dot[h], sc[h]);
            if constexpr (KAFF) {
              const float kb = load_param(prow + (g * 2 + 1) * kpb, a.kl.param);
#pragma unroll
              for (int h = 0; h < G; ++h) sc[h] = fmaf(kb, qsum[h][r], sc[h]);
            }
          }
        }
      }
#pragma unroll
      for (int o = 1; o < TPT; o <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
      if (kpart == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) s_s[warp][tt][h] = valid ? sc[h] : -INFINITY;
      }
    }
    __syncwarp();
    // ---- online softmax over the block's 16 tokens (lanes 16..31 mirror 0..15)
    {
      const int tt = lane & (P - 1);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float s = s_s[warp][tt][h];
        float bm = s;
#pragma unroll
        for (int o = P / 2; o >= 1; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        const float mn = fmaxf(m[h], bm);
        float p = 0.f, corr = 1.f;
        if (mn != -INFINITY) {
          p = exp2f(s - mn);
          corr = exp2f(m[h] - mn);
        }
        float sum = p;
#pragma unroll
        for (int o = P / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        l[h] = l[h] * corr + sum;
        m[h] = mn;
        if (lane < P) p_s[warp][tt][h] = p;
#pragma unroll
        for (int j = 0; j < DPV; ++j) acc[h][j] *= corr;
        accb[h] *= corr;
      }
    }
    __syncwarp();
    // ---- P.V
#pragma unroll 2
    for (int st = 0; st < P / VTW; ++st) {
      const int tt = st * VTW + lane / VT;
      float p[G];
      bool any = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        p[h] = p_s[warp][tt][h];
        any |= p[h] != 0.f;
      }
      if (any) {  // p > 0 only for tokens whose page id was checked above
        const int t = tb + tt;
        const int row = a.ring_rows > 0 ? t % a.ring_rows : t;
        const int page = bt[row / P];
        const int slot = row % P;
        const uint8_t* sub = vbase + (int64_t)page * a.vl.page_bytes;
        uint32_t w[(VNB + 3) / 4];
        load_words<VNB>(sub + slot * a.vl.code_bytes + vpart * VNB, w);
        const uint8_t* prow = sub + P * a.vl.code_bytes + slot * a.vl.param_row_bytes;
        const float vs = load_param(prow + vgroup_idx * a.vl.n_params * vpb, a.vl.param);
        float vb = 0.f;
        if constexpr (VAFF) vb = load_param(prow + (vgroup_idx * 2 + 1) * vpb, a.vl.param);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float wgt = p[h] * vs;
#pragma unroll
          for (int j = 0; j < DPV; ++j) acc[h][j] = fmaf(wgt, code_at<VK>(w, j), acc[h][j]);
          if constexpr (VAFF) accb[h] = fmaf(p[h], vb, accb[h]);
        }
      }
    }
    __syncwarp();
  }

  // Merge the lanes that handled different tokens in P.V.
  if constexpr (VTW == 2) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int j = 0; j < DPV; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], 16);
      accb[h] += __shfl_xor_sync(0xffffffffu, accb[h], 16);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wm_s[warp][h] = m[h];
      wl_s[warp][h] = l[h];
    }
  }
  if (lane < VT) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < DPV; ++j) acc_s[warp][h][vpart * DPV + j] = acc[h][j] + (VAFF ? accb[h] : 0.f);
  }
  __syncthreads();

  // Merge the 4 warps and write the chunk's partial state.
  const int64_t cidx = ((int64_t)b * a.n_kv_heads + kvh) * a.n_chunks + chunk;
  for (int i = threadIdx.x; i < G * HD; i += blockDim.x) {
    const int h = i / HD, d = i % HD;
    float M = wm_s[0][h];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, wm_s[w][h]);
    float o = 0.f, ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(wm_s[w][h] - M);
        o = fmaf(f, acc_s[w][h][d], o);
        ls = fmaf(f, wl_s[w][h], ls);
      }
    }
    a.ws_acc[(cidx * G + h) * HD + d] = o;
    if (d == 0) {
      a.ws_ml[(cidx * G + h) * 2] = M;
      a.ws_ml[(cidx * G + h) * 2 + 1] = ls;
    }
  }
}

template <int KK, int VK>
kvq_status launch_decode_kinds(const DecodeArgs& a, int head_dim, int G, dim3 grid, cudaStream_t s) {
#define KVQ_LAUNCH(HD_, G_)                                                   \
  if (head_dim == HD_ && G == G_) {                                           \
    decode_chunk_kernel<KK, VK, HD_, G_><<<grid, 128, 0, s>>>(a);             \
    return KVQ_OK;                                                            \
  }
  KVQ_LAUNCH(64, 1) KVQ_LAUNCH(64, 2) KVQ_LAUNCH(64, 4) KVQ_LAUNCH(64, 8)
  KVQ_LAUNCH(128, 1) KVQ_LAUNCH(128, 2) KVQ_LAUNCH(128, 4) KVQ_LAUNCH(128, 8)
  KVQ_LAUNCH(256, 1) KVQ_LAUNCH(256, 2) KVQ_LAUNCH(256, 4) KVQ_LAUNCH(256, 8)
#undef KVQ_LAUNCH
  return fail(KVQ_ERR_UNSUPPORTED, "no decode kernel for head_dim %d, G %d", head_dim, G);
}

// Launchers, one translation unit per K/V kind pair.
kvq_status launch_decode_s4s4(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s);
kvq_status launch_decode_s8s8(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s);
kvq_status launch_decode_s8s4(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s);
kvq_status launch_decode_a4a4(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s);

}  // namespace kvq
