// Tensor-core split-K GQA decode attention over a paged, group-quantized KV
// cache, with the log-sum-exp combine fused into the last CTA of each
// (sequence, kv head).
//
// Method: softmax(q K^T * s) V straight from the packed codes through a block
// table ([airllm] §2.2: dequantize inside the kernel after the load, with no
// temporary tensor; §2.3: queries span fixed-size blocks; §3.4: fp32
// softmax).
//
// Why tensor cores here: each code takes part in G multiply-adds for q.K
// and G for p.V.  Done on the fp32 CUDA cores, that arithmetic plus the
// dequantization issues more instructions per byte than the SMs can retire
// at HBM speed.  So the codes go to mma.sync as exact fp16 integers, straight
// from registers.  The packed nibbles are turned into fp16 fragments with a
// mantissa trick and are never written back to shared memory.
//
// Data movement: each warp (a warp pair for hd = 256) owns a ring of D page
// slots in shared memory and takes every fourth (second) page of the chunk.
// Its lane 0 issues the copies of a page and refills the slot as soon as the
// warp is done with it, so D pages per warp stay in flight and no warp waits
// for another.  Code rows use a 3-D TMA tiled copy with hardware swizzle, so
// ldmatrix reads are free of bank conflicts.  Scales use a 1-D bulk copy.
// Each slot completes on an mbarrier, and every wait has a time limit.
//
// Per warp and 16-token page (the G <= 8 query heads share one kv head):
//   Q.K : S[16 x 16] = Qhl[16 x hd] * Khat^T.  Row g < G holds the fp16 high
//         part of query head g (rotated, pre-scaled), row 8+g the low part
//         (q = hi + lo * 2^-12), so the dot products keep about fp32 precision.
//         Codes are exact in fp16.  Each scale group accumulates separately,
//         and its scale (and affine bias * sum q) is applied in fp32 afterwards.
//   softmax: online, base 2, in registers (4 scores per lane).  The running
//         maximum is raised only when a page exceeds it by 2^8, so the
//         accumulators are rescaled on few pages, and p <= 2^8.
//   P.V : O[16 x hd] += W[16 x 16] * Vhat.  Rows g and 8+g hold hi and lo of
//         w = p * scale * 2^7 / R (w = hi + lo * 2^-12), where R is the running
//         maximum V scale of the group, so w stays inside fp16's range.
// Warps own different pages and merge through shared memory at the end.
// hd = 256 splits each page's dimensions over a pair of warps.  The pair
// exchanges partial scores through shared memory under a 64-thread named
// barrier.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "kvq_decode_impl.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tc_ptx.cuh"

namespace kvq {

struct TcArgs {
  DecodeArgs d;
  void* out;
  int32_t* counters;         // [batch][n_kv_heads] arrival tickets (zero between calls)
  int32_t G;                 // query heads per kv head (1..8)
  int32_t blocks_per_chunk;  // 16-token blocks per chunk
  int32_t kc_bytes, vc_bytes, kp_bytes, vp_bytes;  // per page in shared memory
  int32_t depth;                                   // ring slots (pages in flight) per warp group
  int32_t ring_bytes;                              // shared memory of one group's ring
  int32_t k_group_shift, v_group_shift;            // log2 of the group sizes
};

constexpr int kMaxDepth = 8;
constexpr int kTcThreads = 128;
constexpr int kMaxChunkBlocks = 256;
constexpr float kQScale = 256.0f;   // q is held x 2^8 in fp16 (hi/lo)
constexpr float kWScale = 128.0f;   // w is held x 2^7 (w <= 2^8 * 2^7 < 65504)
constexpr float kLazyMax = 8.0f;    // raise the running max only past +2^8

// Shared-memory offset of 16-byte chunk `c` of row `r` in a TMA box of rows of
// ROWB bytes (32/64/128) written with the matching swizzle.
template <int ROWB>
__device__ __forceinline__ int swz(int r, int c) {
  constexpr int SH = ROWB == 128 ? 0 : (ROWB == 64 ? 1 : 2);
  constexpr int MASK = ROWB / 16 - 1;
  return r * ROWB + ((c ^ ((r >> SH) & MASK)) << 4);
}

// Element of the head dimension held by lane (tig) in Q.K k-step `ks`,
// fragment half f (0: k = 2tig, 2tig+1; 1: k = 2tig+8, 2tig+9), element e.
template <int KK>
__device__ __forceinline__ int qk_dim(int ks, int f, int e, int tig) {
  if constexpr (KK == KVQ_SYM_INT8) {  // k-step = one 16-byte chunk = 16 elements
    return 16 * ks + 4 * tig + f + 2 * e;
  } else {  // two k-steps per 16-byte chunk of 32 nibbles
    return 32 * (ks >> 1) + 8 * tig + 2 * (ks & 1) + f + 4 * e;
  }
}

// Element of the head dimension of P.V n-tile j (0..3) of unit v, column n.
template <int VK>
__device__ __forceinline__ int pv_dim(int v, int j, int n) {
  if constexpr (VK == KVQ_SYM_INT8) {
    return 32 * v + 16 * (j >> 1) + 2 * n + (j & 1);
  } else {
    return 32 * v + 4 * n + j;
  }
}

// A stored scale or bias of type PT (kvq_float) read from shared memory.
template <int PT>
__device__ __forceinline__ float ld_param(const uint8_t* p) {
  if constexpr (PT == KVQ_F32) {
    return *reinterpret_cast<const float*>(p);
  } else if constexpr (PT == KVQ_F16) {
    return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(p)));
  } else {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(p)) << 16);
  }
}

// ONEG: one K scale group and one V scale group cover all of a warp's
// dimensions, so each token has one K and one V scale per warp.
// PT: the stored type of the scales (and biases) of both K and V.
template <int KK, int VK, int HD, bool ONEG, int PT>
__global__ void __launch_bounds__(kTcThreads, 3)
decode_tc_kernel(const __grid_constant__ TcArgs A, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int P = 16;
  constexpr int DS = HD == 256 ? 2 : 1;          // warps per page (dimension split)
  constexpr int HDW = HD / DS;                   // dimensions per warp
  constexpr int NU = HDW / 32;                   // 32-element units per warp
  constexpr int KRB = KK == KVQ_SYM_INT8 ? HD : HD / 2;   // K code row bytes
  constexpr int VRB = VK == KVQ_SYM_INT8 ? HD : HD / 2;
  constexpr int KCH = KRB / 16 / DS;             // K 16-byte chunks per warp
  constexpr int VCH = VRB / 16 / DS;
  constexpr int KS = KK == KVQ_SYM_INT8 ? KCH : 2 * KCH;  // Q.K k-steps per warp
  constexpr int NSA = ONEG ? 1 : NU;             // score accumulators per n-tile
  constexpr bool KAFF = KK == KVQ_AFFINE_INT4;
  constexpr bool VAFF = VK == KVQ_AFFINE_INT4;
  constexpr int PB = PT == KVQ_F32 ? 4 : 2;      // bytes of a stored scale
  static_assert(NU >= 2 && KCH % 2 == 0, "units");

  const DecodeArgs& a = A.d;
  const int G = A.G;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[4][kMaxDepth];   // a ring slot landed (TMA bytes)
  __shared__ int32_t page_s[kMaxChunkBlocks];
  __shared__ float q_s[8 * HD];                  // rotated, scaled queries
  __shared__ float xs_s[2][2][P][8];             // hd = 256: partial scores of a warp pair
  __shared__ int32_t flag_s;

  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;

  tc::grid_dependency_wait();   // inputs may come from the kernel before this one

  // Page ids of the chunk's blocks (-1: not readable).  With the whole
  // context attended, a chunk's blocks do not depend on the length, so the
  // block-table entries are read together with seq_lens (one round trip).
  const int32_t* bt = a.block_table + (int64_t)b * a.max_pages;
  const int CB = A.blocks_per_chunk;
  const int ring = a.ring_rows, npp = a.n_pool_pages;
  const bool whole = a.window == 0 && ring == 0;
  int pg_pre[2] = {-1, -1};
  if (whole) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = tid + k * kTcThreads;
      const int blk = chunk * CB + j;
      if (j < CB && blk < a.max_pages) pg_pre[k] = bt[blk];
    }
  }
  const int L = a.seq_lens[b];
  int lo = 0, bad = 0;
  const int n_att = attended(a, L, &lo, &bad);
  const int64_t obase = ((int64_t)b * a.n_heads + (int64_t)kvh * G) * HD;
  if (n_att <= 0) {
    if (chunk == 0) {
      if (bad && tid == 0 && kvh == 0) report(a.status, bad);
      for (int i = tid; i < G * HD; i += kTcThreads) store_act(A.out, a.act, obase + i, 0.f);
    }
    return;
  }
  const int blk_lo = lo / P, blk_hi = (L + P - 1) / P;
  const int nch = (blk_hi - blk_lo + CB - 1) / CB;
  if (chunk >= nch) return;
  const int cb0 = blk_lo + chunk * CB;
  const int ncb = min(CB, blk_hi - cb0);

  // 1024-aligned start of the dynamic region (TMA swizzle atoms), kept as an
  // offset from the shared array so accesses stay in the shared space.
  const int align = (1024 - (int)(tc::smem_u32(smem_raw) & 1023)) & 1023;
  uint8_t* smem = smem_raw + align;
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = tc::smem_u32(&full_bar[0][0]);
  if (tid == 0) {
    for (int s = 0; s < 4 * kMaxDepth; ++s) tc::mbar_init(bar0 + 8 * s, 1);
    tc::fence_barrier_init();
    tc::prefetch_tensormap(&tmap_k);
    tc::prefetch_tensormap(&tmap_v);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int j = tid + k * kTcThreads;
    if (j >= ncb) continue;
    int pg;
    if (whole) {
      pg = pg_pre[k];
    } else {
      const int blk = cb0 + j;
      const int row = ring > 0 ? (int)(((int64_t)blk * P) % ring) : blk * P;
      pg = bt[row / P];
    }
    const bool ok = pg >= 0 && pg < npp;
    if (!ok) report(a.status, KVQ_DEV_BAD_PAGE);
    page_s[j] = ok ? pg : -1;
  }
  __syncthreads();

  // ---- page rings: group g (a warp, or a warp pair for hd = 256) takes the
  // chunk's pages g, g + NGRP, ...; its lane 0 keeps `depth` of them in flight.
  constexpr int NGRP = 4 / DS;
  const int depth = A.depth;
  const int kc_bytes = A.kc_bytes, vc_bytes = A.vc_bytes, kp_bytes = A.kp_bytes, vp_bytes = A.vp_bytes;
  const int grp = warp / DS;
  const int n_local = grp < ncb ? (ncb - grp + NGRP - 1) / NGRP : 0;
  const uint32_t rbase = sbase + grp * A.ring_bytes;       // [depth kc][depth vc][depth kp][depth vp]
  const uint32_t gbar = bar0 + 8 * kMaxDepth * grp;
  const bool producer = lane == 0 && (warp % DS) == 0;
  const int64_t kpage = a.kl.page_bytes, vpage = a.vl.page_bytes;
  const uint8_t* kbase = a.k_pool + (int64_t)kvh * a.kl.sub_bytes + P * a.kl.code_bytes;   // params of page 0
  const uint8_t* vbase = a.v_pool + (int64_t)kvh * a.vl.sub_bytes + P * a.vl.code_bytes;
  const int n_kv = a.n_kv_heads;
  const uint32_t page_tx = (uint32_t)(kc_bytes + vc_bytes + kp_bytes + vp_bytes);

  // Copy local page i of this group into slot i % depth.  The fence orders
  // this group's earlier shared-memory reads of the slot before the copy.
  auto issue = [&](int i) {
    const int slot = i % depth;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bar = gbar + 8 * slot;
    const int pg = page_s[grp + i * NGRP];
    if (pg < 0) {                       // unreadable page: complete the phase with no bytes
      tc::mbar_arrive_expect_tx(bar, 0);
      return;
    }
    tc::mbar_arrive_expect_tx(bar, page_tx);
    const int z = pg * n_kv + kvh;
    tc::tma_load_3d(rbase + slot * kc_bytes, &tmap_k, 0, 0, z, bar);
    tc::tma_load_3d(rbase + depth * kc_bytes + slot * vc_bytes, &tmap_v, 0, 0, z, bar);
    tc::bulk_load(rbase + depth * (kc_bytes + vc_bytes) + slot * kp_bytes, kbase + pg * kpage,
                  (uint32_t)kp_bytes, bar);
    tc::bulk_load(rbase + depth * (kc_bytes + vc_bytes + kp_bytes) + slot * vp_bytes, vbase + pg * vpage,
                  (uint32_t)vp_bytes, bar);
  };
  if (producer) {
    for (int i = 0; i < min(n_local, depth); ++i) issue(i);
  }

  // rotated queries at position L-1, scaled by alpha * log2(e) * 2^8 (while
  // the first stages are in flight)
  {
    const float2* cs = reinterpret_cast<const float2*>(a.rope_tab) + (int64_t)(L - 1) * (HD / 2);
    const float sc = a.score_scale * kQScale;
    const int rope = a.rope, act = a.act;
    const bool neox = rope == KVQ_ROPE_NEOX;
    for (int i = tid; i < G * (HD / 2); i += kTcThreads) {
      const int h = i / (HD / 2), pi = i - h * (HD / 2);
      const int d0 = neox ? pi : 2 * pi;
      const int d1 = neox ? pi + HD / 2 : 2 * pi + 1;
      float x0 = load_act(a.q, act, obase + h * HD + d0);
      float x1 = load_act(a.q, act, obase + h * HD + d1);
      if (rope != KVQ_ROPE_NONE) {
        const float2 t = cs[pi];
        const float r0 = x0 * t.x - x1 * t.y;
        const float r1 = x0 * t.y + x1 * t.x;
        x0 = r0;
        x1 = r1;
      }
      q_s[h * HD + d0] = x0 * sc;
      q_s[h * HD + d1] = x1 * sc;
    }
  }
  __syncthreads();

  // ---- this lane's query fragments (fp16 hi/lo) and per-unit query sums.
  // 4-bit K: the codes in fragment half f = 1 come as 16 * code, so the
  // query elements they meet are divided by 16 here.
  const int half = DS == 2 ? (warp & 1) : 0;     // which half of the dims this warp owns
  const int dim0 = half * HDW;
  const bool live = gid < G;
  uint32_t qa[KS][4];
  float qsum[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) qsum[u] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    float hv[2][2], lv[2][2];
#pragma unroll
    for (int f = 0; f < 2; ++f)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float x = live ? q_s[gid * HD + dim0 + qk_dim<KK>(ks, f, e, tig)] : 0.f;
        qsum[ks >> 1] += x;
        const float xs = (KK != KVQ_SYM_INT8 && f == 1) ? x * (1.0f / 16.0f) : x;
        tc::split_half(xs, hv[f][e], lv[f][e]);
      }
    qa[ks][0] = tc::pack_half2(hv[0][0], hv[0][1]);   // row gid     : hi, k = 2tig, 2tig+1
    qa[ks][1] = tc::pack_half2(lv[0][0], lv[0][1]);   // row gid + 8 : lo
    qa[ks][2] = tc::pack_half2(hv[1][0], hv[1][1]);   // row gid     : hi, k = 2tig+8, 2tig+9
    qa[ks][3] = tc::pack_half2(lv[1][0], lv[1][1]);   // row gid + 8 : lo
  }
  if constexpr (KAFF) {
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      qsum[u] += __shfl_xor_sync(0xffffffffu, qsum[u], 1);
      qsum[u] += __shfl_xor_sync(0xffffffffu, qsum[u], 2);
      qsum[u] *= 1.0f / kQScale;
    }
  }

  // ---- per-lane constants of the main loop
  const int kprb = a.kl.param_row_bytes, vprb = a.vl.param_row_bytes;
  const int kstep = a.kl.n_params * PB, vstep = a.vl.n_params * PB;   // bytes per group in a param row
  const int mi = lane >> 3;
  const int trow = 8 * (mi & 1) + (lane & 7);    // token row this lane addresses in ldmatrix
  const int tok0 = 2 * tig;                      // the lane's tokens: tok0, tok0+1, tok0+8, tok0+9
  int gk[NU], gv[NU];                            // scale-group index of each unit
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    gk[u] = (dim0 + 32 * u) >> A.k_group_shift;
    gv[u] = (dim0 + 32 * u) >> A.v_group_shift;
  }
  int kpo[4], vpo[4];                            // param-row offsets of the lane's tokens
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = tok0 + (i & 1) + 8 * (i >> 1);
    kpo[i] = t * kprb + (ONEG ? gk[0] * kstep : 0);
    vpo[i] = t * vprb + (ONEG ? gv[0] * vstep : 0);
  }
  const int pair = warp >> 1;
  // ldmatrix lane offsets within a page's code rows (chunk pair c, c+1)
  int kls[KCH / 2], vls[(VK == KVQ_SYM_INT8 ? VCH : VCH) / 2];
#pragma unroll
  for (int c = 0; c < KCH; c += 2) kls[c / 2] = swz<KRB>(trow, half * KCH + c + (mi >> 1));
#pragma unroll
  for (int c = 0; c < VCH; c += 2) vls[c / 2] = swz<VRB>(trow, half * VCH + c + (mi >> 1));
  // ---- per-warp running state
  float m = -INFINITY, l = 0.f;
  float oacc[NU][4][4];
  float pb[NU];       // affine V: sum of p * bias per unit
  float vref[NU];     // reference V scale of each unit's group (w = p * scale * 2^7 / vref)
  float vinv[NU];     // 2^7 / vref (0 before the first page)
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    pb[u] = 0.f;
    vref[u] = 0.f;
    vinv[u] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[u][j][e] = 0.f;
  }
  bool timed_out = false;

  for (int i = 0; i < n_local; ++i) {
    const int slot = i % depth;
    if (!tc::mbar_wait(gbar + 8 * slot, (uint32_t)((i / depth) & 1))) timed_out = true;
    const int blk = grp + i * NGRP;
    {
      const bool have = page_s[blk] >= 0;
      const uint32_t kc = rbase + slot * kc_bytes;
      const uint32_t vc = rbase + depth * kc_bytes + slot * vc_bytes;
      const uint8_t* kp = smem + grp * A.ring_bytes + depth * (kc_bytes + vc_bytes) + slot * kp_bytes;
      const uint8_t* vp = smem + grp * A.ring_bytes + depth * (kc_bytes + vc_bytes + kp_bytes) + slot * vp_bytes;
      const int tb = (cb0 + blk) * P;           // absolute token index of the page's slot 0

      float s[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (have) {
        // ---- Q.K on tensor cores
        float sacc[NSA][2][4];
#pragma unroll
        for (int u = 0; u < NSA; ++u)
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[u][n][e] = 0.f;
#pragma unroll
        for (int c = 0; c < KCH; c += 2) {
          uint32_t r[4];   // (tokens 0-7, chunk c), (8-15, c), (0-7, c+1), (8-15, c+1)
          tc::ldsm_x4(kc + kls[c / 2], r);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = c + cc;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
              if constexpr (KK == KVQ_SYM_INT8) {
                uint32_t h[2];
                tc::q8_codes(r[2 * cc + n], h);
                tc::mma_16816(sacc[ONEG ? 0 : (ch >> 1)][n], qa[ch], h[0], h[1]);
              } else {
                uint32_t h[4];
                tc::q4_codes<KAFF>(r[2 * cc + n], h);
                tc::mma_16816(sacc[ONEG ? 0 : ch][n], qa[2 * ch], h[0], h[1]);
                tc::mma_16816(sacc[ONEG ? 0 : ch][n], qa[2 * ch + 1], h[2], h[3]);
              }
            }
          }
        }
        // ---- scores of the lane's 4 tokens for head gid
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = i >> 1, e = i & 1;
          if constexpr (ONEG) {
            const float ks = ld_param<PT>(kp + kpo[i]) * (1.0f / kQScale);
            float v = ks * fmaf(sacc[0][n][e + 2], 1.0f / tc::kLoScale, sacc[0][n][e]);
            if constexpr (KAFF) {
              float qs = 0.f;
#pragma unroll
              for (int u = 0; u < NU; ++u) qs += qsum[u];
              v = fmaf(ld_param<PT>(kp + kpo[i] + PB), qs, v);
            }
            s[i] = v;
          } else {
            float acc = 0.f, part = 0.f, qs = 0.f;
#pragma unroll
            for (int u = 0; u < NU; ++u) {
              part += fmaf(sacc[u][n][e + 2], 1.0f / tc::kLoScale, sacc[u][n][e]);
              if constexpr (KAFF) qs += qsum[u];
              if (u == NU - 1 || gk[u + 1] != gk[u]) {   // end of a group's units
                const uint8_t* pg = kp + kpo[i] + gk[u] * kstep;
                acc = fmaf(ld_param<PT>(pg) * (1.0f / kQScale), part, acc);
                if constexpr (KAFF) acc = fmaf(ld_param<PT>(pg + PB), qs, acc);
                part = 0.f;
                qs = 0.f;
              }
            }
            s[i] = acc;
          }
        }
      }
      if constexpr (DS == 2) {   // add the partner warp's half of each dot product
#pragma unroll
        for (int i = 0; i < 4; ++i) xs_s[pair][half][tok0 + (i & 1) + 8 * (i >> 1)][gid] = s[i];
        asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += xs_s[pair][half ^ 1][tok0 + (i & 1) + 8 * (i >> 1)][gid];
        asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
      }
      if (tb < lo || tb + P > L) {   // a page at the window start or the context end
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = tb + tok0 + (i & 1) + 8 * (i >> 1);
          if (t < lo || t >= L) s[i] = -INFINITY;
        }
      }
      // ---- online softmax (base 2), running max raised lazily
      float bm = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      if (bm > m + kLazyMax) {
        if (m != -INFINITY) {
          const float corr = tc::ex2(m - bm);
          l *= corr;
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            pb[u] *= corr;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) oacc[u][j][e] *= corr;
          }
        }
        m = bm;
      }
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = tc::ex2(s[i] - m);   // 0 for masked tokens (s = -inf)
      if (m == -INFINITY) p[0] = p[1] = p[2] = p[3] = 0.f;
      float ps = (p[0] + p[1]) + (p[2] + p[3]);
      ps += __shfl_xor_sync(0xffffffffu, ps, 1);
      ps += __shfl_xor_sync(0xffffffffu, ps, 2);
      l += ps;
      // ---- P.V on tensor cores (one weight fragment per V group)
      if (have && __any_sync(0xffffffffu, ps > 0.f)) {
        uint32_t wa[4] = {0u, 0u, 0u, 0u};
        uint32_t r[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          if (u == 0 || (!ONEG && gv[u] != gv[u - 1])) {   // weights of this V group
            float sc[4], vb4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint8_t* pg = vp + vpo[i] + (ONEG ? 0 : gv[u] * vstep);
              sc[i] = ld_param<PT>(pg);
              vb4[i] = VAFF ? ld_param<PT>(pg + PB) : 0.f;
            }
            float smax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
            if (smax > vref[u]) {   // raise the group's reference (2x headroom), rescale its sums
              const float nref = 2.0f * smax;
              if (vref[u] > 0.f) {
                const float ratio = vref[u] / nref;
#pragma unroll
                for (int uu = 0; uu < NU; ++uu) {
                  if (gv[uu] != gv[u]) continue;
#pragma unroll
                  for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) oacc[uu][j][e] *= ratio;
                }
              }
              const float ninv = kWScale / nref;
#pragma unroll
              for (int uu = 0; uu < NU; ++uu)
                if (gv[uu] == gv[u]) {
                  vref[uu] = nref;
                  vinv[uu] = ninv;
                }
            }
            const float inv = vinv[u];
            float wh[4], wl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tc::split_half(p[i] * (sc[i] * inv), wh[i], wl[i]);
            wa[0] = tc::pack_half2(wh[0], wh[1]);   // row gid     : hi, tokens tok0, tok0+1
            wa[1] = tc::pack_half2(wl[0], wl[1]);   // row gid + 8 : lo
            wa[2] = tc::pack_half2(wh[2], wh[3]);   // row gid     : hi, tokens tok0+8, tok0+9
            wa[3] = tc::pack_half2(wl[2], wl[3]);   // row gid + 8 : lo
            if constexpr (VAFF) {
              const float add = (p[0] * vb4[0] + p[1] * vb4[1]) + (p[2] * vb4[2] + p[3] * vb4[3]);
#pragma unroll
              for (int uu = 0; uu < NU; ++uu)
                if (gv[uu] == gv[u]) pb[uu] += add;
            }
          }
          if constexpr (VK == KVQ_SYM_INT8) {   // unit = two 16-byte chunks
            tc::ldsm_x4_trans(vc + vls[u], r);
#pragma unroll
            for (int kap = 0; kap < 2; ++kap) {
              uint32_t ha[2], hb[2];
              tc::q8_codes(r[2 * kap], ha);
              tc::q8_codes(r[2 * kap + 1], hb);
              tc::mma_16816(oacc[u][2 * kap], wa, ha[0], hb[0]);
              tc::mma_16816(oacc[u][2 * kap + 1], wa, ha[1], hb[1]);
            }
          } else {                              // unit = one chunk; one ldmatrix per unit pair
            if ((u & 1) == 0) tc::ldsm_x4_trans(vc + vls[u / 2], r);
            const int o = 2 * (u & 1);
            uint32_t bp[4][2];
            tc::q4_pairs<VAFF>(r[o], r[o + 1], bp);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) tc::mma_16816(oacc[u][s4], wa, bp[s4][0], bp[s4][1]);
          }
        }
      }
    }
    // the slot is free once this warp (both warps of a pair) is done with it
    if constexpr (DS == 2) {
      asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory");
    } else {
      __syncwarp();
    }
    if (producer && !timed_out && i + depth < n_local) issue(i + depth);
  }
  tc::grid_dependents_launch();

  // A wait that timed out: flag it, then give every issued copy of this group
  // one more bounded wait so none is still writing the ring when it is reused.
  if (timed_out) {
    if (lane == 0) report(a.status, KVQ_DEV_TIMEOUT);
    for (int i = max(0, n_local - depth); i < n_local; ++i)
      tc::mbar_wait(gbar + 8 * (i % depth), (uint32_t)((i / depth) & 1));
  }
  __syncthreads();

  // ---- merge the warps' states (shared memory reused)
  constexpr int NST = 4 / DS;
  float* ows = reinterpret_cast<float*>(smem);   // [NST][G][HD]
  float* mws = ows + NST * G * HD;               // [NST][G]
  float* lws = mws + NST * G;                    // [NST][G]
  const int state = warp / DS;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    float pbu = pb[u];
    pbu += __shfl_xor_sync(0xffffffffu, pbu, 1);
    pbu += __shfl_xor_sync(0xffffffffu, pbu, 2);
    const float sc = vref[u] * (1.0f / kWScale);
    if (live) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // 4-bit V: n-tiles 1 and 3 hold 16 * code
        const float scj = (VK != KVQ_SYM_INT8 && (j & 1)) ? sc * (1.0f / 16.0f) : sc;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = dim0 + pv_dim<VK>(u, j, 2 * tig + e);
          ows[(state * G + gid) * HD + d] = fmaf(oacc[u][j][e + 2], 1.0f / tc::kLoScale, oacc[u][j][e]) * scj + pbu;
        }
      }
    }
  }
  if (tig == 0 && live && half == 0) {
    mws[state * G + gid] = m;
    lws[state * G + gid] = l;
  }
  __syncthreads();

  const int64_t cidx = ((int64_t)b * a.n_kv_heads + kvh) * a.n_chunks + chunk;
  for (int i = tid; i < G * HD; i += kTcThreads) {
    const int h = i / HD, d = i - h * HD;
    float M = mws[h];
#pragma unroll
    for (int st2 = 1; st2 < NST; ++st2) M = fmaxf(M, mws[st2 * G + h]);
    float o = 0.f, ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int st2 = 0; st2 < NST; ++st2) {
        const float f = exp2f(mws[st2 * G + h] - M);
        o = fmaf(f, ows[(st2 * G + h) * HD + d], o);
        ls = fmaf(f, lws[st2 * G + h], ls);
      }
    }
    if (nch == 1) {
      store_act(A.out, a.act, obase + i, ls > 0.f ? o / ls : 0.f);
    } else {
      a.ws_acc[(cidx * G + h) * HD + d] = o;
      if (d == 0) {
        a.ws_ml[(cidx * G + h) * 2] = M;
        a.ws_ml[(cidx * G + h) * 2 + 1] = ls;
      }
    }
  }
  if (nch == 1) return;

  // ---- fused log-sum-exp combine: the last chunk of (b, kvh) to finish merges all
  __threadfence();
  __syncthreads();
  int32_t* counter = A.counters + (int64_t)b * a.n_kv_heads + kvh;
  if (tid == 0) flag_s = atomicAdd(counter, 1) == nch - 1;
  __syncthreads();
  if (!flag_s) return;
  __threadfence();
  const int64_t cbase = ((int64_t)b * a.n_kv_heads + kvh) * a.n_chunks;
  // (m, l) of every chunk and head in one parallel round, then the weights
  // 2^(m_c - M) / sum_c 2^(m_c - M) l_c per head in shared memory.
  float* wts = reinterpret_cast<float*>(smem);   // [nch][G] m, then weights
  float* lts = wts + nch * G;                    // [nch][G] l
  for (int i = tid; i < nch * G; i += kTcThreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml) + cbase * G + i);
    wts[i] = ml.x;
    lts[i] = ml.y;
  }
  __syncthreads();
  if (tid < G) {
    float mx = -INFINITY;
    for (int c = 0; c < nch; ++c) mx = fmaxf(mx, wts[c * G + tid]);
    float den = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float mc = wts[c * G + tid];
      const float w = (mx == -INFINITY || mc == -INFINITY) ? 0.f : exp2f(mc - mx);
      wts[c * G + tid] = w;
      den = fmaf(w, lts[c * G + tid], den);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int c = 0; c < nch; ++c) wts[c * G + tid] *= inv;
  }
  __syncthreads();
  // out = sum_c w_c acc_c: float4 loads, eight chunks in flight per thread
  const int NV4 = G * HD / 4;
  const float4* acc4 = reinterpret_cast<const float4*>(a.ws_acc) + cbase * NV4;
  for (int e = tid; e < NV4; e += kTcThreads) {
    const int h = (4 * e) / HD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int c = 0;
    for (; c + 8 <= nch; c += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldcg(acc4 + (int64_t)(c + k) * NV4 + e);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w = wts[(c + k) * G + h];
        o.x = fmaf(w, v[k].x, o.x);
        o.y = fmaf(w, v[k].y, o.y);
        o.z = fmaf(w, v[k].z, o.z);
        o.w = fmaf(w, v[k].w, o.w);
      }
    }
    for (; c < nch; ++c) {
      const float4 v = __ldcg(acc4 + (int64_t)c * NV4 + e);
      const float w = wts[c * G + h];
      o.x = fmaf(w, v.x, o.x);
      o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z);
      o.w = fmaf(w, v.w, o.w);
    }
    store_act(A.out, a.act, obase + 4 * e, o.x);
    store_act(A.out, a.act, obase + 4 * e + 1, o.y);
    store_act(A.out, a.act, obase + 4 * e + 2, o.z);
    store_act(A.out, a.act, obase + 4 * e + 3, o.w);
  }
  if (tid == 0) *counter = 0;   // ready for the next call
}

// Host launcher of one instantiation (dynamic shared memory, optional PDL).
template <int KK, int VK, int HD, bool ONEG, int PT>
kvq_status launch_tc_one(const TcArgs& t, const CUtensorMap& mk, const CUtensorMap& mv, dim3 grid, size_t smem,
                         cudaStream_t stream, bool pdl) {
  auto kern = decode_tc_kernel<KK, VK, HD, ONEG, PT>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, t, mk, mv);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

template <int KK, int VK, int PT>
kvq_status launch_tc_pt(const TcArgs& t, const CUtensorMap& mk, const CUtensorMap& mv, int head_dim, bool oneg,
                        dim3 grid, size_t smem, cudaStream_t stream, bool pdl) {
#define KVQ_TC(HD_)                                                                               \
  if (head_dim == HD_)                                                                            \
    return oneg ? launch_tc_one<KK, VK, HD_, true, PT>(t, mk, mv, grid, smem, stream, pdl)        \
                : launch_tc_one<KK, VK, HD_, false, PT>(t, mk, mv, grid, smem, stream, pdl);
  KVQ_TC(64)
  KVQ_TC(128)
  if constexpr (KK != KVQ_SYM_INT8 && VK != KVQ_SYM_INT8) {   // 8-bit rows of 256 B have no TMA swizzle
    KVQ_TC(256)
  }
#undef KVQ_TC
  return fail(KVQ_ERR_UNSUPPORTED, "no tensor-core decode kernel for head_dim %d", head_dim);
}

template <int KK, int VK>
kvq_status launch_tc_kinds(const TcArgs& t, const CUtensorMap& mk, const CUtensorMap& mv, int head_dim,
                           bool oneg, int param, dim3 grid, size_t smem, cudaStream_t stream, bool pdl) {
  if (param == KVQ_F32) return launch_tc_pt<KK, VK, KVQ_F32>(t, mk, mv, head_dim, oneg, grid, smem, stream, pdl);
  if (param == KVQ_F16) return launch_tc_pt<KK, VK, KVQ_F16>(t, mk, mv, head_dim, oneg, grid, smem, stream, pdl);
  return launch_tc_pt<KK, VK, KVQ_BF16>(t, mk, mv, head_dim, oneg, grid, smem, stream, pdl);
}

kvq_status launch_tc_s4s4(const TcArgs&, const CUtensorMap&, const CUtensorMap&, int, bool, int, dim3, size_t,
                          cudaStream_t, bool);
kvq_status launch_tc_s8s8(const TcArgs&, const CUtensorMap&, const CUtensorMap&, int, bool, int, dim3, size_t,
                          cudaStream_t, bool);
kvq_status launch_tc_s8s4(const TcArgs&, const CUtensorMap&, const CUtensorMap&, int, bool, int, dim3, size_t,
                          cudaStream_t, bool);
kvq_status launch_tc_a4a4(const TcArgs&, const CUtensorMap&, const CUtensorMap&, int, bool, int, dim3, size_t,
                          cudaStream_t, bool);

}  // namespace kvq
