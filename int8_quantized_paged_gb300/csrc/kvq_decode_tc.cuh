// Tensor-core split-K GQA decode attention over a paged, group-quantized KV
// cache, with the log-sum-exp combine fused in: by the last CTA of each
// (sequence, kv head) through a global workspace, or, for a few short
// sequences, inside a thread-block cluster per (sequence, kv head) whose CTAs
// push their partials into each other's shared memory.  The same kernel can
// also write the step's new K/V row first (the fused append).
//
// Method: softmax(q K^T * s) V straight from the packed codes through a block
// table ([airllm] §2.2: dequantize inside the kernel after the load, with no
// temporary tensor; §2.3: queries span fixed-size blocks; §3.4: fp32
// softmax).
//
// Why tensor cores: every code takes part in G multiply-adds for q.K and G
// for p.V.  On the fp32 CUDA cores that arithmetic, plus the dequantization,
// needs more instructions per byte than the SMs retire at HBM speed.  So the
// codes go to mma.sync as exact fp16 integers, converted in registers by a
// mantissa trick and never written back to shared memory.
//
// CTA = kWarps warps over one chunk of a (sequence, kv head).  Warp w takes
// the chunk's pages w, w + kWarps, ... and keeps the next D of them in flight
// in a private ring of page slots in shared memory: every lane issues 16-byte
// cp.async copies of the page's K and V sub-blocks (codes and scales), one
// commit group per page, so the warp waits only for its own oldest page.  The
// code rows are written with an XOR swizzle of their 16-byte chunks, so the
// ldmatrix reads below are free of bank conflicts.  A ring per warp, filled
// by all of its lanes, keeps many independent copy streams per SM; a single
// issuing thread per CTA refilling slots in page order does not saturate HBM
// with 2 KB pages.
//
// Per warp and 16-token page (the G <= 8 query heads of one kv head):
//   Q.K : S = Khat * Qhl, m16n8k16 with A = 16 tokens x 16 dims of codes and
//         B = 16 dims x 8 columns.  Column 2h holds the fp16 high part of
//         query head h (rotated, pre-scaled), column 2h+1 the low part
//         (q = hi + lo * 2^-12), so the dot products keep about fp32
//         precision.  A lane ends up with both parts of head h = lane % 4 for
//         tokens lane/4 and lane/4 + 8.  Each scale group accumulates
//         separately; its scale (and affine bias * sum q) applies in fp32.
//   softmax: online, base 2.  The running maximum is raised only when a page
//         exceeds it by 2^8, so the accumulators are rescaled on few pages,
//         and p <= 2^8.
//   P.V : O^T = Vhat^T * W, A = 16 dims x 16 tokens of codes (ldmatrix.trans),
//         B = 16 tokens x 8 columns: column 2h the high part of
//         w = p * scale * 2^7 / R, column 2h+1 the low part, where R is the
//         running maximum V scale of the group (w stays inside fp16's range).
//         w is formed where p lives and moved into the B layout with four
//         shuffles.
// Each warp keeps its own (m, l, O); the warps merge through shared memory at
// the end.  G = 8 (NT = 2) puts the 8 heads in the 8 columns of one tile and
// runs the high and the low parts as two passes into the same accumulators.
// 4-bit codes are symmetric (two's complement), affine (unsigned) or offset
// binary (stored as code + 8); unquantised f16 rows go to the MMAs as loaded.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "kvq_decode_impl.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"
#include "kvq_tc_ptx.cuh"

namespace kvq {

struct TcArgs {
  DecodeArgs d;
  void* out;
  int32_t* counters;         // [batch][n_kv_heads] arrival tickets (zero between calls)
  int32_t G;                 // query heads per kv head (1..8)
  int32_t blocks_per_chunk;  // 16-token blocks per chunk
  int32_t kc_bytes, vc_bytes, kp_bytes, vp_bytes;  // code and scale bytes of a page (one kv head)
  int32_t cluster;           // 0: split-K partials through the workspace; else CTAs per
                             // thread-block cluster (= gridDim.x), combined in shared memory
  int32_t recv_off;          // cluster mode: byte offset of the receive buffers (past every
                             // other use of shared memory; tc_recv_bytes after it)
  int32_t early;             // 1: launch the kernel that reads the lengths, positions,
                             // table, RoPE rows and first pages before waiting for the
                             // kernel before it (the EARLY instantiation)
};

constexpr int kWarps = 4;                 // warps per CTA, split-K through the workspace
constexpr int kTcThreads = 32 * kWarps;
constexpr int kClusterWarps = 8;          // warps per CTA in the cluster mode
constexpr int kMaxCluster = 16;           // CTAs per cluster (a non-portable size)
// Cluster-mode receive buffers of a CTA: the (M, l) pair of every head of
// every CTA of the cluster [kMaxCluster][G], then the partial o of this CTA's
// slice of the G * hd outputs from every CTA [cluster][per].
constexpr int kRecvMl = kMaxCluster * 8 * 8;
// Outputs a cluster CTA combines: its slice of the G * hd outputs, a multiple
// of 4 (the partials move four outputs a store).
__host__ __device__ inline int tc_per(int G, int hd, int cluster) { return ((G * hd + cluster - 1) / cluster + 3) & ~3; }
inline size_t tc_recv_bytes(int G, int hd, int cluster) {
  return kRecvMl + (size_t)cluster * tc_per(G, hd, cluster) * sizeof(float);
}
constexpr float kQScale = 256.0f;   // q is held x 2^8 in fp16 (hi/lo)
constexpr float kWScale = 128.0f;   // w is held x 2^7 (w <= 2^8 * 2^7 < 65504)
constexpr float kLazyMax = 8.0f;    // raise the running max only past +2^8

// Pages in flight per warp, and CTAs per SM (the launch bounds), by shape.
// f16 K/V pages are 4 times larger: 2 in flight per warp at hd 128 (4 at hd 64),
// 3 CTAs per SM.  4-bit pages at head_dim <= 128 keep 4 in flight in the
// cluster mode (one CTA per SM: 8 warps carry the whole page stream; measured
// 9.4 against 8.6 us per llama8b layer with 3) and 3 in the workspace mode,
// where 20 warps per SM do (continuous batch +0.9 % against 4).
__host__ __device__ constexpr int tc_depth(int hd, int nt, int kind = KVQ_SYM_INT4, bool cl = false) {
  return kind == KVQ_F16_KV ? (hd == 128 ? 2 : 4) : ((hd == 256 || nt == 2) ? 3 : (cl ? 4 : 3));
}
__host__ __device__ constexpr int tc_min_blocks(int hd, int nt, int kind = KVQ_SYM_INT4) {
  return kind == KVQ_F16_KV ? 3 : (hd <= 128 ? (nt == 1 ? 5 : 4) : 3);
}
// Shapes with a cluster-mode instantiation (one 8-column tile: G <= 4), and
// the cluster-mode CTAs resident per SM.
__host__ __device__ constexpr bool tc_cluster_shape(int hd, int nt) { return nt == 1; }
__host__ __device__ constexpr int tc_cluster_min_blocks(int hd) { return 1; }
// Shared memory of the query fragments (the same for every warp of a CTA):
// NT tiles x hd/16 k-steps x 2 words x 32 lanes.
__host__ __device__ constexpr int tc_qfrag_bytes(int hd, int nt) { return nt * hd * 16; }
// Shared memory after the page rings: the query fragments, the RoPE row of
// the query's position (hd / 2 cos/sin pairs), the affine-K per-group q sums
// ([nt][ng][4 heads]) and, for a fused append, the new K and V rows (up to
// fp32) with the RoPE row of their position, then their quantized rows (code
// rows up to 2 hd bytes (f16), parameter rows up to 64 bytes).
// The affine-K q sums: [group][4 heads] floats (NT = 1), [group][8] (NT = 2),
// or in the cluster mode, where several warps build the fragments,
// [32-dim unit][4 heads].
__host__ __device__ constexpr int tc_qsum_bytes(int hd, int nt, int ng, bool cl) {
  return cl && hd > 16 * nt * ng ? hd : 16 * nt * ng;
}
__host__ __device__ constexpr int tc_pre_bytes(int hd, int nt, int ng, bool cl) {
  return tc_qfrag_bytes(hd, nt) + 4 * hd + tc_qsum_bytes(hd, nt, ng, cl) + 16 * hd + 128;
}

// Fused append: quantizes the staged row (K rotated at its position) exactly
// as the append kernel does.
template <int HD, int KIND, int PT>
__device__ __forceinline__ RowCodes tc_append_row(const uint8_t* row, int act, const float2* cs, int rope,
                                                  const PoolLayout& L, int lane) {
  constexpr int DPL = HD / 32;
  float x[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) x[j] = load_act(row, act, lane * DPL + j);
  if (cs) rope_rotate_row<DPL>(x, cs, rope, lane);
  return quantize_row<DPL, KIND, PT>(x, L, lane);
}

// Shared-memory offset of 16-byte chunk `c` of row `r` in a block of rows of
// ROWB bytes (32..256), with the chunk index XORed by a function of the row:
// the eight rows an ldmatrix reads at one chunk land in eight different
// 16-byte bank groups.
template <int ROWB>
__device__ __forceinline__ int swz(int r, int c) {
  if constexpr (ROWB >= 128) {
    return r * ROWB + ((c ^ (r & 7)) << 4);
  } else {
    constexpr int SH = ROWB == 64 ? 1 : 2;
    constexpr int MASK = ROWB / 16 - 1;
    return r * ROWB + ((c ^ ((r >> SH) & MASK)) << 4);
  }
}

// A stored scale or bias of type PT (kvq_float) at shared address `addr`.
template <int PT>
__device__ __forceinline__ float ld_param(uint32_t addr) {
  if constexpr (PT == KVQ_F32) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
  } else {
    unsigned short u;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(u) : "r"(addr) : "memory");
    if constexpr (PT == KVQ_F16) return __half2float(__ushort_as_half(u));
    return __uint_as_float((uint32_t)u << 16);
  }
}

// Scale (and bias) bytes of one page of one kv head with ng groups per head.
__host__ __device__ constexpr int tc_scale_bytes(int kind, int ng, int pt) {
  return kind == KVQ_F16_KV ? 0 : 16 * ng * (kind == KVQ_AFFINE_INT4 ? 2 : 1) * (pt == KVQ_F32 ? 4 : 2);
}
// Bytes of one code row of a kind (hd elements).
__host__ __device__ constexpr int tc_row_bytes(int kind, int hd) {
  return kind == KVQ_F16_KV ? 2 * hd : (kind == KVQ_SYM_INT8 ? hd : hd / 2);
}
__host__ __device__ constexpr int tc_slot_bytes(int kk, int vk, int hd, int ng, int pt) {
  return 16 * tc_row_bytes(kk, hd) + 16 * tc_row_bytes(vk, hd) + tc_scale_bytes(kk, ng, pt) +
         tc_scale_bytes(vk, ng, pt);
}

// N consecutive activation elements (f32 / f16 / bf16) from element `off` of
// `p`, with vector loads; `off` is a multiple of N and the base 16-byte aligned.
template <int N>
__device__ __forceinline__ void load_run(const void* p, int act, int64_t off, float (&v)[N]) {
  static_assert(N == 2 || N == 4 || N == 8, "run");
  if (act == KVQ_F32) {
    if constexpr (N == 2) {
      const float2 x = *reinterpret_cast<const float2*>(static_cast<const float*>(p) + off);
      v[0] = x.x;
      v[1] = x.y;
    } else {
      const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(p) + off);
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        const float4 x = s[i];
        v[4 * i] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
      }
    }
  } else {
    uint32_t u[N / 2];
    const unsigned short* s = static_cast<const unsigned short*>(p) + off;
    if constexpr (N == 8) {
      const uint4 x = *reinterpret_cast<const uint4*>(s);
      u[0] = x.x; u[1] = x.y; u[2] = x.z; u[3] = x.w;
    } else if constexpr (N == 4) {
      const uint2 x = *reinterpret_cast<const uint2*>(s);
      u[0] = x.x; u[1] = x.y;
    } else {
      u[0] = *reinterpret_cast<const uint32_t*>(s);
    }
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      if (act == KVQ_F16) {
        v[2 * i] = __half2float(__ushort_as_half((unsigned short)(u[i] & 0xFFFFu)));
        v[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(u[i] >> 16)));
      } else {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    }
  }
}

// (hi, lo) fp16 parts of x packed as (low half, high half): x = hi + lo * 2^-12.
__device__ __forceinline__ uint32_t hilo_pack(float x) {
  const float hi = __half2float(__float2half_rn(x));
  return tc::pack_half2(x, (x - hi) * tc::kLoScale);
}

// The high (part 0) or low (part 1) fp16 part of x, as a float.
__device__ __forceinline__ float hilo_part(float x, int part) {
  const float hi = __half2float(__float2half_rn(x));
  return part ? (x - hi) * tc::kLoScale : x;
}
// The same with the low part x - hi not scaled up (it is added to the high
// part's products in one accumulator).
__device__ __forceinline__ float hilo_part_unscaled(float x, int part) {
  const float hi = __half2float(__float2half_rn(x));
  return part ? x - hi : x;
}

// KK / VK: code kinds of K and V.  HD: head dim.  NT: 1 for G <= 4 (one
// 8-column tile: column 2h the high and 2h+1 the low part of head h), 2 for
// 4 < G <= 8 (one 8-column tile of the 8 heads, column h head h, run twice:
// the high parts, then the low parts into the same accumulators).  NG: scale
// groups per head (the same for K and V), so every group index below is a
// compile-time constant.
// PT: stored type of the scales (and biases) of K and V.
// CL: the cluster mode (kClusterWarps warps per CTA, the chunks of a
// (sequence, kv head) one cluster of A.cluster CTAs); else kWarps warps.
template <int KK, int VK, int HD, int NT, int NG, int PT, bool CL, bool EARLY>
__global__ void __launch_bounds__(32 * (CL ? kClusterWarps : kWarps),
                                   CL ? tc_cluster_min_blocks(HD) : tc_min_blocks(HD, NT, KK))
decode_tc_kernel(const __grid_constant__ TcArgs A) {
  constexpr int P = 16;
  constexpr int NW = CL ? kClusterWarps : kWarps;
  constexpr int D = tc_depth(HD, NT, KK, CL);   // pages in flight per warp
  constexpr bool K8 = KK == KVQ_SYM_INT8, V8 = VK == KVQ_SYM_INT8;
  constexpr bool KAFF = KK == KVQ_AFFINE_INT4, VAFF = VK == KVQ_AFFINE_INT4;
  // 4-bit conversion modes (kvq_tc_ptx.cuh): 0 symmetric, 1 affine, 2 offset-binary (shimmy4)
  constexpr int KQ4 = KAFF ? 1 : (KK == KVQ_SHIMMY_INT4 ? 2 : 0);
  constexpr int VQ4 = VAFF ? 1 : (VK == KVQ_SHIMMY_INT4 ? 2 : 0);
  // F16: unquantised fp16 K and V (no scales): the ldmatrix fragments are the
  // MMA operands as they are, and the stored scales below read as 1
  constexpr bool F16 = KK == KVQ_F16_KV;
  static_assert(F16 == (VK == KVQ_F16_KV), "f16 K goes with f16 V");
  constexpr int KRB = tc_row_bytes(KK, HD);      // K code row bytes
  constexpr int VRB = tc_row_bytes(VK, HD);
  constexpr int KCH = KRB / 16;                  // 16-byte chunks per K row
  constexpr int VCH = VRB / 16;
  constexpr int KDC = F16 ? 8 : (K8 ? 16 : 32);  // dims per K chunk
  constexpr int VDC = F16 ? 8 : (V8 ? 16 : 32);
  constexpr int KSTEPS = F16 ? KCH / 2 : (K8 ? KCH : 2 * KCH);   // Q.K k-steps
  constexpr int MT = HD / 16;                    // P.V m-tiles
  constexpr int RUN = F16 ? 2 : (K8 ? 4 : 8);    // contiguous q dims a lane holds per K chunk
  constexpr int PB = PT == KVQ_F32 ? 4 : 2;      // bytes of a stored scale
  constexpr bool ONEG = NG == 1;
  constexpr int GS = HD / NG;                    // dims per scale group
  constexpr int KNG = NG, VNG = NG;
  // Ring slot: [K codes KC][V codes VC][K scales <= KPMAX][V scales <= VPMAX]
  constexpr int KC = 16 * KRB, VC = 16 * VRB;
  constexpr int KPMAX = tc_scale_bytes(KK, NG, PT), VPMAX = tc_scale_bytes(VK, NG, PT);
  constexpr int SLOT = KC + VC + KPMAX + VPMAX;
  // 16-byte copies per lane and page: lanes 0-15 copy the K sub-block, 16-31 the V one
  constexpr int NCP = cmax((KC + KPMAX) / 16, (VC + VPMAX) / 16) / 16 + 1;
  static_assert(KCH % 2 == 0 && VCH % 2 == 0, "chunk pairs");
  // MRG (G > 4): the 8 heads share one tile, the high and low parts are two
  // passes (the B fragments of pass 0 and 1 take the place of tiles 0 and 1).
  // A lane's two head slots h2 = 0, 1 are then heads 2 tig + h2 instead of
  // tig (and 4 + tig), and the P.V accumulators are one tile (NO = 1).
  constexpr bool MRG = NT == 2;
  constexpr int NO = MRG ? 1 : NT;
  // Query fragments in units of 32 dims (one uint4 of a lane: k-steps 2u,
  // 2u+1; CPU K chunks).  In the cluster mode (8 warps; the appenders are
  // warps 6 and 7) four warps build them, unit u by warp owner(u), each with
  // its own slice of the RoPE row (and, for affine K, per-unit q sums the
  // readers add up per group); elsewhere warp 0 builds them all.  A NeoX
  // pair (u, u + NU/2) stays with one warp.
  constexpr int CPU = F16 ? 4 : (K8 ? 2 : 1);
  constexpr int NU = KCH / CPU;
  constexpr int NBLD = CL ? cmin(4, NU) : 1;
  static_assert(KSTEPS / 2 == NU, "one uint4 of fragments a unit");
  static_assert(NBLD == 1 || !MRG, "several builders only with one tile");

  const DecodeArgs& a = A.d;
  const int G = A.G;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int32_t flag_s;

  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // Inputs may come from the kernel before this one.  Kernels launched after
  // this one may start their launch once every CTA is past the wait; each
  // waits for this grid to finish before it reads anything it writes.
  // EARLY: before its wait a thread reads only inputs the caller guarantees
  // that kernel does not write (lengths, positions, table, RoPE rows, pages).
  // The fragment builders (warp 0; warps 0-3 in the cluster mode), which
  // need q, wait for a whole-context decode once their page-id loads are
  // issued and before they use them (a CTA that starts while that kernel runs
  // has its ids by the end of the wait; one that starts later loads q
  // together with them), and for a ring or a window, whose page ids need the
  // length first, once their first page copies are issued (measured faster
  // there: 8.75 against 9.19 us per window layer).  The appender warps, which
  // need the new rows, wait once their roles are known.  The other warps
  // read nothing that kernel writes; they wait after the barrier that ends
  // the prologue (past the builders' waits), before any write.  A thread
  // triggers its dependents only after its own wait.
  auto wait_inputs = [&]() {
    tc::grid_dependency_wait();
    tc::grid_dependents_launch();
  };
  if constexpr (!EARLY) wait_inputs();

  // One round of independent loads: the length, (builders) this lane's raw q
  // elements (see the fragments below) and, for a whole-context decode, the
  // block-table entries of the warp's pages, which do not depend on the length.
  const int64_t obase = ((int64_t)b * a.n_heads + (int64_t)kvh * G) * HD;
  const int L = a.seq_lens[b];
  const int apos = a.app_pos ? a.app_pos[b] : -1;   // fused append: position of the new row
  float qv[NT][KCH][RUN];
  const bool neox = a.rope == KVQ_ROPE_NEOX;
  auto owner = [&](int u) { return (neox ? u % (NU / 2) : u) % NBLD; };   // builder of unit u
  const bool builder = NBLD == 1 ? warp == 0 : warp < NBLD;
  auto load_q = [&]() {   // this warp's units
    // column gid of the B fragments: head (gid / 2) mod G (NT = 1) or head
    // gid (MRG: both passes, zero for a column past the last head)
    const int hq = MRG ? gid : (gid >> 1) % G;
    if (!MRG || hq < G) {
#pragma unroll
      for (int c = 0; c < KCH; ++c)
        if (NBLD == 1 || owner(c / CPU) == warp)
          load_run<RUN>(a.q, a.act, obase + (int64_t)hq * HD + KDC * c + RUN * tig, qv[0][c]);
    } else {
#pragma unroll
      for (int c = 0; c < KCH; ++c)
#pragma unroll
        for (int k = 0; k < RUN; ++k) qv[0][c][k] = 0.f;
    }
  };
  if (!EARLY && builder) load_q();
  const int CB = A.blocks_per_chunk;
  const int w = warp;
  const int32_t* bt = a.block_table + (int64_t)b * a.max_pages;
  const bool whole = a.window == 0 && a.ring_rows == 0;
  int ids = -1;   // page ids of this warp's pages 32q .. 32q+31 (lane k % 32)
  if (whole) {
    const int blk = chunk * CB + w + NW * lane;
    if (blk < a.max_pages) ids = bt[blk];
  }
  if (EARLY && builder && whole) {
    wait_inputs();
    load_q();
  }

  int lo = 0, bad = 0;
  const int n_att = attended(a, L, &lo, &bad);
  if (n_att <= 0) {   // the same for every CTA of a (sequence, kv head), so of a cluster
    if (EARLY) tc::grid_dependency_wait();   // no write before the kernel before this one ends
    if (chunk == 0) {
      if (bad && tid == 0 && kvh == 0) report(a.status, bad);
      for (int i = tid; i < G * HD; i += NW * 32) store_act(A.out, a.act, obase + i, 0.f);
    }
    return;
  }
  // cluster mode: this CTA has started; the wait before the first store into
  // a peer's shared memory makes sure every peer has too
  if constexpr (CL) tc::cluster_arrive_relaxed();
  const int blk_lo = lo / P, blk_hi = (L + P - 1) / P;
  const int nch = (blk_hi - blk_lo + CB - 1) / CB;
  // In the cluster mode every CTA of the cluster reaches every cluster
  // barrier below: a CTA past the sequence's last chunk reads no page and
  // contributes an empty partial.
  if (chunk >= nch && !CL) return;
  const int cb0 = blk_lo + chunk * CB;
  const int ncb = chunk < nch ? min(CB, blk_hi - cb0) : 0;
  const int n_local = w < ncb ? (ncb - w + NW - 1) / NW : 0;   // pages w, w + NW, ... of the chunk

  // ---- page ring of this warp: D slots of SLOT bytes.  Lane (hl = lane % 16)
  // copies 16-byte chunks j = hl + 16 m of the page's K sub-block (lanes
  // 0-15) or V sub-block (lanes 16-31): codes, then scales.
  const uint32_t wring = tc::smem_u32(smem) + (uint32_t)(w * D * SLOT);
  const bool vlane = lane >= 16;
  const int hl = lane & 15;
  constexpr int KSUB = (KC + KPMAX) / 16, VSUB = (VC + VPMAX) / 16;   // 16-byte chunks of a sub-block
  constexpr int NCP_ALL = cmin(KSUB, VSUB) / 16;                       // copies every lane makes
  const int n_sub = vlane ? VSUB : KSUB;
  const int cnt = n_sub > hl ? (n_sub - hl + 15) / 16 : 0;             // this lane's copies
  // f16 rows: 16 copies a lane of rows with no scales, the destinations
  // computed as they go (keeping them would take 16 registers)
  constexpr int NCPR = F16 ? 1 : NCP;
  uint32_t cp_dst[NCPR];
#pragma unroll
  for (int m = 0; m < NCPR; ++m) {
    const int j = hl + 16 * m;
    uint32_t d;
    if (!vlane) d = j < KC / 16 ? swz<KRB>(j / KCH, j % KCH) : KC + VC + 16 * (j - KC / 16);
    else d = j < VC / 16 ? KC + swz<VRB>(j / VCH, j % VCH) : KC + VC + KPMAX + 16 * (j - VC / 16);
    cp_dst[m] = wring + d;
  }
  const uint32_t lane_sub = wring + (vlane ? KC : 0);   // f16: this lane's sub-block in slot 0
  const int ring = a.ring_rows, npp = a.n_pool_pages;
  auto page_of = [&](int k) -> int {   // page id of this warp's k-th page (k < n_local)
    const int blk = cb0 + w + NW * k;
    const int idx = ring > 0 ? (int)(((int64_t)blk * P) % ring) / P : blk;
    return bt[idx];
  };
  auto checked = [&](int pg, int k) -> int {   // -1 (and a flag) for an id outside the pool
    const bool ok = pg >= 0 && pg < npp;
    if (!ok && k < n_local) report(a.status, KVQ_DEV_BAD_PAGE);
    return ok ? pg : -1;
  };
  const uint8_t* pool_lane = (vlane ? a.v_pool + (int64_t)kvh * a.vl.sub_bytes
                                    : a.k_pool + (int64_t)kvh * a.kl.sub_bytes) + 16 * hl;
  const int64_t page_lane = vlane ? a.vl.page_bytes : a.kl.page_bytes;
  if (!whole && lane < n_local) ids = page_of(lane);
  ids = checked(ids, lane);
  // The builders copy the RoPE row of position L - 1 into shared memory ahead
  // of every page copy (each its units' part, as its own oldest commit group),
  // so the row does not queue behind the pages and the query fragments are
  // ready before they are.
  const uint32_t qfs = tc::smem_u32(smem) + (uint32_t)(NW * D * SLOT);   // fragments
  const uint32_t rope_s = qfs + tc_qfrag_bytes(HD, NT);                  // RoPE row
  const uint32_t qsum_s = rope_s + 4 * HD;                                // affine-K q sums
  if (builder && a.rope != KVQ_ROPE_NONE) {
    const uint8_t* row = reinterpret_cast<const uint8_t*>(a.rope_tab) + (int64_t)(L - 1) * (4 * HD);
    if (NBLD == 1) {
      for (int j = lane; j < HD / 4; j += 32)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(rope_s + 16 * j), "l"(row + 16 * j) : "memory");
    } else {
      // unit u's entries: bytes [128 u, 128 u + 128) (pairs inside the unit's
      // dims), or for NeoX [256 u, 256 u + 256) for u < NU / 2
      const int ub = neox ? 256 : 128;
#pragma unroll
      for (int u = 0; u < NU; ++u)
        if ((!neox || u < NU / 2) && owner(u) == warp && lane < ub / 16)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(rope_s + ub * u + 16 * lane),
                       "l"(row + ub * u + 16 * lane)
                       : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  // ---- fused append.  The CTA whose chunk holds the page of absolute block
  // apos / P (for a ring, the ring page that block lives in, whose other rows
  // a window no longer than the ring reads only through the same block)
  // writes the new row; for a position outside the attended blocks, chunk 0
  // does.  Two of its warps that build no query fragments share the work:
  // warp NW-1 stages the K row and the RoPE row of its position, warp NW-2 the
  // V row, each as its own commit group ahead of its pages; while the pages
  // are in flight each quantizes its row (tc_append_row, the append kernel's
  // arithmetic) into the pool and into a row buffer in shared memory.  The
  // warp that reads the page copies the buffers over the row's stale copy in
  // its slot when it gets there (after the barrier that ends the prologue),
  // so no read of the pool waits for the write.
  const int app_off = NW * D * SLOT + tc_qfrag_bytes(HD, NT) + 4 * HD + tc_qsum_bytes(HD, NT, NG, CL);   // [K][V][RoPE]
  int k_app = -1;    // the page warp: its page index of the new row
  int app_role = 0;  // 1: this warp quantizes the K row, 2: the V row
  int app_pg = -1;   // page id of the new row's block
  if (a.app_pos) {
    const bool pos_ok = apos >= 0 && (ring > 0 || apos / P < a.max_pages) &&
                        (a.rope == KVQ_ROPE_NONE || apos < a.rope_max_pos);
    const int bp = apos / P;
    bool writer = false;   // this CTA writes the row
    if (!pos_ok) {
      if (chunk == 0 && tid == 0) report(a.status, KVQ_DEV_BAD_POS);
    } else if (bp >= blk_lo && bp < blk_hi) {
      writer = chunk == (bp - blk_lo) / CB;
      if (writer && w == (bp - cb0) % NW) k_app = (bp - cb0) / NW;
    } else {
      writer = chunk == 0;
    }
    if (writer) {
      app_pg = bt[ring > 0 ? (int)(((int64_t)bp * P) % ring) / P : bp];   // a ring keeps the block in a ring page
      if (app_pg < 0 || app_pg >= npp) {
        if (tid == 0) report(a.status, KVQ_DEV_BAD_PAGE);
        k_app = -1;
      } else {
        app_role = w == NW - 1 ? 1 : (w == NW - 2 ? 2 : 0);
      }
    }
    if (app_role != 0) {
      if (EARLY) wait_inputs();   // the new rows may come from the kernel before this one
      const int actb = a.act == KVQ_F32 ? 4 : 2;
      const int64_t row = ((int64_t)b * a.n_kv_heads + kvh) * HD * actb;
      const uint8_t* src = static_cast<const uint8_t*>(app_role == 1 ? a.app_k : a.app_v) + row;
      const uint32_t dst = tc::smem_u32(smem) + app_off + (app_role == 1 ? 0 : 4 * HD);
      for (int j = lane; j < HD * actb / 16; j += 32)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * j), "l"(src + 16 * j) : "memory");
      if (app_role == 1 && a.rope != KVQ_ROPE_NONE) {
        const uint8_t* cs = reinterpret_cast<const uint8_t*>(a.rope_tab) + (int64_t)apos * (4 * HD);
        const uint32_t cdst = tc::smem_u32(smem) + app_off + 8 * HD;
        for (int j = lane; j < HD / 4; j += 32)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(cdst + 16 * j), "l"(cs + 16 * j) : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  }
  // The quantized rows, in the pool's row format, after the staged rows:
  // K codes [KRB], V codes [VRB], K parameter row, V parameter row.
  const int qk_off = app_off + 12 * HD, qv_off = qk_off + KRB, qkp_off = qv_off + VRB, qvp_off = qkp_off + 64;
  // Quantizes this warp's staged row (its copies have landed) into the pool
  // and into its row buffer above.
  auto quantize_app = [&]() {
    const uint8_t* st = smem + app_off;
    const int r = apos % P;
    if (app_role == 1) {
      const float2* cs = a.rope != KVQ_ROPE_NONE ? reinterpret_cast<const float2*>(st + 8 * HD) : nullptr;
      const RowCodes kq = tc_append_row<HD, KK, PT>(st, a.act, cs, a.rope, a.kl, lane);
      store_row<KK, PT>(kq, a.kl,
                const_cast<uint8_t*>(a.k_pool) + (int64_t)app_pg * a.kl.page_bytes + (int64_t)kvh * a.kl.sub_bytes,
                r, lane);
      store_code_bytes(smem + qk_off + lane * kq.nbytes, kq.w, kq.nbytes);
      if (kq.leader) {
        store_param(smem + qkp_off + param_scale_offset<KK, PT>(a.kl, kq.group), PT, kq.scale);
        if (KAFF) store_param(smem + qkp_off + param_bias_offset<PT>(a.kl, kq.group), PT, kq.bias);
      }
    } else {
      const RowCodes vq = tc_append_row<HD, VK, PT>(st + 4 * HD, a.act, nullptr, a.rope, a.vl, lane);
      store_row<VK, PT>(vq, a.vl,
                const_cast<uint8_t*>(a.v_pool) + (int64_t)app_pg * a.vl.page_bytes + (int64_t)kvh * a.vl.sub_bytes,
                r, lane);
      store_code_bytes(smem + qv_off + lane * vq.nbytes, vq.w, vq.nbytes);
      if (vq.leader) {
        store_param(smem + qvp_off + param_scale_offset<VK, PT>(a.vl, vq.group), PT, vq.scale);
        if (VAFF) store_param(smem + qvp_off + param_bias_offset<PT>(a.vl, vq.group), PT, vq.bias);
      }
    }
  };
  // Writes the quantized rows over row apos % P of slot s (codes swizzled
  // like the page copies).
  auto place_app = [&](int s) {
    uint8_t* slot = smem + (w * D + s) * SLOT;
    const int r = apos % P;
    if (lane < KCH) {
      const uint4 x = *reinterpret_cast<const uint4*>(smem + qk_off + 16 * lane);
      *reinterpret_cast<uint4*>(slot + swz<KRB>(r, lane)) = x;
    } else if (lane >= 16 && lane - 16 < VCH) {
      const uint4 x = *reinterpret_cast<const uint4*>(smem + qv_off + 16 * (lane - 16));
      *reinterpret_cast<uint4*>(slot + KC + swz<VRB>(r, lane - 16)) = x;
    }
    constexpr int kprb_ = F16 ? 0 : NG * (KAFF ? 2 : 1) * PB, vprb_ = F16 ? 0 : NG * (VAFF ? 2 : 1) * PB;
    for (int j = lane; j < kprb_; j += 32) slot[KC + VC + r * kprb_ + j] = smem[qkp_off + j];
    for (int j = lane; j < vprb_; j += 32) slot[KC + VC + KPMAX + r * vprb_ + j] = smem[qvp_off + j];
  };

  uint32_t valid = 0;   // bit s: slot s holds a page
  auto issue = [&](int k, int s) {   // all lanes: copies of page k into slot s
    if ((k & 31) == 0 && k > 0) ids = checked(k + lane < n_local ? page_of(k + lane) : -1, k + lane);
    const int pg = __shfl_sync(0xffffffffu, ids, k & 31);
    valid = pg >= 0 ? (valid | (1u << s)) : (valid & ~(1u << s));
    if (pg < 0) return;
    const uint8_t* src = pool_lane + pg * page_lane;
    const uint32_t so = s * SLOT;
    if constexpr (F16) {   // K and V sub-blocks alike: KSUB chunks, rows of KCH chunks
#pragma unroll
      for (int m = 0; m < KSUB / 16; ++m) {
        const int j = hl + 16 * m;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(lane_sub + so + swz<KRB>(j / KCH, j % KCH)),
                     "l"(src + 256 * m)
                     : "memory");
      }
    } else {
#pragma unroll
      for (int m = 0; m < NCP; ++m)
        if (m < NCP_ALL || m < cnt)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(cp_dst[m] + so), "l"(src + 256 * m)
                       : "memory");
    }
  };
#pragma unroll
  for (int k = 0; k < D; ++k) {
    if (k < n_local) issue(k, k);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (EARLY && builder && !whole) {
    wait_inputs();
    load_q();
  }

  // ---- query fragments (the builders).  Lane (gid, tig) holds, for column gid
  // (head hq = gid / 2, part gid % 2), the q elements its K k-steps meet: the
  // runs of RUN dims starting at KDC*c + RUN*tig of every K chunk c.  They are
  // the same for every warp of the CTA, so the builders keep them in shared
  // memory, [uint4 i][lane] with uint4 i = words of k-steps 2i, 2i+1 (unit i),
  // and every warp reloads the ones it needs per page (fewer live registers).
  if (builder) {
    // the RoPE row: the oldest of this lane's D + 1 commit groups
    asm volatile("cp.async.wait_group %0;" ::"n"(D) : "memory");
    __syncwarp();
    const float sc = a.score_scale * kQScale;
    const int rope = a.rope;
    auto mine = [&](int c) { return NBLD == 1 || owner(c / CPU) == warp; };   // chunk c is this warp's
    if (rope == KVQ_ROPE_NORMAL) {   // pairs (2i, 2i+1) lie inside a run
#pragma unroll
      for (int c = 0; c < KCH; ++c)
        if (mine(c))
#pragma unroll
        for (int k = 0; k < RUN; k += 2) {
          float2 t;
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                       : "=f"(t.x), "=f"(t.y) : "r"(rope_s + 4 * (KDC * c + RUN * tig + k)) : "memory");
          const float x0 = qv[0][c][k], x1 = qv[0][c][k + 1];
          qv[0][c][k] = x0 * t.x - x1 * t.y;
          qv[0][c][k + 1] = x0 * t.y + x1 * t.x;
        }
    } else if (rope == KVQ_ROPE_NEOX) {   // pairs (i, i + HD/2): chunk c with chunk c + KCH/2
#pragma unroll
      for (int c = 0; c < KCH / 2; ++c)
        if (mine(c))
#pragma unroll
        for (int k = 0; k < RUN; ++k) {
          float2 t;
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                       : "=f"(t.x), "=f"(t.y) : "r"(rope_s + 8 * (KDC * c + RUN * tig + k)) : "memory");
          const float x0 = qv[0][c][k], x1 = qv[0][c + KCH / 2][k];
          qv[0][c][k] = x0 * t.x - x1 * t.y;
          qv[0][c + KCH / 2][k] = x0 * t.y + x1 * t.x;
        }
    }
#pragma unroll
    for (int c = 0; c < KCH; ++c)
      if (mine(c))
#pragma unroll
      for (int k = 0; k < RUN; ++k) qv[0][c][k] *= sc;
    // B fragments of tile (NT = 1) or pass (MRG) nt: 4-bit K chunk c, parity p
    // (p = 1 meets 16 * code, so q / 16):
    //   b0 = q at dims KDC*c + 8tig + p + {0, 4},  b1 = dims + {2, 6}
    // 8-bit K chunk c:  b0 = dims 16c + 4tig + {0, 2},  b1 = dims + {1, 3}
    // f16 K k-step s (chunks 2s, 2s+1 of 8 dims): b0 = dims 16s + 2tig + {0, 1},
    // b1 = dims 16s + 8 + 2tig + {0, 1}
    // The part: high or low by the column's parity (NT = 1) or by the pass
    // (MRG, where the low part is not scaled up: both passes add into one
    // accumulator).
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int part = MRG ? nt : (gid & 1);
      auto qp = [&](float x) { return MRG ? hilo_part_unscaled(x, part) : hilo_part(x, part); };
      uint32_t qb[KSTEPS][2];
#pragma unroll
      for (int c = 0; c < KCH; ++c) {
        if (!mine(c)) continue;
        if constexpr (F16) {
          qb[c / 2][c & 1] = tc::pack_half2(qp(qv[0][c][0]), qp(qv[0][c][1]));
        } else if constexpr (K8) {
          qb[c][0] = tc::pack_half2(qp(qv[0][c][0]), qp(qv[0][c][2]));
          qb[c][1] = tc::pack_half2(qp(qv[0][c][1]), qp(qv[0][c][3]));
        } else {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const float f = p ? 1.0f / 16.0f : 1.0f;
            qb[2 * c + p][0] = tc::pack_half2(qp(qv[0][c][p] * f), qp(qv[0][c][p + 4] * f));
            qb[2 * c + p][1] = tc::pack_half2(qp(qv[0][c][p + 2] * f), qp(qv[0][c][p + 6] * f));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < KSTEPS / 2; ++i)
        if (NBLD == 1 || owner(i) == warp)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qfs + ((nt * (KSTEPS / 2) + i) * 32 + lane) * 16),
                     "r"(qb[2 * i][0]), "r"(qb[2 * i][1]), "r"(qb[2 * i + 1][0]), "r"(qb[2 * i + 1][1])
                     : "memory");
    }
    // affine K: per-group q sums of the columns' heads: [g][4] at lane 8h for
    // head h (gid = 2h, NT = 1), [g][8] at lane 4h for head h (MRG); with
    // several builders, per-unit sums [u][4], which the readers add per group
    if constexpr (KAFF && NBLD > 1) {
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        if (owner(u) != warp) continue;
        float v = 0.f;
#pragma unroll
        for (int c = u * CPU; c < (u + 1) * CPU; ++c)
#pragma unroll
          for (int k = 0; k < RUN; ++k) v += qv[0][c][k];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (tig == 0 && (gid & 1) == 0)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(qsum_s + 4 * (u * 4 + (gid >> 1))), "f"(v * (1.0f / kQScale))
                       : "memory");
      }
    } else if constexpr (KAFF) {
      float part_sum[KNG];
#pragma unroll
      for (int g = 0; g < KNG; ++g) part_sum[g] = 0.f;
#pragma unroll
      for (int c = 0; c < KCH; ++c) {
        const int g = (KDC * c) / GS;
#pragma unroll
        for (int gg = 0; gg < KNG; ++gg)
          if (gg == g)
#pragma unroll
            for (int k = 0; k < RUN; ++k) part_sum[gg] += qv[0][c][k];
      }
#pragma unroll
      for (int g = 0; g < KNG; ++g) {
        float v = part_sum[g];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (tig == 0 && (MRG || (gid & 1) == 0)) {
          const int slot = MRG ? g * 8 + gid : g * 4 + (gid >> 1);
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(qsum_s + 4 * slot), "f"(v * (1.0f / kQScale)) : "memory");
        }
      }
    }
  }
  // The new row is quantized now, while the pages are still arriving, by the
  // two appender warps in parallel with the builders' fragments; the barrier below
  // publishes the row buffers to the page warp.
  if (app_role != 0) {
    asm volatile("cp.async.wait_group %0;" ::"n"(D) : "memory");   // the staged row: older than the pages
    __syncwarp();
    quantize_app();
    __syncwarp();
  }
  __syncthreads();
  if (EARLY && !builder && app_role == 0) wait_inputs();
  // affine K: the q sums of this lane's score heads: tig (mod G) for NT = 1,
  // 2 tig + h2 for head slot h2 (MRG)
  float qsum[NT][KNG];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int g = 0; g < KNG; ++g) {
      qsum[nt][g] = 0.f;
      if constexpr (KAFF && NBLD > 1) {   // the group's units: GS / 32 of them
#pragma unroll
        for (int u = g * (GS / 32); u < (g + 1) * (GS / 32); ++u) {
          float x;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(x) : "r"(qsum_s + 4 * (u * 4 + tig % G)) : "memory");
          qsum[nt][g] += x;
        }
      } else if constexpr (KAFF) {
        const int slot = MRG ? g * 8 + 2 * tig + nt : g * 4 + tig % G;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(qsum[nt][g]) : "r"(qsum_s + 4 * slot) : "memory");
      }
    }

  // ---- per-lane constants of the main loop
  // parameter rows: per group a scale (and an affine bias) of PB bytes; the
  // host checks that the pools' rows have this layout
  constexpr int kstep = F16 ? 0 : (KAFF ? 2 : 1) * PB, vstep = F16 ? 0 : (VAFF ? 2 : 1) * PB;   // per group
  constexpr int kprb = NG * kstep, vprb = NG * vstep;                                          // per row
  const int mi = lane >> 3;
  const int trow = 8 * (mi & 1) + (lane & 7);    // token row this lane addresses in ldmatrix
  int kls[KCH / 2], vls[VCH / 2];
#pragma unroll
  for (int c = 0; c < KCH; c += 2) kls[c / 2] = swz<KRB>(trow, c + (mi >> 1));
#pragma unroll
  for (int c = 0; c < VCH; c += 2) vls[c / 2] = swz<VRB>(trow, c + (mi >> 1));
  // P.V transposition: the B column of this lane is head (gid / 2) mod G,
  // part gid % 2 (NT = 1), or head gid (MRG); its tokens 2tig, 2tig+1 (+8)
  // come from lanes src0, src1, which hold them for heads 2 src_tig, +1 (MRG)
  // or the head's two parts (NT = 1) in the two halves of one word.
  const int src_tig = MRG ? (gid >> 1) : (gid >> 1) % G;
  const int src0 = 8 * tig + src_tig, src1 = src0 + 4;
  const uint32_t psel = (gid & 1) ? 0x7632u : 0x5410u;

  // ---- running state of head slot h2 of this lane: head tig (mod G) for
  // NT = 1, head 2 tig + h2 for MRG
  float m[NT], l[NT];
  float oacc[MT][NO][4];   // MRG: elements e of head slot e & 1
  float pbias[NT][VNG];   // affine V: sum of p * bias per group
  float vinv[VNG];        // 2^7 / R, R the reference V scale of the group (0: none yet)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt] = -INFINITY;
    l[nt] = 0.f;
#pragma unroll
    for (int g = 0; g < VNG; ++g) pbias[nt][g] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int o = 0; o < NO; ++o)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[t][o][e] = 0.f;
  // the P.V accumulators of head slot h2 scaled by f
  auto scale_slot = [&](int h2, float f) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (MRG) {
          if ((e & 1) == h2) oacc[t][0][e] *= f;
        } else {
          oacc[t][h2][e] *= f;
        }
      }
  };
#pragma unroll
  for (int g = 0; g < VNG; ++g) vinv[g] = 0.f;

  // ---- one page (16 tokens) of a slot: its scores, then its P.V.
  // Q.K of the page in slot sl, whose row 0 is absolute token tb.
  auto page_scores = [&](int sl, int tb, bool edge, float (&sc)[NT][2]) {
    const uint32_t kc = wring + sl * SLOT;
    const uint32_t kp = kc + KC + VC;
    // ---- Q.K: A = codes of tokens (gid, gid+8), B = q fragments
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = 0.f;
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    // fold the accumulated dots of K group g into the scores
    auto fold = [&](int g) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t pr = kp + (gid + 8 * j) * kprb + g * kstep;
        const float ks = F16 ? 1.0f / kQScale : ld_param<PT>(pr) * (1.0f / kQScale);
        float kb = 0.f;
        if constexpr (KAFF) kb = ld_param<PT>(pr + PB);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          // MRG: pass 0 (high) and pass 1 (low) of head slot nt; NT = 1: the
          // high and the (scaled) low column of the head
          float v = MRG ? ks * (sacc[0][2 * j + nt] + sacc[1][2 * j + nt])
                        : ks * fmaf(sacc[nt][2 * j + 1], 1.0f / tc::kLoScale, sacc[nt][2 * j]);
          if constexpr (KAFF) {
            float qs = qsum[nt][0];
#pragma unroll
            for (int gg = 1; gg < KNG; ++gg)
              if (gg == g) qs = qsum[nt][gg];
            v = fmaf(kb, qs, v);
          }
          sc[nt][j] += v;
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
    };
#pragma unroll
    for (int c2 = 0; c2 < KCH / 2; ++c2) {
      uint32_t r[4];   // (tokens 0-7, chunk c), (8-15, c), (0-7, c+1), (8-15, c+1)
      tc::ldsm_x4(kc + kls[c2], r);
      if constexpr (F16) {
        // k-step c2: the fragment as loaded, B = words 2 (c2 % 2), +1 of uint4 c2 / 2
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t b0, b1;
          asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                       : "=r"(b0), "=r"(b1)
                       : "r"(qfs + ((nt * (KSTEPS / 2) + c2 / 2) * 32 + lane) * 16 + (c2 & 1) * 8));
          tc::mma_16816(sacc[nt], r, b0, b1);
        }
        continue;
      }
      // query fragments of chunks 2c2, 2c2+1: uint4s (K8: one for both, 4-bit: one each)
      uint32_t qf[NT][2][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int cc = 0; cc < (K8 ? 1 : 2); ++cc) {
          const int i = K8 ? c2 : 2 * c2 + cc;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(qf[nt][cc][0]), "=r"(qf[nt][cc][1]), "=r"(qf[nt][cc][2]), "=r"(qf[nt][cc][3])
                       : "r"(qfs + ((nt * (KSTEPS / 2) + i) * 32 + lane) * 16));
        }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * c2 + cc;
        // codes of tokens gid / gid+8 -> fp16 fragments -> MMAs, in one PTX block
        if constexpr (K8) {   // k-step c: words 2cc, 2cc+1 of the uint4
          const uint32_t b0[2] = {qf[0][0][2 * cc], qf[0][0][2 * cc + 1]};
          if constexpr (NT == 1) {
            tc::qk8(r[2 * cc], r[2 * cc + 1], b0, sacc[0]);
          } else {
            const uint32_t b1[2] = {qf[1][0][2 * cc], qf[1][0][2 * cc + 1]};
            tc::qk8x2(r[2 * cc], r[2 * cc + 1], b0, b1, sacc[0], sacc[1]);
          }
        } else {              // k-steps 2c, 2c+1: the uint4 of chunk c
          const uint32_t be0[2] = {qf[0][cc][0], qf[0][cc][1]}, bo0[2] = {qf[0][cc][2], qf[0][cc][3]};
          if constexpr (NT == 1) {
            tc::qk4<KQ4>(r[2 * cc], r[2 * cc + 1], be0, bo0, sacc[0]);
          } else {
            const uint32_t be1[2] = {qf[1][cc][0], qf[1][cc][1]}, bo1[2] = {qf[1][cc][2], qf[1][cc][3]};
            tc::qk4x2<KQ4>(r[2 * cc], r[2 * cc + 1], be0, bo0, be1, bo1, sacc[0], sacc[1]);
          }
        }
        if constexpr (!ONEG) {
          if ((KDC * (c + 1)) % GS == 0) fold((KDC * c) / GS);
        }
      }
    }
    if constexpr (ONEG) fold(0);
    if (edge) {   // the page at the window start or the context end
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t = tb + gid + 8 * j;
        if (t < lo || t >= L)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) sc[nt][j] = -INFINITY;
      }
    }

  };
  // The running max, raised (lazily) when this lane's scores bm pass it.
  auto raise_max = [&](const float (&bm)[NT]) {
    bool raise = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) raise |= bm[nt] > m[nt] + kLazyMax;
    if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float x = bm[nt];
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
        if (x > m[nt] + kLazyMax) {
          const float corr = m[nt] == -INFINITY ? 0.f : tc::ex2(m[nt] - x);
          l[nt] *= corr;
#pragma unroll
          for (int g = 0; g < VNG; ++g) pbias[nt][g] *= corr;
          scale_slot(nt, corr);
          m[nt] = x;
        }
      }
    }
  };
  // p = 2^(s - m) (0 for masked tokens, s = -inf), added to l.
  auto probs = [&](const float (&sc)[NT][2], float (&p)[NT][2]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float mu = m[nt] == -INFINITY ? 0.f : m[nt];
      p[nt][0] = tc::ex2(sc[nt][0] - mu);
      p[nt][1] = tc::ex2(sc[nt][1] - mu);
      l[nt] += p[nt][0] + p[nt][1];
    }
  };
  // P.V of the page in slot sl with probabilities p.
  auto page_pv = [&](int sl, int tb, bool edge, const float (&p)[NT][2]) {
    const uint32_t vc = wring + sl * SLOT + KC;
    const uint32_t vp = wring + sl * SLOT + KC + VC + KPMAX;
    // ---- P.V: A = V^T codes (ldmatrix.trans), B = weights of V group g.
    // Entering group g: its scales for the lane's tokens (gid, gid+8), a
    // raise of its reference when a scale passes half of it (2x headroom),
    // then w = p * scale * vinv formed here and moved to the B layout.
    uint32_t bw[NT][2];
    auto weights = [&](int g) {
      float vs[2], vb[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t pr = vp + (gid + 8 * j) * vprb + g * vstep;
        vs[j] = F16 ? 1.0f : ld_param<PT>(pr);
        if constexpr (VAFF) vb[j] = ld_param<PT>(pr + PB);
        if (edge) {
          const int t = tb + gid + 8 * j;
          if (t < lo || t >= L) vs[j] = vb[j] = 0.f;
        }
      }
      float vig = vinv[0];
#pragma unroll
      for (int gg = 1; gg < VNG; ++gg)
        if (gg == g) vig = vinv[gg];
      // a scale above half the reference: 2 * scale * vinv > kWScale
      if (__any_sync(0xffffffffu, 2.0f * fmaxf(vs[0], vs[1]) * vig > kWScale || vig == 0.f)) {
        float sm = fmaxf(vs[0], vs[1]);
        sm = fmaxf(sm, __shfl_xor_sync(0xffffffffu, sm, 4));
        sm = fmaxf(sm, __shfl_xor_sync(0xffffffffu, sm, 8));
        sm = fmaxf(sm, __shfl_xor_sync(0xffffffffu, sm, 16));
        if (sm > 0.f && (vig == 0.f || 2.0f * sm * vig > kWScale)) {
          const float nvi = kWScale / (2.0f * sm);
          if (vig > 0.f) {
            const float ratio = nvi / vig;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              const int c = V8 ? t : (t >> 1);
              if ((VDC * c) / GS == g)
#pragma unroll
                for (int o = 0; o < NO; ++o)
#pragma unroll
                  for (int e = 0; e < 4; ++e) oacc[t][o][e] *= ratio;
            }
          }
          vig = nvi;
#pragma unroll
          for (int gg = 0; gg < VNG; ++gg)
            if (gg == g) vinv[gg] = nvi;
        }
      }
      if constexpr (VAFF) {
#pragma unroll
        for (int gg = 0; gg < VNG; ++gg)
          if (gg == g)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              pbias[nt][gg] = fmaf(p[nt][0], vb[0], fmaf(p[nt][1], vb[1], pbias[nt][gg]));
      }
      const float w0 = vs[0] * vig, w1 = vs[1] * vig;
      // MRG: words of pass nt hold the part nt of heads 2tig, 2tig+1 (the
      // low part not scaled up); NT = 1: both parts of head tig
      uint32_t rp[NT][2];
      if constexpr (MRG) {
        const float x00 = p[0][0] * w0, x10 = p[1][0] * w0;   // token gid, heads 2tig, 2tig+1
        const float x01 = p[0][1] * w1, x11 = p[1][1] * w1;   // token gid + 8
        const float h00 = __half2float(__float2half_rn(x00)), h10 = __half2float(__float2half_rn(x10));
        const float h01 = __half2float(__float2half_rn(x01)), h11 = __half2float(__float2half_rn(x11));
        rp[0][0] = tc::pack_half2(h00, h10);
        rp[0][1] = tc::pack_half2(h01, h11);
        rp[1][0] = tc::pack_half2(x00 - h00, x10 - h10);
        rp[1][1] = tc::pack_half2(x01 - h01, x11 - h11);
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          rp[nt][0] = hilo_pack(p[nt][0] * w0);   // token gid
          rp[nt][1] = hilo_pack(p[nt][1] * w1);   // token gid + 8
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t r0 = rp[nt][0], r1 = rp[nt][1];
        const uint32_t u00 = __shfl_sync(0xffffffffu, r0, src0);  // token 2tig
        const uint32_t u10 = __shfl_sync(0xffffffffu, r0, src1);  // token 2tig + 1
        const uint32_t u01 = __shfl_sync(0xffffffffu, r1, src0);  // token 2tig + 8
        const uint32_t u11 = __shfl_sync(0xffffffffu, r1, src1);  // token 2tig + 9
        bw[nt][0] = __byte_perm(u00, u10, psel);
        bw[nt][1] = __byte_perm(u01, u11, psel);
      }
    };
    if constexpr (ONEG) weights(0);
#pragma unroll
    for (int c2 = 0; c2 < VCH / 2; ++c2) {
      uint32_t y[4];   // (tokens 0-7, chunk c), (8-15, c), (0-7, c+1), (8-15, c+1)
      tc::ldsm_x4_trans(vc + vls[c2], y);
      if constexpr (F16) {
        // m-tile c2 (dims of chunks 2c2, 2c2+1): A = V^T as loaded, rows dims
        const uint32_t av[4] = {y[0], y[2], y[1], y[3]};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) tc::mma_16816(oacc[c2][MRG ? 0 : nt], av, bw[nt][0], bw[nt][1]);
        continue;
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * c2 + cc;
        if constexpr (!ONEG) {
          if ((VDC * c) % GS == 0) weights((VDC * c) / GS);
        }
        // V^T codes of chunk c -> fp16 fragments -> MMAs, in one PTX block
        if constexpr (V8) {   // MRG: both passes into tile 0
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) tc::pv8(y[2 * cc], y[2 * cc + 1], bw[nt], oacc[c][MRG ? 0 : nt]);
        } else {
          if constexpr (NT == 1)
            tc::pv4<VQ4>(y[2 * cc], y[2 * cc + 1], bw[0], oacc[2 * c][0], oacc[2 * c + 1][0]);
          else
            tc::pv4m<VQ4>(y[2 * cc], y[2 * cc + 1], bw[0], bw[1], oacc[2 * c][0], oacc[2 * c + 1][0]);
        }
      }
    }
  };
  auto tok0 = [&](int k) { return (cb0 + w + k * NW) * P; };   // absolute token of row 0 of page k
  auto is_edge = [&](int tb) { return tb < lo || tb + P > L; };
  // The whole page k in slot sl.
  auto one_page = [&](int k, int sl) {
    const int tb = tok0(k);
    const bool edge = is_edge(tb);
    float sc[NT][2], p[NT][2], bm[NT];
    page_scores(sl, tb, edge, sc);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) bm[nt] = fmaxf(sc[nt][0], sc[nt][1]);
    raise_max(bm);
    probs(sc, p);
    page_pv(sl, tb, edge, p);
  };

  int s = 0;   // slot of page k: k % D
  int k = 0;
  // Two pages a step where the page's code is small (4-bit K and V, head_dim
  // <= 128): their Q.K chains are independent, one softmax update covers 32
  // tokens, and the wait and the loop control come once per pair.  The step
  // doubles the unrolled page code, so for f16, 8-bit or head_dim-256 pages the
  // one-page loop, which stays in the instruction cache, is faster (measured:
  // f16 llama8b shape 11.2 -> 10.2 us per layer, gemma mix +1 %; the 4-bit
  // llama8b shape 2.6 % slower without the step).
  constexpr bool PAIR_STEP = CL && !F16 && !K8 && !V8 && HD <= 128;
  if constexpr (PAIR_STEP) {
    // Pages k, k+1 landed: at most D - 2 younger commit groups pending.
#pragma unroll 1
    for (; k + 1 < n_local; k += 2) {
      const int s1 = s + 1 == D ? 0 : s + 1;
      asm volatile("cp.async.wait_group %0;" ::"n"(D - 2) : "memory");
      __syncwarp();
      if (k == k_app || k + 1 == k_app) {
        place_app(k == k_app ? s : s1);
        __syncwarp();
      }
      {
        // A page with a bad id (no copy: its slot holds stale data) goes
        // through as an edge page whose rows all start at L, so every row is
        // masked: its scores -inf, its V scales 0 (4-bit codes convert to
        // finite values whatever the bytes).
        const bool oka = ((valid >> s) & 1u) != 0, okb = ((valid >> s1) & 1u) != 0;
        const int ta = oka ? tok0(k) : L, tb1 = okb ? tok0(k + 1) : L;
        const bool ea = !oka || is_edge(ta), eb = !okb || is_edge(tb1);
        float sa[NT][2], sb[NT][2], pa[NT][2], pb[NT][2], bm[NT];
        page_scores(s, ta, ea, sa);
        page_scores(s1, tb1, eb, sb);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) bm[nt] = fmaxf(fmaxf(sa[nt][0], sa[nt][1]), fmaxf(sb[nt][0], sb[nt][1]));
        raise_max(bm);
        probs(sa, pa);
        probs(sb, pb);
        page_pv(s, ta, ea, pa);
        page_pv(s1, tb1, eb, pb);
      }
      // both slots are free once every lane is done reading them
      __syncwarp();
      if (k + D < n_local) issue(k + D, s);
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (k + 1 + D < n_local) issue(k + 1 + D, s1);
      asm volatile("cp.async.commit_group;" ::: "memory");
      s = s1 + 1 == D ? 0 : s1 + 1;
    }
  }
#pragma unroll 1
  for (; k < n_local; ++k) {
    // page k landed: at most D - 1 younger commit groups of this lane pending,
    // and the warp's lanes see each other's copies after the sync
    asm volatile("cp.async.wait_group %0;" ::"n"(D - 1) : "memory");
    __syncwarp();
    if (k == k_app) {   // the new row's page: its stale copy of the row is replaced
      place_app(s);
      __syncwarp();
    }
    if ((valid >> s) & 1u) one_page(k, s);
    // the slot is free once every lane is done reading it: refill it with page k + D
    __syncwarp();
    if (k + D < n_local) issue(k + D, s);
    asm volatile("cp.async.commit_group;" ::: "memory");
    s = s + 1 == D ? 0 : s + 1;
  }

  // ---- merge the warps' states (shared memory reused once every warp is
  // past its ring; no copies are pending).  First the warps' running maxima,
  // then each warp's partial (o, l) scaled by 2^(m_w - M) with M the CTA's
  // maximum (0 for a warp that saw no key), so the merge itself is a sum.
  // Output d of head h is kept at d ^ sw(h) of its row: the low two bits are
  // XORed with the lane's head index, so the 32 lanes of one store hit 32
  // different banks; readers take aligned groups of four and undo the XOR.
  __syncthreads();
  float* ows = reinterpret_cast<float*>(smem);   // [NW][G][HD]
  float* mws = ows + NW * G * HD;                // [NW][G]
  float* lws = mws + NW * G;                     // [NW][G]
  float* Mh = lws + NW * G;                      // [G]
  auto sw = [&](int h) { return MRG ? (h >> 1) & 3 : h & 3; };
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = MRG ? 2 * tig + nt : 4 * nt + tig;   // head of slot nt (valid when < G)
    if (h < G && gid == 0) mws[w * G + h] = m[nt];
  }
  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float lt = l[nt];
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    float pbs[VNG];
#pragma unroll
    for (int g = 0; g < VNG; ++g) {
      float v = pbias[nt][g];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      pbs[g] = v;
    }
    const int h = MRG ? 2 * tig + nt : 4 * nt + tig;
    if (h < G) {
      float M = mws[h];
#pragma unroll
      for (int w2 = 1; w2 < NW; ++w2) M = fmaxf(M, mws[w2 * G + h]);
      const float fw = m[nt] == -INFINITY ? 0.f : exp2f(m[nt] - M);   // this warp's weight
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        int d0, d1;
        float f;
        if constexpr (F16) {   // rows gid / gid+8 of tile t: dims 16t + gid, + 8
          d0 = 16 * t + gid;
          d1 = d0 + 8;
          f = 1.0f;
        } else if constexpr (V8) {
          d0 = 16 * t + 2 * gid;
          d1 = d0 + 1;
          f = 1.0f;
        } else {
          d0 = 32 * (t >> 1) + 4 * gid + (t & 1);
          d1 = d0 + 2;
          f = (t & 1) ? 1.0f / 16.0f : 1.0f;
        }
        const int c = V8 ? t : (t >> 1);
        const int g = (VDC * c) / GS;
        float vi = vinv[0], pbg = pbs[0];
#pragma unroll
        for (int gg = 1; gg < VNG; ++gg)
          if (gg == g) {
            vi = vinv[gg];
            pbg = pbs[gg];
          }
        const float sc = vi > 0.f ? f / vi : 0.f;   // R / 2^7, with 1/16 for 16 * code
        // rows gid / gid+8 of the tile are dims d0 / d1; MRG: columns 2tig, 2tig+1
        // are heads 2tig, 2tig+1; NT = 1: the high and the low part of head tig
        float o0, o1;
        if constexpr (MRG) {
          o0 = oacc[t][0][nt];
          o1 = oacc[t][0][2 + nt];
        } else {
          o0 = fmaf(oacc[t][nt][1], 1.0f / tc::kLoScale, oacc[t][nt][0]);
          o1 = fmaf(oacc[t][nt][3], 1.0f / tc::kLoScale, oacc[t][nt][2]);
        }
        ows[(w * G + h) * HD + (d0 ^ sw(h))] = fw * fmaf(o0, sc, pbg);
        ows[(w * G + h) * HD + (d1 ^ sw(h))] = fw * fmaf(o1, sc, pbg);
      }
      if (gid == 0) {
        lws[w * G + h] = fw * lt;
        if (w == 0) Mh[h] = M;
      }
    }
  }
  __syncthreads();

  const int64_t cidx = ((int64_t)b * a.n_kv_heads + kvh) * a.n_chunks + chunk;
  // cluster mode: the CTA's merged partial goes straight into the receive
  // buffers of the CTAs that combine it: outputs [i, i + 4) to CTA i / per,
  // and every head's (M, l) to every CTA
  const int ncl = CL ? A.cluster : 1;
  const int per = tc_per(G, HD, ncl);   // outputs combined per CTA
  const uint32_t rml = tc::smem_u32(smem) + (uint32_t)A.recv_off;
  const uint32_t rbo = rml + kRecvMl;
  const int rank = CL ? (int)tc::cluster_rank() : 0;
  if constexpr (CL) {
    tc::cluster_wait();
    // the (M, l) of head h to CTA c: one store for each of ncl * G threads
    if (tid < ncl * G) {
      const int h = tid % G, c = tid / G;
      float ls = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < NW; ++w2) ls += lws[w2 * G + h];
      tc::st_cluster_f2(tc::cluster_addr(rml + 8 * (rank * G + h), c), Mh[h], ls);
    }
  }
  for (int i = 4 * tid; i < G * HD; i += 4 * NW * 32) {
    const int h = i / HD, d = i - h * HD;
    const float M = Mh[h];
    float o[4] = {0.f, 0.f, 0.f, 0.f}, ls = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) {
      const float4 x = *reinterpret_cast<const float4*>(ows + (w2 * G + h) * HD + d);
      o[0] += x.x;
      o[1] += x.y;
      o[2] += x.z;
      o[3] += x.w;
      ls += lws[w2 * G + h];
    }
    // stored position j holds output d + (j ^ sw(h)): undo the XOR by swaps
    const int k = sw(h);
    float r0 = o[0], r1 = o[1], r2 = o[2], r3 = o[3];
    if (k & 1) {
      const float t0 = r0, t2 = r2;
      r0 = r1;
      r1 = t0;
      r2 = r3;
      r3 = t2;
    }
    if (k & 2) {
      const float t0 = r0, t1 = r1;
      r0 = r2;
      r1 = r3;
      r2 = t0;
      r3 = t1;
    }
    if constexpr (CL) {
      const int own = i / per;
      tc::st_cluster_f4(tc::cluster_addr(rbo + 4 * (rank * per + i - own * per), own), r0, r1, r2, r3);
    } else if (nch == 1) {
      store_act(A.out, a.act, obase + i, ls > 0.f ? r0 / ls : 0.f);
      store_act(A.out, a.act, obase + i + 1, ls > 0.f ? r1 / ls : 0.f);
      store_act(A.out, a.act, obase + i + 2, ls > 0.f ? r2 / ls : 0.f);
      store_act(A.out, a.act, obase + i + 3, ls > 0.f ? r3 / ls : 0.f);
    } else {
      *reinterpret_cast<float4*>(a.ws_acc + (cidx * G + h) * HD + d) = make_float4(r0, r1, r2, r3);
      if (d == 0) {
        a.ws_ml[(cidx * G + h) * 2] = M;
        a.ws_ml[(cidx * G + h) * 2 + 1] = ls;
      }
    }
  }

  // ---- cluster mode: log-sum-exp combine.  After the cluster barrier every
  // CTA's partials are in the receive buffers of the CTAs that combine them;
  // CTA r combines outputs [r per, (r + 1) per) from its own shared memory and
  // may exit: no CTA touches another's shared memory after the barrier.
  if constexpr (CL) {
    tc::cluster_barrier();
    // four threads an output, sources c = part, part + 4, ... each; the four
    // lanes of a group are consecutive, so xor 1 and 2 reach the others
    const int e0 = rank * per;
    const int e1 = min(G * HD, e0 + per);
    const int part = tid & 3;
    for (int base = e0; base < e1; base += NW * 8) {   // the same trip count for every thread
      const int e = base + (tid >> 2);
      const bool ok = e < e1;
      const int h = (ok ? e : e0) / HD;
      constexpr int NS = kMaxCluster / 4;
      float2 ml[NS];
      float v[NS];
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        const int c = part + 4 * j;
        ml[j] = make_float2(-INFINITY, 0.f);
        v[j] = 0.f;
        if (ok && c < ncl) {
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(ml[j].x), "=f"(ml[j].y) : "r"(rml + 8 * (c * G + h)));
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[j]) : "r"(rbo + 4 * (c * per + e - e0)));
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < NS; ++j) mx = fmaxf(mx, ml[j].x);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      float num = 0.f, den = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
          const float wt = tc::ex2(ml[j].x - mx);   // 0 for an empty partial (-inf)
          num = fmaf(wt, v[j], num);
          den = fmaf(wt, ml[j].y, den);
        }
      }
      num += __shfl_xor_sync(0xffffffffu, num, 1);
      den += __shfl_xor_sync(0xffffffffu, den, 1);
      num += __shfl_xor_sync(0xffffffffu, num, 2);
      den += __shfl_xor_sync(0xffffffffu, den, 2);
      if (ok && part == 0) store_act(A.out, a.act, obase + e, den > 0.f ? num / den : 0.f);
    }
    return;
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
  // Weights 2^(m_c - M) / sum_c 2^(m_c - M) l_c per head into shared memory:
  // warp w takes heads w, w + NW, ...; its lanes hold chunks lane + 32 i
  // (up to 4 per lane in registers, later ones are read again).
  float* wts = reinterpret_cast<float*>(smem);   // [nch][G]
  const float2* mlp = reinterpret_cast<const float2*>(a.ws_ml) + cbase * G;
  for (int h = w; h < G; h += NW) {
    float2 ml[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      ml[i] = c < nch ? __ldcg(mlp + (int64_t)c * G + h) : make_float2(-INFINITY, 0.f);
    }
    float mx = fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x));
    for (int c = lane + 128; c < nch; c += 32) mx = fmaxf(mx, __ldcg(mlp + (int64_t)c * G + h).x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float wt = (mx == -INFINITY || ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - mx);
      ml[i].x = wt;
      den = fmaf(wt, ml[i].y, den);
    }
    for (int c = lane + 128; c < nch; c += 32) {
      const float2 v = __ldcg(mlp + (int64_t)c * G + h);
      const float wt = (mx == -INFINITY || v.x == -INFINITY) ? 0.f : exp2f(v.x - mx);
      wts[c * G + h] = wt;
      den = fmaf(wt, v.y, den);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      if (c < nch) wts[c * G + h] = ml[i].x * inv;
    }
    for (int c = lane + 128; c < nch; c += 32) wts[c * G + h] *= inv;
  }
  __syncthreads();
  // out = sum_c w_c acc_c.  The float4 columns of the partials are spread over
  // the threads, and when there are fewer columns than threads the chunks are
  // split into NGRP groups summed separately, then added through shared memory.
  // Each thread keeps up to 16 partial loads in flight.
  const int NV4 = G * HD / 4;
  const int NGRP = NV4 >= kTcThreads ? 1 : kTcThreads / NV4;
  const float4* acc4 = reinterpret_cast<const float4*>(a.ws_acc) + cbase * NV4;
  float4* red = reinterpret_cast<float4*>(smem + ((8 * nch * G + 15) & ~15));   // [NGRP][NV4], 16-byte aligned
  for (int t = tid; t < NV4 * NGRP; t += kTcThreads) {
    const int e = t % NV4, grp = t / NV4;
    const int h = (4 * e) / HD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int c = grp;
    for (; c + 15 * NGRP < nch; c += 16 * NGRP) {
      float4 v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = __ldcg(acc4 + (int64_t)(c + k * NGRP) * NV4 + e);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float wt = wts[(c + k * NGRP) * G + h];
        o.x = fmaf(wt, v[k].x, o.x);
        o.y = fmaf(wt, v[k].y, o.y);
        o.z = fmaf(wt, v[k].z, o.z);
        o.w = fmaf(wt, v[k].w, o.w);
      }
    }
    for (; c < nch; c += NGRP) {
      const float4 v = __ldcg(acc4 + (int64_t)c * NV4 + e);
      const float wt = wts[c * G + h];
      o.x = fmaf(wt, v.x, o.x);
      o.y = fmaf(wt, v.y, o.y);
      o.z = fmaf(wt, v.z, o.z);
      o.w = fmaf(wt, v.w, o.w);
    }
    if (NGRP == 1) {
      store_act(A.out, a.act, obase + 4 * e, o.x);
      store_act(A.out, a.act, obase + 4 * e + 1, o.y);
      store_act(A.out, a.act, obase + 4 * e + 2, o.z);
      store_act(A.out, a.act, obase + 4 * e + 3, o.w);
    } else {
      red[grp * NV4 + e] = o;
    }
  }
  if (NGRP > 1) {
    __syncthreads();
    for (int e = tid; e < NV4; e += kTcThreads) {
      float4 o = red[e];
      for (int g2 = 1; g2 < NGRP; ++g2) {
        const float4 x = red[g2 * NV4 + e];
        o.x += x.x;
        o.y += x.y;
        o.z += x.z;
        o.w += x.w;
      }
      store_act(A.out, a.act, obase + 4 * e, o.x);
      store_act(A.out, a.act, obase + 4 * e + 1, o.y);
      store_act(A.out, a.act, obase + 4 * e + 2, o.z);
      store_act(A.out, a.act, obase + 4 * e + 3, o.w);
    }
  }
  if (tid == 0) *counter = 0;   // ready for the next call
}

// How to launch the kernel: grid and dynamic shared memory, warps per CTA,
// CTAs per cluster (0: no cluster), PDL.  With max_active set, nothing is
// launched: it receives how many such clusters can be resident at once.
struct TcLaunchCfg {
  dim3 grid;
  size_t smem;
  cudaStream_t stream;
  bool pdl;
  int warps;
  int cluster;
  int* max_active;
};

// Host launcher of one instantiation.
template <int KK, int VK, int HD, int NT, int NG, int PT, bool CL, bool EARLY>
kvq_status launch_tc_one(const TcArgs& t, const TcLaunchCfg& lc) {
  auto kern = decode_tc_kernel<KK, VK, HD, NT, NG, PT, CL, EARLY>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = lc.grid;
  cfg.blockDim = dim3(32 * lc.warps);
  cfg.dynamicSmemBytes = lc.smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (lc.cluster > 0) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = (unsigned)lc.cluster;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (lc.pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  if (lc.max_active) {
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) {
      cudaGetLastError();   // a refused configuration is an answer, not a sticky error
      n = 0;
    }
    *lc.max_active = n;
    return KVQ_OK;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, t);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

// The shapes a K kind is instantiated for: f16 K/V at head_dim 64 and 128
// with one (unused) scale group; the quantised kinds at every shape below.
constexpr bool tc_kind_shape(int kk, int hd, int ng) { return kk != KVQ_F16_KV || (hd <= 128 && ng == 1); }

// Shapes with a tensor-core instantiation: head_dim 64 and 256 with G <= 4,
// head_dim 128 with any G; ng = head_dim / group scale groups per head, with
// groups of at least 32 elements.
inline bool tc_has_shape(int head_dim, int nt, int ng) {
  const bool ng_ok = ng == 1 || ng == 2 || ng == 4 || ng == 8;
  return ng_ok && head_dim / ng >= 32 && (head_dim == 128 || ((head_dim == 64 || head_dim == 256) && nt == 1));
}

template <int KK, int VK, int PT>
kvq_status launch_tc_pt(const TcArgs& t, int head_dim, int nt, int ng, const TcLaunchCfg& lc) {
#define KVQ_TC(HD_, NT_, NG_)                                                                      \
  if constexpr (tc_kind_shape(KK, HD_, NG_))                                                       \
    if (head_dim == HD_ && nt == NT_ && ng == NG_) {                                               \
      if constexpr (tc_cluster_shape(HD_, NT_))                                                     \
        if (lc.cluster > 0)                                                                        \
          return t.early ? launch_tc_one<KK, VK, HD_, NT_, NG_, PT, true, true>(t, lc)             \
                         : launch_tc_one<KK, VK, HD_, NT_, NG_, PT, true, false>(t, lc);           \
      if (lc.cluster > 0) return fail(KVQ_ERR_UNSUPPORTED, "no cluster-mode kernel for this shape"); \
      return t.early ? launch_tc_one<KK, VK, HD_, NT_, NG_, PT, false, true>(t, lc)                \
                     : launch_tc_one<KK, VK, HD_, NT_, NG_, PT, false, false>(t, lc);              \
    }
  KVQ_TC(64, 1, 1)
  KVQ_TC(64, 1, 2)
  KVQ_TC(128, 1, 1)
  KVQ_TC(128, 1, 2)
  KVQ_TC(128, 1, 4)
  KVQ_TC(128, 2, 1)
  KVQ_TC(128, 2, 2)
  KVQ_TC(128, 2, 4)
  KVQ_TC(256, 1, 1)
  KVQ_TC(256, 1, 2)
  KVQ_TC(256, 1, 4)
  KVQ_TC(256, 1, 8)
#undef KVQ_TC
  return fail(KVQ_ERR_UNSUPPORTED, "no tensor-core decode kernel for head_dim %d", head_dim);
}

// One launcher per (K/V kind pair, scale type), each its own translation unit.
typedef kvq_status (*TcLaunch)(const TcArgs&, int, int, int, const TcLaunchCfg&);
#define KVQ_TC_DECLARE(NAME) kvq_status NAME(const TcArgs&, int, int, int, const TcLaunchCfg&);
KVQ_TC_DECLARE(launch_tc_s4s4_f32)
KVQ_TC_DECLARE(launch_tc_s4s4_f16)
KVQ_TC_DECLARE(launch_tc_s4s4_bf16)
KVQ_TC_DECLARE(launch_tc_s8s8_f32)
KVQ_TC_DECLARE(launch_tc_s8s8_f16)
KVQ_TC_DECLARE(launch_tc_s8s8_bf16)
KVQ_TC_DECLARE(launch_tc_s8s4_f32)
KVQ_TC_DECLARE(launch_tc_s8s4_f16)
KVQ_TC_DECLARE(launch_tc_s8s4_bf16)
KVQ_TC_DECLARE(launch_tc_a4a4_f32)
KVQ_TC_DECLARE(launch_tc_a4a4_f16)
KVQ_TC_DECLARE(launch_tc_a4a4_bf16)
KVQ_TC_DECLARE(launch_tc_h16)
KVQ_TC_DECLARE(launch_tc_o4o4_f32)
#undef KVQ_TC_DECLARE

}  // namespace kvq
