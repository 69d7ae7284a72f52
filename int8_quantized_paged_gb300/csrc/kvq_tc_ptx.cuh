// Inline-PTX helpers for the tensor-core decode kernel: TMA (tiled and bulk)
// copies completed on mbarriers, bounded mbarrier waits, ldmatrix, mma.sync,
// programmatic dependent launch, and exact code -> fp16 conversion.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace kvq {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `phase` of the barrier for at most `limit_ns` of
// %globaltimer (a step of the timer backwards restarts the count); false on
// timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase, uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, phase)) return true;
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, phase)) {
    const uint64_t t = global_timer_ns();
    if (t < t0) t0 = t;
    if (t - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled copy of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Contiguous copy (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22, results
// below 2^-126 flushed to zero); used for softmax weights in base 2.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters

// Every thread of every CTA of the cluster arrives (releasing its earlier
// shared-memory writes to the cluster) and waits for all the others.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of shared-memory location `addr` of this CTA in the CTA of the
// cluster with rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- ldmatrix / mma

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// D += A(16x16, row) * B(16x8, col); fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- codes -> fp16

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  __half2 y = *reinterpret_cast<__half2*>(&b);
  __half2 r = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Codes of a packed word as exact half2 values, placed in the mantissa of
// 1024 (0x6400) and the offset subtracted.  Symmetric 4-bit nibbles are XORed
// with 8 (offset binary), affine nibbles are unsigned, and 8-bit codes are
// XORed with 0x80.
//
// 4-bit, word x = nibbles n0..n7 (n_j at bits 4j):
//   q4<0>(x) = (n0, n4)        q4<1>(x) = 16 * (n1, n5)
//   q4<2>(x) = (n2, n6)        q4<3>(x) = 16 * (n3, n7)
// The odd nibbles are taken where they lie (bits 4..7 of each half), which
// gives 16 times the code, still exact in fp16.  The caller folds the 1/16
// into the other operand or the result.  One shift (x >> 8) serves n2, n3,
// n6 and n7.
// 8-bit, word x = bytes b0..b3:  q8<0>(x) = (b0, b2),  q8<1>(x) = (b1, b3).
template <bool AFF>
__device__ __forceinline__ void q4_codes(uint32_t x, uint32_t (&h)[4]) {
  const uint32_t y = x >> 8;
  constexpr uint32_t X0 = AFF ? 0x64006400u : 0x64086408u;   // offset of n at bits 0..3
  constexpr uint32_t X1 = AFF ? 0x64006400u : 0x64806480u;   // offset of n at bits 4..7
  h[0] = hsub2_u32((x & 0x000F000Fu) ^ X0, X0);
  h[1] = hsub2_u32((x & 0x00F000F0u) ^ X1, X1);
  h[2] = hsub2_u32((y & 0x000F000Fu) ^ X0, X0);
  h[3] = hsub2_u32((y & 0x00F000F0u) ^ X1, X1);
}

// The B operand pairs of P.V from two ldmatrix.trans words: b[s] = (q4<s>(xa),
// q4<s>(xb)), produced pairwise so each pair can live in adjacent registers.
template <bool AFF>
__device__ __forceinline__ void q4_pairs(uint32_t xa, uint32_t xb, uint32_t (&b)[4][2]) {
  const uint32_t ya = xa >> 8, yb = xb >> 8;
  constexpr uint32_t X0 = AFF ? 0x64006400u : 0x64086408u;
  constexpr uint32_t X1 = AFF ? 0x64006400u : 0x64806480u;
  b[0][0] = hsub2_u32((xa & 0x000F000Fu) ^ X0, X0);
  b[0][1] = hsub2_u32((xb & 0x000F000Fu) ^ X0, X0);
  b[1][0] = hsub2_u32((xa & 0x00F000F0u) ^ X1, X1);
  b[1][1] = hsub2_u32((xb & 0x00F000F0u) ^ X1, X1);
  b[2][0] = hsub2_u32((ya & 0x000F000Fu) ^ X0, X0);
  b[2][1] = hsub2_u32((yb & 0x000F000Fu) ^ X0, X0);
  b[3][0] = hsub2_u32((ya & 0x00F000F0u) ^ X1, X1);
  b[3][1] = hsub2_u32((yb & 0x00F000F0u) ^ X1, X1);
}

__device__ __forceinline__ void q8_codes(uint32_t x, uint32_t (&h)[2]) {
  h[0] = hsub2_u32((x & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
  h[1] = hsub2_u32(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}

// ---------------------------------------------------------------- fused code conversion + mma
// Each helper converts two code words to exact fp16 fragments inside one PTX
// block and feeds them to mma.sync, so the conversion results go straight into
// the MMA operand registers.  Offsets: symmetric 4-bit nibbles are XORed with 8
// (n + 8 in the mantissa of 1024), affine nibbles are taken as they are, 8-bit
// codes are XORed with 0x80; the odd nibbles come as 16 * code.
//
// 4-bit K (A = tokens): x0 = codes of token gid, x8 = token gid + 8 (one 32-bit
// word each, 8 nibbles).  k-step "even" uses nibbles (0,4 | 2,6), "odd" uses
// (1,5 | 3,7); B fragments be / bo; D += A * B.
#define KVQ_Q4_PRE(K0, K1, X0, X8)                                        \
  " .reg .b32 u0, u1, t, a0, a1, a2, a3, e0, e1, e2, e3;\n"              \
  " shr.b32 u0, " X0 ", 8;\n shr.b32 u1, " X8 ", 8;\n"                   \
  " lop3.b32 t, " X0 ", 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a0, t, " K0 ";\n" \
  " lop3.b32 t, " X8 ", 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a1, t, " K0 ";\n" \
  " lop3.b32 t, u0, 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a2, t, " K0 ";\n"   \
  " lop3.b32 t, u1, 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a3, t, " K0 ";\n"   \
  " lop3.b32 t, " X0 ", 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e0, t, " K1 ";\n" \
  " lop3.b32 t, " X8 ", 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e1, t, " K1 ";\n" \
  " lop3.b32 t, u0, 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e2, t, " K1 ";\n"   \
  " lop3.b32 t, u1, 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e3, t, " K1 ";\n"
#define KVQ_MMA(D, A0, A1, A2, A3, B0, B1)                                                       \
  " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {" D "}, {" A0 "," A1 "," A2 "," A3 "}, {" B0 \
  "," B1 "}, {" D "};\n"
// lop3 immediate 0x6a = (a & b) ^ c.  Symmetric nibbles: offsets 8 (bits 0..3)
// and 0x80 (bits 4..7), i.e. n + 8 and 16 * (n + 8) in the mantissa of 1024;
// affine nibbles: no offset.
// The two constants are register operands: the caller's loop holds them in
// registers instead of every block materializing them.
template <bool AFF>
__device__ __forceinline__ uint32_t q4_magic_lo() { return AFF ? 0x64006400u : 0x64086408u; }
template <bool AFF>
__device__ __forceinline__ uint32_t q4_magic_hi() { return AFF ? 0x64006400u : 0x64806480u; }

// Q.K, 4-bit K, one 8-column tile: 2 MMAs into d.
template <bool AFF>
__device__ __forceinline__ void qk4(uint32_t x0, uint32_t x8, const uint32_t (&be)[2], const uint32_t (&bo)[2],
                                    float (&d)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%10", "%11", "%4", "%5") KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%6", "%7")
               KVQ_MMA("%0,%1,%2,%3", "e0", "e1", "e2", "e3", "%8", "%9") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(x0), "r"(x8), "r"(be[0]), "r"(be[1]), "r"(bo[0]), "r"(bo[1]), "r"(q4_magic_lo<AFF>()),
                 "r"(q4_magic_hi<AFF>()));
}

// Q.K, 4-bit K, two 8-column tiles: 4 MMAs into d / f.
template <bool AFF>
__device__ __forceinline__ void qk4x2(uint32_t x0, uint32_t x8, const uint32_t (&be)[2], const uint32_t (&bo)[2],
                                      const uint32_t (&ce)[2], const uint32_t (&co)[2], float (&d)[4], float (&f)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%18", "%19", "%8", "%9") KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%10", "%11")
               KVQ_MMA("%0,%1,%2,%3", "e0", "e1", "e2", "e3", "%12", "%13")
               KVQ_MMA("%4,%5,%6,%7", "a0", "a1", "a2", "a3", "%14", "%15")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e1", "e2", "e3", "%16", "%17") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]), "+f"(f[0]), "+f"(f[1]), "+f"(f[2]), "+f"(f[3])
               : "r"(x0), "r"(x8), "r"(be[0]), "r"(be[1]), "r"(bo[0]), "r"(bo[1]), "r"(ce[0]), "r"(ce[1]),
                 "r"(co[0]), "r"(co[1]), "r"(q4_magic_lo<AFF>()), "r"(q4_magic_hi<AFF>()));
}

// P.V, 4-bit V (A = V^T from ldmatrix.trans): y0 = the tokens 0-7 word, y8 =
// the tokens 8-15 word.  With the names of KVQ_Q4_PRE (x0 = y0, x8 = y8),
// the even output tile (16-dim rows 4g, 4g+2) takes A = {a0, a2, a1, a3} and
// the odd one (16 x code, rows 4g+1, 4g+3) A = {e0, e2, e1, e3}.
template <bool AFF>
__device__ __forceinline__ void pv4(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], float (&de)[4], float (&dodd)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%12", "%13", "%8", "%9") KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%10", "%11")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%10", "%11") "}\n"
               : "+f"(de[0]), "+f"(de[1]), "+f"(de[2]), "+f"(de[3]), "+f"(dodd[0]), "+f"(dodd[1]),
                 "+f"(dodd[2]), "+f"(dodd[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), "r"(q4_magic_lo<AFF>()), "r"(q4_magic_hi<AFF>()));
}

// P.V, 4-bit V, two 8-column tiles (weights b for tile 0, c for tile 1).
template <bool AFF>
__device__ __forceinline__ void pv4x2(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], const uint32_t (&c)[2],
                                      float (&de)[4], float (&dodd)[4], float (&fe)[4], float (&fodd)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%22", "%23", "%16", "%17")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%18", "%19")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%18", "%19")
               KVQ_MMA("%8,%9,%10,%11", "a0", "a2", "a1", "a3", "%20", "%21")
               KVQ_MMA("%12,%13,%14,%15", "e0", "e2", "e1", "e3", "%20", "%21") "}\n"
               : "+f"(de[0]), "+f"(de[1]), "+f"(de[2]), "+f"(de[3]), "+f"(dodd[0]), "+f"(dodd[1]),
                 "+f"(dodd[2]), "+f"(dodd[3]), "+f"(fe[0]), "+f"(fe[1]), "+f"(fe[2]), "+f"(fe[3]),
                 "+f"(fodd[0]), "+f"(fodd[1]), "+f"(fodd[2]), "+f"(fodd[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), "r"(c[0]), "r"(c[1]), "r"(q4_magic_lo<AFF>()),
                 "r"(q4_magic_hi<AFF>()));
}

// P.V, 4-bit V, one tile run twice (weights b, then c) into the same
// accumulators: the high and the low parts of the weights.
template <bool AFF>
__device__ __forceinline__ void pv4m(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], const uint32_t (&c)[2],
                                     float (&de)[4], float (&dodd)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%14", "%15", "%8", "%9")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%10", "%11")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%10", "%11")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%12", "%13")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%12", "%13") "}\n"
               : "+f"(de[0]), "+f"(de[1]), "+f"(de[2]), "+f"(de[3]), "+f"(dodd[0]), "+f"(dodd[1]),
                 "+f"(dodd[2]), "+f"(dodd[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), "r"(c[0]), "r"(c[1]), "r"(q4_magic_lo<AFF>()),
                 "r"(q4_magic_hi<AFF>()));
}

// 8-bit codes: x = bytes b0..b3 -> (b0, b2) and (b1, b3) as fp16 (XOR 0x80,
// mantissa of 1024, minus 1152).
#define KVQ_Q8_PRE(K0, X0, X8)                                               \
  " .reg .b32 u0, u1, t, a0, a1, a2, a3;\n"                                  \
  " shr.b32 u0, " X0 ", 8;\n shr.b32 u1, " X8 ", 8;\n"                       \
  " lop3.b32 t, " X0 ", 0x00FF00FF, " K0 ", 0x6a;\n sub.rn.f16x2 a0, t, " K0 ";\n" \
  " lop3.b32 t, " X8 ", 0x00FF00FF, " K0 ", 0x6a;\n sub.rn.f16x2 a1, t, " K0 ";\n" \
  " lop3.b32 t, u0, 0x00FF00FF, " K0 ", 0x6a;\n sub.rn.f16x2 a2, t, " K0 ";\n"     \
  " lop3.b32 t, u1, 0x00FF00FF, " K0 ", 0x6a;\n sub.rn.f16x2 a3, t, " K0 ";\n"
constexpr uint32_t kQ8Magic = 0x64806480u;

// Q.K, 8-bit K: A = {x0.(b0,b2), x8.(b0,b2), x0.(b1,b3), x8.(b1,b3)}; one or two tiles.
__device__ __forceinline__ void qk8(uint32_t x0, uint32_t x8, const uint32_t (&b)[2], float (&d)[4]) {
  asm volatile("{\n" KVQ_Q8_PRE("%8", "%4", "%5") KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%6", "%7") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(x0), "r"(x8), "r"(b[0]), "r"(b[1]), "r"(kQ8Magic));
}
__device__ __forceinline__ void qk8x2(uint32_t x0, uint32_t x8, const uint32_t (&b)[2], const uint32_t (&c)[2],
                                      float (&d)[4], float (&f)[4]) {
  asm volatile("{\n" KVQ_Q8_PRE("%14", "%8", "%9") KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%10", "%11")
               KVQ_MMA("%4,%5,%6,%7", "a0", "a1", "a2", "a3", "%12", "%13") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]), "+f"(f[0]), "+f"(f[1]), "+f"(f[2]), "+f"(f[3])
               : "r"(x0), "r"(x8), "r"(b[0]), "r"(b[1]), "r"(c[0]), "r"(c[1]), "r"(kQ8Magic));
}
// P.V, 8-bit V: A = {y0.(b0,b2), y0.(b1,b3), y8.(b0,b2), y8.(b1,b3)}.
__device__ __forceinline__ void pv8(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], float (&d)[4]) {
  asm volatile("{\n" KVQ_Q8_PRE("%8", "%4", "%5") KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%6", "%7") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), "r"(kQ8Magic));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// x = hi + lo * 2^-12 with both parts in fp16: hi = fp16(x) and
// lo = fp16((x - hi) * 2^12).  The low part is stored 2^12 times larger so it
// stays in fp16's normal range as long as hi does; its products are scaled
// back by 2^-12 in fp32.
constexpr float kLoScale = 4096.0f;
__device__ __forceinline__ void split_half(float x, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(x));
  lo = (x - hi) * kLoScale;
}

}  // namespace tc
}  // namespace kvq
