// Inline-PTX helpers for the tensor-core decode kernel: ldmatrix, mma.sync,
// programmatic dependent launch, thread-block clusters, and exact code ->
// fp16 conversion fused with the MMAs.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace kvq {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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
// The two halves of a cluster barrier: arrive without ordering any memory
// access (a CTA announces that it has started), and wait for the phase.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }
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
__device__ __forceinline__ void st_cluster_f(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
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
#define KVQ_Q4_PRE(K0, K1, S0, S1, X0, X8)                                \
  " .reg .b32 u0, u1, t, a0, a1, a2, a3, e0, e1, e2, e3;\n"              \
  " shr.b32 u0, " X0 ", 8;\n shr.b32 u1, " X8 ", 8;\n"                   \
  " lop3.b32 t, " X0 ", 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a0, t, " S0 ";\n" \
  " lop3.b32 t, " X8 ", 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a1, t, " S0 ";\n" \
  " lop3.b32 t, u0, 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a2, t, " S0 ";\n"   \
  " lop3.b32 t, u1, 0x000F000F, " K0 ", 0x6a;\n sub.rn.f16x2 a3, t, " S0 ";\n"   \
  " lop3.b32 t, " X0 ", 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e0, t, " S1 ";\n" \
  " lop3.b32 t, " X8 ", 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e1, t, " S1 ";\n" \
  " lop3.b32 t, u0, 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e2, t, " S1 ";\n"   \
  " lop3.b32 t, u1, 0x00F000F0, " K1 ", 0x6a;\n sub.rn.f16x2 e3, t, " S1 ";\n"
#define KVQ_MMA(D, A0, A1, A2, A3, B0, B1)                                                       \
  " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {" D "}, {" A0 "," A1 "," A2 "," A3 "}, {" B0 \
  "," B1 "}, {" D "};\n"
// lop3 immediate 0x6a = (a & b) ^ c.  4-bit modes Q4: 0 symmetric (two's
// complement nibbles, flipped to offset binary by the XOR: K = S = n + 8 and
// 16 * (n + 8) in the mantissa of 1024), 1 affine (unsigned nibbles, no
// offset), 2 offset-binary nibbles (stored as code + 8: no flip, the offset
// subtracted).  The constants are register operands: the caller's loop holds
// them in registers instead of every block materializing them.
template <int Q4>
__device__ __forceinline__ uint32_t q4_magic_lo() { return Q4 == 0 ? 0x64086408u : 0x64006400u; }
template <int Q4>
__device__ __forceinline__ uint32_t q4_magic_hi() { return Q4 == 0 ? 0x64806480u : 0x64006400u; }
template <int Q4>
__device__ __forceinline__ uint32_t q4_sub_lo() { return Q4 == 1 ? 0x64006400u : 0x64086408u; }
template <int Q4>
__device__ __forceinline__ uint32_t q4_sub_hi() { return Q4 == 1 ? 0x64006400u : 0x64806480u; }

// The four constants of mode Q4 as input operands %N .. %N+3.
#define KVQ_Q4_IN(Q4) "r"(q4_magic_lo<Q4>()), "r"(q4_magic_hi<Q4>()), "r"(q4_sub_lo<Q4>()), "r"(q4_sub_hi<Q4>())

// Q.K, 4-bit K, one 8-column tile: 2 MMAs into d.
template <int Q4>
__device__ __forceinline__ void qk4(uint32_t x0, uint32_t x8, const uint32_t (&be)[2], const uint32_t (&bo)[2],
                                    float (&d)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%10", "%11", "%12", "%13", "%4", "%5")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%6", "%7")
               KVQ_MMA("%0,%1,%2,%3", "e0", "e1", "e2", "e3", "%8", "%9") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(x0), "r"(x8), "r"(be[0]), "r"(be[1]), "r"(bo[0]), "r"(bo[1]), KVQ_Q4_IN(Q4));
}

// Q.K, 4-bit K, B fragments of two tiles (or two passes): 4 MMAs into d / f.
template <int Q4>
__device__ __forceinline__ void qk4x2(uint32_t x0, uint32_t x8, const uint32_t (&be)[2], const uint32_t (&bo)[2],
                                      const uint32_t (&ce)[2], const uint32_t (&co)[2], float (&d)[4], float (&f)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%18", "%19", "%20", "%21", "%8", "%9")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a1", "a2", "a3", "%10", "%11")
               KVQ_MMA("%0,%1,%2,%3", "e0", "e1", "e2", "e3", "%12", "%13")
               KVQ_MMA("%4,%5,%6,%7", "a0", "a1", "a2", "a3", "%14", "%15")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e1", "e2", "e3", "%16", "%17") "}\n"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]), "+f"(f[0]), "+f"(f[1]), "+f"(f[2]), "+f"(f[3])
               : "r"(x0), "r"(x8), "r"(be[0]), "r"(be[1]), "r"(bo[0]), "r"(bo[1]), "r"(ce[0]), "r"(ce[1]),
                 "r"(co[0]), "r"(co[1]), KVQ_Q4_IN(Q4));
}

// P.V, 4-bit V (A = V^T from ldmatrix.trans): y0 = the tokens 0-7 word, y8 =
// the tokens 8-15 word.  With the names of KVQ_Q4_PRE (x0 = y0, x8 = y8),
// the even output tile (16-dim rows 4g, 4g+2) takes A = {a0, a2, a1, a3} and
// the odd one (16 x code, rows 4g+1, 4g+3) A = {e0, e2, e1, e3}.
template <int Q4>
__device__ __forceinline__ void pv4(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], float (&de)[4], float (&dodd)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%12", "%13", "%14", "%15", "%8", "%9")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%10", "%11")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%10", "%11") "}\n"
               : "+f"(de[0]), "+f"(de[1]), "+f"(de[2]), "+f"(de[3]), "+f"(dodd[0]), "+f"(dodd[1]),
                 "+f"(dodd[2]), "+f"(dodd[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), KVQ_Q4_IN(Q4));
}

// P.V, 4-bit V, one tile run twice (weights b, then c) into the same
// accumulators: the high and the low parts of the weights.
template <int Q4>
__device__ __forceinline__ void pv4m(uint32_t y0, uint32_t y8, const uint32_t (&b)[2], const uint32_t (&c)[2],
                                     float (&de)[4], float (&dodd)[4]) {
  asm volatile("{\n" KVQ_Q4_PRE("%14", "%15", "%16", "%17", "%8", "%9")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%10", "%11")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%10", "%11")
               KVQ_MMA("%0,%1,%2,%3", "a0", "a2", "a1", "a3", "%12", "%13")
               KVQ_MMA("%4,%5,%6,%7", "e0", "e2", "e1", "e3", "%12", "%13") "}\n"
               : "+f"(de[0]), "+f"(de[1]), "+f"(de[2]), "+f"(de[3]), "+f"(dodd[0]), "+f"(dodd[1]),
                 "+f"(dodd[2]), "+f"(dodd[3])
               : "r"(y0), "r"(y8), "r"(b[0]), "r"(b[1]), "r"(c[0]), "r"(c[1]), KVQ_Q4_IN(Q4));
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

}  // namespace tc
}  // namespace kvq
