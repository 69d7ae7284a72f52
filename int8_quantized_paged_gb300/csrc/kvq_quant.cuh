// Quantization of one (token, kv head) row, shared by the append kernel and
// the fused append + decode path, so both write the same bytes.
//
// Method: [airllm] §4.2 group_quantize (scale = amax / (2^(bits-1) - 1),
// clamp_min, round, clamp, two codes per byte with the even element low);
// [Fieldfare] "量化和精度" (affine 4-bit with bf16 scale and bias) and
// "KV Cache 的双布局设计" (K rotated before caching, V not).
//
// A warp holds the row, head_dim/32 consecutive elements per lane.  A group's
// amax (or min/max) is a butterfly over the lanes that hold it.  Every
// arithmetic step uses an explicitly rounded intrinsic, so nothing contracts
// into an FMA and the codes are bit-exact against the fp32 specification.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

// Rotates K elements lane*DPL .. lane*DPL + DPL-1 of a row at one position,
// in fp32 with one rounding per operation.  cs points at that position's
// head_dim/2 (cos, sin) pairs (a generic address: global or shared memory).
template <int DPL>
__device__ __forceinline__ void rope_rotate_row(float (&x)[DPL], const float2* cs, int rope, int lane) {
  if (rope == KVQ_ROPE_NORMAL) {   // pairs (2i, 2i+1) inside the lane's run
#pragma unroll
    for (int j = 0; j < DPL; j += 2) {
      const float2 t = cs[(lane * DPL + j) / 2];
      const float x0 = x[j], x1 = x[j + 1];
      x[j] = __fsub_rn(__fmul_rn(x0, t.x), __fmul_rn(x1, t.y));
      x[j + 1] = __fadd_rn(__fmul_rn(x0, t.y), __fmul_rn(x1, t.x));
    }
  } else if (rope == KVQ_ROPE_NEOX) {
    // Element d pairs with d + head_dim/2, which sits 16 lanes away.
    const bool low = lane < 16;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, x[j], 16);
      const float2 t = cs[(lane & 15) * DPL + j];
      if (low) {
        x[j] = __fsub_rn(__fmul_rn(x[j], t.x), __fmul_rn(other, t.y));
      } else {
        x[j] = __fadd_rn(__fmul_rn(other, t.y), __fmul_rn(x[j], t.x));
      }
    }
  }
}

// rint(fl(x / s)) (round half to even of the correctly rounded quotient), for
// |x / s| <= 2^7 + 1 and s > 0, mostly without a division: y = fl(x * r) with
// r = fl(1 / s) is within 2^-23 |x / s| + 2^-24 |x / s| of fl(x / s), under
// 2^-15 for these quotients.  So unless y lies within 2^-14 of a rounding
// boundary n + 1/2, both round to the same integer; near one the quotient is
// taken exactly.
__device__ __forceinline__ float rint_quotient(float x, float s, float r) {
  const float y = __fmul_rn(x, r);
  const float t = y - floorf(y);   // exact for |y| < 2^23
  if (fabsf(t - 0.5f) > 6.103515625e-05f) return rintf(y);
  return rintf(__fdiv_rn(x, s));
}
// The same with round half away from zero (roundf): its boundaries are the
// same half-integers.
__device__ __forceinline__ float round_quotient(float x, float s, float r) {
  const float y = __fmul_rn(x, r);
  const float t = y - floorf(y);
  if (fabsf(t - 0.5f) > 6.103515625e-05f) return roundf(y);
  return roundf(__fdiv_rn(x, s));
}

// The lane's quantized row piece: its packed code bytes (DPL/2 for 4-bit
// kinds, DPL for 8-bit, little-endian in w) and its group's parameters.
struct RowCodes {
  uint4 w;        // packed codes, low bytes first
  int nbytes;     // bytes of w that hold codes
  float scale;    // the group's stored scale (rounded to its type)
  float bias;     // affine: the group's stored bias
  int group;      // group of the lane
  bool leader;    // the first lane of its group: writes the parameters
};

// KIND, PT: the row's kind and parameter type when the caller knows them at
// compile time (the decode kernel: only that kind's code is compiled in),
// else -1 for L.kind and L.param.
template <int DPL, int KIND = -1, int PT = -1>
__device__ __forceinline__ RowCodes quantize_row(const float (&x)[DPL], const PoolLayout& L, int lane) {
  const int kind = KIND >= 0 ? KIND : L.kind;
  const int param = PT >= 0 ? PT : L.param;
  const int lpg = L.group / DPL;   // lanes per group (a power of two)
  RowCodes r;
  r.group = lane / lpg;
  r.leader = lane % lpg == 0;
  r.bias = 0.f;
  if (kind == KVQ_F16_KV) {   // unquantised: the fp16 rounding of each element, no parameters
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < DPL; ++j)
      w[j / 2] |= (uint32_t)__half_as_ushort(__float2half_rn(x[j])) << (16 * (j % 2));
    r.w = make_uint4(w[0], w[1], w[2], w[3]);
    r.nbytes = 2 * DPL;
    r.scale = 1.f;
    r.leader = false;
    return r;
  }
  int c[DPL];
  if (kind == KVQ_AFFINE_INT4) {
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int j = 1; j < DPL; ++j) { mn = fminf(mn, x[j]); mx = fmaxf(mx, x[j]); }
    for (int o = 1; o < lpg; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float scale = round_param(__fdiv_rn(__fsub_rn(mx, mn), 15.0f), param);
    const float bias = round_param(mn, param);
    const float rs = scale == 0.0f ? 0.0f : __frcp_rn(scale);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      float y = scale == 0.0f ? 0.0f : rint_quotient(__fsub_rn(x[j], bias), scale, rs);
      y = fminf(fmaxf(y, 0.0f), 15.0f);
      c[j] = (int)y;
    }
    r.scale = scale;
    r.bias = bias;
  } else if (kind == KVQ_SHIMMY_INT4) {
    // [Shimmy] §3.2: scale = max|x| / 7.5, code = clamp(round(x / scale), -8, 7)
    // (half away from zero), stored as code + 8; a zero scale gives code 0
    float amax = fabsf(x[0]);
#pragma unroll
    for (int j = 1; j < DPL; ++j) amax = fmaxf(amax, fabsf(x[j]));
    for (int o = 1; o < lpg; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = round_param(__fdiv_rn(amax, 7.5f), param);
    const float rs = scale == 0.0f ? 0.0f : __frcp_rn(scale);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      float y = scale == 0.0f ? 0.0f : round_quotient(x[j], scale, rs);
      y = fminf(fmaxf(y, -8.0f), 7.0f);
      c[j] = (int)y + 8;
    }
    r.scale = scale;
  } else {
    const float qmax = kind == KVQ_SYM_INT8 ? 127.0f : 7.0f;
    float amax = fabsf(x[0]);
#pragma unroll
    for (int j = 1; j < DPL; ++j) amax = fmaxf(amax, fabsf(x[j]));
    for (int o = 1; o < lpg; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float floor_s = param == KVQ_F16 ? 6.103515625e-05f : 1e-8f;
    const float scale = round_param(fmaxf(__fdiv_rn(amax, qmax), floor_s), param);
    const float rs = __frcp_rn(scale);
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      float y = rint_quotient(x[j], scale, rs);
      y = fminf(fmaxf(y, -qmax), qmax);
      c[j] = (int)y;
    }
    r.scale = scale;
  }
  uint32_t w[2] = {0u, 0u};
  if (kind == KVQ_SYM_INT8) {
#pragma unroll
    for (int j = 0; j < DPL; ++j) w[j / 4] |= ((uint32_t)c[j] & 0xFFu) << (8 * (j % 4));
    r.nbytes = DPL;
  } else {
#pragma unroll
    for (int j = 0; j < DPL; ++j) w[0] |= ((uint32_t)c[j] & 0xFu) << (4 * j);
    r.nbytes = DPL / 2;
  }
  r.w = make_uint4(w[0], w[1], 0u, 0u);
  return r;
}

// Byte offsets of a group's scale and (affine) bias inside a parameter row
// (KIND, PT as for quantize_row).
template <int KIND = -1, int PT = -1>
__device__ __forceinline__ int param_scale_offset(const PoolLayout& L, int g) {
  const int kind = KIND >= 0 ? KIND : L.kind;
  return (kind == KVQ_AFFINE_INT4 ? 2 * g : g) * param_bytes(PT >= 0 ? PT : L.param);
}
template <int PT = -1>
__device__ __forceinline__ int param_bias_offset(const PoolLayout& L, int g) {
  return (2 * g + 1) * param_bytes(PT >= 0 ? PT : L.param);
}

// Writes `nbytes` (1, 2, 4, 8 or 16) low bytes of w at p, which is aligned to nbytes.
__device__ __forceinline__ void store_code_bytes(uint8_t* p, uint4 w, int nbytes) {
  if (nbytes == 1) {
    *p = (uint8_t)w.x;
  } else if (nbytes == 2) {
    *reinterpret_cast<unsigned short*>(p) = (unsigned short)w.x;
  } else if (nbytes == 4) {
    *reinterpret_cast<uint32_t*>(p) = w.x;
  } else if (nbytes == 8) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w.x, w.y);
  } else {
    *reinterpret_cast<uint4*>(p) = w;
  }
}

// Writes the lane's codes and (group leaders) parameters of token row `slot`
// into a page sub-block in global memory: [P][code_bytes] then
// [P][param_row_bytes] (KIND, PT as for quantize_row).
template <int KIND = -1, int PT = -1>
__device__ __forceinline__ void store_row(const RowCodes& r, const PoolLayout& L, uint8_t* sub, int slot,
                                          int lane) {
  constexpr int P = 16;
  const int kind = KIND >= 0 ? KIND : L.kind;
  const int param = PT >= 0 ? PT : L.param;
  store_code_bytes(sub + slot * L.code_bytes + lane * r.nbytes, r.w, r.nbytes);
  uint8_t* prow = sub + P * L.code_bytes + slot * L.param_row_bytes;
  if (r.leader) {
    store_param(prow + param_scale_offset<KIND, PT>(L, r.group), param, r.scale);
    if (kind == KVQ_AFFINE_INT4) store_param(prow + param_bias_offset<PT>(L, r.group), param, r.bias);
  }
}

}  // namespace kvq
