// Device-side helpers shared by the kvq kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {

__device__ __forceinline__ float load_act(const void* p, int act, int64_t i) {
  if (act == KVQ_F32) return static_cast<const float*>(p)[i];
  if (act == KVQ_F16) return __half2float(static_cast<const __half*>(p)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ void store_act(void* p, int act, int64_t i, float v) {
  if (act == KVQ_F32) {
    static_cast<float*>(p)[i] = v;
  } else if (act == KVQ_F16) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
}

// A stored scale or bias (little-endian f32 / f16 / bf16) as float.
__device__ __forceinline__ float load_param(const uint8_t* p, int param) {
  if (param == KVQ_F32) return *reinterpret_cast<const float*>(p);
  const unsigned short u = *reinterpret_cast<const unsigned short*>(p);
  if (param == KVQ_F16) return __half2float(__ushort_as_half(u));
  return __uint_as_float((uint32_t)u << 16);
}

// Round an fp32 value to the stored parameter type (nearest, ties to even).
__device__ __forceinline__ float round_param(float v, int param) {
  if (param == KVQ_F32) return v;
  if (param == KVQ_F16) return __half2float(__float2half_rn(v));
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void store_param(uint8_t* p, int param, float v) {
  if (param == KVQ_F32) {
    *reinterpret_cast<float*>(p) = v;
  } else if (param == KVQ_F16) {
    *reinterpret_cast<unsigned short*>(p) = __half_as_ushort(__float2half_rn(v));
  } else {
    *reinterpret_cast<unsigned short*>(p) = (unsigned short)(__float_as_uint(v) >> 16);
  }
}

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Integer code value of element k of a packed word as float, exactly.  The
// code is placed in the mantissa of 2^23 and 2^23 (+ offset) subtracted.
// Symmetric 4-bit: two's-complement nibble; XOR 8 maps it to offset binary.
__device__ __forceinline__ float code_sym4(uint32_t w, int k) {
  const uint32_t n = ((w >> (4 * k)) & 0xFu) ^ 0x8u;
  return __uint_as_float(0x4B000000u | n) - 8388616.0f;   // 2^23 + 8
}
__device__ __forceinline__ float code_aff4(uint32_t w, int k) {
  const uint32_t n = (w >> (4 * k)) & 0xFu;
  return __uint_as_float(0x4B000000u | n) - 8388608.0f;   // 2^23
}
__device__ __forceinline__ float code_sym8(uint32_t w, int k) {
  const uint32_t n = ((w >> (8 * k)) & 0xFFu) ^ 0x80u;
  return __uint_as_float(0x4B000000u | n) - 8388736.0f;   // 2^23 + 128
}

template <int KIND>
__device__ __forceinline__ float code_at(const uint32_t* w, int i) {
  if constexpr (KIND == KVQ_SYM_INT8) {
    return code_sym8(w[i >> 2], i & 3);
  } else if constexpr (KIND == KVQ_AFFINE_INT4) {
    return code_aff4(w[i >> 3], i & 7);
  } else {
    return code_sym4(w[i >> 3], i & 7);
  }
}

// Load NB bytes (2, 4, 8 or a multiple of 16; naturally aligned) into words.
template <int NB>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t* w) {
  if constexpr (NB >= 16) {
#pragma unroll
    for (int i = 0; i < NB / 16; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  } else if constexpr (NB == 8) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (NB == 4) {
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  } else {
    static_assert(NB == 2, "NB");
    w[0] = __ldg(reinterpret_cast<const unsigned short*>(p));
  }
}

}  // namespace kvq
