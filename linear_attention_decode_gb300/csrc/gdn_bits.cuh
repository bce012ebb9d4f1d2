// Window input loads as raw storage bits: a loop over a window's tokens issues
// every load first and converts afterwards, so the loads are in flight together
// (a conversion right after each load would make the thread wait for it before
// the next token's loads).
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Raw storage bits of one element (fp32, or bf16 / fp16 zero-extended): a
// loop can issue many such loads before converting any, so they are in flight
// together (a conversion right after each load would wait for it).
__device__ __forceinline__ uint32_t load_bits(const void *p, int64_t i, int dtype) {
  if (dtype == GDN_F32) return reinterpret_cast<const uint32_t *>(p)[i];
  return reinterpret_cast<const uint16_t *>(p)[i];
}

__device__ __forceinline__ float bits_to_f32(uint32_t x, int dtype) {
  if (dtype == GDN_BF16) return __uint_as_float(x << 16);  // bf16 is the high half of an fp32
  if (dtype == GDN_F16) return __half2float(__ushort_as_half((unsigned short)x));
  return __uint_as_float(x);
}

// The same inputs as raw storage bits (converted by bits_to_f32 later).
struct QkvBits {
  uint32_t q, k, v;
};

template <int D>
__device__ __forceinline__ QkvBits load_qkv_bits(const DecodeParams &P, int b, int hv) {
  const int t = threadIdx.x;
  const int hk = hv / P.G;
  const int64_t base = (int64_t)b * P.qkv_stride;
  QkvBits x{0u, 0u, 0u};
  if (t < D) {
    x.q = load_bits(P.qkv, base + (int64_t)hk * D + t, P.qkv_dtype);
    x.k = load_bits(P.qkv, base + (int64_t)P.HK * D + (int64_t)hk * D + t, P.qkv_dtype);
    x.v = load_bits(P.qkv, base + 2 * (int64_t)P.HK * D + (int64_t)hv * D + t, P.qkv_dtype);
  }
  return x;
}

__device__ __forceinline__ QkvRaw qkv_from_bits(QkvBits x, int dtype) {
  return QkvRaw{bits_to_f32(x.q, dtype), bits_to_f32(x.k, dtype), bits_to_f32(x.v, dtype)};
}

}  // namespace gdn
