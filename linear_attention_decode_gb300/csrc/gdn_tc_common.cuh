// Helpers shared by the tensor-core decode kernels: shared-memory layout of the
// one-CTA-per-head kernel, tcgen05 instruction / shared-memory descriptors, and
// the writers of the no-swizzle K-major operand tiles.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms per barrier wait

// kind: 0 f16 operands, 1 bf16 operands, 2 tf32 operands.
struct TcLayout {
  int KD;        // padded replay depth (multiple of the per-instruction K)
  int KC;        // 16-byte chunks per operand row
  size_t tA, tB, fl, bars, total;
};

__host__ __device__ inline TcLayout tc_layout(int D, int kind, int L) {
  TcLayout t;
  const int es = kind == 2 ? 4 : 2;
  const int kstep = 32 / es;
  t.KD = L > 1 ? ((L - 1 + kstep - 1) / kstep) * kstep : 0;
  t.KC = t.KD * es / 16;
  t.tA = (size_t)D * D * 4;                       // S0 boxes first (1024-aligned)
  t.tB = t.tA + (size_t)128 * t.KD * es;          // A: 128 rows (M)
  t.fl = t.tB + (size_t)D * t.KD * es;            // B: D rows (N)
  t.bars = t.fl + (size_t)(5 * D + 8 + 64) * 4;   // q k v a Acol | red | w
  t.total = t.bars + 32;                          // 2 mbarriers + TMEM address
  return t;
}

// Instruction descriptor: D fp32, A/B f16 (0) / bf16 (1) / tf32 (2), both
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t make_idesc(int kind, int n) {
  const uint32_t ab = (uint32_t)kind;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Shared-memory matrix descriptor, no swizzle: core matrices of 8 rows x 16 B
// stored as 128 contiguous bytes; `lbo` = byte step between core matrices along
// K, `sbo` = byte step between 8-row groups.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  return d;
}

__device__ __forceinline__ uint32_t tile_off(int m, int j, int KC, int es) {
  return (uint32_t)((m >> 3) * (KC * 128) + ((j * es) >> 4) * 128 + (m & 7) * 16 + ((j * es) & 15));
}

template <int KIND>
__device__ __forceinline__ void put_elem(uint8_t *tile, uint32_t off, float x) {
  if constexpr (KIND == 0) *reinterpret_cast<__half *>(tile + off) = __float2half_rn(x);
  else if constexpr (KIND == 1) *reinterpret_cast<__nv_bfloat16 *>(tile + off) = __float2bfloat16_rn(x);
  else *reinterpret_cast<float *>(tile + off) = round_tf32(x);
}

__device__ __forceinline__ void zero_row(uint8_t *tile, int m, int KC) {
  uint8_t *row = tile + (m >> 3) * (KC * 128) + (m & 7) * 16;
  for (int h = 0; h < KC; ++h) *reinterpret_cast<uint4 *>(row + h * 128) = make_uint4(0, 0, 0, 0);
}

}  // namespace gdn
