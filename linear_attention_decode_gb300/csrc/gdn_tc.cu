// ReplaySSM decode with the replay sum on the 5th-generation tensor cores.
//
// One CTA of 128 threads per (row, value head).  Per CTA:
//  1. thread 0 starts the TMA stream of the fp32 checkpoint S0 [V, K] as K/32
//     boxes of [V rows x 32 columns], 128-byte swizzled in shared memory;
//  2. meanwhile all threads load q, k, v, the gates and the first p ring entries
//     and write the two replay operands in the tensor core's no-swizzle K-major
//     layout ([P1] Design 1 and 7):
//       GDN  A[v][j] = w_j d_j[v],  B[c][j] = k_j[c];
//       KDA  A[v][j] = d_j[v],      B[c][j] = w_j[c] k_j[c];
//     entries j >= p are zero (stale ring entries are never read);
//  3. one thread issues tcgen05.mma: dS[v][c] = sum_j A[v][j] B[c][j] into
//     tensor memory (M = 128 lanes = state rows, N = K columns, fp32), the L-deep
//     reconstruction contraction of [P1] Design 2;
//  4. thread r owns state row r: it reads dS[r][:] from its TMEM lane and S0[r][:]
//     from shared memory, forms S = A S0 + dS (KDA: S0 Diag(A) + dS) and
//     contracts it with q and k in registers — no cross-thread reduction;
//  5. d = beta (v - alpha Sk), out = alpha Sq + d k^T q; a flush row rewrites
//     its shared-memory S0 row with alpha S + d k^T and one TMA store per box
//     writes the new checkpoint; otherwise (d, k, g) go to the ring.
// Waits on the TMA and MMA barriers are bounded; a CTA that runs out of time
// records GDN_DEV_TIMEOUT, frees its tensor memory and returns.
#include <mutex>

#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

// KIND: tensor-core operand type (0 f16, 1 bf16, 2 tf32); RING_DT: ring storage type.
template <int D, int GATE, int KIND, int RING_DT>
__global__ void __launch_bounds__(128, 3) tc_decode_kernel(const DecodeParams P,
                                                           const __grid_constant__ CUtensorMap tmap) {
  constexpr int ES = KIND == 2 ? 4 : 2;
  constexpr int KSTEP = 32 / ES;
  constexpr int NBOX = D / 32;
  constexpr int BOX_BYTES = D * 128;
  const TcLayout lay = tc_layout(D, KIND, P.L);
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t *s0 = smem;
  uint8_t *tA = smem + lay.tA, *tB = smem + lay.tB;
  float *q = reinterpret_cast<float *>(smem + lay.fl);
  float *k = q + D, *vv = k + D, *a = vv + D, *Acol = a + D, *red = Acol + D, *wv = red + 8;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);

  const int b = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, warp = t >> 5;
  const int64_t bh = (int64_t)b * P.HV + hv;

  const RowInfo ri = resolve_row(P, b, hv == 0 && t == 0);
  if (hv == 0 && t == 0 && P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
  if (!ri.live) {  // padding row: zeros, no cache access
    if (t < D) store_from_f32(P.out, bh * D + t, P.out_dtype, 0.f);
    return;
  }
  const int slot = ri.slot, p = ri.p, hk = hv / P.G;

  if (smem_addr(smem) & 1023u) {  // the 128-byte swizzle below assumes a 1024-byte aligned base
    if (t == 0) set_status(P.status, GDN_DEV_INTERNAL);
    return;
  }
  const uint32_t bar_load = smem_addr(&bars[0]), bar_mma = smem_addr(&bars[1]);
  if (t == 0) {
    prefetch_tensormap(&tmap);
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), D);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // 1. Checkpoint stream (rows (slot*HV + hv)*V .. +V of the [N*HV*V, K] view).
  const int row0 = (slot * P.HV + hv) * D;
  if (t == 0) {
    mbar_arrive_expect_tx(bar_load, (uint32_t)(D * D * 4));
#pragma unroll
    for (int c = 0; c < NBOX; ++c) tma_load_2d(smem_addr(s0 + c * BOX_BYTES), &tmap, 32 * c, row0, bar_load);
  }

  // 2. Inputs, gates and the replay operands.
  const float kq = load_qkv<D>(P, b, hv, q, k, vv, red);  // ends with a CTA barrier
  const float v_r = t < D ? vv[t] : 0.f;
  const float beta = P.beta[bh];
  float alpha = 1.f, A = 1.f;
  if (GATE == GDN_GATE_SCALAR) alpha = expf(P.g[bh]);

  if (GATE == GDN_GATE_SCALAR) {
    if (p > 0 && t == 0)
      wv[63] = replay_decays(P.ring_g + ((int64_t)slot * P.HV + hv) * P.L, 1, p, wv, 1);
    __syncthreads();
    if (p > 0) {
      A = wv[63];
      const int64_t dbase = ((int64_t)slot * P.HV + hv) * P.L * D;
      const int64_t kbase = ((int64_t)slot * P.HK + hk) * P.L * D;
      zero_row(tA, t, lay.KC);  // A has 128 rows; rows >= D stay zero
      if (t < D) {
        zero_row(tB, t, lay.KC);
        for (int j = 0; j < p; ++j) {
          put_elem<KIND>(tA, tile_off(t, j, lay.KC, ES), wv[j] * load_as_f32(P.ring_d, dbase + (int64_t)j * D + t, RING_DT));
          put_elem<KIND>(tB, tile_off(t, j, lay.KC, ES), load_as_f32(P.ring_k, kbase + (int64_t)j * D + t, RING_DT));
        }
      }
    }
  } else {
    if (t < D) {
      const float at = expf(P.g[bh * D + t]);
      a[t] = at;
      float s = 0.f;
      if (p > 0) {
        const int64_t dbase = ((int64_t)slot * P.HV + hv) * P.L * D;
        const int64_t kbase = ((int64_t)slot * P.HK + hk) * P.L * D;
        const float *g = P.ring_g + ((int64_t)slot * P.HV + hv) * P.L * D + t;
        zero_row(tB, t, lay.KC);
        for (int j = p - 1; j >= 0; --j) {  // w_j[c] from the newest entry backwards
          const float w = expf(s);
          s += g[(int64_t)j * D];
          put_elem<KIND>(tB, tile_off(t, j, lay.KC, ES), w * load_as_f32(P.ring_k, kbase + (int64_t)j * D + t, RING_DT));
        }
        zero_row(tA, t, lay.KC);
        for (int j = 0; j < p; ++j)
          put_elem<KIND>(tA, tile_off(t, j, lay.KC, ES), load_as_f32(P.ring_d, dbase + (int64_t)j * D + t, RING_DT));
      }
      Acol[t] = expf(s);
      q[t] *= at;   // q <- a o q
      vv[t] = at * k[t];  // v slot now holds a o k (v_r is already in a register)
    } else if (p > 0) {
      zero_row(tA, t, lay.KC);
    }
  }
  fence_proxy_async_smem();  // operand tiles -> tensor-core (async) proxy
  __syncthreads();

  // 3. Replay contraction on the tensor cores.
  if (p > 0 && t == 0) {
    tc_fence_after();
    const uint32_t idesc = make_idesc(KIND, D);
    const uint32_t sbo = (uint32_t)lay.KC * 128;
    const int nsteps = (p + KSTEP - 1) / KSTEP;
    for (int i = 0; i < nsteps; ++i) {
      const uint64_t ad = make_sdesc(smem_addr(tA) + 256 * i, 128, sbo);
      const uint64_t bd = make_sdesc(smem_addr(tB) + 256 * i, 128, sbo);
      tc_mma<KIND == 2 ? 1 : 0>(tmem, ad, bd, idesc, i > 0 ? 1u : 0u);
    }
    tc_commit(bar_mma);
  }

  bool ok = mbar_wait_bounded(bar_load, 0, kWaitLimitNs);
  if (p > 0) ok = mbar_wait_bounded(bar_mma, 0, kWaitLimitNs) && ok;
  if (__syncthreads_or(!ok)) {
    if (t == 0) set_status(P.status, GDN_DEV_TIMEOUT);
    mbar_wait_bounded(bar_load, 0, kWaitLimitNs);  // let copies in flight land
    if (p > 0) mbar_wait_bounded(bar_mma, 0, kWaitLimitNs);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, D);
    return;
  }
  tc_fence_after();

  // 4./5. Row epilogue: thread t owns state row t (TMEM lane t).
  const float *qe = q;                               // GDN: q, KDA: a o q
  const float *ke = GATE == GDN_GATE_SCALAR ? k : vv;  // GDN: k, KDA: a o k
  float d = 0.f;
  if (warp < D / 32) {
    const int r = t;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float sq = 0.f, sk = 0.f;
#pragma unroll 1
    for (int c = 0; c < NBOX; ++c) {
      float acc[32];
      if (p > 0) {
        tmem_ld32(trow + 32 * c, acc);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      }
      const uint8_t *rowp = s0 + c * BOX_BYTES + r * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = *reinterpret_cast<const float4 *>(rowp + ((j ^ (r & 7)) << 4));
        const int col = 32 * c + 4 * j;
        const float4 q4 = *reinterpret_cast<const float4 *>(qe + col);
        const float4 k4 = *reinterpret_cast<const float4 *>(ke + col);
        float4 A4 = make_float4(A, A, A, A);
        if (GATE == GDN_GATE_PER_K) A4 = *reinterpret_cast<const float4 *>(Acol + col);
        const float e0 = fmaf(A4.x, x.x, acc[4 * j + 0]);
        const float e1 = fmaf(A4.y, x.y, acc[4 * j + 1]);
        const float e2 = fmaf(A4.z, x.z, acc[4 * j + 2]);
        const float e3 = fmaf(A4.w, x.w, acc[4 * j + 3]);
        sq = fmaf(e0, q4.x, sq); sk = fmaf(e0, k4.x, sk);
        sq = fmaf(e1, q4.y, sq); sk = fmaf(e1, k4.y, sk);
        sq = fmaf(e2, q4.z, sq); sk = fmaf(e2, k4.z, sk);
        sq = fmaf(e3, q4.w, sq); sk = fmaf(e3, k4.w, sk);
      }
    }
    if (GATE == GDN_GATE_SCALAR) {
      sq *= alpha;
      sk *= alpha;
    }
    d = beta * (v_r - sk);
    store_from_f32(P.out, bh * D + r, P.out_dtype, fmaf(d, kq, sq));

    if (ri.flush) {  // rebuild the row once more and overwrite S0 in place
#pragma unroll 1
      for (int c = 0; c < NBOX; ++c) {
        float acc[32];
        if (p > 0) {
          tmem_ld32(trow + 32 * c, acc);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        }
        uint8_t *rowp = s0 + c * BOX_BYTES + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 *px = reinterpret_cast<float4 *>(rowp + ((j ^ (r & 7)) << 4));
          const float4 x = *px;
          const int col = 32 * c + 4 * j;
          const float4 k4 = *reinterpret_cast<const float4 *>(k + col);
          float4 A4 = make_float4(A, A, A, A);
          float4 g4 = make_float4(alpha, alpha, alpha, alpha);
          if (GATE == GDN_GATE_PER_K) {
            A4 = *reinterpret_cast<const float4 *>(Acol + col);
            g4 = *reinterpret_cast<const float4 *>(a + col);
          }
          float4 n;
          n.x = fmaf(d, k4.x, fmaf(A4.x, x.x, acc[4 * j + 0]) * g4.x);
          n.y = fmaf(d, k4.y, fmaf(A4.y, x.y, acc[4 * j + 1]) * g4.y);
          n.z = fmaf(d, k4.z, fmaf(A4.z, x.z, acc[4 * j + 2]) * g4.z);
          n.w = fmaf(d, k4.w, fmaf(A4.w, x.w, acc[4 * j + 3]) * g4.w);
          *px = n;
        }
      }
    } else {
      store_from_f32(P.ring_d, (((int64_t)slot * P.HV + hv) * P.L + p) * D + r, RING_DT, d);
    }
  }

  if (ri.flush) {
    fence_proxy_async_smem();  // new rows -> TMA (async) proxy
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int c = 0; c < NBOX; ++c) tma_store_2d(&tmap, 32 * c, row0, smem_addr(s0 + c * BOX_BYTES));
      bulk_commit();
      bulk_wait_read_all();
    }
  } else {  // ring append of g and, once per key head, k
    if (GATE == GDN_GATE_SCALAR) {
      if (t == 0) P.ring_g[((int64_t)slot * P.HV + hv) * P.L + p] = P.g[bh];
    } else if (t < D) {
      P.ring_g[(((int64_t)slot * P.HV + hv) * P.L + p) * D + t] = P.g[bh * D + t];
    }
    if (hv % P.G == 0 && t < D)
      store_from_f32(P.ring_k, (((int64_t)slot * P.HK + hk) * P.L + p) * D + t, RING_DT, k[t]);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, D);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Operand type of the replay contraction follows the ring type: f16, bf16, or
// tf32 for an fp32 ring ([P1] Design 2).
static int kind_of(int ring_dtype) { return ring_dtype == GDN_F16 ? 0 : (ring_dtype == GDN_BF16 ? 1 : 2); }

size_t tc_smem_bytes(int D, int gate, int ring_dtype, int L) {
  (void)gate;
  return tc_layout(D, kind_of(ring_dtype), L).total;
}

template <int D, int GATE, int KIND, int RING_DT>
static cudaError_t launch_t(const DecodeParams &P, const CUtensorMap &map, size_t smem, cudaStream_t s) {
  auto kern = tc_decode_kernel<D, GATE, KIND, RING_DT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)P.B * P.HV, 128, smem, s>>>(P, map);
  return cudaGetLastError();
}

template <int D, int GATE>
static cudaError_t launch_kind(const DecodeParams &P, const CUtensorMap &map, size_t smem, int kind,
                               cudaStream_t s) {
  (void)kind;
  if (P.ring_dtype == GDN_F16) return launch_t<D, GATE, 0, GDN_F16>(P, map, smem, s);
  if (P.ring_dtype == GDN_BF16) return launch_t<D, GATE, 1, GDN_BF16>(P, map, smem, s);
  return launch_t<D, GATE, 2, GDN_F32>(P, map, smem, s);
}

cudaError_t make_state_tmap(const DecodeParams &P, int D, CUtensorMap *map, const char **why) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  // The checkpoint as a 2-D tensor [N*HV*V rows, K fp32 columns]; one box is
  // [V rows x 32 columns] = 128-byte rows, 128-byte swizzle.
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)P.N * P.HV * D};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)D};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.state, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected the checkpoint tensor";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t make_tmap_2d(const void *base, int dtype, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_rows, CUtensorMap *map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = dtype == GDN_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_tc_decode(const DecodeParams &P, int D, int gate, cudaStream_t s, const char **why,
                             bool *fused) {
  *fused = false;
  if (slab_decode_takes(P, gate)) {  // few items: the small-batch kernel spreads them over the GPU
    const cudaError_t e = launch_slab_decode(P, D, gate, s);
    *fused = e == cudaSuccess && P.sync != nullptr;
    return e;
  }
  CUtensorMap map;
  const cudaError_t em = make_state_tmap(P, D, &map, why);
  if (em != cudaSuccess) return em;
  const cudaError_t e = launch_tcp_decode(P, D, gate, map, s);
  if (e != cudaErrorNotSupported) {
    *fused = e == cudaSuccess && P.sync != nullptr;
    return e;
  }
  const int kind = kind_of(P.ring_dtype);
  const size_t smem = tc_layout(D, kind, P.L).total;
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_kind<128, 0>(P, map, smem, kind, s)
                                   : launch_kind<128, 1>(P, map, smem, kind, s);
  return gate == GDN_GATE_SCALAR ? launch_kind<64, 0>(P, map, smem, kind, s)
                                 : launch_kind<64, 1>(P, map, smem, kind, s);
}

}  // namespace gdn
