// Persistent, warp-specialised ReplaySSM decode on the 5th-generation tensor
// cores.  One CTA per SM walks a round-robin share of the (row, value head)
// items.
//
// Roles (448 threads):
//   warp 0       producer: for each item, once its info stage is free, bulk-copies
//                the first p ring entries (d, k; KDA also g) and, when aligned,
//                the q, k, v vectors into the stage's landing zone (land barrier),
//                then streams the fp32 checkpoint S0 [V, K] by TMA one [V x 32]
//                box (128-byte swizzled) at a time through a ring of NB box slots
//                (box_full / box_empty barriers);
//   warp 1       allocates 2 x K TMEM columns (two accumulators) and issues the
//                replay contraction tcgen05.mma for each item into one of them;
//   warps 2-9    two prep warpgroups taking alternate items: from the landing
//                zone they compute the replay decays and write the two K-major
//                operand tiles ([P1] Design 1 and 7)
//                      GDN  A[v][j] = w_j d_j[v],  B[c][j] = k_j[c]
//                      KDA  A[v][j] = d_j[v],      B[c][j] = w_j[c] k_j[c]
//                plus the epilogue's vectors (info_full barrier);
//   warps 10-13  epilogue: thread r owns state row r (TMEM lane r).  It adds
//                A S0[r][:] (KDA: S0[r][:] o A) to dS[r][:] from TMEM, contracts
//                with q and k in registers, writes out[r] = alpha Sq + d (k^T q)
//                with d = beta (v - alpha Sk); a flush item rewrites its box rows
//                with alpha S + d k^T and TMA-stores them, otherwise (d, k, g) are
//                appended to the ring.  It then frees the stage (info_empty).
// Every wait is bounded: a wait that runs out raises a CTA-wide abort flag and
// GDN_DEV_TIMEOUT; all roles then leave their loops, the producer and the MMA
// thread wait (bounded) for their own copies and contraction still in flight,
// and the CTA frees its TMEM and returns.
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

constexpr int kTcpThreads = 448;
constexpr int kItemsMax = 256;  // items one CTA may own (sets the table size)
#ifndef GDN_TCP_STAGES
#define GDN_TCP_STAGES 3  // info stages (operand tiles + landing zone) in flight
#endif


struct TcpLayout {
  int KD, KC, NI, NB;
  int qkv_bulk;  // 1: q, k, v arrive by bulk copy (16-byte aligned rows)
  uint32_t box_bytes, stage_bytes;
  uint32_t off_stage, off_table, off_bars, total;
  // offsets inside an info stage
  uint32_t st_A, st_B, st_f, st_ld, st_lk, st_lg, st_lq;
};

// Shared memory: NB checkpoint boxes | NI info stages | item table | barriers.
// An info stage: A tile | B tile | fp32 vectors | landing zone (d rows, k rows,
// KDA g rows, q k v).
static TcpLayout tcp_layout(int D, int kind, int gate, int L, int ring_bytes, int qkv_bytes, int qkv_bulk,
                            int smem_budget) {
  TcpLayout t{};
  const int es = kind == 2 ? 4 : 2;
  const int kstep = 32 / es;
  const int depth = L > 1 ? L - 1 : 0;
  t.KD = depth ? ((depth + kstep - 1) / kstep) * kstep : 0;
  t.KC = t.KD * es / 16;
  t.qkv_bulk = qkv_bulk;
  t.box_bytes = (uint32_t)D * 128;
  t.st_A = 0;
  t.st_B = (uint32_t)(128 * t.KD * es);
  t.st_f = t.st_B + (uint32_t)(D * t.KD * es);
  t.st_ld = t.st_f + (uint32_t)(7 * D + 144) * 4;
  t.st_lk = t.st_ld + (uint32_t)(depth * D * ring_bytes);
  t.st_lg = t.st_lk + (uint32_t)(depth * D * ring_bytes);
  t.st_lq = t.st_lg + (uint32_t)(gate == GDN_GATE_PER_K ? depth * D * 4 : 0);
  t.stage_bytes = t.st_lq + (uint32_t)(qkv_bulk ? 3 * D * qkv_bytes : 0);
  t.stage_bytes = (t.stage_bytes + 127) & ~127u;
  const uint32_t table = (uint32_t)kItemsMax * 8;
  const uint32_t bars = 512;
  t.NI = GDN_TCP_STAGES;
  const long rest = (long)smem_budget - (long)t.NI * t.stage_bytes - table - bars;
  t.NB = rest > 0 ? (int)(rest / t.box_bytes) : 0;
  if (t.NB > 16) t.NB = 16;
  t.off_stage = (uint32_t)t.NB * t.box_bytes;
  t.off_table = t.off_stage + (uint32_t)t.NI * t.stage_bytes;
  t.off_bars = t.off_table + table;
  t.total = t.off_bars + bars;
  return t;
}

struct TcpBars {
  uint32_t box_full, box_empty, land, info_full, info_empty, tmem_full, tmem_empty;
  __device__ uint32_t bf(int i) const { return box_full + 8 * i; }
  __device__ uint32_t be(int i) const { return box_empty + 8 * i; }
  __device__ uint32_t ld(int i) const { return land + 8 * i; }
  __device__ uint32_t inf(int i) const { return info_full + 8 * i; }
  __device__ uint32_t ine(int i) const { return info_empty + 8 * i; }
  __device__ uint32_t tf(int i) const { return tmem_full + 8 * i; }
  __device__ uint32_t te(int i) const { return tmem_empty + 8 * i; }
};

// Bounded wait that also gives up when another thread raised the abort flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1u;
      set_status(status, GDN_DEV_TIMEOUT);
      return false;
    }
  }
}

// Sum of x and y over one 128-thread warpgroup (named barrier `bar_id`).
__device__ __forceinline__ float2 group_sum2(float x, float y, float *red, uint32_t bar_id, int pt) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  if ((pt & 31) == 0) {
    red[pt >> 5] = x;
    red[4 + (pt >> 5)] = y;
  }
  named_bar_sync(bar_id, 128);
  float2 r = make_float2((red[0] + red[1]) + (red[2] + red[3]), (red[4] + red[5]) + (red[6] + red[7]));
  named_bar_sync(bar_id, 128);
  return r;
}

template <int KIND>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (KIND == 0) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// Writes one 16-byte chunk (elements h*EPC .. h*EPC+EPC-1 of K-major row m).
template <int KIND, int EPC>
__device__ __forceinline__ void put_chunk(uint8_t *tile, int m, int h, int KC, const float (&x)[EPC]) {
  uint4 v;
  if constexpr (KIND == 2) {
    v = make_uint4(__float_as_uint(round_tf32(x[0])), __float_as_uint(round_tf32(x[1])),
                   __float_as_uint(round_tf32(x[2])), __float_as_uint(round_tf32(x[3])));
  } else {
    v = make_uint4(pack2<KIND>(x[0], x[1]), pack2<KIND>(x[2], x[3]), pack2<KIND>(x[4], x[5]),
                   pack2<KIND>(x[6], x[7]));
  }
  *reinterpret_cast<uint4 *>(tile + (m >> 3) * (KC * 128) + h * 128 + (m & 7) * 16) = v;
}

template <int D, int GATE, int KIND, int RING_DT>
__global__ void __launch_bounds__(kTcpThreads, 1)
    tcp_decode_kernel(const DecodeParams P, const __grid_constant__ CUtensorMap tmap, const TcpLayout lay) {
  constexpr int ES = KIND == 2 ? 4 : 2;
  constexpr int KSTEP = 32 / ES;
  constexpr int EPC = 16 / ES;  // operand elements per 16-byte chunk
  constexpr int NBOX = D / 32;
  constexpr int BOX_BYTES = D * 128;
  constexpr int RB = RING_DT == GDN_F32 ? 4 : 2;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Items (row b, value head hv) = b * HV + hv are dealt round-robin: CTA c takes
  // c, c + G, c + 2G, ...  A flushing row's heads (about twice the work) thus
  // spread over HV different CTAs instead of piling up on one or two.
  const int T = P.B * P.HV;
  const int G = gridDim.x;
  const int n = (int)blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / G + 1 : 0;
  const int NB = lay.NB, NI = lay.NI;
  const int qes = P.qkv_dtype == GDN_F32 ? 4 : 2;

  if (smem_addr(smem) & 1023u) {  // the 128-byte swizzle assumes a 1024-byte aligned base
    if (tid == 0) set_status(P.status, GDN_DEV_INTERNAL);
    return;
  }
  int2 *table = reinterpret_cast<int2 *>(smem + lay.off_table);
  uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + lay.off_bars);
  const uint32_t bar0 = smem_addr(bar_mem);
  const TcpBars bars{bar0,
                     bar0 + 8u * NB,
                     bar0 + 16u * NB,
                     bar0 + 16u * NB + 8u * NI,
                     bar0 + 16u * NB + 16u * NI,
                     bar0 + 16u * NB + 24u * NI,
                     bar0 + 16u * NB + 24u * NI + 16u};
  // Two flush barriers, used by alternate flush items: an epilogue thread can
  // run one item ahead of another, and its arrival for the next flush item must
  // not count toward the current one.
  const uint32_t flush_bar0 = bar0 + 16u * NB + 24u * NI + 32u;
  // misc[0] TMEM base, misc[1] abort flag, misc[2..3] prep-group go/stop words
  uint32_t *misc = reinterpret_cast<uint32_t *>(bar_mem + 2 * NB + 3 * NI + 6);
  volatile uint32_t *abort_flag = misc + 1;

  // --- item table: slot, cursor, flush decision of every item of this CTA ---
  for (int j = tid; j < n; j += kTcpThreads) {
    const int item = (int)blockIdx.x + j * G, b = item / P.HV, hv = item % P.HV;
    const RowInfo ri = resolve_row(P, b, hv == 0);
    if (hv == 0 && P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
    table[j] = make_int2(ri.slot, ri.p | (ri.flush << 8) | ((ri.live ? 1 : 0) << 9));
  }
  if (tid == 0) {
    for (int i = 0; i < NB; ++i) {
      mbar_init(bars.bf(i), 1);
      mbar_init(bars.be(i), 128);
    }
    for (int i = 0; i < NI; ++i) {
      mbar_init(bars.ld(i), 1);
      mbar_init(bars.inf(i), 1);
      mbar_init(bars.ine(i), 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.tf(i), 1);
      mbar_init(bars.te(i), 128);
    }
    mbar_init(flush_bar0, 128);
    mbar_init(flush_bar0 + 8u, 128);
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(misc), 2 * D);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  uint8_t *boxes = smem;
  uint8_t *stages = smem + lay.off_stage;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap);
      uint32_t use = 0;
      int li = 0, land_issued = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int2 e = table[j];
        if (!(e.y & 512)) continue;
        const int item = (int)blockIdx.x + j * G, b = item / P.HV, hv = item % P.HV, hk = hv / P.G;
        const int p = e.y & 255, slot = e.x, s = li % NI;
        const uint32_t u = (uint32_t)(li / NI);
        // landing zone of the item's info stage
        if (u > 0 && !(ok = wait_bar(bars.ine(s), (u - 1) & 1, abort_flag, P.status))) break;
        uint8_t *st = stages + s * lay.stage_bytes;
        const uint32_t ring_bytes = (uint32_t)(p * D * RB);
        const uint32_t gbytes = GATE == GDN_GATE_PER_K ? (uint32_t)(p * D * 4) : 0u;
        const uint32_t qbytes = lay.qkv_bulk ? (uint32_t)(3 * D * qes) : 0u;
        mbar_arrive_expect_tx(bars.ld(s), 2 * ring_bytes + gbytes + qbytes);
        if (p > 0) {
          const int64_t drow = ((int64_t)slot * P.HV + hv) * P.L;
          const int64_t krow = ((int64_t)slot * P.HK + hk) * P.L;
          bulk_load(smem_addr(st + lay.st_ld), (const uint8_t *)P.ring_d + drow * D * RB, ring_bytes, bars.ld(s));
          bulk_load(smem_addr(st + lay.st_lk), (const uint8_t *)P.ring_k + krow * D * RB, ring_bytes, bars.ld(s));
          if (GATE == GDN_GATE_PER_K)
            bulk_load(smem_addr(st + lay.st_lg), P.ring_g + drow * D, gbytes, bars.ld(s));
        }
        if (lay.qkv_bulk) {
          const uint8_t *row = (const uint8_t *)P.qkv + (int64_t)b * P.qkv_stride * qes;
          const uint32_t vb = (uint32_t)(D * qes);
          bulk_load(smem_addr(st + lay.st_lq), row + (int64_t)hk * vb, vb, bars.ld(s));
          bulk_load(smem_addr(st + lay.st_lq + vb), row + ((int64_t)P.HK + hk) * vb, vb, bars.ld(s));
          bulk_load(smem_addr(st + lay.st_lq + 2 * vb), row + (2 * (int64_t)P.HK + hv) * vb, vb, bars.ld(s));
        }
        ++land_issued;
        // checkpoint boxes
        const int row0 = (slot * P.HV + hv) * D;
        for (int c = 0; c < NBOX; ++c, ++use) {
          const int bs = (int)(use % NB);
          const uint32_t ub = use / NB;
          if (ub > 0 && !(ok = wait_bar(bars.be(bs), (ub - 1) & 1, abort_flag, P.status))) break;
          mbar_arrive_expect_tx(bars.bf(bs), BOX_BYTES);
          tma_load_2d(smem_addr(boxes + bs * BOX_BYTES), &tmap, 32 * c, row0, bars.bf(bs));
        }
        ++li;
      }
      if (*abort_flag) {  // let this thread's copies still in flight land first
        for (uint32_t k = use > (uint32_t)NB ? use - NB : 0u; k < use; ++k)
          mbar_wait_bounded(bars.bf((int)(k % NB)), (k / NB) & 1, kWaitLimitNs);
        for (int k = land_issued > NI ? land_issued - NI : 0; k < land_issued; ++k)
          mbar_wait_bounded(bars.ld(k % NI), (uint32_t)(k / NI) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc(KIND, D);
      const uint32_t sbo = (uint32_t)lay.KC * 128;
      int li = 0;
      for (int j = 0; j < n; ++j) {
        const int2 e = table[j];
        if (!(e.y & 512)) continue;
        const int p = e.y & 255, s = li % NI, tb = li & 1;
        const uint32_t u = (uint32_t)(li / NI), ut = (uint32_t)(li >> 1);
        if (!wait_bar(bars.inf(s), u & 1, abort_flag, P.status)) break;
        if (ut > 0 && !wait_bar(bars.te(tb), (ut - 1) & 1, abort_flag, P.status)) break;
        tc_fence_after();
        if (p > 0) {
          const uint32_t a0 = smem_addr(stages + s * lay.stage_bytes + lay.st_A);
          const uint32_t b0 = smem_addr(stages + s * lay.stage_bytes + lay.st_B);
          const int nsteps = (p + KSTEP - 1) / KSTEP;
          for (int i = 0; i < nsteps; ++i)
            tc_mma<KIND == 2 ? 1 : 0>(tmem + tb * D, make_sdesc(a0 + 256 * i, 128, sbo),
                                      make_sdesc(b0 + 256 * i, 128, sbo), idesc, i > 0 ? 1u : 0u);
          tc_commit(bars.tf(tb));
        } else {
          mbar_arrive(bars.tf(tb));
        }
        ++li;
      }
      if (*abort_flag && li > 0)  // the last contraction must finish before TMEM is freed
        mbar_wait_bounded(bars.tf((li - 1) & 1), (uint32_t)((li - 1) >> 1) & 1, kWaitLimitNs);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ prep (2 groups)
    const int grp = (warp - 2) >> 2;
    const int pt = tid - 64 - 128 * grp;
    const uint32_t bar_id = 1 + grp;
    int li = 0;
    for (int j = 0; j < n; ++j) {
      const int2 e = table[j];
      if (!(e.y & 512)) continue;
      if ((li & 1) != grp) {
        ++li;
        continue;
      }
      const int p = e.y & 255, slot = e.x, s = li % NI;
      const uint32_t u = (uint32_t)(li / NI);
      const int item = (int)blockIdx.x + j * G, b = item / P.HV, hv = item % P.HV, hk = hv / P.G;
      const int64_t bh = (int64_t)b * P.HV + hv;
      // small loads first, so their latency overlaps the landing wait
      float gc = 0.f, gj = 0.f, qv = 0.f, kv = 0.f, vv = 0.f;
      if (GATE == GDN_GATE_SCALAR) {
        gc = P.g[bh];
        if (pt < p) gj = P.ring_g[((int64_t)slot * P.HV + hv) * P.L + pt];
      } else if (pt < D) {
        gc = P.g[bh * D + pt];
      }
      const float beta = P.beta[bh];
      if (!lay.qkv_bulk && pt < D) {
        const int64_t qbase = (int64_t)b * P.qkv_stride;
        qv = load_as_f32(P.qkv, qbase + (int64_t)hk * D + pt, P.qkv_dtype);
        kv = load_as_f32(P.qkv, qbase + (int64_t)P.HK * D + (int64_t)hk * D + pt, P.qkv_dtype);
        vv = load_as_f32(P.qkv, qbase + 2 * (int64_t)P.HK * D + (int64_t)hv * D + pt, P.qkv_dtype);
      }
      // Only the group leader waits for the landing zone; the go/stop word it
      // leaves before the group barrier keeps every later group barrier uniform.
      volatile uint32_t *go = misc + 2 + grp;
      if (pt == 0) *go = wait_bar(bars.ld(s), u & 1, abort_flag, P.status) ? 1u : 0u;
      named_bar_sync(bar_id, 128);
      if (*go == 0u) break;
      uint8_t *st = stages + s * lay.stage_bytes;
      uint8_t *tA = st + lay.st_A, *tB = st + lay.st_B;
      float *f = reinterpret_cast<float *>(st + lay.st_f);
      float *fq = f, *fk = f + D, *fke = f + 2 * D, *fa = f + 3 * D, *fA = f + 4 * D, *fv = f + 5 * D,
            *fg = f + 6 * D, *gsc = f + 7 * D, *wsc = gsc + 64, *scal = wsc + 64, *red = scal + 8;
      const uint8_t *land_d = st + lay.st_ld, *land_k = st + lay.st_lk;
      const float *land_g = reinterpret_cast<const float *>(st + lay.st_lg);
      if (lay.qkv_bulk && pt < D) {
        const uint8_t *lq = st + lay.st_lq;
        qv = load_as_f32(lq, pt, P.qkv_dtype);
        kv = load_as_f32(lq, D + pt, P.qkv_dtype);
        vv = load_as_f32(lq, 2 * D + pt, P.qkv_dtype);
      }
      if (P.qk_l2norm) {
        const float2 nn = group_sum2(qv * qv, kv * kv, red, bar_id, pt);
        qv = qv / sqrtf(nn.x + 1e-6f);
        kv = kv / sqrtf(nn.y + 1e-6f);
      }
      qv *= P.q_scale;
      if (GATE == GDN_GATE_SCALAR && pt < p) gsc[pt] = gj;
      const float kq = group_sum2(kv * qv, 0.f, red, bar_id, pt).x;  // also publishes gsc

      float A = 1.f;
      if (GATE == GDN_GATE_SCALAR) {
        // w_j = exp(sum_{j<i<p} g_i), summed from the newest entry backwards
        if (pt < p) {
          float sfx = 0.f;
          for (int i = p - 1; i > pt; --i) sfx += gsc[i];
          wsc[pt] = expf(sfx);
          if (pt == 0) scal[2] = expf(sfx + gsc[0]);
        }
        named_bar_sync(bar_id, 128);
        if (p > 0) A = scal[2];
        // A row pt: w_j d_j[pt];  B row pt: k_j[pt]
        for (int h = 0; h < lay.KC; ++h) {
          float xa[EPC], xb[EPC];
#pragma unroll
          for (int e2 = 0; e2 < EPC; ++e2) {
            const int jj = h * EPC + e2;
            xa[e2] = xb[e2] = 0.f;
            if (jj < p && pt < D) {
              xa[e2] = wsc[jj] * load_as_f32(land_d, (int64_t)jj * D + pt, RING_DT);
              xb[e2] = load_as_f32(land_k, (int64_t)jj * D + pt, RING_DT);
            }
          }
          put_chunk<KIND, EPC>(tA, pt, h, lay.KC, xa);
          if (pt < D) put_chunk<KIND, EPC>(tB, pt, h, lay.KC, xb);
        }
      } else {
        // channel c = pt: w_j[c] by a backward sum over the channel's gates, so
        // the chunks of B are filled from the newest entry down
        float sfx = 0.f;
        for (int h = lay.KC - 1; h >= 0; --h) {
          float xa[EPC], xb[EPC];
#pragma unroll
          for (int e2 = EPC - 1; e2 >= 0; --e2) {
            const int jj = h * EPC + e2;
            xa[e2] = xb[e2] = 0.f;
            if (jj < p && pt < D) {
              const float wj = expf(sfx);
              sfx += land_g[jj * D + pt];
              xa[e2] = load_as_f32(land_d, (int64_t)jj * D + pt, RING_DT);
              xb[e2] = wj * load_as_f32(land_k, (int64_t)jj * D + pt, RING_DT);
            }
          }
          put_chunk<KIND, EPC>(tA, pt, h, lay.KC, xa);
          if (pt < D) put_chunk<KIND, EPC>(tB, pt, h, lay.KC, xb);
        }
        A = expf(sfx);
      }
      // Epilogue inputs.
      if (pt < D) {
        const float at = GATE == GDN_GATE_PER_K ? expf(gc) : 1.f;
        fq[pt] = GATE == GDN_GATE_PER_K ? at * qv : qv;
        fk[pt] = kv;
        fke[pt] = GATE == GDN_GATE_PER_K ? at * kv : kv;
        fa[pt] = at;
        fA[pt] = A;
        fv[pt] = vv;
        fg[pt] = gc;
      }
      if (pt == 0) {
        scal[0] = GATE == GDN_GATE_SCALAR ? expf(gc) : 1.f;
        scal[1] = beta;
        scal[2] = A;
        scal[3] = kq;
      }
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (pt == 0) mbar_arrive(bars.inf(s));
      ++li;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;  // state row = TMEM lane
    const bool row_live = r < D;   // warp-uniform
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    int li = 0;
    uint32_t use = 0, nflush = 0;
    for (int j = 0; j < n; ++j) {
      const int2 e = table[j];
      const int item = (int)blockIdx.x + j * G, b = item / P.HV, hv = item % P.HV;
      const int64_t bh = (int64_t)b * P.HV + hv;
      if (!(e.y & 512)) {
        if (row_live) store_from_f32(P.out, bh * D + r, P.out_dtype, 0.f);
        continue;
      }
      const int p = e.y & 255, slot = e.x, flush = (e.y >> 8) & 1, s = li % NI, tb = li & 1;
      const uint32_t u = (uint32_t)(li / NI), ut = (uint32_t)(li >> 1);
      if (!wait_bar(bars.inf(s), u & 1, abort_flag, P.status)) break;
      if (!wait_bar(bars.tf(tb), ut & 1, abort_flag, P.status)) break;
      tc_fence_after();
      const float *f = reinterpret_cast<const float *>(stages + s * lay.stage_bytes + lay.st_f);
      const float *fq = f, *fk = f + D, *fke = f + 2 * D, *fa = f + 3 * D, *fA = f + 4 * D, *fv = f + 5 * D,
                  *fg = f + 6 * D, *scal = f + 7 * D + 128;
      const float alpha = scal[0], beta = scal[1], A = scal[2], kq = scal[3];
      const uint32_t trow = tmem + tb * D + lane_off;
      float sq[4] = {0.f, 0.f, 0.f, 0.f}, sk[4] = {0.f, 0.f, 0.f, 0.f};
      bool ok = true;
      for (int c = 0; c < NBOX; ++c) {
        const int bs = (int)((use + c) % NB);
        if (!(ok = wait_bar(bars.bf(bs), ((use + c) / NB) & 1, abort_flag, P.status))) break;
        if (row_live) {
          float acc[32];
          if (p > 0) {
            tmem_ld32(trow + 32 * c, acc);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
          }
          const uint8_t *rowp = boxes + bs * BOX_BYTES + r * 128;
#pragma unroll
          for (int jc = 0; jc < 8; ++jc) {
            const float4 x = *reinterpret_cast<const float4 *>(rowp + ((jc ^ (r & 7)) << 4));
            const int col = 32 * c + 4 * jc;
            const float4 q4v = *reinterpret_cast<const float4 *>(fq + col);
            const float4 k4v = *reinterpret_cast<const float4 *>(fke + col);
            float4 A4 = make_float4(A, A, A, A);
            if (GATE == GDN_GATE_PER_K) A4 = *reinterpret_cast<const float4 *>(fA + col);
            const float e0 = fmaf(A4.x, x.x, acc[4 * jc + 0]);
            const float e1 = fmaf(A4.y, x.y, acc[4 * jc + 1]);
            const float e2 = fmaf(A4.z, x.z, acc[4 * jc + 2]);
            const float e3 = fmaf(A4.w, x.w, acc[4 * jc + 3]);
            sq[0] = fmaf(e0, q4v.x, sq[0]); sk[0] = fmaf(e0, k4v.x, sk[0]);
            sq[1] = fmaf(e1, q4v.y, sq[1]); sk[1] = fmaf(e1, k4v.y, sk[1]);
            sq[2] = fmaf(e2, q4v.z, sq[2]); sk[2] = fmaf(e2, k4v.z, sk[2]);
            sq[3] = fmaf(e3, q4v.w, sq[3]); sk[3] = fmaf(e3, k4v.w, sk[3]);
          }
        }
        if (!flush) mbar_arrive(bars.be(bs));
      }
      if (!ok) break;
      float sqt = (sq[0] + sq[1]) + (sq[2] + sq[3]);
      float skt = (sk[0] + sk[1]) + (sk[2] + sk[3]);
      if (GATE == GDN_GATE_SCALAR) {
        sqt *= alpha;
        skt *= alpha;
      }
      const float v_r = row_live ? fv[r] : 0.f;
      const float d = beta * (v_r - skt);
      if (row_live) store_from_f32(P.out, bh * D + r, P.out_dtype, fmaf(d, kq, sqt));
      const int hk = hv / P.G;
      if (flush) {
        if (row_live) {
          for (int c = 0; c < NBOX; ++c) {
            const int bs = (int)((use + c) % NB);
            float acc[32];
            if (p > 0) {
              tmem_ld32(trow + 32 * c, acc);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            }
            uint8_t *rowp = boxes + bs * BOX_BYTES + r * 128;
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {
              float4 *px = reinterpret_cast<float4 *>(rowp + ((jc ^ (r & 7)) << 4));
              const float4 x = *px;
              const int col = 32 * c + 4 * jc;
              const float4 k4 = *reinterpret_cast<const float4 *>(fk + col);
              float4 A4 = make_float4(A, A, A, A), g4 = make_float4(alpha, alpha, alpha, alpha);
              if (GATE == GDN_GATE_PER_K) {
                A4 = *reinterpret_cast<const float4 *>(fA + col);
                g4 = *reinterpret_cast<const float4 *>(fa + col);
              }
              float4 nv;
              nv.x = fmaf(d, k4.x, fmaf(A4.x, x.x, acc[4 * jc + 0]) * g4.x);
              nv.y = fmaf(d, k4.y, fmaf(A4.y, x.y, acc[4 * jc + 1]) * g4.y);
              nv.z = fmaf(d, k4.z, fmaf(A4.z, x.z, acc[4 * jc + 2]) * g4.z);
              nv.w = fmaf(d, k4.w, fmaf(A4.w, x.w, acc[4 * jc + 3]) * g4.w);
              *px = nv;
            }
          }
        }
        fence_proxy_async_smem();
        const uint32_t fbar = flush_bar0 + 8u * (nflush & 1);
        mbar_arrive(fbar);
        if (tid == 320) {  // one thread stores the rewritten boxes once all rows are in
          if (!wait_bar(fbar, (nflush >> 1) & 1, abort_flag, P.status)) break;
          const int row0 = (slot * P.HV + hv) * D;
          for (int c = 0; c < NBOX; ++c)
            tma_store_2d(&tmap, 32 * c, row0, smem_addr(boxes + (int)((use + c) % NB) * BOX_BYTES));
          bulk_commit();
          bulk_wait_read_all();
          for (int c = 0; c < NBOX; ++c) mbar_arrive_count(bars.be((int)((use + c) % NB)), 128);
        }
        ++nflush;
      } else {
        if (row_live) {
          store_from_f32(P.ring_d, (((int64_t)slot * P.HV + hv) * P.L + p) * D + r, RING_DT, d);
          if (GATE == GDN_GATE_PER_K) P.ring_g[(((int64_t)slot * P.HV + hv) * P.L + p) * D + r] = fg[r];
          if (hv % P.G == 0)
            store_from_f32(P.ring_k, (((int64_t)slot * P.HK + hk) * P.L + p) * D + r, RING_DT, fk[r]);
        }
        if (GATE == GDN_GATE_SCALAR && tid == 320) P.ring_g[((int64_t)slot * P.HV + hv) * P.L + p] = fg[0];
      }
      tc_fence_before();
      mbar_arrive(bars.te(tb));
      mbar_arrive(bars.ine(s));
      use += NBOX;
      ++li;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * D);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

static int device_attr(cudaDeviceAttr a) {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, a, dev);
  return v;
}

template <int D, int GATE, int KIND, int RING_DT>
static cudaError_t launch_tcp_t(const DecodeParams &P, const CUtensorMap &map, const TcpLayout &lay,
                                int grid, cudaStream_t s) {
  auto kern = tcp_decode_kernel<D, GATE, KIND, RING_DT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcpThreads, lay.total, s>>>(P, map, lay);
  return cudaGetLastError();
}

template <int D, int GATE>
static cudaError_t launch_tcp_ring(const DecodeParams &P, const CUtensorMap &map, const TcpLayout &lay,
                                   int grid, cudaStream_t s) {
  if (P.ring_dtype == GDN_F16) return launch_tcp_t<D, GATE, 0, GDN_F16>(P, map, lay, grid, s);
  if (P.ring_dtype == GDN_BF16) return launch_tcp_t<D, GATE, 1, GDN_BF16>(P, map, lay, grid, s);
  return launch_tcp_t<D, GATE, 2, GDN_F32>(P, map, lay, grid, s);
}

// Returns cudaErrorNotSupported (nothing launched) when the persistent layout
// does not fit; the caller then uses the one-CTA-per-head kernel.
cudaError_t launch_tcp_decode(const DecodeParams &P, int D, int gate, const CUtensorMap &map,
                              cudaStream_t s) {
  static const int sms = device_attr(cudaDevAttrMultiProcessorCount);
  static const int optin = device_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin);
  const int kind = P.ring_dtype == GDN_F16 ? 0 : (P.ring_dtype == GDN_BF16 ? 1 : 2);
  const int ring_bytes = P.ring_dtype == GDN_F32 ? 4 : 2;
  const int qes = P.qkv_dtype == GDN_F32 ? 4 : 2;
  // q, k, v rows can be bulk-copied when every vector starts on 16 bytes
  const int qkv_bulk =
      ((reinterpret_cast<uintptr_t>(P.qkv) & 15u) == 0 && ((P.qkv_stride * qes) & 15) == 0) ? 1 : 0;
  if (gate == GDN_GATE_PER_K && (reinterpret_cast<uintptr_t>(P.ring_g) & 15u) != 0) return cudaErrorNotSupported;
  const int T = P.B * P.HV;
  int grid = sms > 0 && sms < T ? sms : T;
  if ((T + grid - 1) / grid > kItemsMax) grid = (T + kItemsMax - 1) / kItemsMax;
  const TcpLayout lay = tcp_layout(D, kind, gate, P.L, ring_bytes, qes, qkv_bulk, optin);
  if (lay.NB < D / 32 + 1 || lay.total > (uint32_t)optin) return cudaErrorNotSupported;
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_tcp_ring<128, 0>(P, map, lay, grid, s)
                                   : launch_tcp_ring<128, 1>(P, map, lay, grid, s);
  return gate == GDN_GATE_SCALAR ? launch_tcp_ring<64, 0>(P, map, lay, grid, s)
                                 : launch_tcp_ring<64, 1>(P, map, lay, grid, s);
}

}  // namespace gdn
