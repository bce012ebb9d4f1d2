// Small-batch ReplaySSM decode: one block per (row, value head, slab of R
// state rows), so a batch with few (row, head) items still spreads over the
// whole GPU (B = 1, HV = 32, K = V = 128: 256 blocks of 16 rows).  A block does
// the whole step for its rows on the CUDA cores in fp32 ([P1] Modifications,
// Design 1/3/5/7; [P2] 3.2, 3.3):
//   S[r] = A S0[r] + sum_{j<p} w_j d_j[r] k_j      (KDA: S0[r] o A + sum_j d_j[r] (w_j o k_j))
//   GDN: Sq_r, Sk_r <- alpha S[r].q, alpha S[r].k;  KDA: S[r].(a o q), S[r].(a o k)
//   d_r = beta (v_r - Sk_r);  out_r = Sq_r + d_r (k^T q)
//   flush: S_new[r] = alpha S[r] + d_r k          (KDA: S[r] o a + d_r k)
//   else:  ring_d[p][r] = d_r; the slab-0 blocks append k (one per key head) and g.
// A small batch is latency-bound, so the block keeps its chain of dependent
// memory round trips short: the step's inputs are requested first (they depend
// on the block alone); as soon as the row's slot is known, one thread issues
// bulk copies of the block's checkpoint rows and of every ring entry the slot
// holds (L - 1 of them, without waiting for the cursor: entries at or past the
// cursor are selected away, never multiplied) into shared memory, beside the
// cursor load.  Thread layout of the readout: 8 lanes per state row (a warp
// holds 4 rows), each lane 4 consecutive columns in every 32-column group, so a
// row's sums over K are 3-step shuffles.
//
// With P.sync (decode + advance in one launch) the thread that read the cursor
// counts the block; the last block to count advances every row's cursor
// ([P1] Design 3) and leaves the counter at zero.
#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

constexpr int kSlabRows = 16;     // state rows the block's threads cover at a time
constexpr int kSlabThreads = 128;

// Shared memory, in bytes: the checkpoint rows [R][D] fp32 (first, 16-byte
// aligned); ring d [L-1][R] and ring k [L-1][D] as copied (ring type); KDA ring
// g [L-1][D] fp32; for a 16-bit ring, fp32 copies of d [L-1][R] and k
// [L-1][D] (an fp32 ring is used in place); then q, k, a, A [D], v [R],
// decays [64], scratch [16] floats; one mbarrier.
struct SlabLayout {
  uint32_t off_d, off_k, off_g, off_d32, off_k32, off_f, off_bar, total;
};
__host__ __device__ inline SlabLayout slab_layout(int D, int R, int L, int rb, int gate) {
  SlabLayout t;
  // entries are padded to a multiple of four (zero operands), for the
  // replay loop's four-entry steps
  const uint32_t depth = L > 1 ? (((uint32_t)(L - 1) + 3u) & ~3u) : 0u;
  t.off_d = (uint32_t)R * D * 4;
  t.off_k = t.off_d + ((depth * R * rb + 15u) & ~15u);
  t.off_g = t.off_k + depth * D * rb;
  t.off_d32 = t.off_g + (gate == GDN_GATE_PER_K ? depth * D * 4 : 0u);
  t.off_k32 = t.off_d32 + (rb == 2 ? depth * R * 4 : 0u);
  t.off_f = t.off_k32 + (rb == 2 ? depth * D * 4 : 0u);
  t.off_bar = t.off_f + (((uint32_t)(4 * D + R + 64 + 16) * 4 + 15u) & ~15u);
  t.total = t.off_bar + 16;
  return t;
}

// Block (item, slab): rows slab * R .. slab * R + R - 1 of item (row b, value
// head hv), R = D / NS.
template <int D, int GATE, int RING_DT>
__global__ void __launch_bounds__(kSlabThreads, 4) slab_decode_kernel(const DecodeParams P, const int NS) {
  constexpr int M = D / 32;  // float4 chunks per lane per row
  constexpr int RB = RING_DT == GDN_F32 ? 4 : 2;
  const int R = D / NS;
  const int item = blockIdx.x / NS, slab = blockIdx.x % NS;
  const int b = item / P.HV, hv = item % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rl = t >> 3, cg = t & 7;  // state row within the 16 at hand, column group
  const int row0 = slab * R;
  const int depth = P.L > 1 ? P.L - 1 : 0;
  constexpr int rb = RB;
  const SlabLayout lay = slab_layout(D, R, P.L, rb, GATE);
  extern __shared__ __align__(16) uint8_t slab_smem[];
  const float *sS0 = reinterpret_cast<const float *>(slab_smem);
  uint8_t *sD = slab_smem + lay.off_d, *sK = slab_smem + lay.off_k;
  const float *sG = reinterpret_cast<const float *>(slab_smem + lay.off_g);
  // the replay operands in fp32: Dw[j][rr] = d_j (GDN: times w_j in the loop),
  // Kw[j][c] = k_j[c] (KDA: w_j[c] k_j[c]); a 16-bit ring is converted into its
  // own arrays, an fp32 ring in place
  float *Dw = reinterpret_cast<float *>(RB == 4 ? sD : slab_smem + lay.off_d32);
  float *Kw = reinterpret_cast<float *>(RB == 4 ? sK : slab_smem + lay.off_k32);
  float *q = reinterpret_cast<float *>(slab_smem + lay.off_f);
  float *k = q + D, *a = k + D, *Acol = a + D, *v = Acol + D, *wv = v + R, *red = wv + 64;
  int *rinfo = reinterpret_cast<int *>(red + 12);
  const uint32_t bar = smem_addr(slab_smem + lay.off_bar);
  const int64_t bh = (int64_t)b * P.HV + hv;
  const int hk = hv / P.G;

  // Without GDN_STEP_OVERLAP_PREVIOUS nothing is read before the previous
  // launch has completed, and the step's inputs are requested first.  With it
  // the row, its cursor, the checkpoint rows and the ring are read first (the
  // caller states that launch leaves them alone); the inputs and every write
  // come after the wait.
  const bool overlap = P.overlap != 0;
  float qt = 0.f, kt = 0.f, gt = 0.f, beta = 0.f, gs = 0.f;
  const int64_t base = (int64_t)b * P.qkv_stride;
  auto load_inputs = [&]() {
    if (t < D) {
      float unused;
      load3_as_f32(P.qkv, base + (int64_t)hk * D + t, base + (int64_t)P.HK * D + (int64_t)hk * D + t,
                   base + (int64_t)P.HK * D + (int64_t)hk * D + t, P.qkv_dtype, qt, kt, unused);
      if (GATE == GDN_GATE_PER_K) gt = P.g[bh * D + t];
    }
    if (t < R) v[t] = load_as_f32(P.qkv, base + 2 * (int64_t)P.HK * D + (int64_t)hv * D + row0 + t, P.qkv_dtype);
    beta = P.beta[bh];
    if (GATE == GDN_GATE_SCALAR) gs = P.g[bh];
  };
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (!overlap) {
    grid_dependency_wait();
    grid_launch_dependents();
    load_inputs();
  }
  // Thread 0 reads the row's slot, starts the copies, then reads the cursor
  // and hands everything to the block (decode + advance counts the block once
  // that read is done: a cursor read by any other thread could come after the
  // last block has moved it).  The count's result is looked at only at the
  // end, so its round trip hides behind the work.
  uint32_t ticket = 0u;
  if (t == 0) {
    const int slot = __ldcg(P.idx + b);
    const bool ok = slot >= 0 && slot < P.N;
    if (ok) {
      const int64_t drow = ((int64_t)slot * P.HV + hv) * P.L, krow = ((int64_t)slot * P.HK + hk) * P.L;
      const uint32_t s0b = (uint32_t)R * D * 4, db = (uint32_t)R * rb, kb = (uint32_t)(depth * D * rb);
      const uint32_t gb = GATE == GDN_GATE_PER_K ? (uint32_t)(depth * D * 4) : 0u;
      mbar_arrive_expect_tx(bar, s0b + (uint32_t)depth * db + kb + gb);
      bulk_load(smem_addr(slab_smem), P.state + (((int64_t)slot * P.HV + hv) * D + row0) * D, s0b, bar);
      for (int j = 0; j < depth; ++j)
        bulk_load(smem_addr(sD + j * db), (const uint8_t *)P.ring_d + ((drow + j) * D + row0) * rb, db, bar);
      if (depth > 0) {
        bulk_load(smem_addr(sK), (const uint8_t *)P.ring_k + krow * D * rb, kb, bar);
        if (GATE == GDN_GATE_PER_K) bulk_load(smem_addr(sG), P.ring_g + drow * D, gb, bar);
      }
    }
    RowInfo r0{-1, 0, 0, false, 0u};
    if (slot >= P.N) {
      r0.bad = GDN_DEV_BAD_SLOT;
    } else if (ok) {
      const int p = __ldcg(P.write_pos + slot);
      if (p < 0 || p >= P.L) {
        r0.bad = GDN_DEV_BAD_WRITE_POS;
      } else {
        r0 = RowInfo{slot, p, (p == P.L - 1) || (P.force_flush != nullptr && __ldcg(P.force_flush + b) != 0), true,
                     0u};
      }
    }
    rinfo[0] = r0.slot;
    rinfo[1] = r0.p | (r0.flush << 8) | ((r0.live ? 1 : 0) << 9) | (ok ? 1 << 10 : 0);
    rinfo[2] = (int)r0.bad;
    if (P.sync && !overlap) ticket = atomic_add_release_gpu(P.sync, 1u);
  }
  __syncthreads();
  RowInfo ri;
  ri.slot = rinfo[0];
  ri.p = rinfo[1] & 255;
  ri.flush = (rinfo[1] >> 8) & 1;
  ri.live = ((rinfo[1] >> 9) & 1) != 0;
  ri.bad = (uint32_t)rinfo[2];
  const bool copied = ((rinfo[1] >> 10) & 1) != 0;  // the copies were issued (and must land)
  const int slot = ri.slot, p = ri.p;
  const int64_t drow = ((int64_t)slot * P.HV + hv) * P.L;  // ring rows of (slot, hv) / (slot, hk)
  const int64_t krow = ((int64_t)slot * P.HK + hk) * P.L;
  float g_lo = 0.f, g_hi = 0.f;  // GDN, warp 0: the cached log-gates l and l + 32
  if (ri.live && GATE == GDN_GATE_SCALAR && warp == 0) {
    if (lane < p) g_lo = P.ring_g[drow + lane];
    if (lane + 32 < p) g_hi = P.ring_g[drow + lane + 32];
  }
  if (overlap) {
    grid_dependency_wait();
    if (t == 0) grid_launch_dependents();
    load_inputs();
    if (P.sync && t == 0) ticket = atomic_add_release_gpu(P.sync, 1u);
  }
  if (hv == 0 && slab == 0 && t == 0) {  // one block reports the row
    if (ri.bad) set_status(P.status, ri.bad);
    if (P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
  }
  // The last block to count moves every row's cursor ([P1] Design 3).
  auto advance_if_last = [&]() {
    if (P.sync && warp == 0) {
      const bool last = __shfl_sync(0xffffffffu, ticket == gridDim.x - 1u ? 1 : 0, 0) != 0;
      if (last) {
        __threadfence();
        for (int bb = lane; bb < P.B; bb += 32) {
          const RowInfo rb2 = resolve_row(P, bb, false);
          if (rb2.live) P.write_pos_w[rb2.slot] = rb2.flush ? 0 : rb2.p + 1;
        }
        if (lane == 0) *P.sync = 0u;
      }
    }
  };
  // every thread waits for the copies (bounded): shared memory must not be
  // left with copies in flight when the block exits
  bool landed = true;
  if (copied) landed = mbar_wait_bounded(bar, 0, kWaitLimitNs);
  if (!landed && t == 0) set_status(P.status, GDN_DEV_TIMEOUT);
  const int64_t obase = bh * D + row0;
  if (!ri.live || !landed) {  // padding (or invalid) row: zeros, no cache access
    for (int rr = t; rr < R; rr += kSlabThreads) store_from_f32(P.out, obase + rr, P.out_dtype, 0.f);
    advance_if_last();
    return;
  }

  if (P.qk_l2norm) {
    const float2 n = block_sum2(qt * qt, kt * kt, red);
    qt = qt / sqrtf(n.x + 1e-6f);
    kt = kt / sqrtf(n.y + 1e-6f);
  }
  qt *= P.q_scale;
  if (t < D) {
    q[t] = qt;
    k[t] = kt;
    if (GATE == GDN_GATE_PER_K) a[t] = expf(gt);
  }
  // Replay decays ([P1] Design 1 and 7), summed from the newest entry back.
  if (GATE == GDN_GATE_SCALAR) {
    if (warp == 0) {
      float t_lo = g_lo, t_hi = g_hi;  // suffix sums: lane l ends with sum_{l<=i<p} g_i
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_down_sync(0xffffffffu, t_hi, o);
        if (lane + o < 32) t_hi += x;
      }
      const float hi_total = __shfl_sync(0xffffffffu, t_hi, 0);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_down_sync(0xffffffffu, t_lo, o);
        if (lane + o < 32) t_lo += x;
      }
      t_lo += hi_total;
      const float nxt_lo = __shfl_down_sync(0xffffffffu, t_lo, 1);
      const float nxt_hi = __shfl_down_sync(0xffffffffu, t_hi, 1);
      wv[lane] = expf(lane == 31 ? hi_total : nxt_lo);  // w_j = exp(sum_{j<i<p} g_i)
      wv[lane + 32] = expf(lane == 31 ? 0.f : nxt_hi);
      if (lane == 0) red[8] = p > 0 ? expf(t_lo) : 1.f;  // A
    }
  }
  const int p4 = (p + 3) & ~3;  // entries p .. p4 - 1 are zero operands
  if (t < D) {  // channel t of the keys (KDA: times w_j[t], summed from the newest entry back)
    if (GATE == GDN_GATE_PER_K) {
      float sg = 0.f;
      for (int j = p - 1; j >= 0; --j) {
        const float kj = load_as_f32(sK, (int64_t)j * D + t, RING_DT);
        Kw[j * D + t] = expf(sg) * kj;
        sg += sG[j * D + t];
      }
      Acol[t] = expf(sg);
    } else if (RB == 2) {
      for (int j0 = 0; j0 < p; j0 += 4) {  // four loads in flight per step
        float kv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) kv[u] = j0 + u < p ? load_as_f32(sK, (int64_t)(j0 + u) * D + t, RING_DT) : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) Kw[(j0 + u) * D + t] = kv[u];
      }
    }
    for (int j = p; j < p4; ++j) Kw[j * D + t] = 0.f;
  }
  // the block's rows of the corrections
  for (int e0 = 0; e0 < p4 * R; e0 += 4 * kSlabThreads) {
    float dv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * kSlabThreads + t;
      dv[u] = e < p * R ? load_as_f32(sD, e, RING_DT) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * kSlabThreads + t;
      if (e < p4 * R) Dw[e] = dv[u];
    }
  }
  __syncthreads();
  const float A = GATE == GDN_GATE_SCALAR ? red[8] : 1.f;
  const float alpha = GATE == GDN_GATE_SCALAR ? expf(gs) : 1.f;

  // This lane's columns of the readout vectors.
  float4 qe[M], ke[M], kraw[M], a4[M], A4[M];
  float kq = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c4 = 8 * m + cg;
    kraw[m] = reinterpret_cast<const float4 *>(k)[c4];
    qe[m] = reinterpret_cast<const float4 *>(q)[c4];
    kq = dot4(kraw[m], qe[m], kq);
    ke[m] = kraw[m];
    a4[m] = A4[m] = make_float4(1.f, 1.f, 1.f, 1.f);
    if (GATE == GDN_GATE_PER_K) {
      a4[m] = reinterpret_cast<const float4 *>(a)[c4];
      A4[m] = reinterpret_cast<const float4 *>(Acol)[c4];
      qe[m] = make_float4(a4[m].x * qe[m].x, a4[m].y * qe[m].y, a4[m].z * qe[m].z, a4[m].w * qe[m].w);
      ke[m] = make_float4(a4[m].x * ke[m].x, a4[m].y * ke[m].y, a4[m].z * ke[m].z, a4[m].w * ke[m].w);
    }
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);  // k.q over the row's 8 lanes

  float4 *S = reinterpret_cast<float4 *>(P.state + ((int64_t)slot * P.HV + hv) * D * D);
  for (int it = 0; it < R / kSlabRows; ++it) {
    const int rr = it * kSlabRows + rl, r = row0 + rr;
    // row r of the pre-token state, then its readout
    float4 s[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4 c = reinterpret_cast<const float4 *>(sS0 + rr * D)[8 * m + cg];
      s[m] = GATE == GDN_GATE_SCALAR ? make_float4(A * c.x, A * c.y, A * c.z, A * c.w)
                                     : make_float4(A4[m].x * c.x, A4[m].y * c.y, A4[m].z * c.z, A4[m].w * c.w);
    }
    for (int j0 = 0; j0 < p4; j0 += 4) {  // four entries a step, their loads in flight together
      float dw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        dw[u] = GATE == GDN_GATE_SCALAR ? wv[j0 + u] * Dw[(j0 + u) * R + rr] : Dw[(j0 + u) * R + rr];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float4 kr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) kr[u] = reinterpret_cast<const float4 *>(Kw + (j0 + u) * D)[8 * m + cg];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          s[m].x = fmaf(dw[u], kr[u].x, s[m].x);
          s[m].y = fmaf(dw[u], kr[u].y, s[m].y);
          s[m].z = fmaf(dw[u], kr[u].z, s[m].z);
          s[m].w = fmaf(dw[u], kr[u].w, s[m].w);
        }
      }
    }
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      sq = dot4(s[m], qe[m], sq);
      sk = dot4(s[m], ke[m], sk);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {  // the row's 8 lanes
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (GATE == GDN_GATE_SCALAR) {
      sq *= alpha;
      sk *= alpha;
    }
    const float d = beta * (v[rr] - sk);
    if (cg == 0) store_from_f32(P.out, bh * D + r, P.out_dtype, fmaf(d, kq, sq));
    if (ri.flush) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float4 x = s[m], kk = kraw[m];
        float4 o;
        if (GATE == GDN_GATE_SCALAR) {
          o = make_float4(fmaf(d, kk.x, alpha * x.x), fmaf(d, kk.y, alpha * x.y), fmaf(d, kk.z, alpha * x.z),
                          fmaf(d, kk.w, alpha * x.w));
        } else {
          o = make_float4(fmaf(d, kk.x, x.x * a4[m].x), fmaf(d, kk.y, x.y * a4[m].y),
                          fmaf(d, kk.z, x.z * a4[m].z), fmaf(d, kk.w, x.w * a4[m].w));
        }
        S[r * (D / 4) + 8 * m + cg] = o;
      }
    } else if (cg == 0) {
      store_from_f32(P.ring_d, (drow + p) * D + r, P.ring_dtype, d);
    }
  }
  if (!ri.flush && slab == 0) {  // the key (once per key head) and the gate
    if (hv % P.G == 0 && t < D) store_from_f32(P.ring_k, (krow + p) * D + t, P.ring_dtype, kt);
    if (GATE == GDN_GATE_SCALAR) {
      if (t == 0) P.ring_g[drow + p] = gs;
    } else if (t < D) {
      P.ring_g[(drow + p) * D + t] = gt;
    }
  }
  advance_if_last();
}

// Slabs per head: as many as keep the launch within about four blocks per SM
// (a small batch's blocks then all run in one wave).
static int slab_count(const DecodeParams &P, int D) {
  static const int sms = [] {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 1;
  }();
  const int64_t items = (int64_t)P.B * P.HV;
  int ns = D / kSlabRows;
  while (ns > 1 && items * ns > 4 * (int64_t)sms) ns >>= 1;
  return ns;
}

bool slab_decode_takes(const DecodeParams &P, int gate) {
  // the bulk copies of a KDA layer's gates start on 16 bytes
  if (gate == GDN_GATE_PER_K && P.L > 1 && (reinterpret_cast<uintptr_t>(P.ring_g) & 15u) != 0) return false;
  if (P.persistent_only) return false;
  const int64_t items = (int64_t)P.B * P.HV;
  if (items <= kSlabMaxItems) return true;
  // A GDN layer with a short ring: up to 256 items this kernel's CUDA-core
  // replay (p ring entries per state element) still costs less than the
  // persistent kernel's per-launch set-up while items x L stays at or below
  // 2048 (at 32 value heads: B = 4 up to L = 16, B = 8 up to L = 8; measured
  // B = 4, L = 4: 6.9 against 10.5 us; B = 8, L = 4: 9.1 against 11.6 us).
  return gate == GDN_GATE_SCALAR && items <= 4 * kSlabMaxItems && items * P.L <= 32 * kSlabMaxItems;
}

template <int D, int GATE, int RING_DT>
static cudaError_t launch_slab_t(const DecodeParams &P, cudaStream_t s) {
  auto kern = slab_decode_kernel<D, GATE, RING_DT>;
  const int ns = slab_count(P, D);
  const size_t smem = slab_layout(D, D / ns, P.L, P.ring_dtype == GDN_F32 ? 4 : 2, GATE).total;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // programmatic stream serialisation, as the persistent kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P.B * P.HV * ns));
  cfg.blockDim = dim3(kSlabThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, P, ns);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int GATE>
static cudaError_t launch_slab_ring(const DecodeParams &P, cudaStream_t s) {
  if (P.ring_dtype == GDN_F16) return launch_slab_t<D, GATE, GDN_F16>(P, s);
  if (P.ring_dtype == GDN_BF16) return launch_slab_t<D, GATE, GDN_BF16>(P, s);
  return launch_slab_t<D, GATE, GDN_F32>(P, s);
}

cudaError_t launch_slab_decode(const DecodeParams &P, int D, int gate, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_slab_ring<128, 0>(P, s) : launch_slab_ring<128, 1>(P, s);
  return gate == GDN_GATE_SCALAR ? launch_slab_ring<64, 0>(P, s) : launch_slab_ring<64, 1>(P, s);
}

}  // namespace gdn
