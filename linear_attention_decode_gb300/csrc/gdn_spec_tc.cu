// Speculative verify window with the checkpoint contraction on the tensor cores
// ([P3] Core concept, Design notes).
//
// Row b with slot s and cursor p verifies T tokens: token t is the non-flush
// decode at cursor p + t, so it needs S_{p+t} q_t and S_{p+t} k_t, where S_{p+t}
// is the state after the committed entries j < p and the window's own tokens
// i < t.  Both are linear in the state, so the window needs only products of
// the checkpoint with 2T vectors, never a rebuilt state:
//
//   a_t  = exp(g_t) (GDN: the same for every channel), P_t = prod_{m<=t} a_m,
//   X'_t = P_t o {q_t, k_t},  A = prod_{i<p} a_i (from the cached log-gates),
//   y    = S0 (A o X')                          one tf32 MMA, M=128, N=2T, K=128
//        + sum_{j<p} d_j [(w_j o k_j) . X']     committed entries (CUDA cores)
//        + sum_{i<t} d^_i [(prod_{i<m<=t} a_m o k^_i) . x_t]  earlier window tokens
//   d_t  = beta_t (v_t - y[k_t]),  o_t = y[q_t] + d_t (k_t . q_t),
//
// where d^_i, k^_i are token i's correction and key as the ring caches them
// (rounded to the ring type), exactly what the decode at cursor p + t would
// replay.  The window's (d, k, g) go to ring positions p .. p+T-1; neither the
// checkpoint nor the cursor changes.
//
// One persistent CTA per SM, 14 warps:
//   warp 0      TMA producer: the checkpoint of each item (row, value head) as
//               four [128 rows x 32 fp32] boxes, 128-byte swizzled, into a ring;
//   warp 1      MMA issuer (one thread): y[:, 0:N] = S0 . B^T, kind::tf32, the
//               accumulator of each worker group in its own TMEM columns;
//   warps 2-13  three worker groups of four warps, items dealt round-robin.  A
//               group loads the window's inputs (thread c = key channel c),
//               writes the B operand A o X' (tf32, K-major), the window's ring
//               entries k and g, and reduces the small dot products
//               (k_j . X', k^_i . x_t, k_t . q_t) over the channels; after the
//               MMA, thread r owns state row r: it reads y[r, :] from its TMEM
//               lane, adds the ring terms and runs the T-token recurrence.
// The MMA is issued only from warp 1, which never reads TMEM.  Every wait is
// bounded; a CTA that runs out of time records GDN_DEV_TIMEOUT, lets its copies
// and contractions land, frees its TMEM and returns.
#include "gdn_bits.cuh"
#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

namespace {

constexpr int kGroups = 3;                         // worker groups
constexpr int kThreadsSpec = 64 + 128 * kGroups;   // producer, MMA, workers
constexpr uint32_t kBoxBytes = 128 * 128;          // [128 rows x 32 fp32]

// Shared-memory layout, computed identically on host and device.  A worker
// group's field holds, in floats: v of the window tokens [T][128], beta [32],
// the per-warp partial sums [4][NBAT][NCOL] (totals land in the first slice),
// and the staged committed entries j < p of the current item: log-gates (GDN
// [64], KDA [PMAX][128] fp32), corrections and keys ([PMAX][128] ring type).
struct SpecLayout {
  int NB;            // checkpoint box slots
  int NBAT;          // reduction batches per item: 1 (k.q) + (T-1) window + p committed <= L-1
  int tmem_cols;
  uint32_t btile;    // kGroups B operands of NCOL rows x 512 bytes
  uint32_t field;    // kGroups fields of field_floats floats
  uint32_t field_floats;
  uint32_t o_part, o_gst, o_dst, o_kst;  // float offsets inside a field
  uint32_t bars;     // full[NB], empty[NB], bready[G], accf[G], ringf[G], fin; tmem address, abort flag
  uint32_t tab;      // the CTA's items, resolved once: {slot or a negative code, cursor}
  int tab_cap;
  uint32_t total;
};

constexpr int kBarsFixed = 3 * kGroups + 1;

__host__ __device__ inline SpecLayout spec_layout(int T, int L, int ncol, int NB, int ring_bytes, int gate,
                                                  int tab_cap) {
  SpecLayout l;
  l.NB = NB;
  l.NBAT = L - 1;
  const int pmax = L - 1 - T;
  const int tc = kGroups * ncol;
  l.tmem_cols = 32;
  while (l.tmem_cols < tc) l.tmem_cols <<= 1;
  l.btile = (uint32_t)NB * kBoxBytes;
  l.field = l.btile + (uint32_t)kGroups * ncol * 512;
  uint32_t f = (uint32_t)(T * 128 + 32);
  l.o_part = f;
  f += (uint32_t)(4 * l.NBAT * ncol);
  l.o_gst = f;
  f += gate == GDN_GATE_PER_K ? (uint32_t)(pmax * 128) : 64u;
  l.o_dst = f;
  f += (uint32_t)(pmax * 128 * ring_bytes / 4);
  l.o_kst = f;
  f += (uint32_t)(pmax * 128 * ring_bytes / 4);
  l.field_floats = f;
  l.bars = l.field + (uint32_t)kGroups * l.field_floats * 4;
  l.bars = (l.bars + 7u) & ~7u;
  l.tab = l.bars + (uint32_t)(2 * NB + kBarsFixed) * 8 + 16;
  l.tab_cap = tab_cap;
  l.total = l.tab + (uint32_t)tab_cap * 8;
  return l;
}

// K-major operand with 128-byte swizzle (what a TMA box of 128-byte rows
// writes): 8-row groups 1024 bytes apart; the start address selects the
// 32-byte K slice inside the swizzle row.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= 1ull << 46;                    // descriptor version for tcgen05
  d |= 2ull << 61;                    // 128-byte swizzle
  return d;
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier of `nthreads` threads on hardware barrier `id` that also ORs a
// predicate over them (every thread gets the result).
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Bounded wait that also gives up once another role has raised the abort flag;
// the first role to run out of time raises it.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// Sum over the 32 lanes of N per-lane values at once (N = 16 or 32): after the
// call lane l holds the warp total of value l % N (a butterfly that halves the
// value count at each step: N - 1 shuffles instead of 5 N).
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  float r = v[0];
  if (N == 16) r += __shfl_xor_sync(0xffffffffu, r, 16);
  return r;
}

__device__ __forceinline__ float round_to_ring(float x, int dtype) {
  if (dtype == GDN_F16) return __half2float(__float2half_rn(x));
  if (dtype == GDN_BF16) return __bfloat162float(__float2bfloat16_rn(x));
  return x;
}

// Item i = (row, value head), its slot and cursor, and whether the window fits.
struct SpecItem {
  int b, hv, slot, p;
  bool live;
  uint32_t bad;
};

__device__ __forceinline__ SpecItem spec_item(const DecodeParams &P, int i) {
  SpecItem it;
  it.b = i / P.HV;
  it.hv = i - it.b * P.HV;
  it.slot = P.idx[it.b];
  it.p = 0;
  it.live = false;
  it.bad = 0;
  if (it.slot < 0) return it;
  if (it.slot >= P.N) {
    it.bad = GDN_DEV_BAD_SLOT;
    return it;
  }
  const int p = P.write_pos[it.slot];
  if (p < 0 || p + P.T > P.L - 1) {
    it.bad = GDN_DEV_BAD_WRITE_POS;
    return it;
  }
  it.p = p;
  it.live = true;
  return it;
}

// Item table entry: {slot, p} for a live item, {-1, 0} padding, {-2, 0} slot
// past the pool, {-3, 0} a window that does not fit.
__device__ __forceinline__ int2 encode_item(const SpecItem &it) {
  if (it.live) return make_int2(it.slot, it.p);
  return make_int2(it.bad == GDN_DEV_BAD_SLOT ? -2 : (it.bad ? -3 : -1), 0);
}

__device__ __forceinline__ SpecItem decode_item(int2 e, int i, int HV) {
  SpecItem it;
  it.b = i / HV;
  it.hv = i - it.b * HV;
  it.slot = e.x;
  it.p = e.y;
  it.live = e.x >= 0;
  it.bad = e.x == -2 ? GDN_DEV_BAD_SLOT : (e.x == -3 ? GDN_DEV_BAD_WRITE_POS : 0u);
  return it;
}

}  // namespace

template <int GATE, int NCOL>
__global__ void __launch_bounds__(kThreadsSpec, 1) spec_tc_kernel(const DecodeParams P,
                                                                 const __grid_constant__ CUtensorMap tmap,
                                                                 const SpecLayout lay) {
  constexpr int D = 128;
  constexpr int TMAX = NCOL / 2;
  constexpr int KC = D * 4 / 16;  // 16-byte chunks per B operand row
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NB = lay.NB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * NB + kBarsFixed);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto full = [&](int s) { return smem_addr(&bars[s]); };
  auto empty = [&](int s) { return smem_addr(&bars[NB + s]); };
  auto bready = [&](int g) { return smem_addr(&bars[2 * NB + g]); };
  auto accf = [&](int g) { return smem_addr(&bars[2 * NB + kGroups + g]); };
  auto ringf = [&](int g) { return smem_addr(&bars[2 * NB + 2 * kGroups + g]); };
  const uint32_t fin = smem_addr(&bars[2 * NB + 3 * kGroups]);

  if (smem_addr(smem) & 1023u) {  // the swizzled boxes need a 1024-byte aligned base
    if (tid == 0) set_status(P.status, GDN_DEV_INTERNAL);
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < NB; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(bready(g), 1);
      mbar_init(accf(g), 1);
      mbar_init(ringf(g), 1);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), (uint32_t)lay.tmem_cols);
    tmem_relinquish();
  }
  const int T = P.T;
  const int items = P.B * P.HV;
  // this CTA's items i = blockIdx.x + li * gridDim.x, resolved in parallel once
  const int nmine = items > (int)blockIdx.x ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  int2 *tab = reinterpret_cast<int2 *>(smem + lay.tab);
  for (int li = tid; li < nmine && li < lay.tab_cap; li += blockDim.x)
    tab[li] = encode_item(spec_item(P, blockIdx.x + li * gridDim.x));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      prefetch_tensormap(&tmap);
      uint32_t n = 0;  // boxes issued
      bool ok = true;
      for (int li = 0; ok && li < nmine; ++li) {
        const SpecItem it = decode_item(tab[li], blockIdx.x + li * gridDim.x, P.HV);
        if (!it.live) continue;
        const int row0 = (it.slot * P.HV + it.hv) * D;
        for (int c = 0; c < D / 32; ++c, ++n) {
          const uint32_t s = n % NB;
          if (n >= (uint32_t)NB && !wait_or_abort(empty(s), ((n / NB) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(s), kBoxBytes);
          tma_load_2d(smem_addr(smem + s * kBoxBytes), &tmap, 32 * c, row0, full(s));
        }
      }
      // every copy issued must have landed before the CTA may exit
      const uint32_t last = n < (uint32_t)NB ? n : (uint32_t)NB;
      for (uint32_t k = 0; k < last; ++k) {
        const uint32_t m = n - 1 - k;
        mbar_wait_bounded(full(m % NB), (m / NB) & 1u, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const uint32_t idesc = make_idesc(2, NCOL);
      uint32_t n = 0, gph = 0;
      bool ok = true;
      for (int li = 0; ok && li < nmine; ++li) {
        const SpecItem it = decode_item(tab[li], blockIdx.x + li * gridDim.x, P.HV);
        if (!it.live) continue;
        const int g = li % kGroups;
        if (!wait_or_abort(bready(g), (gph >> g) & 1u, abort_flag)) break;
        gph ^= 1u << g;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(g * NCOL);
        const uint32_t bt = smem_addr(smem + lay.btile + g * NCOL * 512);
        for (int c = 0; c < D / 32; ++c, ++n) {
          const uint32_t s = n % NB;
          if (!wait_or_abort(full(s), (n / NB) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t box = smem_addr(smem + s * kBoxBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma<1>(acc, make_sdesc_sw128(box + 32 * kk),
                      make_sdesc(bt + 256 * (4 * c + kk), 128, KC * 128), idesc, (c | kk) != 0 ? 1u : 0u);
          tc_commit(empty(s));  // the box slot is free once these MMAs have read it
        }
        if (ok) tc_commit(accf(g));
      }
      tc_commit(fin);  // nothing of ours may still run when TMEM is freed
      mbar_wait_bounded(fin, 0, kWaitLimitNs);
    }
  } else {
    // ---- worker groups ----
    const int g = (warp - 2) >> 2;
    const int wq = warp & 3;              // warp slot in the group (TMEM lanes 32 wq ..)
    const int r = 32 * wq + lane;         // key channel in the prologue, state row in the epilogue
    const uint32_t bar_id = 1 + g;
    const uint32_t row_bytes = (uint32_t)D * (P.ring_dtype == GDN_F32 ? 4u : 2u);
    float *F = reinterpret_cast<float *>(smem + lay.field) + g * lay.field_floats;
    float *Vs = F;                        // [T][128] v of the window tokens
    float *Bt = F + T * D;                // [32] beta
    float *part = F + lay.o_part;         // [4][NBAT][NCOL] per-warp partial sums; totals in part[0]
    float *gst = F + lay.o_gst;           // cached log-gates j < p (GDN [p], KDA [p][128])
    const void *dst = F + lay.o_dst;      // cached corrections d_j [p][128], ring type
    const void *kst = F + lay.o_kst;      // cached keys k_j [p][128], ring type
    const int pstride = lay.NBAT * NCOL;
    uint8_t *bt = smem + lay.btile + g * NCOL * 512;
    const uint32_t ringbar = ringf(g);
    uint32_t accph = 0, ringph = 0;
    bool ring_pending = false;
    for (int li = g; li < nmine; li += kGroups) {
      const SpecItem it = decode_item(tab[li], blockIdx.x + li * gridDim.x, P.HV);
      if (!it.live) {  // padding or unusable row: zeros for every window token
        if (it.bad && it.hv == 0 && r == 0) set_status(P.status, it.bad);
        for (int t = 0; t < T; ++t)
          store_from_f32(P.out, (((int64_t)it.b * T + t) * P.HV + it.hv) * D + r, P.out_dtype, 0.f);
        continue;
      }
      const int b = it.b, hv = it.hv, slot = it.slot, p = it.p, hk = hv / P.G;
      const int64_t hrow = (int64_t)slot * P.HV + hv;
      const int64_t krow = (int64_t)slot * P.HK + hk;

      // 1. the committed entries j < p, staged by bulk copies (one round trip);
      // a GDN group's committed gates go through registers and reach shared
      // memory only after the window loads below have been issued
      float gate_r = 0.f;
      if (p > 0) {
        if (r == 0) {
          const uint32_t bytes = 2u * p * row_bytes + (GATE == GDN_GATE_PER_K ? (uint32_t)p * D * 4u : 0u);
          mbar_arrive_expect_tx(ringbar, bytes);
          bulk_load(smem_addr(dst), static_cast<const uint8_t *>(P.ring_d) + hrow * P.L * row_bytes,
                    p * row_bytes, ringbar);
          bulk_load(smem_addr(kst), static_cast<const uint8_t *>(P.ring_k) + krow * P.L * row_bytes,
                    p * row_bytes, ringbar);
          if (GATE == GDN_GATE_PER_K)
            bulk_load(smem_addr(gst), P.ring_g + hrow * P.L * D, (uint32_t)p * D * 4u, ringbar);
        }
        if (GATE == GDN_GATE_SCALAR && r < p) gate_r = P.ring_g[hrow * P.L + r];
        ring_pending = true;
      }

      // 2. window inputs of channel r: every load first (raw bits, so none waits
      // for the one before), then the conversions and the stores
      float q[TMAX], k[TMAX], a[TMAX], vv[TMAX];
      {
        uint32_t bq[TMAX], bk[TMAX], bv[TMAX];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          bq[t] = bk[t] = bv[t] = 0u;
          a[t] = 0.f;  // log-gate; tokens past the window keep exp(0) = 1
          if (t < T) {
            const int64_t row = (int64_t)b * T + t;
            const int64_t base = row * P.qkv_stride;
            bq[t] = load_bits(P.qkv, base + (int64_t)hk * D + r, P.qkv_dtype);
            bk[t] = load_bits(P.qkv, base + (int64_t)(P.HK + hk) * D + r, P.qkv_dtype);
            bv[t] = load_bits(P.qkv, base + (int64_t)2 * P.HK * D + (int64_t)hv * D + r, P.qkv_dtype);
            const int64_t bh = row * P.HV + hv;
            a[t] = GATE == GDN_GATE_PER_K ? P.g[bh * D + r] : P.g[bh];
          }
        }
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          q[t] = bits_to_f32(bq[t], P.qkv_dtype);
          k[t] = bits_to_f32(bk[t], P.qkv_dtype);
          vv[t] = bits_to_f32(bv[t], P.qkv_dtype);
        }
      }
      const float beta_r = r < T ? P.beta[((int64_t)b * T + r) * P.HV + hv] : 0.f;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          Vs[t * D + r] = vv[t];
          // the window's ring entries: g here, k once per key head after the norm
          if (GATE == GDN_GATE_PER_K) P.ring_g[(hrow * P.L + p + t) * D + r] = a[t];
          else if (r == 0) P.ring_g[hrow * P.L + p + t] = a[t];
        }
      }
      if (r < T) Bt[r] = beta_r;
      if (GATE == GDN_GATE_SCALAR && r < p) gst[r] = gate_r;
      if (P.qk_l2norm) {
        float v[NCOL];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          v[2 * t] = q[t] * q[t];
          v[2 * t + 1] = k[t] * k[t];
        }
        const float s = warp_reduce_scatter<NCOL>(v, lane);
        if (lane < NCOL) part[wq * pstride + lane] = s;
        named_bar_sync(bar_id, 128);
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          if (t < T) {
            const float nq = (part[2 * t] + part[pstride + 2 * t]) +
                             (part[2 * pstride + 2 * t] + part[3 * pstride + 2 * t]);
            const float nk = (part[2 * t + 1] + part[pstride + 2 * t + 1]) +
                             (part[2 * pstride + 2 * t + 1] + part[3 * pstride + 2 * t + 1]);
            q[t] = q[t] / sqrtf(nq + 1e-6f);
            k[t] = k[t] / sqrtf(nk + 1e-6f);
          }
        }
        named_bar_sync(bar_id, 128);  // part is written again below
      }
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        q[t] *= P.q_scale;
        a[t] = expf(a[t]);
        if (t < T && hv % P.G == 0)
          store_from_f32(P.ring_k, (krow * P.L + p + t) * D + r, P.ring_dtype, k[t]);
      }

      // 3. the committed gates are in shared memory (the barrier publishes the
      // GDN gates; KDA's come with the staged copies).  A GDN group waits for
      // the staged corrections and keys only where it first reads them (the
      // committed dot products), so its operand for the contraction, which
      // needs only the gates, is not held up by those copies.
      bool ok = true;
      if (GATE == GDN_GATE_PER_K && p > 0) ok = wait_or_abort(ringbar, ringph, abort_flag);
      if (named_bar_or(bar_id, 128, !ok)) break;
      if (GATE == GDN_GATE_PER_K && p > 0) {
        ringph ^= 1u;
        ring_pending = false;
      }
      // committed decay A = prod_{i<p} a_i (summed newest first, as every replay does)
      float gsum = 0.f;
      for (int j = p - 1; j >= 0; --j) gsum += GATE == GDN_GATE_PER_K ? gst[j * D + r] : gst[j];
      const float A = expf(gsum);

      // 4. B operand: row x of A o X' (x = 2t: q_t, x = 2t + 1: k_t), tf32, column r
      float xp[NCOL];
      {
        float Pt = 1.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
          Pt *= a[t];
          xp[2 * t] = t < T ? Pt * q[t] : 0.f;
          xp[2 * t + 1] = t < T ? Pt * k[t] : 0.f;
        }
      }
#pragma unroll
      for (int x = 0; x < NCOL; ++x)
        *reinterpret_cast<float *>(bt + tile_off(x, r, KC, 4)) = round_tf32(A * xp[x]);
      fence_proxy_async_smem();  // operand rows -> tensor-core (async) proxy
      tc_fence_before();         // this group's previous TMEM reads are done
      named_bar_sync(bar_id, 128);
      if (r == 0) mbar_arrive(bready(g));

      // 5. dot products over the channels, one batch of NCOL values per warp shuffle pass
      {  // batch 0: k_t . q_t
        float v[NCOL];
#pragma unroll
        for (int x = 0; x < NCOL; ++x) v[x] = 0.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) v[t] = k[t] * q[t];
        const float s = warp_reduce_scatter<NCOL>(v, lane);
        if (lane < NCOL) part[wq * pstride + lane] = s;
      }
#pragma unroll
      for (int i2 = 0; i2 < TMAX - 1; ++i2) {  // batches 1 + i2: window entry i2 against later tokens
        if (i2 < T - 1) {
          const float kh = round_to_ring(k[i2], P.ring_dtype);
          float v[NCOL];
          float run = 1.f;
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t > i2) run *= a[t];
            v[2 * t] = t > i2 ? run * kh * q[t] : 0.f;
            v[2 * t + 1] = t > i2 ? run * kh * k[t] : 0.f;
          }
          const float s = warp_reduce_scatter<NCOL>(v, lane);
          if (lane < NCOL) part[wq * pstride + (1 + i2) * NCOL + lane] = s;
        }
      }
      if (GATE == GDN_GATE_SCALAR && p > 0) {  // the staged corrections and keys
        ok = wait_or_abort(ringbar, ringph, abort_flag);
        if (named_bar_or(bar_id, 128, !ok)) break;
        ringph ^= 1u;
        ring_pending = false;
      }
      {  // batches T + j: committed entry j, weight w_j = prod_{j<i<p} a_i
        float s = 0.f;
        for (int j = p - 1; j >= 0; --j) {
          const float wk = expf(s) * load_as_f32(kst, (int64_t)j * D + r, P.ring_dtype);
          s += GATE == GDN_GATE_PER_K ? gst[j * D + r] : gst[j];
          float v[NCOL];
#pragma unroll
          for (int x = 0; x < NCOL; ++x) v[x] = wk * xp[x];
          const float red = warp_reduce_scatter<NCOL>(v, lane);
          if (lane < NCOL) part[wq * pstride + (T + j) * NCOL + lane] = red;
        }
      }
      named_bar_sync(bar_id, 128);
      for (int e = r; e < (T + p) * NCOL; e += 128)
        part[e] = (part[e] + part[pstride + e]) + (part[2 * pstride + e] + part[3 * pstride + e]);
      named_bar_sync(bar_id, 128);

      // 6. epilogue: thread r owns state row r
      ok = wait_or_abort(accf(g), accph, abort_flag);
      accph ^= 1u;
      if (named_bar_or(bar_id, 128, !ok)) break;
      tc_fence_after();
      float y[NCOL];
      {
        const uint32_t taddr = tmem + ((uint32_t)(32 * wq) << 16) + (uint32_t)(g * NCOL);
        if constexpr (NCOL == 16) {
          tmem_ld16(taddr, y);
        } else {
          float y0[16], y1[16];
          tmem_ld16(taddr, y0);
          tmem_ld16(taddr + 16, y1);
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            y[x] = y0[x];
            y[16 + x] = y1[x];
          }
        }
      }
      for (int j = 0; j < p; ++j) {
        const float dj = load_as_f32(dst, (int64_t)j * D + r, P.ring_dtype);
        const float4 *z = reinterpret_cast<const float4 *>(part + (T + j) * NCOL);
#pragma unroll
        for (int x4 = 0; x4 < NCOL / 4; ++x4) {
          const float4 c = z[x4];
          y[4 * x4 + 0] = fmaf(dj, c.x, y[4 * x4 + 0]);
          y[4 * x4 + 1] = fmaf(dj, c.y, y[4 * x4 + 1]);
          y[4 * x4 + 2] = fmaf(dj, c.z, y[4 * x4 + 2]);
          y[4 * x4 + 3] = fmaf(dj, c.w, y[4 * x4 + 3]);
        }
      }
      const int64_t dbase = hrow * P.L * D + r;
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          const float d = Bt[t] * (Vs[t * D + r] - y[2 * t + 1]);
          const int64_t orow = ((int64_t)b * T + t) * P.HV + hv;
          store_from_f32(P.out, orow * D + r, P.out_dtype, fmaf(d, part[t], y[2 * t]));
          store_from_f32(P.ring_d, dbase + (int64_t)(p + t) * D, P.ring_dtype, d);
          if (t < T - 1) {
            const float dh = round_to_ring(d, P.ring_dtype);
            const float4 *e = reinterpret_cast<const float4 *>(part + (1 + t) * NCOL);
#pragma unroll
            for (int x4 = 0; x4 < NCOL / 4; ++x4) {
              const float4 c = e[x4];
              y[4 * x4 + 0] = fmaf(dh, c.x, y[4 * x4 + 0]);
              y[4 * x4 + 1] = fmaf(dh, c.y, y[4 * x4 + 1]);
              y[4 * x4 + 2] = fmaf(dh, c.z, y[4 * x4 + 2]);
              y[4 * x4 + 3] = fmaf(dh, c.w, y[4 * x4 + 3]);
            }
          }
        }
      }
      tc_fence_before();
      named_bar_sync(bar_id, 128);  // the field is rewritten by the next item
    }
    // a staged copy that was not waited for must land before the CTA may exit
    if (ring_pending && r == 0) mbar_wait_bounded(ringbar, ringph, kWaitLimitNs);
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) set_status(P.status, GDN_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)lay.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

static int spec_device_attr(cudaDeviceAttr a) {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, a, dev);
  return v;
}

template <int GATE, int NCOL>
static cudaError_t launch_spec_tc_t(const DecodeParams &P, const CUtensorMap &map, const SpecLayout &lay,
                                    int grid, cudaStream_t s) {
  auto kern = spec_tc_kernel<GATE, NCOL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreadsSpec, lay.total, s>>>(P, map, lay);
  return cudaGetLastError();
}

// Checkpoint box slots (16 KB each, four per item) when shared memory allows.
#ifndef GDN_SPEC_BOX_SLOTS
#define GDN_SPEC_BOX_SLOTS 8
#endif
constexpr int kSpecBoxSlots = GDN_SPEC_BOX_SLOTS;

cudaError_t launch_spec_tc(const DecodeParams &P, int D, int gate, cudaStream_t s, const char **why) {
  static const int sms = spec_device_attr(cudaDevAttrMultiProcessorCount);
  static const int optin = spec_device_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin);
  if (D != 128 || P.T > 16) return cudaErrorNotSupported;
  if ((int64_t)P.N * P.HV * D >= ((int64_t)1 << 31)) return cudaErrorNotSupported;  // TMA row coordinate
  // the per-channel gates are staged by bulk copies (16-byte aligned rows)
  if (gate == GDN_GATE_PER_K && (reinterpret_cast<uintptr_t>(P.ring_g) & 15u) != 0) return cudaErrorNotSupported;
  const int ncol = P.T <= 8 ? 16 : 32;
  const int rb = P.ring_dtype == GDN_F32 ? 4 : 2;
  const int items = P.B * P.HV;
  const int grid = sms > 0 && sms < items ? sms : items;
  const int cap = (items + grid - 1) / grid;
  SpecLayout lay = spec_layout(P.T, P.L, ncol, kSpecBoxSlots, rb, gate, cap);
  while (lay.NB > 4 && lay.total > (uint32_t)optin) lay = spec_layout(P.T, P.L, ncol, lay.NB - 1, rb, gate, cap);
  if (lay.total > (uint32_t)optin) return cudaErrorNotSupported;
  CUtensorMap map;
  cudaError_t e = make_state_tmap(P, D, &map, why);
  if (e != cudaSuccess) return e;
  if (gate == GDN_GATE_SCALAR)
    return ncol == 16 ? launch_spec_tc_t<0, 16>(P, map, lay, grid, s) : launch_spec_tc_t<0, 32>(P, map, lay, grid, s);
  return ncol == 16 ? launch_spec_tc_t<1, 16>(P, map, lay, grid, s) : launch_spec_tc_t<1, 32>(P, map, lay, grid, s);
}

}  // namespace gdn
