// Persistent, warp-specialised ReplaySSM decode on the 5th-generation tensor
// cores.  One CTA per SM walks a round-robin share of the (row, value head)
// items.
//
// Roles (544 threads):
//   warp 0       producer: streams each item's fp32 checkpoint S0 [V, K] by TMA,
//                one [V x 32] box (128-byte swizzled) at a time, through a ring
//                of NB box slots (box_full / box_empty); it also allocates the
//                4 x K TMEM columns (four accumulators, two per group);
//   warps 1-8    two prep warpgroups taking alternate items.  A group's leader
//                bulk-copies the first p ring entries (d, k; KDA also g) and,
//                when aligned, q, k, v of its items two group-items ahead into
//                the group's landing slots (land_full).  From a landed slot the
//                group computes the replay decays and the two K-major operand tiles
//                ([P1] Design 1 and 7)
//                      GDN  A[v][j] = w_j d_j[v],  B[c][j] = k_j[c]
//                      KDA  A[v][j] = d_j[v],      B[c][j] = w_j[c] k_j[c]
//                into a tile stage, plus the epilogue's vectors into a field
//                stage (info_full / info_empty); the group leader then issues the
//                replay contraction tcgen05.mma into one of the group's two
//                accumulators (alternating), so the contraction of the group's
//                next item overlaps the epilogue of its current one;
//   warps 9-16   two epilogue warpgroups, group g taking the items of prep group
//                g and reading accumulator g: thread r owns state row r (TMEM
//                lane r).  It adds A S0[r][:] (KDA: S0[r][:] o A) to dS[r][:],
//                contracts with q and k in registers (packed fp32x2 FMAs), writes
//                out[r] = alpha Sq + d (k^T q) with d = beta (v - alpha Sk); a
//                flush item reads its box row and accumulator a second time and
//                stores row r of alpha S + d k^T straight to the checkpoint,
//                otherwise (d, k, g) are appended to the ring.
// Every wait is bounded: a wait that runs out raises a CTA-wide abort flag and
// GDN_DEV_TIMEOUT; all roles then leave their loops, the producer and the MMA
// issuers wait (bounded) for their own copies and contractions still in
// flight, and the CTA frees its TMEM and returns.
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

constexpr int kTcpThreads = 544;  // 17 warps
constexpr int kItemsMax = 256;    // items one CTA may own (sets the table size)
// Ring entries per landing slot and per operand tile stage when the whole
// replay depth does not fit the shared-memory layout: the replay then runs in
// chunks of kChunk entries that accumulate into the same TMEM accumulator;
// chunks past the first come straight from the ring in global memory.  A KDA
// layer with an fp32 ring takes chunks of 8 entries (one tf32 K-step): that
// halves its operand tiles and landing slots (d, k and the per-channel gates,
// 4 bytes each) so that two items' checkpoint boxes still fit beside them.
constexpr int kChunk = 16;
__host__ __device__ constexpr int chunk_entries(int kind, int gate) {
  return kind == 2 && gate == GDN_GATE_PER_K ? 8 : kChunk;
}

struct TcpLayout {
  int KD, KC, NT, NF, NL, NB;
  int CH;        // ring entries per replay chunk (>= the deepest replay: one chunk)
  int qkv_bulk;  // 1: q, k, v arrive by bulk copy (16-byte aligned rows)
  uint32_t box_bytes, tile_bytes, field_bytes, land_bytes;
  uint32_t off_tile, off_field, off_land, off_table, off_adv, off_bars, total;
  uint32_t t_B;                     // B operand inside a tile stage (A at 0)
  uint32_t ld_d, ld_k, ld_g, ld_q;  // inside a landing slot
};

// Epilogue vectors of an item (floats): q, k, v for GDN; KDA adds a o k, a, the
// total decay per channel and the current log-gate.  Then 16 scalars: alpha,
// beta, A, the current log-gate, and at 8..11 the four prep warps' partial
// sums of k.q.
__host__ __device__ inline int field_floats(int D, int gate) { return (gate == GDN_GATE_PER_K ? 7 : 3) * D + 16; }

// Shared memory: NB checkpoint boxes | NT operand tile stages | NF field stages
// | NL landing slots | item table | barriers.
static TcpLayout tcp_layout(int D, int kind, int gate, int L, int ring_bytes, int qkv_bytes, int qkv_bulk,
                            int NT, int NL, int smem_budget, bool chunked) {
  TcpLayout t{};
  const int es = kind == 2 ? 4 : 2;
  const int kstep = 32 / es;
  const int depth = L > 1 ? L - 1 : 0;
  const int chunk = chunk_entries(kind, gate);
  const int ldep = chunked && depth > chunk ? chunk : depth;  // ring entries of one chunk
  t.CH = chunked && depth > chunk ? chunk : (depth > 0 ? depth : 1);
  t.KD = ldep ? ((ldep + kstep - 1) / kstep) * kstep : 0;
  t.KC = t.KD * es / 16;
  t.qkv_bulk = qkv_bulk;
  t.box_bytes = (uint32_t)D * 128;
  t.t_B = (uint32_t)(128 * t.KD * es);
  t.tile_bytes = (t.t_B + (uint32_t)(D * t.KD * es) + 127) & ~127u;
  t.field_bytes = ((uint32_t)field_floats(D, gate) * 4 + 127) & ~127u;
  t.ld_d = 0;
  t.ld_k = t.ld_d + (uint32_t)(ldep * D * ring_bytes);
  t.ld_g = t.ld_k + (uint32_t)(ldep * D * ring_bytes);
  t.ld_q = t.ld_g + (uint32_t)(gate == GDN_GATE_PER_K ? ldep * D * 4 : 0);
  t.land_bytes = (t.ld_q + (uint32_t)(qkv_bulk ? 3 * D * qkv_bytes : 0) + 127) & ~127u;
  const uint32_t table = (uint32_t)kItemsMax * 16;  // item table
  const uint32_t adv = (uint32_t)kTcpThreads * 4;  // the rows' next cursors (decode + advance)
  const uint32_t bars = 1024;  // barriers, then misc words and the dealing's counters
  t.NT = NT;
  t.NF = NT + 4;  // a group's fields live from its prep until its epilogue, up to NT + 4 items later
  t.NL = NL;
  const long rest = (long)smem_budget - (long)t.NT * t.tile_bytes - (long)t.NF * t.field_bytes -
                    (long)t.NL * t.land_bytes - table - adv - bars;
  t.NB = rest > 0 ? (int)(rest / t.box_bytes) : 0;
  if (t.NB > 16) t.NB = 16;
  t.off_tile = (uint32_t)t.NB * t.box_bytes;
  t.off_field = t.off_tile + (uint32_t)t.NT * t.tile_bytes;
  t.off_land = t.off_field + (uint32_t)t.NF * t.field_bytes;
  t.off_table = t.off_land + (uint32_t)t.NL * t.land_bytes;
  t.off_adv = t.off_table + table;
  t.off_bars = t.off_adv + adv;
  t.total = t.off_bars + bars;
  return t;
}

// The first (tile stages, landing slots) choice that leaves room for two items'
// checkpoint boxes plus one more; else the one with the most boxes.  The whole
// replay depth in one chunk first (one contraction per item, nothing loaded
// past the landing); chunks only when that leaves too few boxes (GDN fp32
// rings beyond L = 17, KDA fp32 rings beyond L = 9, any ring beyond L = 33).
static TcpLayout tcp_pick_layout(int D, int kind, int gate, int L, int ring_bytes, int qkv_bytes, int qkv_bulk,
                                 int smem_budget) {
  static const int cand[4][2] = {{4, 4}, {2, 4}, {4, 2}, {2, 2}};
  const int want = 2 * (D / 32) + 1;
  TcpLayout best{};
  for (int chunked = 0; chunked < 2; ++chunked) {
    for (const auto &c : cand) {
      const TcpLayout t =
          tcp_layout(D, kind, gate, L, ring_bytes, qkv_bytes, qkv_bulk, c[0], c[1], smem_budget, chunked != 0);
      if (t.NB >= want) return t;
      if (t.NB > best.NB) best = t;
    }
    if (best.NB >= 2 * (D / 32)) return best;  // enough for the pipeline without chunks
  }
  return best;
}

struct TcpBars {
  uint32_t box_full, box_empty, land_full, info_full, info_empty, tile_empty, tmem_full, tmem_empty;
  __device__ uint32_t bf(int i) const { return box_full + 8 * i; }
  __device__ uint32_t be(int i) const { return box_empty + 8 * i; }
  __device__ uint32_t lf(int i) const { return land_full + 8 * i; }
  __device__ uint32_t inf(int i) const { return info_full + 8 * i; }
  __device__ uint32_t ine(int i) const { return info_empty + 8 * i; }
  __device__ uint32_t tle(int i) const { return tile_empty + 8 * i; }
  __device__ uint32_t tf(int i) const { return tmem_full + 8 * i; }
  __device__ uint32_t te(int i) const { return tmem_empty + 8 * i; }
};

// Position in a ring of n slots walked in order, packed in one register:
// bits 0-15 the slot, bit 16 the lap's parity (the mbarrier phase in which the
// slot's "full" barrier completes), bit 17 set once past the first lap (a slot
// must then first be released).
struct RingPos {
  uint32_t v;
  __device__ int i() const { return (int)(v & 0xffffu); }
  __device__ uint32_t ph() const { return (v >> 16) & 1u; }
  __device__ bool lapped() const { return (v >> 17) != 0u; }
  __device__ void init(int start, int n) {
    v = 0u;
    advance(start, n);
  }
  __device__ void advance(int k, int n) {
    int i = (int)(v & 0xffffu) + k;
    uint32_t hi = v & 0x30000u;
    while (i >= n) {
      i -= n;
      hi = (hi ^ 0x10000u) | 0x20000u;
    }
    v = hi | (uint32_t)i;
  }
};

// An item table entry: x slot, y p | flush << 8 | live << 9 | writes-k << 10,
// z row b, w value head hv | key head hk << 16.
__device__ __forceinline__ int tab_p(const int4 &e) { return e.y & 255; }
__device__ __forceinline__ int tab_flush(const int4 &e) { return (e.y >> 8) & 1; }
__device__ __forceinline__ bool tab_live(const int4 &e) { return (e.y & 512) != 0; }
__device__ __forceinline__ bool tab_kw(const int4 &e) { return (e.y & 1024) != 0; }
__device__ __forceinline__ int tab_hv(const int4 &e) { return e.w & 0xffff; }
__device__ __forceinline__ int tab_hk(const int4 &e) { return e.w >> 16; }

// Bounded wait that also gives up when another thread raised the abort flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         uint32_t *status);

// The same for a whole warp: lane 0 polls, the warp follows with its verdict
// (fewer threads hammering the barrier unit).
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                              uint32_t *status) {
  if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity) ? 1 : 0)) return true;
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, status);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// A completed phase is caught by the non-blocking test: a blocking try_wait on
// a phase that is already complete was measured at ~240 ns on GB300.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                         uint32_t *status) {
  if (mbar_test_wait(bar, parity)) return true;
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

// One arrival for the whole warp once all its lanes are past this point (the
// consumer barriers count warps, not threads: fewer atomics on one word).
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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
  constexpr int NVEC = GATE == GDN_GATE_PER_K ? 7 : 3;  // epilogue vectors per item
  constexpr int kCh = chunk_entries(KIND, GATE);  // ring entries per replay chunk
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Items are the (row b, value head hv) pairs, laid out in one sequence and
  // dealt round-robin: CTA c takes positions c, c + G, c + 2G, ... (see the
  // dealing below).
  const int T = P.B * P.HV;
  const int G = gridDim.x;
  const int n = (int)blockIdx.x < T ? (T - 1 - (int)blockIdx.x) / G + 1 : 0;
  const int NB = lay.NB, NT = lay.NT, NF = lay.NF, NL = lay.NL;
  const int NBg = NB / 2;  // checkpoint box slots per epilogue group
  const int qes = P.qkv_dtype == GDN_F32 ? 4 : 2;

  if (smem_addr(smem) & 1023u) {  // the 128-byte swizzle assumes a 1024-byte aligned base
    // No item runs.  A decode + advance launch still counts this block, so the
    // counter ends the launch at zero, and the last block to count moves the
    // cursors as the call promises (every other block has read them by then).
    grid_dependency_wait();
    grid_launch_dependents();
    uint32_t last = 0u;
    if (tid == 0) {
      set_status(P.status, GDN_DEV_INTERNAL);
      if (P.sync) {
        __threadfence();
        last = atomicAdd(P.sync, 1u) == gridDim.x - 1u ? 1u : 0u;
      }
    }
    if (__syncthreads_or(last != 0u)) {
      __threadfence();
      for (int b = tid; b < P.B; b += kTcpThreads) {
        const RowInfo ri = resolve_row(P, b, false);
        if (ri.live) P.write_pos_w[ri.slot] = ri.flush ? 0 : ri.p + 1;
      }
      if (tid == 0) *P.sync = 0u;
    }
    return;
  }
  int4 *table = reinterpret_cast<int4 *>(smem + lay.off_table);
  // decode + advance: row b's slot << 7 | next cursor, or -1 (single-pass dealing)
  int *advq = reinterpret_cast<int *>(smem + lay.off_adv);
  uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + lay.off_bars);
  const uint32_t bar0 = smem_addr(bar_mem);
  TcpBars bars;
  bars.box_full = bar0;
  bars.box_empty = bars.box_full + 8u * NB;
  bars.land_full = bars.box_empty + 8u * NB;
  bars.info_full = bars.land_full + 8u * NL;
  bars.info_empty = bars.info_full + 8u * NF;
  bars.tile_empty = bars.info_empty + 8u * NF;
  bars.tmem_full = bars.tile_empty + 8u * NT;
  bars.tmem_empty = bars.tmem_full + 32u;  // four accumulators
  // misc[0] TMEM base, misc[1] abort flag, misc[2..3] prep-group go/stop words,
  // misc[4] number of live items, misc[7] last CTA to finish (decode +
  // advance), misc[8..] the dealing's counters
  uint32_t *misc = reinterpret_cast<uint32_t *>(bar_mem + 2 * NB + NL + 2 * NF + NT + 8);
  volatile uint32_t *abort_flag = misc + 1;

  // Set-up that reads nothing an earlier kernel writes: barriers, TMEM, the
  // tensor map.  With a programmatic dependency on the previous launch in the
  // stream it overlaps that launch's tail; everything after the dependency
  // wait sees the previous launch complete.  Without GDN_STEP_OVERLAP_PREVIOUS
  // every thread waits before the dealing; with it the dealing (rows, cursors)
  // and the producer's checkpoint stream run first, and the other roles wait
  // before they read the step's inputs or write anything.  The next launch is
  // let in only after this block has waited, so a launch never starts while
  // the one two places ahead of it is still running.
  // The last warp does this set-up, its lanes side by side, while the others
  // start dealing the rows (it holds rows only when B > 512).  Barriers in
  // address order: box full / empty, land full, info full / empty, tile
  // empty, TMEM full / empty; the "empty" ones count one arrival per consumer
  // warp, the others one arrival (or the transaction bytes).
  constexpr int kSetupWarp = kTcpThreads / 32 - 1;
  if (warp == kSetupWarp) {
    const int nbar = 2 * NB + NL + 2 * NF + NT + 8;
    for (int i = lane; i < nbar; i += 32) {
      int k = i;
      uint32_t count = 1;
      if (k >= NB && k < 2 * NB) count = 4;  // one arrival per epilogue warp
      k -= 2 * NB + NL;
      if (k >= NF && k < 2 * NF) count = 4;
      k -= 2 * NF + NT;
      if (k >= 4 && k < 8) count = 4;
      mbar_init(bar0 + 8u * (uint32_t)i, count);
    }
    if (lane == 0) misc[1] = 0u;
    fence_mbar_init();
    tmem_alloc(smem_addr(misc), 4 * D);
    tmem_relinquish();
  }
  if (tid == 32) prefetch_tensormap(&tmap);
  const bool overlap = P.overlap != 0;
  if (!overlap) {
    grid_dependency_wait();
    grid_launch_dependents();
  }

  // --- dealing: the item table of this CTA ---
  // Every CTA classifies every row: live without flush (0), live with flush (1)
  // or dead (2: padding, or an invalid slot or cursor).  Items (b, hv) form one
  // sequence: the flush items, then the other live ones, then the dead ones,
  // each group in row order; item t goes to CTA t % G.  Every CTA thus gets
  // the same share (to one) of flush items, each about 1.5x the work of
  // another.  Inside a CTA the flush items are spread evenly among its other
  // live items (a merge of the two by (2 rank + 1) / count, non-flush first on
  // a tie) and the dead ones come last.
  int *cnt = reinterpret_cast<int *>(misc + 8);  // [3] row counts, [3] carries, [3][32] per warp
  int *carry = cnt + 3, *wc = cnt + 6;
  constexpr int NW = kTcpThreads / 32;
  // Enters row b (category cat, rank among its category's rows) into the table
  // if this CTA holds some of its heads.  Sizes here stay far below 2^31.
  auto place = [&](const RowInfo &ri, int b, int cat, int rank, int NNF, int NFL) {
    const int F = NFL * P.HV, M = NNF * P.HV, c = (int)blockIdx.x;
    const int t_lo = rank * P.HV + (cat == 1 ? 0 : (cat == 0 ? F : F + M));
    const int nf = c < F ? (F - 1 - c) / G + 1 : 0;              // this CTA's flush items
    const int nn = (c < F + M ? (F + M - 1 - c) / G + 1 : 0) - nf;  // and its other live items
    for (int t = t_lo + ((c - t_lo) % G + G) % G; t < t_lo + P.HV; t += G) {
      const int q = (t - c) / G;  // rank among this CTA's items of the sequence
      int j = q;
      if (cat == 1) {  // other live items ahead: (2r + 1) nf <= (2q + 1) nn
        const int z = (2 * q + 1) * nn / nf;
        j = q + (z >= 1 ? min(nn, (z - 1) / 2 + 1) : 0);
      } else if (cat == 0) {  // flush items ahead: (2f + 1) nn < (2r + 1) nf, r = q - nf
        const int r = q - nf, y = ((2 * r + 1) * nf - 1) / nn;
        j = r + (y >= 1 ? min(nf, (y - 1) / 2 + 1) : 0);
      }
      const int hv = t - t_lo;
      if (hv == 0 && !overlap) {  // the CTA holding head 0 reports the row (with overlap: block 0, later)
        if (ri.bad) set_status(P.status, ri.bad);
        if (P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
      }
      table[j] = make_int4(ri.slot, ri.p | (ri.flush << 8) | ((ri.live ? 1 : 0) << 9) | ((hv % P.G == 0) << 10), b,
                           hv | ((hv / P.G) << 16));
    }
  };
  // category of row b (3: past the end) and its rank within the warp
  auto classify = [&](const RowInfo &ri, bool in, int &rank) {
    const int cat = in ? (ri.live ? ri.flush : 2) : 3;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const uint32_t m = __ballot_sync(0xffffffffu, cat == k);
      if (cat == k) rank = __popc(m & ((1u << lane) - 1u));
      if (lane == 0) wc[k * 32 + warp] = __popc(m);
    }
    return cat;
  };
  int NNF = 0, NFL = 0;
  if (P.B <= kTcpThreads) {  // one row per thread: one pass, one barrier
    const bool in = tid < P.B;
    const RowInfo ri = in ? resolve_row(P, tid, false) : RowInfo{-1, 0, 0, false, 0u};
    // row tid: slot << 7 | next cursor when live (next == 0: flush), else -1
    // (padding) or -1 - its status bit (an invalid slot or cursor)
    advq[tid] = ri.live ? ((ri.slot << 7) | (ri.flush ? 0 : ri.p + 1)) : -1 - (int)ri.bad;
    int rank = 0;
    const int cat = classify(ri, in, rank);
    __syncthreads();
    {
      // lane w holds warp w's counts; totals and this warp's offset by shuffles
      const int c0 = lane < NW ? wc[lane] : 0, c1 = lane < NW ? wc[32 + lane] : 0,
                c2 = lane < NW ? wc[64 + lane] : 0;
      NNF = c0;
      NFL = c1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        NNF += __shfl_xor_sync(0xffffffffu, NNF, o);
        NFL += __shfl_xor_sync(0xffffffffu, NFL, o);
      }
      // counts of each category in the warps ahead of this one
      int b0 = lane < warp ? c0 : 0, b1 = lane < warp ? c1 : 0, b2 = lane < warp ? c2 : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        b0 += __shfl_xor_sync(0xffffffffu, b0, o);
        b1 += __shfl_xor_sync(0xffffffffu, b1, o);
        b2 += __shfl_xor_sync(0xffffffffu, b2, o);
      }
      if (cat < 3) rank += cat == 0 ? b0 : (cat == 1 ? b1 : b2);
    }
    if (cat < 3) place(ri, tid, cat, rank, NNF, NFL);
  } else {  // a pass to count the categories, then one to rank and place the rows
    if (tid < 6) cnt[tid] = 0;
    __syncthreads();
    for (int base = 0; base < P.B; base += kTcpThreads) {
      const bool in = base + tid < P.B;
      const RowInfo ri = in ? resolve_row(P, base + tid, false) : RowInfo{-1, 0, 0, false, 0u};
      int rank = 0;
      const int cat = classify(ri, in, rank);
      if (lane == 0)
        for (int k = 0; k < 3; ++k)
          if (wc[k * 32 + warp]) atomicAdd(&cnt[k], wc[k * 32 + warp]);
      __syncthreads();  // wc is reused by the next chunk
    }
    NNF = cnt[0];
    NFL = cnt[1];
    for (int base = 0; base < P.B; base += kTcpThreads) {
      const bool in = base + tid < P.B;
      const RowInfo ri = in ? resolve_row(P, base + tid, false) : RowInfo{-1, 0, 0, false, 0u};
      int rank = 0;
      const int cat = classify(ri, in, rank);
      __syncthreads();
      if (cat < 3) {
        rank += carry[cat];
        for (int w = 0; w < warp; ++w) rank += wc[cat * 32 + w];
        place(ri, base + tid, cat, rank, NNF, NFL);
      }
      __syncthreads();
      if (tid < 3) {
        int t = 0;
        for (int w = 0; w < NW; ++w) t += wc[tid * 32 + w];
        carry[tid] += t;
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    const int lv = (NNF + NFL) * P.HV;  // live positions come first
    misc[4] = (int)blockIdx.x < lv ? (uint32_t)((lv - 1 - (int)blockIdx.x) / G + 1) : 0u;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  uint8_t *boxes = smem;
  uint8_t *tiles = smem + lay.off_tile;
  uint8_t *fields = smem + lay.off_field;
  uint8_t *lands = smem + lay.off_land;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (never waits for the previous launch with overlap: it reads only this
    // layer's checkpoint, which that launch does not write)
    if (lane == 0) {
      // each checkpoint box is read once: let it leave L2 first, so the rows,
      // cursors and inputs of the next launches stay there
      const uint64_t policy = l2_policy_evict_first();
      // Each epilogue group has its own NBg box slots (its items' boxes only),
      // so consecutive users of a slot are always the same group: a slot's
      // barrier can then never be waited on a lap ahead of its last phase.
      uint32_t ug[2] = {0u, 0u};
      RingPos bpg[2];
      bpg[0].init(0, NBg);
      bpg[1].init(0, NBg);
      int li = 0;  // live items seen so far
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int4 e = table[j];
        if (!tab_live(e)) continue;
        // checkpoint boxes
        const int row0 = (e.x * P.HV + tab_hv(e)) * D;
        const int g = li & 1;
        for (int c = 0; c < NBOX; ++c, ++ug[g]) {
          RingPos &bp = bpg[g];
          const int bs = g * NBg + bp.i();
          if (bp.lapped() && !(ok = wait_bar(bars.be(bs), bp.ph() ^ 1u, abort_flag, P.status))) break;
          mbar_arrive_expect_tx(bars.bf(bs), BOX_BYTES);
          tma_load_2d_hint(smem_addr(boxes + bs * BOX_BYTES), &tmap, 32 * c, row0, bars.bf(bs), policy);
          bp.advance(1, NBg);
        }
        ++li;
      }
      if (*abort_flag)  // let this thread's copies still in flight land first
        for (int g = 0; g < 2; ++g)
          for (uint32_t k = ug[g] > (uint32_t)NBg ? ug[g] - NBg : 0u; k < ug[g]; ++k)
            mbar_wait_bounded(bars.bf(g * NBg + (int)(k % NBg)), (k / NBg) & 1, kWaitLimitNs);
    }
  } else if (warp < 9) {
    // ------------------------------------------------------------ prep + MMA
    // Group pg takes the live items with li % 2 == pg; its leader also issues
    // the item's contraction into TMEM accumulator 2 pg + (li / 2) % 2.
    if (overlap) {  // the step's inputs come from the previous launch's stream order
      grid_dependency_wait();
      if (tid == 32) grid_launch_dependents();
    }
    const int pg = (warp - 1) >> 2;
    const int pt = tid - 32 - 128 * pg;  // 0..127: operand row / key channel
    const uint32_t bar_id = 1 + pg;
    const uint32_t idesc = make_idesc(KIND, D);
    volatile uint32_t *go = misc + 2 + pg;
    bool leader_ok = true;  // leader only: false after a wait ran out
    int li = 0, land_next = pg;  // leader: next live item to land
    int last_acc = -1;           // leader: accumulator and use count of its last contraction
    uint32_t last_use = 0;
    bool last_committed = true;  // leader: that contraction's completion is signalled on tmem_full
    const int nlive = (int)misc[4];
    // The group's landing slots (li % NL with NL = 4: two per group) are filled
    // by its own leader two group-items ahead: right after the group has read a
    // slot, the copies for the item that uses it next are issued.
    RingPos lp;  // landing slot of the next item to land
    lp.init(pg, NL);
    auto land = [&](int lj) {
      const int4 el = table[lj];  // the live items are the table's first entries
      const int bl = el.z, hvl = tab_hv(el), hkl = tab_hk(el);
      const int pl0 = tab_p(el), sl = el.x, l = lp.i();
      const int pl = pl0 < lay.CH ? pl0 : lay.CH;  // the first chunk's entries
      lp.advance(2, NL);
      uint8_t *ld = lands + l * lay.land_bytes;
      const uint32_t ring_bytes = (uint32_t)(pl * D * RB);
      const uint32_t gbytes = GATE == GDN_GATE_PER_K ? (uint32_t)(pl * D * 4) : 0u;
      const uint32_t qbytes = lay.qkv_bulk ? (uint32_t)(3 * D * qes) : 0u;
      mbar_arrive_expect_tx(bars.lf(l), 2 * ring_bytes + gbytes + qbytes);
      if (pl > 0) {
        const int64_t drow = ((int64_t)sl * P.HV + hvl) * P.L;
        const int64_t krow = ((int64_t)sl * P.HK + hkl) * P.L;
        bulk_load(smem_addr(ld + lay.ld_d), (const uint8_t *)P.ring_d + drow * D * RB, ring_bytes, bars.lf(l));
        bulk_load(smem_addr(ld + lay.ld_k), (const uint8_t *)P.ring_k + krow * D * RB, ring_bytes, bars.lf(l));
        if (GATE == GDN_GATE_PER_K) bulk_load(smem_addr(ld + lay.ld_g), P.ring_g + drow * D, gbytes, bars.lf(l));
      }
      if (lay.qkv_bulk) {
        const uint8_t *row = (const uint8_t *)P.qkv + (int64_t)bl * P.qkv_stride * qes;
        const uint32_t vb = (uint32_t)(D * qes);
        bulk_load(smem_addr(ld + lay.ld_q), row + (int64_t)hkl * vb, vb, bars.lf(l));
        bulk_load(smem_addr(ld + lay.ld_q + vb), row + ((int64_t)P.HK + hkl) * vb, vb, bars.lf(l));
        bulk_load(smem_addr(ld + lay.ld_q + 2 * vb), row + (2 * (int64_t)P.HK + hvl) * vb, vb, bars.lf(l));
      }
    };
    if (pt == 0)
      for (; land_next < nlive && land_next < pg + NL; land_next += 2) land(land_next);
    RingPos fp, tp, cp;  // field stage, tile stage, landing slot of this group's next item
    fp.init(pg, NF);
    tp.init(pg, NT);
    cp.init(pg, NL);
    for (int j = 0; j < n; ++j) {
      const int4 e = table[j];
      if (!tab_live(e)) continue;
      if ((li & 1) != pg) {
        ++li;
        continue;
      }
      const int p = tab_p(e), slot = e.x, s = fp.i(), t = tp.i(), l = cp.i();
      const uint32_t ph_f = fp.ph(), ph_t = tp.ph(), ph_l = cp.ph();
      const bool lap_f = fp.lapped(), lap_t = tp.lapped();
      fp.advance(2, NF);
      tp.advance(2, NT);
      cp.advance(2, NL);
      const int b = e.z, hv = tab_hv(e), hk = tab_hk(e);
      const int64_t bh = (int64_t)b * P.HV + hv;
      // GDN with an fp32 ring, chunk c >= 1 of a long replay: this thread's
      // row of the chunk's raw d and k goes by 4-byte async copies straight
      // into its place in the chunk's tile stage; the thread later rewrites
      // its own row in place (w_j d_j and k_j, rounded to tf32).
      constexpr bool kStaged = RING_DT == GDN_F32 && GATE == GDN_GATE_SCALAR;
      constexpr int KCC = kCh * ES / 16;  // 16-byte column chunks of a full chunk
      auto stage_rows = [&](int c, int tc) {
        uint8_t *sA = tiles + tc * lay.tile_bytes, *sB = sA + lay.t_B;
        const float *rd = reinterpret_cast<const float *>(P.ring_d) + ((int64_t)slot * P.HV + hv) * P.L * D + pt;
        const float *rk = reinterpret_cast<const float *>(P.ring_k) + ((int64_t)slot * P.HK + hk) * P.L * D + pt;
        if (pt < D) {
#pragma unroll
          for (int e2 = 0; e2 < kCh; ++e2) {
            const int jj = c * kCh + e2, jc = jj < p - 1 ? jj : p - 1;
            cp_async4(smem_addr(sA + tile_off(pt, e2, KCC, 4)), rd + (int64_t)jc * D);
            cp_async4(smem_addr(sB + tile_off(pt, e2, KCC, 4)), rk + (int64_t)jc * D);
          }
        }
      };
      // small loads first, so their latency overlaps the waits
      float gc = 0.f, qv = 0.f, kv = 0.f, vv = 0.f, g_lo = 0.f, g_hi = 0.f;
      if (GATE == GDN_GATE_SCALAR) {
        gc = P.g[bh];
        // every warp holds the cursor's log-gates: lane l has entries l and l + 32
        const float *grow = P.ring_g + ((int64_t)slot * P.HV + hv) * P.L;
        if (lane < p) g_lo = grow[lane];
        if (lane + 32 < p) g_hi = grow[lane + 32];
      } else if (pt < D) {
        gc = P.g[bh * D + pt];
      }
      const float beta = P.beta[bh];
      if (!lay.qkv_bulk && pt < D) {
        const int64_t qbase = (int64_t)b * P.qkv_stride;
        load3_as_f32(P.qkv, qbase + (int64_t)hk * D + pt, qbase + (int64_t)P.HK * D + (int64_t)hk * D + pt,
                     qbase + 2 * (int64_t)P.HK * D + (int64_t)hv * D + pt, P.qkv_dtype, qv, kv, vv);
      }
      // Only the leader waits (landing slot filled, tile stage read by its last
      // contraction, field stage free); the
      // go/stop word it leaves before the group barrier makes the whole group
      // leave together, so the group's barriers stay uniform.
      if (pt == 0)
        *go = (leader_ok && wait_bar(bars.lf(l), ph_l, abort_flag, P.status) &&
               (!lap_t || wait_bar(bars.tle(t), ph_t ^ 1u, abort_flag, P.status)) &&
               (!lap_f || wait_bar(bars.ine(s), ph_f ^ 1u, abort_flag, P.status)))
                  ? 1u
                  : 0u;
      named_bar_sync(bar_id, 128);
      if (*go == 0u) break;
      // the newest chunk's stage is free now (checked with the landing): its
      // copies overlap the work below
      if constexpr (kStaged) {
        if (p > lay.CH) stage_rows((p - 1) / kCh, t);
      }
      float *f = reinterpret_cast<float *>(fields + s * lay.field_bytes);
      float *fq = f, *fk = f + D, *fv = f + 2 * D, *fke = f + 3 * D, *fa = f + 4 * D, *fA = f + 5 * D,
            *fg = f + 6 * D, *scal = f + NVEC * D;
      const uint8_t *ld = lands + l * lay.land_bytes;
      const uint8_t *land_d = ld + lay.ld_d, *land_k = ld + lay.ld_k, *lq = ld + lay.ld_q;
      const float *land_g = reinterpret_cast<const float *>(ld + lay.ld_g);
      if (lay.qkv_bulk && pt < D) load3_as_f32(lq, pt, D + pt, 2 * D + pt, P.qkv_dtype, qv, kv, vv);
      float kq;
      if (!P.qk_l2norm) {
        // k.q: this thread's channel, summed over the warp; the epilogue adds
        // the four warps' partial sums
        qv *= P.q_scale;
        kq = qv * kv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
      } else {
        // in-kernel norm: q.q, k.k and k.q over the whole head, computed
        // redundantly by every warp (lane l takes the channels l, l + 32, ...);
        // warp 0 carries the sum of k.q
        float qq = 0.f, kk = 0.f;
        kq = 0.f;
        for (int c = lane; c < D; c += 32) {
          float qc, kc, unused;
          if (lay.qkv_bulk) {
            load3_as_f32(lq, c, D + c, D + c, P.qkv_dtype, qc, kc, unused);
          } else {
            const int64_t qbase = (int64_t)b * P.qkv_stride;
            load3_as_f32(P.qkv, qbase + (int64_t)hk * D + c, qbase + (int64_t)P.HK * D + (int64_t)hk * D + c,
                         qbase + (int64_t)P.HK * D + (int64_t)hk * D + c, P.qkv_dtype, qc, kc, unused);
          }
          qq = fmaf(qc, qc, qq);
          kk = fmaf(kc, kc, kk);
          kq = fmaf(kc, qc, kq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          qq += __shfl_xor_sync(0xffffffffu, qq, o);
          kk += __shfl_xor_sync(0xffffffffu, kk, o);
          kq += __shfl_xor_sync(0xffffffffu, kq, o);
        }
        const float nq = sqrtf(qq + 1e-6f), nk = sqrtf(kk + 1e-6f);
        qv = qv / nq * P.q_scale;
        kv = kv / nk;
        kq = (pt >> 5) == 0 ? kq / (nq * nk) * P.q_scale : 0.f;
      }

      // Operand rows, in chunks of kCh ring entries, the newest chunk first
      // (GDN: A row pt w_j d_j[pt], B row pt k_j[pt]; KDA: A row pt d_j[pt],
      // B row pt w_j[pt] k_j[pt]).  Chunk 0 comes from the landing slot, later
      // chunks straight from the ring in global memory; each chunk fills one
      // tile stage and is contracted into the item's accumulator.  Entries
      // j >= p are zero (selected, never multiplied: stale ring rows may hold
      // anything); their loads read row min(j, p - 1) of the slot.  The
      // weights w_j are rounded to the operand type right after, so the fast
      // exponential's error (of order 1e-6 relative for the sums seen here) is
      // far below that rounding; A, which scales the fp32 checkpoint, uses
      // the accurate one.
      float A = 1.f;
      const int jmax = p > 0 ? p - 1 : 0;
      const int ptc = pt < D ? pt : 0;
      const int nch = p > lay.CH ? (p + kCh - 1) / kCh : 1;  // lay.CH is kCh when it chunks
      const int acc = 2 * pg + ((li >> 1) & 1);
      const uint32_t ua = (uint32_t)(li >> 2);
      const int64_t drow = ((int64_t)slot * P.HV + hv) * P.L;  // ring rows of (slot, hv) / (slot, hk)
      const int64_t krow = ((int64_t)slot * P.HK + hk) * P.L;
      float w_lo = 0.f, w_hi = 0.f;  // GDN: w_j of entry j sits in lane j (lo: j < 32, hi: j >= 32)
      if (GATE == GDN_GATE_SCALAR) {
        // Suffix sums of the log-gates by a warp scan (each warp on its own):
        // afterwards lane l holds T_l = sum_{l<=i<p} g_i; w_j = exp(T_{j+1}),
        // A = exp(T_0).
        float t_lo = g_lo, t_hi = g_hi;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float a = __shfl_down_sync(0xffffffffu, t_hi, o);
          if (lane + o < 32) t_hi += a;
        }
        const float hi_total = __shfl_sync(0xffffffffu, t_hi, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float a = __shfl_down_sync(0xffffffffu, t_lo, o);
          if (lane + o < 32) t_lo += a;
        }
        t_lo += hi_total;
        A = p > 0 ? expf(__shfl_sync(0xffffffffu, t_lo, 0)) : 1.f;
        const float nxt_lo = __shfl_down_sync(0xffffffffu, t_lo, 1);
        w_lo = __expf(lane == 31 ? hi_total : nxt_lo);
        const float nxt_hi = __shfl_down_sync(0xffffffffu, t_hi, 1);
        w_hi = __expf(lane == 31 ? 0.f : nxt_hi);
      }
      // Epilogue inputs (KDA: all but the total decay per channel, which comes
      // out of the chunk loop, are written before it; GDN writes them after,
      // which the register allocation of that variant prefers).
      auto write_fields = [&]() {
      if (pt < D) {
        fk[pt] = kv;
        fv[pt] = vv;
        if (GATE == GDN_GATE_PER_K) {
          const float at = expf(gc);
          fq[pt] = at * qv;
          fke[pt] = at * kv;
          fa[pt] = at;
          fg[pt] = gc;
        } else {
          fq[pt] = qv;
        }
      }
      if (lane == 0) scal[8 + (pt >> 5)] = kq;
      if (pt == 0) {
        scal[0] = GATE == GDN_GATE_SCALAR ? expf(gc) : 1.f;
        scal[1] = beta;
        scal[4] = gc;
      }
      };
      if (GATE == GDN_GATE_PER_K) write_fields();
      float sfx = 0.f;  // KDA: the sum of this channel's gates newer than the entry at hand
      bool stop = false;
      for (int c = nch - 1; c >= 0; --c) {
        int tc = t;
        if (c != nch - 1) {  // a later chunk: the next tile stage, once its last contraction is done
          tc = tp.i();
          const uint32_t phc = tp.ph();
          const bool lapc = tp.lapped();
          tp.advance(2, NT);
          if (pt == 0)
            *go = (leader_ok && (!lapc || wait_bar(bars.tle(tc), phc ^ 1u, abort_flag, P.status))) ? 1u : 0u;
          named_bar_sync(bar_id, 128);
          if (*go == 0u) {
            stop = true;
            break;
          }
        }
        uint8_t *tA = tiles + tc * lay.tile_bytes, *tB = tA + lay.t_B;
        const int j0 = c * kCh;
        if (c == 0) {
          if (GATE == GDN_GATE_SCALAR) {
            for (int h = 0; h < lay.KC; ++h) {
              float xa[EPC], xb[EPC];
#pragma unroll
              for (int e2 = 0; e2 < EPC; ++e2) {
                const int jj = h * EPC + e2;
                const int jc = jj < jmax ? jj : jmax;
                const bool valid = jj < p && pt < D;
                const float wj = __shfl_sync(0xffffffffu, jj < 32 ? w_lo : w_hi, jj & 31);
                const float dj = load_as_f32(land_d, (int64_t)jc * D + ptc, RING_DT);
                const float kj = load_as_f32(land_k, (int64_t)jc * D + ptc, RING_DT);
                xa[e2] = valid ? wj * dj : 0.f;
                xb[e2] = valid ? kj : 0.f;
              }
              put_chunk<KIND, EPC>(tA, pt, h, lay.KC, xa);
              if (pt < D) put_chunk<KIND, EPC>(tB, pt, h, lay.KC, xb);
            }
          } else {
            // channel c = pt: w_j[c] by a backward sum over the channel's
            // gates, so the chunks of B are filled from the newest entry down
            for (int h = lay.KC - 1; h >= 0; --h) {
              float xa[EPC], xb[EPC];
#pragma unroll
              for (int e2 = EPC - 1; e2 >= 0; --e2) {
                const int jj = h * EPC + e2;
                const int jc = jj < jmax ? jj : jmax;
                const bool valid = jj < p && pt < D;
                const float wj = __expf(sfx);
                const float gj = land_g[jc * D + ptc];
                const float dj = load_as_f32(land_d, (int64_t)jc * D + ptc, RING_DT);
                const float kj = load_as_f32(land_k, (int64_t)jc * D + ptc, RING_DT);
                sfx += valid ? gj : 0.f;
                xa[e2] = valid ? dj : 0.f;
                xb[e2] = valid ? wj * kj : 0.f;
              }
              put_chunk<KIND, EPC>(tA, pt, h, lay.KC, xa);
              if (pt < D) put_chunk<KIND, EPC>(tB, pt, h, lay.KC, xb);
            }
          }
        } else if constexpr (kStaged) {
          // a chunk past the landed one, staged by async copies: rewrite this
          // thread's own row in place
          if (c != nch - 1) stage_rows(c, tc);
          cp_async_wait_all();
#pragma unroll
          for (int h = 0; h < KCC; ++h) {
            const uint32_t off = (uint32_t)((pt >> 3) * (KCC * 128) + h * 128 + (pt & 7) * 16);
            float4 ra = make_float4(0.f, 0.f, 0.f, 0.f), rb = ra;
            if (pt < D) {
              ra = *reinterpret_cast<const float4 *>(tA + off);
              rb = *reinterpret_cast<const float4 *>(tB + off);
            }
            const float rav[4] = {ra.x, ra.y, ra.z, ra.w}, rbv[4] = {rb.x, rb.y, rb.z, rb.w};
            float xa[EPC], xb[EPC];
#pragma unroll
            for (int e2 = 0; e2 < EPC; ++e2) {
              const int jj = j0 + h * EPC + e2;
              const bool valid = jj < p && pt < D;
              const float wj = __shfl_sync(0xffffffffu, jj < 32 ? w_lo : w_hi, jj & 31);
              xa[e2] = valid ? wj * rav[e2] : 0.f;
              xb[e2] = valid ? rbv[e2] : 0.f;
            }
            put_chunk<KIND, EPC>(tA, pt, h, KCC, xa);
            if (pt < D) put_chunk<KIND, EPC>(tB, pt, h, KCC, xb);
          }
        } else {
          // a chunk past the landed one, straight from global memory in two
          // halves, each half's loads in flight at once (registers allow no more)
          constexpr int HALF = kCh / 2;
          constexpr int HPC = KCC / 2;           // column chunks per half
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int half = GATE == GDN_GATE_SCALAR ? hf : 1 - hf;  // KDA walks newest first
            float dr[HALF], kr[HALF], gr[HALF];
#pragma unroll
            for (int e = 0; e < HALF; ++e) {
              const int jj = j0 + half * HALF + e, jc = jj < jmax ? jj : jmax;
              dr[e] = load_as_f32(P.ring_d, (drow + jc) * D + ptc, RING_DT);
              kr[e] = load_as_f32(P.ring_k, (krow + jc) * D + ptc, RING_DT);
              gr[e] = GATE == GDN_GATE_PER_K ? P.ring_g[(drow + jc) * D + ptc] : 0.f;
            }
            if (GATE == GDN_GATE_SCALAR) {
#pragma unroll
              for (int hh = 0; hh < HPC; ++hh) {
                float xa[EPC], xb[EPC];
#pragma unroll
                for (int e2 = 0; e2 < EPC; ++e2) {
                  const int e = hh * EPC + e2, jj = j0 + half * HALF + e;
                  const bool valid = jj < p && pt < D;
                  const float wj = __shfl_sync(0xffffffffu, jj < 32 ? w_lo : w_hi, jj & 31);
                  xa[e2] = valid ? wj * dr[e] : 0.f;
                  xb[e2] = valid ? kr[e] : 0.f;
                }
                put_chunk<KIND, EPC>(tA, pt, half * HPC + hh, KCC, xa);
                if (pt < D) put_chunk<KIND, EPC>(tB, pt, half * HPC + hh, KCC, xb);
              }
            } else {
#pragma unroll
              for (int hh = HPC - 1; hh >= 0; --hh) {
                float xa[EPC], xb[EPC];
#pragma unroll
                for (int e2 = EPC - 1; e2 >= 0; --e2) {
                  const int e = hh * EPC + e2, jj = j0 + half * HALF + e;
                  const bool valid = jj < p && pt < D;
                  const float wj = __expf(sfx);
                  sfx += valid ? gr[e] : 0.f;
                  xa[e2] = valid ? dr[e] : 0.f;
                  xb[e2] = valid ? wj * kr[e] : 0.f;
                }
                put_chunk<KIND, EPC>(tA, pt, half * HPC + hh, KCC, xa);
                if (pt < D) put_chunk<KIND, EPC>(tB, pt, half * HPC + hh, KCC, xb);
              }
            }
          }
        }
        if (c == 0) {  // the last chunk: the rest of the epilogue's inputs go with its tiles
          if (GATE == GDN_GATE_PER_K) {
            A = expf(sfx);
            if (pt < D) fA[pt] = A;
          } else {
            write_fields();
          }
          if (pt == 0) scal[2] = A;
        }
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (pt == 0 && c == 0) mbar_arrive(bars.inf(s));
        if (pt == 0 && leader_ok) {
          // the first chunk's contraction waits until the epilogue has read
          // the accumulator's previous item out
          if (c == nch - 1 && ua > 0 && !wait_bar(bars.te(acc), (ua - 1) & 1, abort_flag, P.status)) {
            leader_ok = false;
          } else {
            tc_fence_after();
            if (p > 0) {
              const uint32_t a0 = smem_addr(tA), b0 = smem_addr(tB);
              const uint32_t sbo = (uint32_t)lay.KC * 128;
              const int cnt = p - j0 < lay.CH ? p - j0 : lay.CH;  // entries of this chunk
              const int nsteps = (cnt + KSTEP - 1) / KSTEP;
              for (int i = 0; i < nsteps; ++i)
                tc_mma<KIND == 2 ? 1 : 0>(tmem + acc * D, make_sdesc(a0 + 256 * i, 128, sbo),
                                          make_sdesc(b0 + 256 * i, 128, sbo), idesc,
                                          (c != nch - 1 || i > 0) ? 1u : 0u);
              last_acc = acc;
              last_use = ua;
              last_committed = false;
              if (c == 0) {
                tc_commit(bars.tf(acc));
                last_committed = true;
              }
              tc_commit(bars.tle(tc));
            } else {
              mbar_arrive(bars.tf(acc));
              mbar_arrive(bars.tle(tc));
            }
            // after the last chunk the landing slot has been read: fill it
            // for the item that uses it next
            if (c == 0 && land_next < nlive) {
              land(land_next);
              land_next += 2;
            }
          }
        }
      }
      if (stop) break;
      ++li;
    }
    // an aborted CTA lets its last contraction and its landings finish first
    if (pt == 0 && *abort_flag) {
      if (last_acc >= 0) {
        if (!last_committed) tc_commit(bars.tf(last_acc));  // chunks issued for an item cut short
        mbar_wait_bounded(bars.tf(last_acc), last_use & 1, kWaitLimitNs);
      }
      for (int k = land_next - 2; k >= 0 && k >= land_next - NL; k -= 2)
        mbar_wait_bounded(bars.lf(k % NL), (uint32_t)(k / NL) & 1, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue (2 groups)
    if (overlap) {
      // nothing is written before the previous launch has completed
      grid_dependency_wait();
      if (warp == 9 && blockIdx.x == 0) {
        // the rows' flush flags and status bits, held back by the dealing
        if (P.B <= kTcpThreads) {
          for (int b = lane; b < P.B; b += 32) {
            const int q = advq[b];
            if (q < -1) set_status(P.status, (uint32_t)(-1 - q));
            if (P.flushed) P.flushed[b] = (q >= 0 && (q & 127) == 0) ? 1 : 0;
          }
        } else {  // read again: nothing moves the cursors before this block has counted
          for (int b = lane; b < P.B; b += 32) {
            const RowInfo ri = resolve_row(P, b, false);
            if (ri.bad) set_status(P.status, ri.bad);
            if (P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
          }
        }
      }
    }
    // Decode + advance with one row per thread ([P1] Design 3): every CTA has
    // read its cursors by the end of the dealing, so the last CTA to get past
    // it may advance them at once.  The first epilogue warp does it while it
    // waits for its first item, off the launch's tail.
    if (warp == 9 && P.sync && P.B <= kTcpThreads) {
      uint32_t last = 0u;
      if (lane == 0) {
        __threadfence();
        last = atomicAdd(P.sync, 1u) == (uint32_t)(G - 1) ? 1u : 0u;
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence();
        for (int b = lane; b < P.B; b += 32) {
          const int q = advq[b];
          if (q >= 0) P.write_pos_w[q >> 7] = q & 127;
        }
        if (lane == 0) *P.sync = 0u;  // every CTA of this launch has counted
      }
    }
    // Group eg takes the items with li % 2 == eg and reads TMEM accumulator
    // 2 eg + (li / 2) % 2.
    const int eg = (warp - 9) >> 2;
    const int etid = tid - 288 - 128 * eg;  // 0 is the group's store thread
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;  // state row = TMEM lane
    const bool row_live = r < D;   // warp-uniform
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    int li = 0;
    RingPos fp, bp;  // field stage and first checkpoint box of this group's next item
    fp.init(eg, NF);
    bp.init(0, NBg);
    for (int j = 0; j < n; ++j) {
      const int4 e = table[j];
      const int b = e.z, hv = tab_hv(e);
      const int64_t bh = (int64_t)b * P.HV + hv;
      if (!tab_live(e)) {
        if ((j & 1) == eg && row_live) store_from_f32(P.out, bh * D + r, P.out_dtype, 0.f);
        continue;
      }
      if ((li & 1) != eg) {
        ++li;
        continue;
      }
      const int p = tab_p(e), slot = e.x, flush = tab_flush(e), s = fp.i();
      const uint32_t ph_f = fp.ph();
      fp.advance(2, NF);
      const int tb = 2 * eg + ((li >> 1) & 1);
      const uint32_t ut = (uint32_t)(li >> 2);
      const RingPos box0 = bp;
      bp.advance(NBOX, NBg);
      if (!wait_bar_warp(bars.inf(s), ph_f, abort_flag, P.status)) break;
      if (!wait_bar_warp(bars.tf(tb), ut & 1, abort_flag, P.status)) break;
      tc_fence_after();
      const float *f = reinterpret_cast<const float *>(fields + s * lay.field_bytes);
      const float *fq = f, *fk = f + D, *fv = f + 2 * D, *fke = GATE == GDN_GATE_PER_K ? f + 3 * D : fk,
                  *fa = f + 4 * D, *fA = f + 5 * D, *fg = f + 6 * D, *scal = f + NVEC * D;
      const float alpha = scal[0], beta = scal[1], A = scal[2], kq = (scal[8] + scal[9]) + (scal[10] + scal[11]);
      const uint32_t trow = tmem + tb * D + lane_off;
      float2 sq01 = make_float2(0.f, 0.f), sq23 = sq01, sk01 = sq01, sk23 = sq01;
      bool ok = true;
      RingPos bq = box0;
      for (int c = 0; c < NBOX; ++c, bq.advance(1, NBg)) {
        const int bs = eg * NBg + bq.i();
        if (!(ok = wait_bar_warp(bars.bf(bs), bq.ph(), abort_flag, P.status))) break;
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
            float2 A01 = make_float2(A, A), A23 = A01;
            if (GATE == GDN_GATE_PER_K) {
              const float4 A4 = *reinterpret_cast<const float4 *>(fA + col);
              A01 = make_float2(A4.x, A4.y);
              A23 = make_float2(A4.z, A4.w);
            }
            const float2 e01 = ffma2(A01, make_float2(x.x, x.y), make_float2(acc[4 * jc], acc[4 * jc + 1]));
            const float2 e23 = ffma2(A23, make_float2(x.z, x.w), make_float2(acc[4 * jc + 2], acc[4 * jc + 3]));
            sq01 = ffma2(e01, make_float2(q4v.x, q4v.y), sq01);
            sq23 = ffma2(e23, make_float2(q4v.z, q4v.w), sq23);
            sk01 = ffma2(e01, make_float2(k4v.x, k4v.y), sk01);
            sk23 = ffma2(e23, make_float2(k4v.z, k4v.w), sk23);
          }
        }
        if (!flush) warp_arrive(bars.be(bs));
      }
      if (!ok) break;
      if (!flush) {  // only a flush item reads its accumulator again
        tc_fence_before();
        warp_arrive(bars.te(tb));
      }
      float sqt = (sq01.x + sq01.y) + (sq23.x + sq23.y);
      float skt = (sk01.x + sk01.y) + (sk23.x + sk23.y);
      if (GATE == GDN_GATE_SCALAR) {
        sqt *= alpha;
        skt *= alpha;
      }
      const float v_r = row_live ? fv[r] : 0.f;
      const float d = beta * (v_r - skt);
      if (row_live) store_from_f32(P.out, bh * D + r, P.out_dtype, fmaf(d, kq, sqt));
      const int hk = tab_hk(e);
      if (flush) {
        // second pass over the boxes: row r of alpha S + d k^T replaces row r of
        // the box; the warp then stores its 32 rows of the box to the checkpoint
        // as whole 128-byte row segments (four per instruction) and hands the
        // box back to the producer
        const float2 d2 = make_float2(d, d);
        float *gwarp = P.state + (((int64_t)slot * P.HV + hv) * D + 32 * q4) * D + 4 * (lane & 7);
        bq = box0;
        for (int c = 0; c < NBOX; ++c, bq.advance(1, NBg)) {
          const int bs = eg * NBg + bq.i();
          if (row_live) {
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
              float2 A01 = make_float2(A, A), A23 = A01, g01 = make_float2(alpha, alpha), g23 = g01;
              if (GATE == GDN_GATE_PER_K) {
                const float4 A4 = *reinterpret_cast<const float4 *>(fA + col);
                const float4 g4 = *reinterpret_cast<const float4 *>(fa + col);
                A01 = make_float2(A4.x, A4.y);
                A23 = make_float2(A4.z, A4.w);
                g01 = make_float2(g4.x, g4.y);
                g23 = make_float2(g4.z, g4.w);
              }
              const float2 e01 = ffma2(A01, make_float2(x.x, x.y), make_float2(acc[4 * jc], acc[4 * jc + 1]));
              const float2 e23 = ffma2(A23, make_float2(x.z, x.w), make_float2(acc[4 * jc + 2], acc[4 * jc + 3]));
              const float2 n01 = ffma2(d2, make_float2(k4.x, k4.y), fmul2(e01, g01));
              const float2 n23 = ffma2(d2, make_float2(k4.z, k4.w), fmul2(e23, g23));
              *px = make_float4(n01.x, n01.y, n23.x, n23.y);
            }
            __syncwarp();
            // lanes 8i .. 8i+7 take the eight 16-byte chunks of one row
            const uint8_t *wbox = boxes + bs * BOX_BYTES + 32 * q4 * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int rr = 4 * k + (lane >> 3);  // row within the warp's 32
              const float4 v = *reinterpret_cast<const float4 *>(wbox + rr * 128 + (((lane & 7) ^ (rr & 7)) << 4));
              *reinterpret_cast<float4 *>(gwarp + (int64_t)rr * D + 32 * c) = v;
            }
          }
          warp_arrive(bars.be(bs));
        }
        tc_fence_before();
        warp_arrive(bars.te(tb));
      } else {
        if (row_live) {
          store_from_f32(P.ring_d, (((int64_t)slot * P.HV + hv) * P.L + p) * D + r, RING_DT, d);
          if (GATE == GDN_GATE_PER_K) P.ring_g[(((int64_t)slot * P.HV + hv) * P.L + p) * D + r] = fg[r];
          if (tab_kw(e))
            store_from_f32(P.ring_k, (((int64_t)slot * P.HK + hk) * P.L + p) * D + r, RING_DT, fk[r]);
        }
        if (GATE == GDN_GATE_SCALAR && etid == 0) P.ring_g[((int64_t)slot * P.HV + hv) * P.L + p] = scal[4];
      }
      warp_arrive(bars.ine(s));
      ++li;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSetupWarp) {  // the warp that allocated
    tc_fence_after();
    tmem_dealloc(tmem, 4 * D);
  }

  // Decode + advance with more rows than threads ([P1] Design 3): every CTA
  // read the cursors while dealing, long before it got here; the last CTA to
  // finish advances them and leaves the counter at zero for the next launch.
  // No CTA waits for another.
  if (P.sync && P.B > kTcpThreads) {
    if (tid == 0) {
      __threadfence();
      misc[7] = atomicAdd(P.sync, 1u) == (uint32_t)(G - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (misc[7]) {
      __threadfence();
      for (int b = tid; b < P.B; b += kTcpThreads) {
        const RowInfo ri = resolve_row(P, b, false);
        if (ri.live) P.write_pos_w[ri.slot] = ri.flush ? 0 : ri.p + 1;
      }
      if (tid == 0) *P.sync = 0u;
    }
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
  // Programmatic stream serialisation: the kernel's set-up may start while the
  // previous launch in the stream finishes; it reads no input before
  // griddepcontrol.wait, which returns once that launch has completed.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcpThreads);
  cfg.dynamicSmemBytes = lay.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, P, map, lay);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int GATE>
static cudaError_t launch_tcp_ring(const DecodeParams &P, const CUtensorMap &map, const TcpLayout &lay,
                                   int grid, cudaStream_t s) {
  if (P.ring_dtype == GDN_F16) return launch_tcp_t<D, GATE, 0, GDN_F16>(P, map, lay, grid, s);
  if (P.ring_dtype == GDN_BF16) return launch_tcp_t<D, GATE, 1, GDN_BF16>(P, map, lay, grid, s);
  return launch_tcp_t<D, GATE, 2, GDN_F32>(P, map, lay, grid, s);
}

// Whether the persistent kernel takes this launch, with its layout and grid.
static bool tcp_plan(const DecodeParams &P, int D, int gate, TcpLayout *lay, int *grid) {
  static const int sms = device_attr(cudaDevAttrMultiProcessorCount);
  static const int optin = device_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin);
  const int kind = P.ring_dtype == GDN_F16 ? 0 : (P.ring_dtype == GDN_BF16 ? 1 : 2);
  const int ring_bytes = P.ring_dtype == GDN_F32 ? 4 : 2;
  const int qes = P.qkv_dtype == GDN_F32 ? 4 : 2;
  // q, k, v rows can be bulk-copied when every vector starts on 16 bytes
  const int qkv_bulk =
      ((reinterpret_cast<uintptr_t>(P.qkv) & 15u) == 0 && ((P.qkv_stride * qes) & 15) == 0) ? 1 : 0;
  if (gate == GDN_GATE_PER_K && (reinterpret_cast<uintptr_t>(P.ring_g) & 15u) != 0) return false;
  if (P.HV >= 32768) return false;       // the item table packs hv and hk into 16 bits each
  if (P.N >= (1 << 24)) return false;    // the dealing packs a row's slot in 24 bits
  const int T = P.B * P.HV;
  *grid = sms > 0 && sms < T ? sms : T;
  if ((T + *grid - 1) / *grid > kItemsMax) *grid = (T + kItemsMax - 1) / kItemsMax;
  *lay = tcp_pick_layout(D, kind, gate, P.L, ring_bytes, qes, qkv_bulk, optin);
  return lay->NB >= 2 * (D / 32) && lay->total <= (uint32_t)optin;
}

bool tcp_decode_fits(const DecodeParams &P, int D, int gate) {
  TcpLayout lay;
  int grid = 0;
  return tcp_plan(P, D, gate, &lay, &grid);
}

// Returns cudaErrorNotSupported (nothing launched) when the persistent layout
// does not fit; the caller then uses the one-CTA-per-head kernel.
cudaError_t launch_tcp_decode(const DecodeParams &P, int D, int gate, const CUtensorMap &map,
                              cudaStream_t s) {
  TcpLayout lay;
  int grid = 0;
  if (!tcp_plan(P, D, gate, &lay, &grid)) return cudaErrorNotSupported;
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_tcp_ring<128, 0>(P, map, lay, grid, s)
                                   : launch_tcp_ring<128, 1>(P, map, lay, grid, s);
  return gate == GDN_GATE_SCALAR ? launch_tcp_ring<64, 0>(P, map, lay, grid, s)
                                 : launch_tcp_ring<64, 1>(P, map, lay, grid, s);
}

}  // namespace gdn
