// Device-side helpers shared by the gdnreplay kernels: kernel parameter block,
// dtype conversion, row resolution (slot, cursor, flush decision), gate prefix,
// and thin inline-PTX wrappers for mbarrier, TMA and tcgen05.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdnreplay.h"

namespace gdn {

// Longest sleep (ns) inside one mbarrier.try_wait.
constexpr uint32_t kTryWaitSuspendNs = 1000000u;

// Parameters of one decode / fold launch, already checked on the host.
struct DecodeParams {
  int N, HV, HK, G, L;         // slots, value heads, key heads, HV/HK, ring length
  float *state;                // [N, HV, V, K]
  void *ring_d;                // [N, HV, L, V]
  void *ring_k;                // [N, HK, L, K]
  float *ring_g;               // [N, HV, L] or [N, HV, L, K]
  int ring_dtype;              // gdn_dtype_t
  const int32_t *write_pos;    // [N]
  const uint8_t *force_flush;  // [B] or null
  const void *qkv;             // [B, row]
  int qkv_dtype;
  int64_t qkv_stride;
  const float *g;              // [B, HV] or [B, HV, K]
  const float *beta;           // [B, HV]
  const int32_t *idx;          // [B]
  int B;
  float q_scale;
  int qk_l2norm;
  void *out;                   // [B, HV, V]
  int out_dtype;
  uint8_t *flushed;            // [B] or null
  uint32_t *status;            // or null
  const int32_t *slots;        // fold: [n]
  // decode + advance in one launch (persistent tensor-core kernel only): a
  // completion counter in caller workspace (zero between launches), and the
  // cursors the last CTA to finish advances; both null otherwise
  uint32_t *sync;
  int32_t *write_pos_w;
  int T;  // speculative verify: tokens per row (token t of row b is input row b * T + t)
  // GDN_STEP_OVERLAP_PREVIOUS (persistent tensor-core kernel only): the launch
  // before this one leaves the cache, cursors, rows and force_flush alone, so
  // they may be read before waiting for it
  int overlap;
  // GDN_STEP_PERSISTENT_KERNEL: tensor-core recon always takes the persistent
  // kernel, never the small-batch one
  int persistent_only;
};

__device__ __forceinline__ float load_as_f32(const void *p, int64_t i, int dtype) {
  if (dtype == GDN_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  if (dtype == GDN_F16) return __half2float(reinterpret_cast<const __half *>(p)[i]);
  return reinterpret_cast<const float *>(p)[i];
}

// Three loads of the same dtype as fp32 (one dtype dispatch for all three).
__device__ __forceinline__ void load3_as_f32(const void *p, int64_t i0, int64_t i1, int64_t i2, int dtype,
                                             float &a, float &b, float &c) {
  if (dtype == GDN_BF16) {
    const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(p);
    a = __bfloat162float(q[i0]);
    b = __bfloat162float(q[i1]);
    c = __bfloat162float(q[i2]);
  } else if (dtype == GDN_F16) {
    const __half *q = reinterpret_cast<const __half *>(p);
    a = __half2float(q[i0]);
    b = __half2float(q[i1]);
    c = __half2float(q[i2]);
  } else {
    const float *q = reinterpret_cast<const float *>(p);
    a = q[i0];
    b = q[i1];
    c = q[i2];
  }
}

// Store with round-to-nearest-even to the destination type.
__device__ __forceinline__ void store_from_f32(void *p, int64_t i, int dtype, float x) {
  if (dtype == GDN_BF16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else if (dtype == GDN_F16) reinterpret_cast<__half *>(p)[i] = __float2half_rn(x);
  else reinterpret_cast<float *>(p)[i] = x;
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Row b's slot, cursor and flush decision ([P1] Design 3 and 5; [P2] 3.1, 3.3).
struct RowInfo {
  int slot;   // >= 0 for a live row
  int p;      // ring entries to replay
  int flush;  // 1: write the checkpoint, no ring append
  bool live;
  uint32_t bad;  // status bit of an invalid slot or cursor, else 0
};

__device__ __forceinline__ RowInfo resolve_row(const DecodeParams &P, int b, bool report) {
  // loads cached in L2 only: a kernel may read these before the launch ahead
  // of it has completed (programmatic dependent launch), and no line of them
  // left in this SM's L1 by an earlier kernel may be used
  RowInfo r{-1, 0, 0, false, 0u};
  int slot = __ldcg(P.idx + b);
  if (slot < 0) return r;
  if (slot >= P.N) {
    r.bad = GDN_DEV_BAD_SLOT;
    if (report) set_status(P.status, r.bad);
    return r;
  }
  int p = __ldcg(P.write_pos + slot);
  if (p < 0 || p >= P.L) {
    r.bad = GDN_DEV_BAD_WRITE_POS;
    if (report) set_status(P.status, r.bad);
    return r;
  }
  r.slot = slot;
  r.p = p;
  r.flush = (p == P.L - 1) || (P.force_flush != nullptr && __ldcg(P.force_flush + b) != 0);
  r.live = true;
  return r;
}

// Replay decays from the cached log-gates of one channel ([P1] Design 1 and 7):
// w_j = exp(sum_{j<i<p} g_i), A = exp(sum_{i<p} g_i), summed from the newest
// entry backwards so no difference of partial sums is ever formed.
// g points at entry 0 of the channel, entries `stride` floats apart.
__device__ __forceinline__ float replay_decays(const float *g, int stride, int p, float *w,
                                               int w_stride) {
  float s = 0.f;
  for (int j = p - 1; j >= 0; --j) {
    w[j * w_stride] = expf(s);
    s += g[(int64_t)j * stride];
  }
  return expf(s);
}

// ---------------------------------------------------------------------------
// Row inputs (CTA of 128 threads).
// ---------------------------------------------------------------------------

__device__ __forceinline__ float dot4(const float4 &a, const float4 &b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  acc = fmaf(a.w, b.w, acc);
  return acc;
}

// Sum of x and of y over the first 128 threads of the CTA, returned to every
// thread (a CTA of more threads passes zeros from the others, which add nothing
// and are not read).
__device__ __forceinline__ float2 block_sum2(float x, float y, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  if (lane == 0 && warp < 4) {
    red[warp] = x;
    red[4 + warp] = y;
  }
  __syncthreads();
  float2 r = make_float2((red[0] + red[1]) + (red[2] + red[3]), (red[4] + red[5]) + (red[6] + red[7]));
  __syncthreads();
  return r;
}

// Row b's raw inputs for thread t = key / value channel t (zeros for t >= D):
// q and k of key head hv / G, v of value head hv ([P2] 3.1 packed input).
struct QkvRaw {
  float q, k, v;
};

template <int D>
__device__ __forceinline__ QkvRaw load_qkv_raw(const DecodeParams &P, int b, int hv) {
  const int t = threadIdx.x;
  const int hk = hv / P.G;
  const int64_t base = (int64_t)b * P.qkv_stride;
  QkvRaw x{0.f, 0.f, 0.f};
  if (t < D)
    load3_as_f32(P.qkv, base + (int64_t)hk * D + t, base + (int64_t)P.HK * D + (int64_t)hk * D + t,
                 base + 2 * (int64_t)P.HK * D + (int64_t)hv * D + t, P.qkv_dtype, x.q, x.k, x.v);
  return x;
}

// Applies the optional L2 norm and q_scale to one token's raw inputs, publishes
// q, k, v to shared memory and returns k^T q (a CTA-wide sum; ends with a CTA
// barrier).  Every rounding is pinned, so kernels that share it agree bit for bit.
template <int D>
__device__ __forceinline__ float finish_qkv(const DecodeParams &P, QkvRaw x, float *q, float *k, float *v,
                                            float *red) {
  const int t = threadIdx.x;
  float qt = x.q, kt = x.k;
  if (t < D) v[t] = x.v;
  if (P.qk_l2norm) {
    float2 n = block_sum2(__fmul_rn(qt, qt), __fmul_rn(kt, kt), red);
    qt = __fdiv_rn(qt, __fsqrt_rn(__fadd_rn(n.x, 1e-6f)));
    kt = __fdiv_rn(kt, __fsqrt_rn(__fadd_rn(n.y, 1e-6f)));
  }
  qt = __fmul_rn(qt, P.q_scale);
  if (t < D) {
    q[t] = qt;
    k[t] = kt;
  }
  float2 kq = block_sum2(__fmul_rn(kt, qt), 0.f, red);  // also publishes q, k, v
  return kq.x;
}

// Loads q, k (key head hv / G) and v (value head hv) of row b as fp32, applies
// the optional L2 norm and q_scale, and returns k^T q ([P2] 3.1 packed input).
template <int D>
__device__ float load_qkv(const DecodeParams &P, int b, int hv, float *q, float *k, float *v,
                          float *red) {
  return finish_qkv<D>(P, load_qkv_raw<D>(P, b, hv), q, k, v, red);
}

// ---------------------------------------------------------------------------
// Inline PTX: shared-memory addresses, mbarrier, TMA, tcgen05.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// atomicAdd with release semantics at GPU scope: this thread's earlier memory
// accesses are performed before the addition is (the result is not waited on
// until it is used).
__device__ __forceinline__ uint32_t atomic_add_release_gpu(uint32_t *addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch: wait until the grid this one depends on has
// completed and its memory is visible (a no-op without such a dependency), and
// allow the grid that depends on this one to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Barrier among `nthreads` threads (whole warps) on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  // The thread may sleep in the instruction until the phase completes, for at
  // most the hint (ns), so a waiting warp takes no issue slots meanwhile.
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, P1;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(kTryWaitSuspendNs)
      : "memory");
  return done != 0;
}

// Non-blocking test of the phase with the given parity (no suspend).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P1;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// limit_ns of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same load with an L2 cache policy (e.g. evict-first for data read once).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy: lines brought in under it are the first to be evicted.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Contiguous bulk copy global -> shared (both 16-byte aligned, size a multiple
// of 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Asynchronous 4-byte copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}

// Waits until every cp.async this thread has issued has landed in shared memory.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One arrival on `bar` once every cp.async this thread issued so far has
// landed; the arrival is not added to the barrier's expected count, so the
// barrier must have been initialised to include it.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2-D tiled TMA store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --- tcgen05 (5th-generation tensor core, accumulator in tensor memory) ---

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction, issued by one thread.
template <int KIND>  // 0: kind::f16 (f16/bf16 operands), 1: kind::tf32
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if constexpr (KIND == 0) {
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "setp.ne.b32 P1, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "setp.ne.b32 P1, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, P1;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Packed fp32x2 arithmetic (two independent round-to-nearest fp32 operations per
// instruction, bit-identical to two fmaf / __fmul_rn calls).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d, ua, ub, uc;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(uc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(ua), "l"(ub), "l"(uc));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d, ua, ub;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ua) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(ub) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(ua), "l"(ub));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// Round an fp32 value to tf32 (nearest, ties away from zero), kept in fp32 bits.
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

}  // namespace gdn
