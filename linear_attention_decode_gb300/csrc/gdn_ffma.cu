// CUDA-core kernels: the packed read+write decode (the baseline), the ReplaySSM
// decode with the replay sum evaluated term by term in fp32 FFMA, the standalone
// ring fold, and the cursor advance / reset kernels.
//
// Thread mapping of the row loops: one CTA per (row, value head), 4 warps.  A
// warp works on 4 state rows at a time; lane = 8 * row_in_group + column_group,
// and a lane owns columns 32*m + 4*column_group + {0..3} (m < K/32), so each
// 16-byte load of a warp covers four 128-byte runs of four rows and a row's
// contraction over K needs only a 3-step shuffle among its 8 lanes.
#include "gdn_bits.cuh"
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

constexpr int kThreads = 128;

// Stages the replay operands of (slot, hv) in shared memory ([P1] Design 1, 7):
//   GDN: Dw[j][r] = w_j d_j[r], Kr[j][c] = k_j[c], returns A;
//   KDA: Dw[j][r] = d_j[r],     Kr[j][c] = w_j[c] k_j[c], Acol[c] = A[c].
// Only entries j < p are read; the ring rows are fetched kStageBatch entries
// at a time so their loads are in flight together.  Ends with a CTA barrier.
constexpr int kStageBatch = 8;

// In-place suffix decays of one channel: on entry x[j * stride] = g_j, on exit
// x[j * stride] = w_j = exp(sum_{j<i<p} g_i); returns A = exp(sum_{i<p} g_i).
// The sums run from the newest entry backwards, as replay_decays does.
__device__ __forceinline__ float decays_in_place(float *x, int stride, int p) {
  float s = 0.f;
  for (int j = p - 1; j >= 0; --j) {
    const float gj = x[j * stride];
    x[j * stride] = expf(s);
    s += gj;
  }
  return expf(s);
}

template <int D, int GATE>
__device__ float stage_replay(const DecodeParams &P, int slot, int hv, int p, float *wv,
                              float *Acol, float *Dw, float *Kr) {
  const int t = threadIdx.x;
  const int hk = hv / P.G;
  const int64_t dbase = ((int64_t)slot * P.HV + hv) * P.L * D;
  const int64_t kbase = ((int64_t)slot * P.HK + hk) * P.L * D;
  float A = 1.f;
  if (GATE == GDN_GATE_SCALAR) {
    if (t < p) wv[t] = P.ring_g[((int64_t)slot * P.HV + hv) * P.L + t];
    __syncthreads();
    if (t == 0) wv[63] = decays_in_place(wv, 1, p);
    __syncthreads();
    A = wv[63];
  } else if (t < D) {
    const float *g = P.ring_g + ((int64_t)slot * P.HV + hv) * P.L * D + t;
    for (int j0 = 0; j0 < p; j0 += kStageBatch) {
      float gv[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) gv[u] = j0 + u < p ? g[(int64_t)(j0 + u) * D] : 0.f;
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u)
        if (j0 + u < p) Kr[(j0 + u) * D + t] = gv[u];
    }
    Acol[t] = decays_in_place(Kr + t, D, p);  // w_j[c] parked in Kr
  }
  if (t < D) {
    for (int j0 = 0; j0 < p; j0 += kStageBatch) {
      float dv[kStageBatch], kv[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        dv[u] = 0.f;
        kv[u] = 0.f;
        if (j0 + u < p) {
          dv[u] = load_as_f32(P.ring_d, dbase + (int64_t)(j0 + u) * D + t, P.ring_dtype);
          kv[u] = load_as_f32(P.ring_k, kbase + (int64_t)(j0 + u) * D + t, P.ring_dtype);
        }
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int j = j0 + u;
        if (j < p) {
          if (GATE == GDN_GATE_SCALAR) {
            Dw[j * D + t] = wv[j] * dv[u];
            Kr[j * D + t] = kv[u];
          } else {
            Dw[j * D + t] = dv[u];
            Kr[j * D + t] *= kv[u];
          }
        }
      }
    }
  }
  __syncthreads();
  return A;
}

// The per-token arithmetic of one state row, shared by the packed decode and
// the lossless verify and commit so that they agree bit for bit: every rounding
// is pinned (mul.rn / sub.rn / fma.rn; nothing the compiler may contract).
//
// token_out: once the row's 8 lanes hold partial sums of S x (x = q, k; KDA
// a o q, a o k), sums them (xor 1, 2, 4) and forms
//   GDN: sq, sk <- alpha sq, alpha sk;   d = beta (v_r - sk);   o = sq + d (k^T q).
template <int GATE>
__device__ __forceinline__ float token_out(float sq, float sk, float alpha, float beta, float vr, float kq,
                                           float &d) {
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  if (GATE == GDN_GATE_SCALAR) {
    sq = __fmul_rn(sq, alpha);
    sk = __fmul_rn(sk, alpha);
  }
  d = __fmul_rn(beta, __fsub_rn(vr, sk));
  return __fmaf_rn(d, kq, sq);
}

// token_update: four columns of the row after the token,
//   GDN: s <- fma(d, k, fl(alpha s));   KDA: s <- fma(d, k, fl(s a))
// (the decayed state is one rounded multiply, the rank-1 update one fma).
// Packed fp32x2 operations round each element exactly as mul.rn / fma.rn do.
template <int GATE>
__device__ __forceinline__ float4 token_update(const float4 &s, const float4 &k, const float4 &a, float alpha,
                                               float d) {
  const float2 dd = make_float2(d, d);
  float2 lo, hi;
  if (GATE == GDN_GATE_SCALAR) {
    const float2 aa = make_float2(alpha, alpha);
    lo = __ffma2_rn(dd, make_float2(k.x, k.y), __fmul2_rn(aa, make_float2(s.x, s.y)));
    hi = __ffma2_rn(dd, make_float2(k.z, k.w), __fmul2_rn(aa, make_float2(s.z, s.w)));
  } else {
    lo = __ffma2_rn(dd, make_float2(k.x, k.y), __fmul2_rn(make_float2(s.x, s.y), make_float2(a.x, a.y)));
    hi = __ffma2_rn(dd, make_float2(k.z, k.w), __fmul2_rn(make_float2(s.z, s.w), make_float2(a.z, a.w)));
  }
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// This lane's partial sum of a state row against x over its M float4 column
// chunks: one fma chain per float4 component (m ascending; two packed fp32x2
// chains), the four chains added pairwise.  Short chains, pinned order.
template <int M>
__device__ __forceinline__ float lane_dot(const float4 (&s)[M], const float4 (&x)[M]) {
  float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    lo = __ffma2_rn(make_float2(s[m].x, s[m].y), make_float2(x[m].x, x[m].y), lo);
    hi = __ffma2_rn(make_float2(s[m].z, s[m].w), make_float2(x[m].z, x[m].w), hi);
  }
  return __fadd_rn(__fadd_rn(lo.x, lo.y), __fadd_rn(hi.x, hi.y));
}

__device__ __forceinline__ float4 mul4(const float4 &a, const float4 &b) {
  return make_float4(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y), __fmul_rn(a.z, b.z), __fmul_rn(a.w, b.w));
}

// REPLAY = false: packed decode (read S, write S every step).
// REPLAY = true:  ReplaySSM decode with the replay sum on the CUDA cores.
// OUT_ONLY (with REPLAY): a non-flush row never forms the replayed state; its
// readout is factored through the ring ([P1] Design 1, the output-only form; [P2] 3.2):
//   GDN: S x = A (S0 x) + sum_j (w_j d_j) (k_j . x),
//   KDA: S x = S0 (A o x) + sum_j d_j ((w_j o k_j) . x),   x = q, k (KDA: a o q, a o k),
// O(V K + p (V + K)) per head instead of O(p V K).  Flush rows rebuild S as above.
template <int D, int GATE, bool REPLAY, bool OUT_ONLY = false>
__global__ void __launch_bounds__(kThreads) ffma_decode_kernel(const DecodeParams P) {
  constexpr int M = D / 32;             // float4 chunks per lane per row
  constexpr int ROWS_PER_WARP = D / 4;  // 4 warps
  constexpr int NIT = ROWS_PER_WARP / 4;
  const int b = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rg = lane >> 3, cg = lane & 7;
  extern __shared__ float4 smem_f4[];
  float *q = reinterpret_cast<float *>(smem_f4);
  float *k = q + D, *v = k + D, *a = v + D, *Acol = a + D, *red = Acol + D, *wv = red + 8;
  float *Dw = wv + 64, *Kr = Dw + (P.L - 1) * D;
  float *zq = Kr + (P.L - 1) * D, *zk = zq + 64;  // OUT_ONLY: k_j . x for the staged entries

  RowInfo ri;
  if (REPLAY) {
    ri = resolve_row(P, b, hv == 0 && t == 0);
  } else {
    int slot = P.idx[b];
    ri = RowInfo{slot, 0, 1, slot >= 0 && slot < P.N};
    if (slot >= P.N && hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
  }
  if (REPLAY && hv == 0 && t == 0 && P.flushed) P.flushed[b] = ri.live ? (uint8_t)ri.flush : 0;
  if (!ri.live) {  // padding row: zeros, no cache access
    if (t < D) store_from_f32(P.out, ((int64_t)b * P.HV + hv) * D + t, P.out_dtype, 0.f);
    return;
  }
  const int slot = ri.slot, p = ri.p;
  const int64_t bh = (int64_t)b * P.HV + hv;

  // the checkpoint's first rows are requested before the inputs and the ring
  float4 *S = reinterpret_cast<float4 *>(P.state + ((int64_t)slot * P.HV + hv) * D * D);
  float4 cur[M], nxt[M];
  {
    const int r0 = warp * ROWS_PER_WARP + rg;
#pragma unroll
    for (int m = 0; m < M; ++m) cur[m] = S[r0 * (D / 4) + 8 * m + cg];
  }

  const float kq = load_qkv<D>(P, b, hv, q, k, v, red);
  const float beta = P.beta[bh];
  float alpha = 1.f, A = 1.f;
  if (GATE == GDN_GATE_SCALAR) {
    alpha = expf(P.g[bh]);
  } else if (t < D) {
    a[t] = expf(P.g[bh * D + t]);
    Acol[t] = 1.f;
  }
  if (REPLAY) {
    A = stage_replay<D, GATE>(P, slot, hv, p, wv, Acol, Dw, Kr);
  } else {
    __syncthreads();
  }
  const bool out_only = OUT_ONLY && !ri.flush;
  if (out_only) {  // zq[j] = Kr[j] . x_q, zk[j] = Kr[j] . x_k, one warp per entry
    for (int j = warp; j < p; j += 4) {
      float zqa = 0.f, zka = 0.f;
      for (int c = lane; c < D; c += 32) {
        const float kr = Kr[j * D + c];
        const float ac = GATE == GDN_GATE_PER_K ? a[c] : 1.f;
        zqa = fmaf(kr, ac * q[c], zqa);
        zka = fmaf(kr, ac * k[c], zka);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        zqa += __shfl_xor_sync(0xffffffffu, zqa, o);
        zka += __shfl_xor_sync(0xffffffffu, zka, o);
      }
      if (lane == 0) {
        zq[j] = zqa;
        zk[j] = zka;
      }
    }
    __syncthreads();
  }

  // Per-lane column constants.
  float4 qe[M], ke[M], kraw[M], a4[M], A4[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c4 = 8 * m + cg;
    kraw[m] = reinterpret_cast<const float4 *>(k)[c4];
    qe[m] = reinterpret_cast<const float4 *>(q)[c4];
    ke[m] = kraw[m];
    a4[m] = A4[m] = make_float4(1.f, 1.f, 1.f, 1.f);
    if (GATE == GDN_GATE_PER_K) {
      a4[m] = reinterpret_cast<const float4 *>(a)[c4];
      A4[m] = reinterpret_cast<const float4 *>(Acol)[c4];
      qe[m] = mul4(a4[m], qe[m]);
      ke[m] = mul4(a4[m], ke[m]);
    }
  }

#pragma unroll 1
  for (int it = 0; it < NIT; ++it) {
    const int r = warp * ROWS_PER_WARP + it * 4 + rg;
    if (it + 1 < NIT) {
#pragma unroll
      for (int m = 0; m < M; ++m) nxt[m] = S[(r + 4) * (D / 4) + 8 * m + cg];
    }
    float sq = 0.f, sk = 0.f;
    float4 s[M];
    if (out_only) {
      // S0 row r against the decayed readout vectors, plus this lane's share
      // (j = cg mod 8) of the ring terms; the row's shuffle sums the rest.
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float4 c = GATE == GDN_GATE_PER_K
                             ? make_float4(A4[m].x * cur[m].x, A4[m].y * cur[m].y, A4[m].z * cur[m].z,
                                           A4[m].w * cur[m].w)
                             : cur[m];
        sq = dot4(c, qe[m], sq);
        sk = dot4(c, ke[m], sk);
      }
      if (GATE == GDN_GATE_SCALAR) {
        sq *= A;
        sk *= A;
      }
      for (int j = cg; j < p; j += 8) {
        const float dw = Dw[j * D + r];
        sq = fmaf(dw, zq[j], sq);
        sk = fmaf(dw, zk[j], sk);
      }
    } else {
    // Replayed row r of the pre-token state.
#pragma unroll
    for (int m = 0; m < M; ++m) {
      if (GATE == GDN_GATE_SCALAR) {
        s[m] = REPLAY ? make_float4(A * cur[m].x, A * cur[m].y, A * cur[m].z, A * cur[m].w) : cur[m];
      } else {
        s[m] = REPLAY ? make_float4(A4[m].x * cur[m].x, A4[m].y * cur[m].y, A4[m].z * cur[m].z,
                                    A4[m].w * cur[m].w)
                      : cur[m];
      }
    }
    if (REPLAY) {
      for (int j = 0; j < p; ++j) {
        const float dw = Dw[j * D + r];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const float4 kr = reinterpret_cast<const float4 *>(Kr + j * D)[8 * m + cg];
          s[m].x = fmaf(dw, kr.x, s[m].x);
          s[m].y = fmaf(dw, kr.y, s[m].y);
          s[m].z = fmaf(dw, kr.z, s[m].z);
          s[m].w = fmaf(dw, kr.w, s[m].w);
        }
      }
    }
    sq = lane_dot<M>(s, qe);
    sk = lane_dot<M>(s, ke);
    }
    float d;
    const float o = token_out<GATE>(sq, sk, alpha, beta, v[r], kq, d);
    if (cg == 0) store_from_f32(P.out, bh * D + r, P.out_dtype, o);
    if (ri.flush) {
#pragma unroll
      for (int m = 0; m < M; ++m) S[r * (D / 4) + 8 * m + cg] = token_update<GATE>(s[m], kraw[m], a4[m], alpha, d);
    } else if (cg == 0) {
      store_from_f32(P.ring_d, (((int64_t)slot * P.HV + hv) * P.L + p) * D + r, P.ring_dtype, d);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) cur[m] = nxt[m];
  }

  if (REPLAY && !ri.flush) {  // ring append of k (one writer per key head) and g
    const int hk = hv / P.G;
    if (GATE == GDN_GATE_SCALAR) {
      if (t == 0) P.ring_g[((int64_t)slot * P.HV + hv) * P.L + p] = P.g[bh];
    } else if (t < D) {
      P.ring_g[(((int64_t)slot * P.HV + hv) * P.L + p) * D + t] = P.g[bh * D + t];
    }
    if (hv % P.G == 0 && t < D)
      store_from_f32(P.ring_k, (((int64_t)slot * P.HK + hk) * P.L + p) * D + t, P.ring_dtype, k[t]);
  }
}

// Standalone fold: state[s, hv] <- replayed state with write_pos[s] entries.
template <int D, int GATE>
__global__ void __launch_bounds__(kThreads) fold_kernel(const DecodeParams P) {
  constexpr int M = D / 32;
  constexpr int ROWS_PER_WARP = D / 4;
  const int i = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rg = lane >> 3, cg = lane & 7;
  extern __shared__ float4 smem_f4[];
  float *Acol = reinterpret_cast<float *>(smem_f4), *wv = Acol + D, *Dw = wv + 64;
  float *Kr = Dw + (P.L - 1) * D;
  const int slot = P.slots[i];
  if (slot < 0) return;
  if (slot >= P.N) {
    if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
    return;
  }
  const int p = P.write_pos[slot];
  if (p < 0 || p >= P.L) {
    if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_WRITE_POS);
    return;
  }
  if (GATE == GDN_GATE_PER_K && t < D) Acol[t] = 1.f;
  const float A = stage_replay<D, GATE>(P, slot, hv, p, wv, Acol, Dw, Kr);
  float4 A4[M];
#pragma unroll
  for (int m = 0; m < M; ++m)
    A4[m] = GATE == GDN_GATE_PER_K ? reinterpret_cast<const float4 *>(Acol)[8 * m + cg]
                                   : make_float4(A, A, A, A);
  float4 *S = reinterpret_cast<float4 *>(P.state + ((int64_t)slot * P.HV + hv) * D * D);
  for (int it = 0; it < ROWS_PER_WARP / 4; ++it) {
    const int r = warp * ROWS_PER_WARP + it * 4 + rg;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4 c = S[r * (D / 4) + 8 * m + cg];
      float4 s = make_float4(A4[m].x * c.x, A4[m].y * c.y, A4[m].z * c.z, A4[m].w * c.w);
      for (int j = 0; j < p; ++j) {
        const float dw = Dw[j * D + r];
        const float4 kr = reinterpret_cast<const float4 *>(Kr + j * D)[8 * m + cg];
        s.x = fmaf(dw, kr.x, s.x);
        s.y = fmaf(dw, kr.y, s.y);
        s.z = fmaf(dw, kr.z, s.z);
        s.w = fmaf(dw, kr.w, s.w);
      }
      S[r * (D / 4) + 8 * m + cg] = s;
    }
  }
}

// Speculative verify window ([P3] Core concept, Design notes): row b's T
// tokens are decoded from the checkpoint and the first p = write_pos[slot]
// ring entries, token t as the non-flush decode at cursor p + t would decode
// it: its output uses the exact correction d_t, and the state carried to token
// t + 1 takes d_t and k_t as they are cached at ring position p + t (rounded
// to the ring type), as a committed entry would be replayed.  Needs
// p + T <= L - 1; neither the checkpoint nor the cursor changes.  The state row
// recurrence is row-separable, so each state row is rebuilt once and carried
// through the window in registers.
template <int D, int GATE>
__global__ void __launch_bounds__(kThreads) spec_verify_kernel(const DecodeParams P) {
  constexpr int M = D / 32;
  constexpr int ROWS_PER_WARP = D / 4;
  const int b = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rg = lane >> 3, cg = lane & 7;
  const int T = P.T;
  extern __shared__ float4 smem_f4[];
  // window vectors: q (a o q for KDA), k, v, a (KDA), k rounded to the ring type; scalars
  float *wq = reinterpret_cast<float *>(smem_f4);
  float *wk = wq + T * D, *wv_ = wk + T * D, *wa = wv_ + T * D, *wkr = wa + T * D;
  float *wsc = wkr + T * D;  // [T][4]: alpha, beta, k.q
  float *Acol = wsc + 4 * T, *red = Acol + D, *wv = red + 8, *Dw = wv + 64;
  float *Kr = Dw + (P.L - 1) * D;
  float *q = Kr + (P.L - 1) * D, *k = q + D, *v = k + D;  // scratch for one token's inputs

  int slot = P.idx[b];
  bool live = slot >= 0;
  int p = 0;
  if (slot >= P.N) {
    if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
    live = false;
  } else if (live) {
    p = P.write_pos[slot];
    if (p < 0 || p + T > P.L - 1) {
      if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_WRITE_POS);
      live = false;
    }
  }
  if (!live) {  // padding row: zeros for every window token, no cache access
    for (int tok = 0; tok < T; ++tok)
      if (t < D) store_from_f32(P.out, (((int64_t)b * T + tok) * P.HV + hv) * D + t, P.out_dtype, 0.f);
    return;
  }

  // Window inputs, token by token (load_qkv reduces over the CTA).
  for (int tok = 0; tok < T; ++tok) {
    const int row = b * T + tok;
    const int64_t bh = (int64_t)row * P.HV + hv;
    const float kq = load_qkv<D>(P, row, hv, q, k, v, red);
    if (t < D) {
      float a = 1.f;
      if (GATE == GDN_GATE_PER_K) a = expf(P.g[bh * D + t]);
      wq[tok * D + t] = GATE == GDN_GATE_PER_K ? a * q[t] : q[t];
      wk[tok * D + t] = k[t];
      wv_[tok * D + t] = v[t];
      wa[tok * D + t] = a;
      // the key as the ring caches it (and as a later token replays it)
      float kr = k[t];
      if (P.ring_dtype == GDN_F16) kr = __half2float(__float2half_rn(kr));
      else if (P.ring_dtype == GDN_BF16) kr = __bfloat162float(__float2bfloat16_rn(kr));
      wkr[tok * D + t] = kr;
    }
    if (t == 0) {
      wsc[4 * tok + 0] = GATE == GDN_GATE_SCALAR ? expf(P.g[bh]) : 1.f;
      wsc[4 * tok + 1] = P.beta[bh];
      wsc[4 * tok + 2] = kq;
    }
    __syncthreads();
  }
  if (GATE == GDN_GATE_PER_K && t < D) Acol[t] = 1.f;
  const float A = stage_replay<D, GATE>(P, slot, hv, p, wv, Acol, Dw, Kr);
  float4 A4[M];
#pragma unroll
  for (int m = 0; m < M; ++m)
    A4[m] = GATE == GDN_GATE_PER_K ? reinterpret_cast<const float4 *>(Acol)[8 * m + cg]
                                   : make_float4(A, A, A, A);

  const float4 *S = reinterpret_cast<const float4 *>(P.state + ((int64_t)slot * P.HV + hv) * D * D);
  for (int it = 0; it < ROWS_PER_WARP / 4; ++it) {
    const int r = warp * ROWS_PER_WARP + it * 4 + rg;
    // row r of the state before the window
    float4 s[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4 c = S[r * (D / 4) + 8 * m + cg];
      s[m] = make_float4(A4[m].x * c.x, A4[m].y * c.y, A4[m].z * c.z, A4[m].w * c.w);
    }
    for (int j = 0; j < p; ++j) {
      const float dw = Dw[j * D + r];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float4 kr = reinterpret_cast<const float4 *>(Kr + j * D)[8 * m + cg];
        s[m].x = fmaf(dw, kr.x, s[m].x);
        s[m].y = fmaf(dw, kr.y, s[m].y);
        s[m].z = fmaf(dw, kr.z, s[m].z);
        s[m].w = fmaf(dw, kr.w, s[m].w);
      }
    }
    // the window, token by token
    for (int tok = 0; tok < T; ++tok) {
      const float alpha = wsc[4 * tok], beta = wsc[4 * tok + 1], kq = wsc[4 * tok + 2];
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c4 = 8 * m + cg;
        const float4 q4 = reinterpret_cast<const float4 *>(wq + tok * D)[c4];
        float4 k4 = reinterpret_cast<const float4 *>(wk + tok * D)[c4];
        if (GATE == GDN_GATE_PER_K) {
          const float4 a4 = reinterpret_cast<const float4 *>(wa + tok * D)[c4];
          k4 = make_float4(a4.x * k4.x, a4.y * k4.y, a4.z * k4.z, a4.w * k4.w);
        }
        sq = dot4(s[m], q4, sq);
        sk = dot4(s[m], k4, sk);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (GATE == GDN_GATE_SCALAR) {
        sq *= alpha;
        sk *= alpha;
      }
      const float d = beta * (wv_[tok * D + r] - sk);
      const int64_t orow = ((int64_t)b * T + tok) * P.HV + hv;
      if (cg == 0) {
        store_from_f32(P.out, orow * D + r, P.out_dtype, fmaf(d, kq, sq));
        store_from_f32(P.ring_d, (((int64_t)slot * P.HV + hv) * P.L + p + tok) * D + r, P.ring_dtype, d);
      }
      // carry row r to the next token with (d, k) as cached
      float dr = d;
      if (P.ring_dtype == GDN_F16) dr = __half2float(__float2half_rn(dr));
      else if (P.ring_dtype == GDN_BF16) dr = __bfloat162float(__float2bfloat16_rn(dr));
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c4 = 8 * m + cg;
        const float4 kr = reinterpret_cast<const float4 *>(wkr + tok * D)[c4];
        if (GATE == GDN_GATE_SCALAR) {
          s[m] = make_float4(fmaf(dr, kr.x, alpha * s[m].x), fmaf(dr, kr.y, alpha * s[m].y),
                             fmaf(dr, kr.z, alpha * s[m].z), fmaf(dr, kr.w, alpha * s[m].w));
        } else {
          const float4 a4 = reinterpret_cast<const float4 *>(wa + tok * D)[c4];
          s[m] = make_float4(fmaf(dr, kr.x, s[m].x * a4.x), fmaf(dr, kr.y, s[m].y * a4.y),
                             fmaf(dr, kr.z, s[m].z * a4.z), fmaf(dr, kr.w, s[m].w * a4.w));
        }
      }
    }
  }
  // k (one writer per key head) and g of every window token
  const int hk = hv / P.G;
  for (int tok = 0; tok < T; ++tok) {
    const int64_t bh = ((int64_t)b * T + tok) * P.HV + hv;
    const int64_t pos = p + tok;
    if (GATE == GDN_GATE_SCALAR) {
      if (t == 0) P.ring_g[((int64_t)slot * P.HV + hv) * P.L + pos] = P.g[bh];
    } else if (t < D) {
      P.ring_g[(((int64_t)slot * P.HV + hv) * P.L + pos) * D + t] = P.g[bh * D + t];
    }
    if (hv % P.G == 0 && t < D)
      store_from_f32(P.ring_k, (((int64_t)slot * P.HK + hk) * P.L + pos) * D + t, P.ring_dtype,
                     wk[tok * D + t]);
  }
}

// Lossless speculative verify ([P5] The idea; Modifications, Verify kernel):
// row b's T tokens (input rows b*T + t) run the packed decode's recurrence from
// the checkpoint, token after token, with the packed decode's lane layout and
// its pinned arithmetic (finish_qkv, token_out, token_update), so token t's
// output and correction are bit-identical to those of the t-th of T successive
// gdn_packed_decode calls.  No state is written: each token's correction u,
// key k and log-gate g go to fp32 tuple buffers instead
//   tup_u [B, T, HV, V],  tup_k [B, T, HK, K] (one writer per key head),
//   tup_g [B, T, HV] (KDA [B, T, HV, K]).
// State rows evolve independently: a thread keeps RG groups of its rows in
// registers for the whole window (token loop outside, row loop inside), so each
// token's readout vectors are read from shared memory once per pass.
template <int D, int GATE, int RG>
__global__ void __launch_bounds__(kThreads) lossless_verify_kernel(const DecodeParams P, float *tup_u,
                                                                   float *tup_k, float *tup_g) {
  constexpr int M = D / 32;
  constexpr int ROWS_PER_WARP = D / 4;
  constexpr int NIT = ROWS_PER_WARP / 4;
  static_assert(NIT % RG == 0, "row groups per pass must divide the row groups of a warp");
  const int b = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rg = lane >> 3, cg = lane & 7;
  const int T = P.T;
  extern __shared__ float4 smem_f4[];
  // per token [T][D]: readout vectors x_q, x_k (KDA a o q, a o k), key, gate a (KDA), v;
  // scalars [T][4]: alpha, beta, k.q; then one token's q, k, v and the reduction scratch
  float *wq = reinterpret_cast<float *>(smem_f4);
  float *wke = wq + T * D, *wk = wke + T * D, *wa = wk + T * D, *wv = wa + T * D, *wsc = wv + T * D;
  float *q = wsc + 4 * T, *k = q + D, *v = k + D, *red = v + D;

  const int slot = P.idx[b];
  if (slot >= P.N && hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
  if (slot < 0 || slot >= P.N) {  // padding row: zeros for every token, tuples untouched
    for (int tok = 0; tok < T; ++tok)
      if (t < D) store_from_f32(P.out, (((int64_t)b * T + tok) * P.HV + hv) * D + t, P.out_dtype, 0.f);
    return;
  }
  const int hk = hv / P.G;
  const float4 *S = reinterpret_cast<const float4 *>(P.state + ((int64_t)slot * P.HV + hv) * D * D);

  // the first pass's rows are requested before the window's inputs
  float4 st[RG][M];
#pragma unroll
  for (int i = 0; i < RG; ++i) {
    const int r = warp * ROWS_PER_WARP + i * 4 + rg;
#pragma unroll
    for (int m = 0; m < M; ++m) st[i][m] = S[r * (D / 4) + 8 * m + cg];
  }

  // window inputs: kStageBatch tokens' loads in flight at once, then each
  // token finished as the packed decode finishes its single token
  for (int tok0 = 0; tok0 < T; tok0 += kStageBatch) {
    QkvBits raw[kStageBatch];
    float graw[kStageBatch], braw[kStageBatch];
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
      raw[u] = QkvBits{0u, 0u, 0u};
      graw[u] = braw[u] = 0.f;
      const int tok = tok0 + u;
      if (tok < T) {
        const int64_t bh = ((int64_t)b * T + tok) * P.HV + hv;
        raw[u] = load_qkv_bits<D>(P, b * T + tok, hv);
        graw[u] = GATE == GDN_GATE_PER_K ? (t < D ? P.g[bh * D + t] : 0.f) : P.g[bh];
        braw[u] = P.beta[bh];
      }
    }
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
      const int tok = tok0 + u;
      if (tok < T) {
        const int64_t row = (int64_t)b * T + tok;
        const float kq = finish_qkv<D>(P, qkv_from_bits(raw[u], P.qkv_dtype), q, k, v, red);
        if (t < D) {
          const float a = GATE == GDN_GATE_PER_K ? expf(graw[u]) : 1.f;
          wq[tok * D + t] = GATE == GDN_GATE_PER_K ? __fmul_rn(a, q[t]) : q[t];
          wke[tok * D + t] = GATE == GDN_GATE_PER_K ? __fmul_rn(a, k[t]) : k[t];
          wk[tok * D + t] = k[t];
          wa[tok * D + t] = a;
          wv[tok * D + t] = v[t];
          if (hv % P.G == 0) tup_k[(row * P.HK + hk) * D + t] = k[t];
          if (GATE == GDN_GATE_PER_K) tup_g[(row * P.HV + hv) * D + t] = graw[u];
        }
        if (t == 0) {
          wsc[4 * tok + 0] = GATE == GDN_GATE_SCALAR ? expf(graw[u]) : 1.f;
          wsc[4 * tok + 1] = braw[u];
          wsc[4 * tok + 2] = kq;
          if (GATE == GDN_GATE_SCALAR) tup_g[row * P.HV + hv] = graw[u];
        }
      }
    }
  }
  __syncthreads();

#pragma unroll 1
  for (int pass = 0; pass < NIT / RG; ++pass) {
    if (pass > 0) {
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const int r = warp * ROWS_PER_WARP + (pass * RG + i) * 4 + rg;
#pragma unroll
        for (int m = 0; m < M; ++m) st[i][m] = S[r * (D / 4) + 8 * m + cg];
      }
    }
#pragma unroll 1
    for (int tok = 0; tok < T; ++tok) {
      const float alpha = wsc[4 * tok], beta = wsc[4 * tok + 1], kq = wsc[4 * tok + 2];
      float4 xq[M], xk[M], kr[M], a4[M];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c4 = 8 * m + cg;
        xq[m] = reinterpret_cast<const float4 *>(wq + tok * D)[c4];
        xk[m] = reinterpret_cast<const float4 *>(wke + tok * D)[c4];
        kr[m] = reinterpret_cast<const float4 *>(wk + tok * D)[c4];
        a4[m] = GATE == GDN_GATE_PER_K ? reinterpret_cast<const float4 *>(wa + tok * D)[c4]
                                       : make_float4(1.f, 1.f, 1.f, 1.f);
      }
      const int64_t orow = ((int64_t)b * T + tok) * P.HV + hv;
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const int r = warp * ROWS_PER_WARP + (pass * RG + i) * 4 + rg;
        const float sq = lane_dot<M>(st[i], xq);
        const float sk = lane_dot<M>(st[i], xk);
        float d;
        const float o = token_out<GATE>(sq, sk, alpha, beta, wv[tok * D + r], kq, d);
        if (cg == 0) {
          store_from_f32(P.out, orow * D + r, P.out_dtype, o);
          tup_u[orow * D + r] = d;
        }
#pragma unroll
        for (int m = 0; m < M; ++m) st[i][m] = token_update<GATE>(st[i][m], kr[m], a4[m], alpha, d);
      }
    }
  }
}

// Exact-order commit ([P5] Modifications, Commit): row b's first a =
// accepted[b] tuples are replayed from state[src], src = ssm_state_indices[b],
// with the packed decode's own update (token_update: fl(alpha s), then one fma
// per element), and the result is stored at state[dst], dst = dst_idx[b] (src
// when dst_idx is null).  The state is therefore bit-identical to the one a
// successive gdn_packed_decode calls leave.  Rows with a negative src, dst or
// a are skipped; src or dst >= N and a > T are reported and skipped.
template <int D, int GATE>
__global__ void __launch_bounds__(kThreads) lossless_commit_kernel(const DecodeParams P, const int32_t *dst_idx,
                                                                   const int32_t *accepted, const float *tup_u,
                                                                   const float *tup_k, const float *tup_g) {
  constexpr int M = D / 32;
  constexpr int ROWS_PER_WARP = D / 4;
  const int b = blockIdx.x / P.HV, hv = blockIdx.x % P.HV;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int rg = lane >> 3, cg = lane & 7;
  const int T = P.T;
  extern __shared__ float4 smem_f4[];
  float *wk = reinterpret_cast<float *>(smem_f4);  // [T][D] keys
  float *wu = wk + T * D, *wa = wu + T * D;        // [T][D] corrections, [T][D] KDA gates
  float *walpha = wa + T * D;                      // [T] GDN decays

  const int src = P.idx[b], dst = dst_idx ? dst_idx[b] : src, a = accepted[b];
  if (src < 0 || dst < 0 || a < 0) return;
  if (src >= P.N || dst >= P.N) {
    if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
    return;
  }
  if (a > T) {
    if (hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_ACCEPTED);
    return;
  }
  if (a == 0 && dst == src) return;  // nothing to replay, nothing moves
  const int hk = hv / P.G;
  const float4 *S = reinterpret_cast<const float4 *>(P.state + ((int64_t)src * P.HV + hv) * D * D);
  float4 *Sd = reinterpret_cast<float4 *>(P.state + ((int64_t)dst * P.HV + hv) * D * D);
  float4 cur[M];
  {
    const int r0 = warp * ROWS_PER_WARP + rg;
#pragma unroll
    for (int m = 0; m < M; ++m) cur[m] = S[r0 * (D / 4) + 8 * m + cg];
  }
  // the accepted tuples, kStageBatch tokens' loads in flight at once
  if (t < D) {
    for (int tok0 = 0; tok0 < a; tok0 += kStageBatch) {
      float ku[kStageBatch], uu[kStageBatch], gg[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        ku[u] = uu[u] = gg[u] = 0.f;
        const int64_t row = (int64_t)b * T + tok0 + u;
        if (tok0 + u < a) {
          ku[u] = tup_k[(row * P.HK + hk) * D + t];
          uu[u] = tup_u[(row * P.HV + hv) * D + t];
          gg[u] = GATE == GDN_GATE_PER_K ? tup_g[(row * P.HV + hv) * D + t] : tup_g[row * P.HV + hv];
        }
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int tok = tok0 + u;
        if (tok < a) {
          wk[tok * D + t] = ku[u];
          wu[tok * D + t] = uu[u];
          wa[tok * D + t] = GATE == GDN_GATE_PER_K ? expf(gg[u]) : 1.f;
          if (GATE == GDN_GATE_SCALAR && t == 0) walpha[tok] = expf(gg[u]);
        }
      }
    }
  }
  __syncthreads();
  for (int it = 0; it < ROWS_PER_WARP / 4; ++it) {
    const int r = warp * ROWS_PER_WARP + it * 4 + rg;
    float4 nxt[M];
    if (it + 1 < ROWS_PER_WARP / 4) {
#pragma unroll
      for (int m = 0; m < M; ++m) nxt[m] = S[(r + 4) * (D / 4) + 8 * m + cg];
    }
    for (int tok = 0; tok < a; ++tok) {
      const float d = wu[tok * D + r];
      const float alpha = GATE == GDN_GATE_SCALAR ? walpha[tok] : 1.f;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c4 = 8 * m + cg;
        cur[m] = token_update<GATE>(cur[m], reinterpret_cast<const float4 *>(wk + tok * D)[c4],
                                    reinterpret_cast<const float4 *>(wa + tok * D)[c4], alpha, d);
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      Sd[r * (D / 4) + 8 * m + cg] = cur[m];
      cur[m] = nxt[m];
    }
  }
}

// Commit after verification ([P3] Core concept: rejecting drafts only moves
// the cursor): the cursor moves over the accepted tokens only; a slot whose
// next window would not fit (p + a + T > L - 1) is listed in flush_slots
// (else -1) for a fold.
__global__ void spec_commit_kernel(const int32_t *idx, const int32_t *accepted, int B, int T, int N, int L,
                                   int32_t *write_pos, int32_t *flush_slots, uint32_t *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  flush_slots[b] = -1;
  const int slot = idx[b];
  if (slot < 0) return;
  if (slot >= N) {
    set_status(status, GDN_DEV_BAD_SLOT);
    return;
  }
  const int p = write_pos[slot], a = accepted[b];
  if (p < 0 || p + T > L - 1) {
    set_status(status, GDN_DEV_BAD_WRITE_POS);
    return;
  }
  if (a < 0 || a > T) {
    set_status(status, GDN_DEV_BAD_ACCEPTED);
    return;
  }
  write_pos[slot] = p + a;
  if (p + a + T > L - 1) flush_slots[b] = slot;
}

__global__ void advance_kernel(const int32_t *idx, int B, const uint8_t *ff, int N, int L,
                               int32_t *write_pos, uint32_t *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int slot = idx[b];
  if (slot < 0) return;
  if (slot >= N) {
    set_status(status, GDN_DEV_BAD_SLOT);
    return;
  }
  const int p = write_pos[slot];
  if (p < 0 || p >= L) {
    set_status(status, GDN_DEV_BAD_WRITE_POS);
    return;
  }
  const bool flush = (p == L - 1) || (ff != nullptr && ff[b] != 0);
  write_pos[slot] = flush ? 0 : p + 1;
}

__global__ void reset_kernel(int32_t *write_pos, int N, const int32_t *slots, int n,
                             uint32_t *status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int slot = slots[i];
  if (slot < 0) return;
  if (slot >= N) {
    set_status(status, GDN_DEV_BAD_SLOT);
    return;
  }
  write_pos[slot] = 0;
}

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------

static size_t ffma_smem_bytes(int D, int L, bool replay, bool out_only = false) {
  size_t floats = 5 * (size_t)D + 8 + 64 + (replay ? 2 * (size_t)(L - 1) * D : 0) + (out_only ? 128 : 0);
  return floats * sizeof(float);
}

template <int D, int GATE, bool REPLAY, bool OUT_ONLY = false>
static cudaError_t launch_decode_t(const DecodeParams &P, cudaStream_t s) {
  const size_t smem = ffma_smem_bytes(D, P.L, REPLAY, OUT_ONLY);
  auto kern = ffma_decode_kernel<D, GATE, REPLAY, OUT_ONLY>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_ffma_decode(const DecodeParams &P, int D, int gate, bool replay, cudaStream_t s) {
  if (D == 128) {
    if (gate == GDN_GATE_SCALAR)
      return replay ? launch_decode_t<128, 0, true>(P, s) : launch_decode_t<128, 0, false>(P, s);
    return replay ? launch_decode_t<128, 1, true>(P, s) : launch_decode_t<128, 1, false>(P, s);
  }
  if (gate == GDN_GATE_SCALAR)
    return replay ? launch_decode_t<64, 0, true>(P, s) : launch_decode_t<64, 0, false>(P, s);
  return replay ? launch_decode_t<64, 1, true>(P, s) : launch_decode_t<64, 1, false>(P, s);
}

cudaError_t launch_output_only_decode(const DecodeParams &P, int D, int gate, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_decode_t<128, 0, true, true>(P, s) : launch_decode_t<128, 1, true, true>(P, s);
  return gate == GDN_GATE_SCALAR ? launch_decode_t<64, 0, true, true>(P, s) : launch_decode_t<64, 1, true, true>(P, s);
}

template <int D, int GATE>
static cudaError_t launch_fold_t(const DecodeParams &P, int n, cudaStream_t s) {
  const size_t smem = (2 * (size_t)D + 64 + 2 * (size_t)(P.L - 1) * D) * sizeof(float);
  auto kern = fold_kernel<D, GATE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)n * P.HV, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_fold(const DecodeParams &P, int D, int gate, int n, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_fold_t<128, 0>(P, n, s) : launch_fold_t<128, 1>(P, n, s);
  return gate == GDN_GATE_SCALAR ? launch_fold_t<64, 0>(P, n, s) : launch_fold_t<64, 1>(P, n, s);
}

template <int D, int GATE>
static cudaError_t launch_spec_t(const DecodeParams &P, cudaStream_t s) {
  const size_t smem = (5 * (size_t)P.T * D + 4 * (size_t)P.T + 4 * (size_t)D + 8 + 64 +
                       2 * (size_t)(P.L - 1) * D) * sizeof(float);
  auto kern = spec_verify_kernel<D, GATE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_spec_verify(const DecodeParams &P, int D, int gate, cudaStream_t s) {
  if (D == 128) return gate == GDN_GATE_SCALAR ? launch_spec_t<128, 0>(P, s) : launch_spec_t<128, 1>(P, s);
  return gate == GDN_GATE_SCALAR ? launch_spec_t<64, 0>(P, s) : launch_spec_t<64, 1>(P, s);
}

// Row groups of four rows a verify thread keeps in registers at once (of 8 for K = 128;
// two measured fastest: more raise the registers per thread and cut occupancy).
#ifndef GDN_VERIFY_ROW_GROUPS
#define GDN_VERIFY_ROW_GROUPS 2
#endif
constexpr int kVerifyRowGroups = GDN_VERIFY_ROW_GROUPS;

template <int D, int GATE>
static cudaError_t launch_lossless_verify_t(const DecodeParams &P, float *tu, float *tk, float *tg,
                                            cudaStream_t s) {
  const size_t smem = (5 * (size_t)P.T * D + 4 * (size_t)P.T + 3 * (size_t)D + 8) * sizeof(float);
  auto kern = lossless_verify_kernel<D, GATE, (D == 128 ? kVerifyRowGroups : 4)>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P, tu, tk, tg);
  return cudaGetLastError();
}

cudaError_t launch_lossless_verify(const DecodeParams &P, int D, int gate, float *tup_u, float *tup_k,
                                   float *tup_g, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_lossless_verify_t<128, 0>(P, tup_u, tup_k, tup_g, s)
                                   : launch_lossless_verify_t<128, 1>(P, tup_u, tup_k, tup_g, s);
  return gate == GDN_GATE_SCALAR ? launch_lossless_verify_t<64, 0>(P, tup_u, tup_k, tup_g, s)
                                 : launch_lossless_verify_t<64, 1>(P, tup_u, tup_k, tup_g, s);
}

template <int D, int GATE>
static cudaError_t launch_lossless_commit_t(const DecodeParams &P, const int32_t *dst, const int32_t *acc,
                                            const float *tu, const float *tk, const float *tg, cudaStream_t s) {
  const size_t smem = (3 * (size_t)P.T * D + (size_t)P.T) * sizeof(float);
  auto kern = lossless_commit_kernel<D, GATE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P, dst, acc, tu, tk, tg);
  return cudaGetLastError();
}

cudaError_t launch_lossless_commit(const DecodeParams &P, int D, int gate, const int32_t *dst_idx,
                                   const int32_t *accepted, const float *tup_u, const float *tup_k,
                                   const float *tup_g, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_lossless_commit_t<128, 0>(P, dst_idx, accepted, tup_u, tup_k, tup_g, s)
                                   : launch_lossless_commit_t<128, 1>(P, dst_idx, accepted, tup_u, tup_k, tup_g, s);
  return gate == GDN_GATE_SCALAR ? launch_lossless_commit_t<64, 0>(P, dst_idx, accepted, tup_u, tup_k, tup_g, s)
                                 : launch_lossless_commit_t<64, 1>(P, dst_idx, accepted, tup_u, tup_k, tup_g, s);
}

cudaError_t launch_spec_commit(const int32_t *idx, const int32_t *accepted, int B, int T, int N, int L,
                               int32_t *write_pos, int32_t *flush_slots, uint32_t *status, cudaStream_t s) {
  spec_commit_kernel<<<(B + 255) / 256, 256, 0, s>>>(idx, accepted, B, T, N, L, write_pos, flush_slots, status);
  return cudaGetLastError();
}

cudaError_t launch_advance(const int32_t *idx, int B, const uint8_t *ff, int N, int L,
                           int32_t *write_pos, uint32_t *status, cudaStream_t s) {
  advance_kernel<<<(B + 255) / 256, 256, 0, s>>>(idx, B, ff, N, L, write_pos, status);
  return cudaGetLastError();
}

cudaError_t launch_reset(int32_t *write_pos, int N, const int32_t *slots, int n, uint32_t *status,
                         cudaStream_t s) {
  reset_kernel<<<(n + 255) / 256, 256, 0, s>>>(write_pos, N, slots, n, status);
  return cudaGetLastError();
}

}  // namespace gdn
