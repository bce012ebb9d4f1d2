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
// token_out: once the row's 8 lanes hold partial sums s_0..s_7 of S x (x = q,
// k; KDA a o q, a o k), sums them (xor 1, 2, 4), which leaves every lane with
// ((s_0 + s_1) + (s_2 + s_3)) + ((s_4 + s_5) + (s_6 + s_7)) (each add is
// commutative, so the lanes agree bit for bit), and calls token_finish:
//   GDN: sq, sk <- alpha sq, alpha sk;   d = beta (v_r - sk);   o = sq + d (k^T q).
template <int GATE>
__device__ __forceinline__ float token_finish(float sq, float sk, float alpha, float beta, float vr, float kq,
                                              float &d) {
  if (GATE == GDN_GATE_SCALAR) {
    sq = __fmul_rn(sq, alpha);
    sk = __fmul_rn(sk, alpha);
  }
  d = __fmul_rn(beta, __fsub_rn(vr, sk));
  return __fmaf_rn(d, kq, sq);
}

template <int GATE>
__device__ __forceinline__ float token_out(float sq, float sk, float alpha, float beta, float vr, float kq,
                                           float &d) {
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  return token_finish<GATE>(sq, sk, alpha, beta, vr, kq, d);
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

// Block sums of NV values at once over the first 128 threads, each summed as
// block_sum2 sums one (a 32-lane xor tree per warp, then the four warps'
// partials as (w0 + w1) + (w2 + w3)), so each result is bit-identical to a
// block_sum2 of that value; two barriers for all NV instead of two each.
// red: NV * 4 floats.
template <int NV>
__device__ __forceinline__ void block_sums(float (&x)[NV], float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < NV; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
  if (lane == 0 && warp < 4)
#pragma unroll
    for (int i = 0; i < NV; ++i) red[4 * i + warp] = x[i];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) x[i] = (red[4 * i] + red[4 * i + 1]) + (red[4 * i + 2] + red[4 * i + 3]);
  __syncthreads();
}

// The same verify with LPR (2 or 4) lanes per state row and two rows per
// thread (K = V = 128 only; D * LPR / 2 threads): lane LPR i + h of warp w holds
// rows R w + i and R w + i + R / 2 (R = 64 / LPR rows per warp), columns of the
// packed decode's column groups l = NL h .. NL h + NL - 1 (NL = 8 / LPR; float4
// chunks 8 m + l).  Each lane forms its partial sums s_l exactly as a
// packed-decode lane does (lane_dot), adds them as the first rounds of the
// packed decode's tree would, and exchanges with its LPR - 1 partners for the
// rest of the tree, so every output and correction is bit-identical to the
// 8-lane form.  A lane's operand loads from shared memory serve two rows, and
// with four lanes per row a thread holds 64 state registers, so two blocks of
// eight warps fit on an SM.
//
// The grid is persistent (items (row, value head) dealt round robin).  One
// thread stages an item with nine TMA loads: the checkpoint as M tiles of
// 128-byte swizzled rows (a quarter warp's reads of its rows' chunks fall in
// distinct banks) and the window's q, k, v, gate and beta tiles.  Once an item's
// rows are in registers and its window's vectors are formed, the staging area
// is free, and the block's next item streams into it while this item's window
// runs: an item starts with its data on chip.
constexpr uint64_t kVerifyWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms per wait

template <int LPR>
__host__ __device__ constexpr int verify_lane_threads() {
  return 128 * LPR / 2;
}

// The tensor maps the verify stages an item with: the checkpoint ([N HV V rows,
// K] fp32, 128-byte swizzle, [V x 32] boxes), mixed_qkv ([B T rows, used
// columns], [T x D] boxes: one key or value head's span for the window's T
// tokens), the log-gates ([B T rows, HV] with [T x 4] boxes for GDN, [B T rows,
// HV K] with [T x K] boxes for KDA) and beta ([B T rows, HV], [T x 4] boxes).
struct VerifyMaps {
  CUtensorMap state, qkv, g, beta;
};

template <int D, int GATE, int LPR>
__global__ void __launch_bounds__(verify_lane_threads<LPR>(), 2)
    lossless_verify_lanes_kernel(const DecodeParams P, float *tup_u, float *tup_k, float *tup_g,
                                 const __grid_constant__ VerifyMaps maps) {
  static_assert(D == 128 && (LPR == 2 || LPR == 4), "a 128-row state, two or four lanes per row");
  constexpr int kT = verify_lane_threads<LPR>();
  constexpr int M = D / 32;
  constexpr int NL = 8 / LPR;        // column groups per lane
  constexpr int RW = 64 / LPR;       // rows per warp
  constexpr int GW = GATE == GDN_GATE_PER_K ? D : 4;  // columns of a staged gate row
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int h = lane % LPR;
  const int row0 = warp * RW + lane / LPR, row1 = row0 + RW / 2;
  const bool stores = h < 2;                   // lane 0 of a row group stores row0, lane 1 row1
  const int my_row = h == 1 ? row1 : row0;
  const int T = P.T;
  const int items = P.B * P.HV;
  const int esz = P.qkv_dtype == GDN_F32 ? 4 : 2;
  extern __shared__ uint8_t verify_smem[];
  // the checkpoint tiles need a 1024-byte aligned base (128-byte swizzle); the
  // allocation has 1024 bytes of slack for it
  uint8_t *sm = verify_smem + (((smem_addr(verify_smem) + 1023u) & ~1023u) - smem_addr(verify_smem));
  // Checkpoint: M tiles of [D rows x 32 columns], row r's 16-byte chunk j of
  // tile m at m * 128 D + 128 r + 16 (j ^ (r mod 8)).  Then the raw window
  // inputs as the maps deliver them (q, k, v: [T][D] of the input type; gates
  // [T][GW] and beta [T][4] fp32), each region 128-byte aligned, then the
  // window's vectors.
  const int qbytes = (T * D * esz + 127) & ~127;
  uint8_t *rq = sm + M * D * 128, *rk = rq + qbytes, *rv = rk + qbytes;
  float *rg = reinterpret_cast<float *>(rv + qbytes);
  float *rb = rg + ((T * GW + 31) & ~31);
  float *wq = rb + ((T * 4 + 31) & ~31);
  float *wk = wq + T * D, *wv = wk + T * D, *wsc = wv + T * D;
  float *wke = GATE == GDN_GATE_PER_K ? wsc + 4 * T : wk;  // KDA: a o k
  float *wa = GATE == GDN_GATE_PER_K ? wke + T * D : wk;   // KDA: a
  float *red = GATE == GDN_GATE_PER_K ? wa + T * D : wsc + 4 * T;  // [2 * kStageBatch][4]
  const uint32_t bar = (smem_addr(red + 8 * kStageBatch) + 7u) & ~7u;  // the mbarrier, 8-byte aligned
  const uint32_t s_base = smem_addr(sm);
  const uint32_t tx_bytes = D * D * 4 + 3 * T * D * esz + T * GW * 4 + T * 16;

  // One thread stages an item: nine TMA loads completing on `bar`.
  auto stage = [&](int slot_, int b_, int hv_) {
    const int hk_ = hv_ / P.G;
    mbar_arrive_expect_tx(bar, tx_bytes);
    const int y = (slot_ * P.HV + hv_) * D;
#pragma unroll
    for (int m = 0; m < M; ++m) tma_load_2d(s_base + m * D * 128, &maps.state, 32 * m, y, bar);
    tma_load_2d(smem_addr(rq), &maps.qkv, hk_ * D, b_ * T, bar);
    tma_load_2d(smem_addr(rk), &maps.qkv, (P.HK + hk_) * D, b_ * T, bar);
    tma_load_2d(smem_addr(rv), &maps.qkv, 2 * P.HK * D + hv_ * D, b_ * T, bar);
    tma_load_2d(smem_addr(rg), &maps.g, GATE == GDN_GATE_PER_K ? hv_ * D : hv_ & ~3, b_ * T, bar);
    tma_load_2d(smem_addr(rb), &maps.beta, hv_ & ~3, b_ * T, bar);
  };
  if (t == 0) {
    prefetch_tensormap(&maps.state);
    prefetch_tensormap(&maps.qkv);
    prefetch_tensormap(&maps.g);
    prefetch_tensormap(&maps.beta);
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  int staged = -1;  // the item whose checkpoint and inputs are in flight to shared memory
  bool failed = false;
  int slot = blockIdx.x < items ? P.idx[blockIdx.x / P.HV] : -1;  // then carried from the item before

#pragma unroll 1
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = item / P.HV, hv = item % P.HV;
    const int next = item + gridDim.x;
    const int next_slot = next < items ? P.idx[next / P.HV] : -1;  // used once this item's inputs are formed
    const int cur = slot;
    slot = next_slot;
    if (cur >= P.N && hv == 0 && t == 0) set_status(P.status, GDN_DEV_BAD_SLOT);
    if (cur < 0 || cur >= P.N) {  // padding row: zeros for every token, tuples untouched
      for (int tok = 0; tok < T; ++tok)
        if (t < D) store_from_f32(P.out, (((int64_t)b * T + tok) * P.HV + hv) * D + t, P.out_dtype, 0.f);
      continue;
    }
    const int hk = hv / P.G;
    if (staged != item && t == 0) stage(cur, b, hv);  // else it arrived during the previous item's window
    staged = item;
    const bool landed = mbar_wait_bounded(bar, phase, kVerifyWaitLimitNs);
    phase ^= 1u;
    if (__syncthreads_or(!landed)) {  // the copies did not land: report, stop this block
      if (t == 0) set_status(P.status, GDN_DEV_TIMEOUT);
      failed = true;
      break;
    }

    for (int tok0 = 0; tok0 < T; tok0 += kStageBatch) {
      // finish_qkv's arithmetic for kStageBatch tokens at once: the optional L2
      // norm, q_scale, k^T q, each block sum formed as block_sum2 forms it
      float qt[kStageBatch], kt[kStageBatch], kq[kStageBatch];
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int tok = tok0 + u;
        qt[u] = kt[u] = 0.f;
        if (t < D && tok < T) {
          const int i = tok * D + t;
          const QkvBits bits = esz == 4 ? QkvBits{reinterpret_cast<const uint32_t *>(rq)[i],
                                                  reinterpret_cast<const uint32_t *>(rk)[i],
                                                  reinterpret_cast<const uint32_t *>(rv)[i]}
                                        : QkvBits{reinterpret_cast<const uint16_t *>(rq)[i],
                                                  reinterpret_cast<const uint16_t *>(rk)[i],
                                                  reinterpret_cast<const uint16_t *>(rv)[i]};
          const QkvRaw x = qkv_from_bits(bits, P.qkv_dtype);
          qt[u] = x.q;
          kt[u] = x.k;
          wv[i] = x.v;
        }
      }
      if (P.qk_l2norm) {
        float n[2 * kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          n[u] = __fmul_rn(qt[u], qt[u]);
          n[kStageBatch + u] = __fmul_rn(kt[u], kt[u]);
        }
        block_sums<2 * kStageBatch>(n, red);
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
          qt[u] = __fdiv_rn(qt[u], __fsqrt_rn(__fadd_rn(n[u], 1e-6f)));
          kt[u] = __fdiv_rn(kt[u], __fsqrt_rn(__fadd_rn(n[kStageBatch + u], 1e-6f)));
        }
      }
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        qt[u] = __fmul_rn(qt[u], P.q_scale);
        kq[u] = __fmul_rn(kt[u], qt[u]);
      }
      block_sums<kStageBatch>(kq, red);
      const bool key_writer = hv % P.G == 0;
#pragma unroll
      for (int u = 0; u < kStageBatch; ++u) {
        const int tok = tok0 + u;
        if (tok < T) {
          const int64_t row = (int64_t)b * T + tok;
          if (t < D) {
            if (GATE == GDN_GATE_PER_K) {
              const float graw = rg[tok * GW + t];
              const float a = expf(graw);
              wq[tok * D + t] = __fmul_rn(a, qt[u]);
              wke[tok * D + t] = __fmul_rn(a, kt[u]);
              wa[tok * D + t] = a;
              tup_g[(row * P.HV + hv) * D + t] = graw;
            } else {
              wq[tok * D + t] = qt[u];
            }
            wk[tok * D + t] = kt[u];
            if (key_writer) tup_k[(row * P.HK + hk) * D + t] = kt[u];
          }
          if (t == tok) {  // the token's scalars, one thread per token
            const float graw = rg[tok * GW + (GATE == GDN_GATE_PER_K ? 0 : (hv & 3))];
            wsc[4 * tok + 0] = GATE == GDN_GATE_SCALAR ? expf(graw) : 1.f;
            wsc[4 * tok + 1] = rb[tok * 4 + (hv & 3)];
            wsc[4 * tok + 2] = kq[u];
            if (GATE == GDN_GATE_SCALAR) tup_g[row * P.HV + hv] = graw;
          }
        }
      }
    }

    float4 st[2][M * NL];  // [row][m * NL + li]: chunk 8 m + NL h + li of the row
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int li = 0; li < NL; ++li) {
        const int j = NL * h + li;
        st[0][m * NL + li] = *reinterpret_cast<const float4 *>(sm + m * D * 128 + row0 * 128 + 16 * (j ^ (row0 & 7)));
        st[1][m * NL + li] = *reinterpret_cast<const float4 *>(sm + m * D * 128 + row1 * 128 + 16 * (j ^ (row1 & 7)));
      }
    // the window's vectors are in place, and the staged checkpoint and raw
    // inputs are free: the next item's stream in under this window
    fence_proxy_async_smem();
    __syncthreads();
    staged = -1;
    if (next_slot >= 0 && next_slot < P.N) {
      if (t == 0) stage(next_slot, next / P.HV, next % P.HV);
      staged = next;
    }

#pragma unroll 1
    for (int tok = 0; tok < T; ++tok) {
      const float alpha = wsc[4 * tok], beta = wsc[4 * tok + 1], kq = wsc[4 * tok + 2];
      const float4 *xq4 = reinterpret_cast<const float4 *>(wq + tok * D);
      const float4 *xk4 = reinterpret_cast<const float4 *>(wke + tok * D);
      const float4 *kr4 = reinterpret_cast<const float4 *>(wk + tok * D);
      const float4 *a44 = reinterpret_cast<const float4 *>(wa + tok * D);
      float pq[2][NL], pk[2][NL];
#pragma unroll
      for (int li = 0; li < NL; ++li) {
        float2 loq[2], hiq[2], lok[2], hik[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) loq[j] = hiq[j] = lok[j] = hik[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const float4 xq = xq4[8 * m + NL * h + li], xk = xk4[8 * m + NL * h + li];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float4 &s = st[j][m * NL + li];
            loq[j] = __ffma2_rn(make_float2(s.x, s.y), make_float2(xq.x, xq.y), loq[j]);
            hiq[j] = __ffma2_rn(make_float2(s.z, s.w), make_float2(xq.z, xq.w), hiq[j]);
            lok[j] = __ffma2_rn(make_float2(s.x, s.y), make_float2(xk.x, xk.y), lok[j]);
            hik[j] = __ffma2_rn(make_float2(s.z, s.w), make_float2(xk.z, xk.w), hik[j]);
          }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pq[j][li] = __fadd_rn(__fadd_rn(loq[j].x, loq[j].y), __fadd_rn(hiq[j].x, hiq[j].y));
          pk[j][li] = __fadd_rn(__fadd_rn(lok[j].x, lok[j].y), __fadd_rn(hik[j].x, hik[j].y));
        }
      }
      float d[2], o[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float sq, sk;
        if constexpr (NL == 4) {
          sq = __fadd_rn(__fadd_rn(pq[j][0], pq[j][1]), __fadd_rn(pq[j][2], pq[j][3]));
          sk = __fadd_rn(__fadd_rn(pk[j][0], pk[j][1]), __fadd_rn(pk[j][2], pk[j][3]));
        } else {
          sq = __fadd_rn(pq[j][0], pq[j][1]);
          sk = __fadd_rn(pk[j][0], pk[j][1]);
        }
#pragma unroll
        for (int x = 1; x < LPR; x <<= 1) {
          sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, x));
          sk = __fadd_rn(sk, __shfl_xor_sync(0xffffffffu, sk, x));
        }
        o[j] = token_finish<GATE>(sq, sk, alpha, beta, wv[tok * D + (j ? row1 : row0)], kq, d[j]);
      }
      const int64_t orow = ((int64_t)b * T + tok) * P.HV + hv;
      if (stores) {
        store_from_f32(P.out, orow * D + my_row, P.out_dtype, h == 1 ? o[1] : o[0]);
        tup_u[orow * D + my_row] = h == 1 ? d[1] : d[0];
      }
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int li = 0; li < NL; ++li) {
          const float4 kr = kr4[8 * m + NL * h + li];
          const float4 a4 = GATE == GDN_GATE_PER_K ? a44[8 * m + NL * h + li] : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            st[j][m * NL + li] = token_update<GATE>(st[j][m * NL + li], kr, a4, alpha, d[j]);
        }
    }
    __syncthreads();  // the next item's inputs overwrite the window's vectors
  }
  if (failed)  // copies may still be in flight: give them the limit again before the block leaves
    mbar_wait_bounded(bar, phase ^ 1u, kVerifyWaitLimitNs);
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

// D = 64: the 8-lane layout with all four row groups of a warp in registers.
template <int GATE>
static cudaError_t launch_lossless_verify_64(const DecodeParams &P, float *tu, float *tk, float *tg,
                                             cudaStream_t s) {
  constexpr int D = 64;
  const size_t smem = (5 * (size_t)P.T * D + 4 * (size_t)P.T + 3 * (size_t)D + 8) * sizeof(float);
  auto kern = lossless_verify_kernel<D, GATE, 4>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P, tu, tk, tg);
  return cudaGetLastError();
}

// D = 128: two lanes per row, two rows per thread; the checkpoint tiles, the
// window's raw tiles and vectors (three of them for GDN, five for KDA) share the
// block's shared memory, at most 203 KB (a 32-token KDA window of fp32 inputs).
// Where the tensor maps cannot describe the inputs (a buffer or row stride not a
// multiple of 16 bytes, HV not a multiple of 4, coordinates past 2^31), the
// 8-lane form runs.
template <int GATE>
static cudaError_t launch_lossless_verify_128(const DecodeParams &P, float *tu, float *tk, float *tg,
                                              cudaStream_t s) {
  constexpr int D = 128;
  constexpr int GW = GATE == GDN_GATE_PER_K ? D : 4;
  const size_t esz = P.qkv_dtype == GDN_F32 ? 4 : 2;
  const int64_t rows = (int64_t)P.B * P.T;
  const int64_t cols = 2 * (int64_t)P.HK * D + (int64_t)P.HV * D;
  const int64_t gcols = (int64_t)P.HV * (GATE == GDN_GATE_PER_K ? D : 1);
  VerifyMaps maps;
  const char *why = nullptr;
  bool ok = (int64_t)P.N * P.HV * D < ((int64_t)1 << 31) && cols < ((int64_t)1 << 31) &&
            rows < ((int64_t)1 << 31) && P.HV % 4 == 0 && ((size_t)P.qkv_stride * esz) % 16 == 0 &&
            reinterpret_cast<uintptr_t>(P.qkv) % 16 == 0 && reinterpret_cast<uintptr_t>(P.g) % 16 == 0 &&
            reinterpret_cast<uintptr_t>(P.beta) % 16 == 0;
  ok = ok && make_state_tmap(P, D, &maps.state, &why) == cudaSuccess;
  ok = ok && make_tmap_2d(P.qkv, P.qkv_dtype, cols, rows, (uint64_t)P.qkv_stride * esz, D, P.T, &maps.qkv) == cudaSuccess;
  ok = ok && make_tmap_2d(P.g, GDN_F32, gcols, rows, gcols * 4, GW, P.T, &maps.g) == cudaSuccess;
  ok = ok && make_tmap_2d(P.beta, GDN_F32, P.HV, rows, (uint64_t)P.HV * 4, 4, P.T, &maps.beta) == cudaSuccess;
  if (!ok) {
    const size_t smem = (5 * (size_t)P.T * D + 4 * (size_t)P.T + 3 * (size_t)D + 8) * sizeof(float);
    auto kern = lossless_verify_kernel<D, GATE, 2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)P.B * P.HV, kThreads, smem, s>>>(P, tu, tk, tg);
    return cudaGetLastError();
  }
  const size_t vecs = GATE == GDN_GATE_PER_K ? 5 : 3;
  const size_t qbytes = ((size_t)P.T * D * esz + 127) & ~(size_t)127;
  const size_t smem = 1024 + (size_t)D * D * 4 + 3 * qbytes +
                      (((size_t)P.T * GW + 31) & ~(size_t)31) * 4 + (((size_t)P.T * 4 + 31) & ~(size_t)31) * 4 +
                      (vecs * (size_t)P.T * D + 4 * (size_t)P.T + 8 * kStageBatch) * sizeof(float) + 16;
  constexpr int LPR = 2;
  constexpr int kT = verify_lane_threads<LPR>();
  auto kern = lossless_verify_lanes_kernel<D, GATE, LPR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // resident blocks on this device for this shared-memory size (the window
  // length and the input width change it), looked up once per (device, window, width)
  static int resident[64][33][2] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const int wide = P.qkv_dtype == GDN_F32;
  int slots = dev < 64 ? resident[dev][P.T][wide] : 0;
  if (slots == 0) {
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kT, smem)) != cudaSuccess) return e;
    slots = (per_sm < 1 ? 1 : per_sm) * sms;
    if (dev < 64) resident[dev][P.T][wide] = slots;
  }
  const int64_t items = (int64_t)P.B * P.HV;
  const int64_t grid = items < slots ? items : slots;
  kern<<<(unsigned)grid, kT, smem, s>>>(P, tu, tk, tg, maps);
  return cudaGetLastError();
}

cudaError_t launch_lossless_verify(const DecodeParams &P, int D, int gate, float *tup_u, float *tup_k,
                                   float *tup_g, cudaStream_t s) {
  if (D == 128)
    return gate == GDN_GATE_SCALAR ? launch_lossless_verify_128<0>(P, tup_u, tup_k, tup_g, s)
                                   : launch_lossless_verify_128<1>(P, tup_u, tup_k, tup_g, s);
  return gate == GDN_GATE_SCALAR ? launch_lossless_verify_64<0>(P, tup_u, tup_k, tup_g, s)
                                 : launch_lossless_verify_64<1>(P, tup_u, tup_k, tup_g, s);
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
