/*
 * CPU oracle for Gated DeltaNet (GDN) / Kimi Delta Attention (KDA) single-token
 * decode with the ReplaySSM checkpoint + ring cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, double-precision C written from the
 * pages' definitions.  It shares no code, header, table or helper with the CUDA
 * library; the product never loads it.  Only the test-suite, the smoke check and
 * the CPU-baseline leg of the benchmark may call it.
 *
 * Sources (page title, then section):
 *  [P1] sglang pull request #28451 "ReplaySSM decode": Modifications (GDN math),
 *       Design 1 (output-only reconstruction), Design 3 (write_pos), Design 5
 *       (force_flush), Design 7 (KDA per-K gate).
 *  [P2] "ReplaySSM" explainer (llm.rainlin.net): section 1 (recurrence),
 *       2.1 (state replay), 2.2 (cache layout), 3.1 (mixed_qkv, padding rows),
 *       3.2 (non-flush step), 3.3 (flush step, L=4 table), 5.2 (KDA).
 *
 * Readings taken where the pages are silent (each also listed in the design notes):
 *  - state orientation [V][K], K contiguous;
 *  - mixed_qkv columns are q | k | v, q and k in HK blocks of K, v in HV blocks of V;
 *  - GQA groups are contiguous: key head = value head / (HV/HK);
 *  - optional q/k L2 norm: x / sqrt(sum x^2 + 1e-6), then q *= q_scale;
 *  - a flush step appends nothing to the ring;
 *  - stored values are rounded (IEEE round-to-nearest-even) to their storage type:
 *    checkpoint to the state type, ring d and k to the ring type; g stays fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gdn_oracle.h"

/* ------------------------------------------------------------------------- */
/* Storage rounding: IEEE binary formats, round to nearest, ties to even.     */
/* ------------------------------------------------------------------------- */

/* Round x to a binary floating format with `mant` fraction bits, minimum normal
 * exponent `emin` and maximum exponent `emax` (IEEE 754 section 4.3.1). */
static double round_binary(double x, int mant, int emin, int emax)
{
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);              /* ax = m * 2^e, m in [0.5, 1) */
    int ex = e - 1;             /* floor(log2(ax)) */
    if (ex < emin) ex = emin;   /* subnormal range keeps the fixed quantum */
    double quantum = ldexp(1.0, ex - mant);
    double r = nearbyint(ax / quantum) * quantum; /* default mode: ties to even */
    /* largest finite value is (2 - 2^-mant) * 2^emax; anything that rounded
     * past it is an overflow to infinity */
    if (r > ldexp(2.0 - ldexp(1.0, -mant), emax)) r = INFINITY;
    return copysign(r, x);
}

double oracle_round(double x, int dtype)
{
    switch (dtype) {
    case ORACLE_F32:  return round_binary(x, 23, -126, 127);
    case ORACLE_F16:  return round_binary(x, 10, -14, 15);
    case ORACLE_BF16: return round_binary(x, 7, -126, 127);
    default:          return x; /* ORACLE_F64: no rounding */
    }
}

void oracle_round_array(double *x, long n, int dtype)
{
    for (long i = 0; i < n; i++) x[i] = oracle_round(x[i], dtype);
}

/* ------------------------------------------------------------------------- */
/* Small dense helpers (row-major, double).                                  */
/* ------------------------------------------------------------------------- */

static double dot(int n, const double *a, const double *b)
{
    double s = 0.0;
    for (int i = 0; i < n; i++) s += a[i] * b[i];
    return s;
}

/* y[r] = sum_c M[r][c] * x[c] for an R x C matrix */
static void matvec(int R, int C, const double *M, const double *x, double *y)
{
    for (int r = 0; r < R; r++) y[r] = dot(C, M + (size_t)r * C, x);
}

/* optional q/k preparation (reading: x / sqrt(sum x^2 + 1e-6)) */
static void prepare_qk(int K, double *q, double *k, double q_scale, int qk_l2norm)
{
    if (qk_l2norm) {
        double nq = sqrt(dot(K, q, q) + 1e-6), nk = sqrt(dot(K, k, k) + 1e-6);
        for (int c = 0; c < K; c++) { q[c] /= nq; k[c] /= nk; }
    }
    for (int c = 0; c < K; c++) q[c] *= q_scale;
}

/* ------------------------------------------------------------------------- */
/* O1: the sequential recurrence, one value head, one token.                 */
/* [P2] section 1: S~ = alpha S, u = beta (v - S~ k), S_t = S~ + u k^T,      */
/*      y = S_t q.  [P1] Design 7: KDA replaces alpha S by S Diag(exp(g)).   */
/* ------------------------------------------------------------------------- */

void oracle_gdn_step(int K, int V, double *S, const double *q, const double *k,
                     const double *v, double g, double beta, double *y, double *u)
{
    double alpha = exp(g);
    double *Sk = (double *)malloc(sizeof(double) * V);
    for (size_t i = 0; i < (size_t)V * K; i++) S[i] *= alpha;       /* S~ = alpha S  */
    matvec(V, K, S, k, Sk);                                          /* S~ k          */
    for (int r = 0; r < V; r++) u[r] = beta * (v[r] - Sk[r]);        /* u             */
    for (int r = 0; r < V; r++)                                      /* S_t = S~+u k^T */
        for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r] * k[c];
    matvec(V, K, S, q, y);                                           /* y = S_t q     */
    free(Sk);
}

void oracle_kda_step(int K, int V, double *S, const double *q, const double *k,
                     const double *v, const double *g, double beta, double *y, double *u)
{
    double *Sk = (double *)malloc(sizeof(double) * V);
    for (int r = 0; r < V; r++)                                      /* S Diag(exp g) */
        for (int c = 0; c < K; c++) S[(size_t)r * K + c] *= exp(g[c]);
    matvec(V, K, S, k, Sk);
    for (int r = 0; r < V; r++) u[r] = beta * (v[r] - Sk[r]);
    for (int r = 0; r < V; r++)
        for (int c = 0; c < K; c++) S[(size_t)r * K + c] += u[r] * k[c];
    matvec(V, K, S, q, y);
    free(Sk);
}

/* ------------------------------------------------------------------------- */
/* Packed input unpacking ([P2] section 3.1): row b of mixed_qkv holds        */
/* q (HK*K) | k (HK*K) | v (HV*V).                                           */
/* ------------------------------------------------------------------------- */

static void unpack_head(const oracle_geom *G, const double *row, int hv,
                        double *q, double *k, double *v)
{
    int group = G->HV / G->HK;
    int hk = hv / group;
    const double *qs = row + (size_t)hk * G->K;
    const double *ks = row + (size_t)G->HK * G->K + (size_t)hk * G->K;
    const double *vs = row + 2 * (size_t)G->HK * G->K + (size_t)hv * G->V;
    memcpy(q, qs, sizeof(double) * G->K);
    memcpy(k, ks, sizeof(double) * G->K);
    memcpy(v, vs, sizeof(double) * G->V);
}

static size_t row_len(const oracle_geom *G)
{
    return 2 * (size_t)G->HK * G->K + (size_t)G->HV * G->V;
}

/* ------------------------------------------------------------------------- */
/* Packed decode (the read + write baseline): O1 per (row, value head), the   */
/* new state stored back every step ([P1] Motivation; [P2] section 1).        */
/* ------------------------------------------------------------------------- */

int oracle_packed_decode(const oracle_geom *G, double *state, int B, const int *indices,
                         const double *mixed_qkv, const double *g, const double *beta,
                         double q_scale, int qk_l2norm, double *o, unsigned *status)
{
    int K = G->K, V = G->V, HV = G->HV;
    double *q = malloc(sizeof(double) * K), *k = malloc(sizeof(double) * K);
    double *v = malloc(sizeof(double) * V), *u = malloc(sizeof(double) * V);
    double *S = malloc(sizeof(double) * (size_t)V * K);
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        for (int hv = 0; hv < HV; hv++) {
            double *ob = o + ((size_t)b * HV + hv) * V;
            if (slot < 0 || slot >= G->N) {              /* padding: zeros */
                if (slot >= G->N) *status |= ORACLE_BAD_SLOT;
                for (int r = 0; r < V; r++) ob[r] = 0.0;
                continue;
            }
            unpack_head(G, mixed_qkv + (size_t)b * row_len(G), hv, q, k, v);
            prepare_qk(K, q, k, q_scale, qk_l2norm);
            double *S0 = state + ((size_t)slot * HV + hv) * V * K;
            memcpy(S, S0, sizeof(double) * (size_t)V * K);
            double bt = beta[(size_t)b * HV + hv];
            if (G->gate == ORACLE_GATE_PER_K)
                oracle_kda_step(K, V, S, q, k, v, g + ((size_t)b * HV + hv) * K, bt, ob, u);
            else
                oracle_gdn_step(K, V, S, q, k, v, g[(size_t)b * HV + hv], bt, ob, u);
            for (size_t i = 0; i < (size_t)V * K; i++) S0[i] = oracle_round(S[i], G->state_dtype);
        }
    }
    free(q); free(k); free(v); free(u); free(S);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* O2: the ReplaySSM state machine.                                          */
/* ------------------------------------------------------------------------- */

/* Pre-token state of (slot, hv) rebuilt from the checkpoint and the first p
 * ring entries ([P2] section 2.1 replay identity; [P1] Design 1):
 *   GDN: S = A S0 + sum_{j<p} w_j d_j k_j^T,  A = prod_{j<p} alpha_j,
 *        w_j = prod_{j<i<p} alpha_i  (empty product = 1);
 *   KDA: S = S0 Diag(A) + sum_{j<p} d_j (w_j o k_j)^T with per-channel A, w_j
 *        ([P1] Design 7). */
void oracle_replay_state(const oracle_geom *G, const double *state, const double *ring_d,
                         const double *ring_k, const double *ring_g, int slot, int hv, int p,
                         double *S)
{
    int K = G->K, V = G->V, HV = G->HV, HK = G->HK, L = G->L;
    int hk = hv / (HV / HK);
    const double *S0 = state + ((size_t)slot * HV + hv) * V * K;
    const double *dr = ring_d + ((size_t)slot * HV + hv) * L * V;
    const double *kr = ring_k + ((size_t)slot * HK + hk) * L * K;
    if (G->gate == ORACLE_GATE_PER_K) {
        const double *gr = ring_g + ((size_t)slot * HV + hv) * L * K;
        for (int c = 0; c < K; c++) {
            double A = 1.0;
            for (int j = 0; j < p; j++) A *= exp(gr[(size_t)j * K + c]);
            for (int r = 0; r < V; r++) S[(size_t)r * K + c] = S0[(size_t)r * K + c] * A;
        }
        for (int j = 0; j < p; j++)
            for (int c = 0; c < K; c++) {
                double w = 1.0;
                for (int i = j + 1; i < p; i++) w *= exp(gr[(size_t)i * K + c]);
                for (int r = 0; r < V; r++)
                    S[(size_t)r * K + c] += dr[(size_t)j * V + r] * (w * kr[(size_t)j * K + c]);
            }
    } else {
        const double *gr = ring_g + ((size_t)slot * HV + hv) * L;
        double A = 1.0;
        for (int j = 0; j < p; j++) A *= exp(gr[j]);
        for (size_t i = 0; i < (size_t)V * K; i++) S[i] = A * S0[i];
        for (int j = 0; j < p; j++) {
            double w = 1.0;
            for (int i = j + 1; i < p; i++) w *= exp(gr[i]);
            for (int r = 0; r < V; r++)
                for (int c = 0; c < K; c++)
                    S[(size_t)r * K + c] += (w * dr[(size_t)j * V + r]) * kr[(size_t)j * K + c];
        }
    }
}

/* One decode launch over B rows ([P1] Modifications + Design 1/3/5/7;
 * [P2] sections 3.2 and 3.3):
 *   p = write_pos[slot]; is_flush = (p == L-1) or force_flush[b];
 *   S = replayed pre-token state (ring entries j < p only);
 *   GDN: Sq = alpha S q, Sk = alpha S k;  KDA: Sq = S (a o q), Sk = S (a o k);
 *   d = beta (v - Sk);  o = Sq + d (k^T q);
 *   flush:     checkpoint <- alpha S + d k^T   (KDA: S Diag(a) + d k^T);
 *   otherwise: ring[p] <- (d, k, g).
 * write_pos itself is only read here; oracle_replay_advance moves it. */
int oracle_replay_decode(const oracle_geom *G, double *state, double *ring_d, double *ring_k,
                         double *ring_g, const int *write_pos, int B, const int *indices,
                         const unsigned char *force_flush, const double *mixed_qkv,
                         const double *g, const double *beta, double q_scale, int qk_l2norm,
                         double *o, unsigned char *flushed, unsigned *status)
{
    int K = G->K, V = G->V, HV = G->HV, HK = G->HK, L = G->L;
    int kda = G->gate == ORACLE_GATE_PER_K;
    double *q = malloc(sizeof(double) * K), *k = malloc(sizeof(double) * K);
    double *v = malloc(sizeof(double) * V), *d = malloc(sizeof(double) * V);
    double *qe = malloc(sizeof(double) * K), *ke = malloc(sizeof(double) * K);
    double *a = malloc(sizeof(double) * K);
    double *Sq = malloc(sizeof(double) * V), *Sk = malloc(sizeof(double) * V);
    double *S = malloc(sizeof(double) * (size_t)V * K);
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        int bad = 0;
        if (slot >= G->N) { *status |= ORACLE_BAD_SLOT; bad = 1; }
        int p = (slot >= 0 && !bad) ? write_pos[slot] : 0;
        if (slot >= 0 && !bad && (p < 0 || p >= L)) { *status |= ORACLE_BAD_WRITE_POS; bad = 1; }
        int is_flush = 0;
        if (slot >= 0 && !bad) is_flush = (p == L - 1) || (force_flush && force_flush[b]);
        if (flushed) flushed[b] = (unsigned char)is_flush;
        for (int hv = 0; hv < HV; hv++) {
            double *ob = o + ((size_t)b * HV + hv) * V;
            if (slot < 0 || bad) {                      /* padding row: zeros, no cache touch */
                for (int r = 0; r < V; r++) ob[r] = 0.0;
                continue;
            }
            int hk = hv / (HV / HK);
            unpack_head(G, mixed_qkv + (size_t)b * row_len(G), hv, q, k, v);
            prepare_qk(K, q, k, q_scale, qk_l2norm);
            double bt = beta[(size_t)b * HV + hv];
            const double *gc = kda ? g + ((size_t)b * HV + hv) * K : g + (size_t)b * HV + hv;
            oracle_replay_state(G, state, ring_d, ring_k, ring_g, slot, hv, p, S);
            if (kda) {
                for (int c = 0; c < K; c++) { a[c] = exp(gc[c]); qe[c] = a[c] * q[c]; ke[c] = a[c] * k[c]; }
                matvec(V, K, S, qe, Sq);
                matvec(V, K, S, ke, Sk);
            } else {
                double alpha = exp(gc[0]);
                matvec(V, K, S, q, Sq);
                matvec(V, K, S, k, Sk);
                for (int r = 0; r < V; r++) { Sq[r] *= alpha; Sk[r] *= alpha; }
            }
            double kq = dot(K, k, q);
            for (int r = 0; r < V; r++) {
                d[r] = bt * (v[r] - Sk[r]);
                ob[r] = Sq[r] + d[r] * kq;
            }
            if (is_flush) {
                double *S0 = state + ((size_t)slot * HV + hv) * V * K;
                for (int r = 0; r < V; r++)
                    for (int c = 0; c < K; c++) {
                        double decayed = kda ? S[(size_t)r * K + c] * a[c]
                                             : exp(gc[0]) * S[(size_t)r * K + c];
                        S0[(size_t)r * K + c] = oracle_round(decayed + d[r] * k[c], G->state_dtype);
                    }
            } else {
                double *dr = ring_d + (((size_t)slot * HV + hv) * L + p) * V;
                double *kr = ring_k + (((size_t)slot * HK + hk) * L + p) * K;
                for (int r = 0; r < V; r++) dr[r] = oracle_round(d[r], G->ring_dtype);
                for (int c = 0; c < K; c++) kr[c] = oracle_round(k[c], G->ring_dtype);
                if (kda) {
                    double *gr = ring_g + (((size_t)slot * HV + hv) * L + p) * K;
                    for (int c = 0; c < K; c++) gr[c] = gc[c];
                } else {
                    ring_g[((size_t)slot * HV + hv) * L + p] = gc[0];
                }
            }
        }
    }
    free(q); free(k); free(v); free(d); free(qe); free(ke); free(a);
    free(Sq); free(Sk); free(S);
    return 0;
}

/* Cursor advance, once per forward after every layer ([P1] Design 3):
 * next = 0 if (write_pos == L-1 or force_flush) else write_pos + 1. */
int oracle_replay_advance(int N, int B, const int *indices, const unsigned char *force_flush,
                          int L, int *write_pos, unsigned *status)
{
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        if (slot < 0) continue;
        if (slot >= N) { *status |= ORACLE_BAD_SLOT; continue; }
        int p = write_pos[slot];
        if (p < 0 || p >= L) { *status |= ORACLE_BAD_WRITE_POS; continue; }
        int ff = force_flush ? force_flush[b] != 0 : 0;
        write_pos[slot] = (p == L - 1 || ff) ? 0 : p + 1;
    }
    return 0;
}

/* Standalone fold of a slot's ring into its checkpoint (the state a snapshot or
 * a copy-on-write must see, [P1] Design 5; [P2] section 4.1):
 * checkpoint <- replayed state with the first write_pos[slot] entries.  The
 * cursor is left as is (the caller resets it). */
int oracle_replay_fold(const oracle_geom *G, double *state, const double *ring_d,
                       const double *ring_k, const double *ring_g, const int *write_pos,
                       int n, const int *slots, unsigned *status)
{
    int K = G->K, V = G->V, HV = G->HV;
    double *S = malloc(sizeof(double) * (size_t)V * K);
    for (int i = 0; i < n; i++) {
        int slot = slots[i];
        if (slot < 0) continue;
        if (slot >= G->N) { *status |= ORACLE_BAD_SLOT; continue; }
        int p = write_pos[slot];
        if (p < 0 || p >= G->L) { *status |= ORACLE_BAD_WRITE_POS; continue; }
        for (int hv = 0; hv < HV; hv++) {
            oracle_replay_state(G, state, ring_d, ring_k, ring_g, slot, hv, p, S);
            double *S0 = state + ((size_t)slot * HV + hv) * V * K;
            for (size_t e = 0; e < (size_t)V * K; e++) S0[e] = oracle_round(S[e], G->state_dtype);
        }
    }
    free(S);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Speculative-decode verify window and commit ([P3] Core concept and       */
/* "Design notes"): one checkpoint plus the ring; a window of T tokens is     */
/* decoded from the committed ring and the window's own earlier tokens, every */
/* token's (d, k, g) goes into the ring after the committed entries, and a    */
/* rejected draft is dropped by not moving the cursor over it.                */
/* ------------------------------------------------------------------------- */

/* Window decode of B rows x T tokens.  Token t of row b is row b*T + t of
 * mixed_qkv / g / beta / o.  For a row with slot s and p = write_pos[s]
 * (requires p + T <= L - 1, the ring's capacity outside a flush step), token t
 * is exactly the non-flush decode of oracle_replay_decode at cursor p + t, so
 * it sees the committed entries and the window's entries p .. p + t - 1; its
 * (d, k, g) is written at ring position p + t.  Neither the checkpoint nor the
 * cursor changes.  A row outside that range sets ORACLE_BAD_WRITE_POS and is
 * treated as padding (zeros). */
int oracle_spec_verify(const oracle_geom *G, double *state, double *ring_d, double *ring_k,
                       double *ring_g, const int *write_pos, int B, int T, const int *indices,
                       const double *mixed_qkv, const double *g, const double *beta,
                       double q_scale, int qk_l2norm, double *o, unsigned *status)
{
    int HV = G->HV, V = G->V, K = G->K;
    size_t gsz = G->gate == ORACLE_GATE_PER_K ? (size_t)HV * K : (size_t)HV;
    int *cursor = malloc(sizeof(int) * (size_t)G->N);
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        int ok = slot >= 0 && slot < G->N;
        if (slot >= G->N) *status |= ORACLE_BAD_SLOT;
        int p = ok ? write_pos[slot] : 0;
        if (ok && (p < 0 || p + T > G->L - 1)) { *status |= ORACLE_BAD_WRITE_POS; ok = 0; }
        for (int t = 0; t < T; t++) {
            size_t row = (size_t)b * T + t;
            if (!ok) {
                for (size_t e = 0; e < (size_t)HV * V; e++) o[row * HV * V + e] = 0.0;
                continue;
            }
            cursor[slot] = p + t;
            int idx1 = slot;
            oracle_replay_decode(G, state, ring_d, ring_k, ring_g, cursor, 1, &idx1, NULL,
                                 mixed_qkv + row * row_len(G), g + row * gsz, beta + row * HV,
                                 q_scale, qk_l2norm, o + row * HV * V, NULL, status);
        }
    }
    free(cursor);
    return 0;
}

/* Commit after verification: row b accepted accepted[b] of its T window
 * tokens (0 <= a <= T).  The cursor moves over the accepted entries only, so
 * the rejected drafts are rolled back by the move itself; when the next window
 * would not fit (cursor + T > L - 1) flush_slots[b] = slot (fold that slot's
 * ring into its checkpoint on every layer, then reset its cursor), else -1.
 * Padding rows get -1. */
int oracle_spec_commit(int N, int L, int T, int B, const int *indices, const int *accepted,
                       int *write_pos, int *flush_slots, unsigned *status)
{
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        flush_slots[b] = -1;
        if (slot < 0) continue;
        if (slot >= N) { *status |= ORACLE_BAD_SLOT; continue; }
        int p = write_pos[slot], a = accepted[b];
        if (p < 0 || p + T > L - 1) { *status |= ORACLE_BAD_WRITE_POS; continue; }
        if (a < 0 || a > T) { *status |= ORACLE_BAD_ACCEPTED; continue; }
        write_pos[slot] = p + a;
        if (p + a + T > L - 1) flush_slots[b] = slot;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Lossless speculative verify and its exact-order commit (sglang pull        */
/* request #42388: "The idea"; Modifications, "Verify kernel" and "Commit").  */
/* Verify updates no state and keeps, per draft token, the fp32 tuple         */
/* (u, k, g) instead of a state snapshot; the commit rebuilds the accepted    */
/* state from the checkpoint by replaying the tuples with the sequential      */
/* kernel's own rounding, so the committed state is bit-identical to it.      */
/* ------------------------------------------------------------------------- */

/* One fp32 step of the sequential recurrence with the rounding the pages give
 * its verify kernel: the decayed state D = fl32(h * a) is formed once and used
 * twice, by the delta reduction and by the update,
 *   Sk_r = sum_c D[r][c] k[c]  (fp32, c ascending),   u_r = fl32(beta * fl32(v_r - Sk_r)),
 *   h[r][c] = fma(k[c], u_r, D[r][c]),                 y_r = sum_c h[r][c] q[c]  (fp32),
 * with a = expf(g) for every channel (GDN, gk == NULL) or a_c = expf(gk[c]) (KDA).
 * h is [V][K] in IEEE binary32. */
void oracle_step_f32(int K, int V, float *h, const float *q, const float *k, const float *v,
                     float g, const float *gk, float beta, float *y, float *u)
{
    float alpha = expf(g);
    for (int r = 0; r < V; r++) {
        float *hr = h + (size_t)r * K;
        for (int c = 0; c < K; c++) hr[c] = hr[c] * (gk ? expf(gk[c]) : alpha);  /* D */
        float sk = 0.0f;
        for (int c = 0; c < K; c++) sk = sk + hr[c] * k[c];
        float diff = v[r] - sk;
        u[r] = beta * diff;
        for (int c = 0; c < K; c++) hr[c] = fmaf(k[c], u[r], hr[c]);
        float yr = 0.0f;
        for (int c = 0; c < K; c++) yr = yr + hr[c] * q[c];
        y[r] = yr;
    }
}

/* Verify of B rows x T tokens that writes no state: row b with slot
 * s = indices[b] runs O1 (oracle_gdn_step / oracle_kda_step) from the
 * checkpoint state[s] over its T tokens (token t at input row b*T + t); token
 * t's output goes to o row b*T + t and its correction u, key k (after the
 * optional norm) and log-gate g, rounded to fp32 (the tuples are always fp32),
 * to
 *   tup_u [B][T][HV][V],  tup_k [B][T][HK][K],  tup_g [B][T][HV] (KDA [B][T][HV][K]).
 * The checkpoint is unchanged.  Padding rows (slot < 0) and slots >= N (which
 * set ORACLE_BAD_SLOT) get zero outputs and leave the tuples alone. */
int oracle_lossless_verify(const oracle_geom *G, const double *state, int B, int T, const int *indices,
                           const double *mixed_qkv, const double *g, const double *beta,
                           double q_scale, int qk_l2norm, double *o, double *tup_u, double *tup_k,
                           double *tup_g, unsigned *status)
{
    int K = G->K, V = G->V, HV = G->HV, HK = G->HK;
    int kda = G->gate == ORACLE_GATE_PER_K;
    size_t gsz = kda ? (size_t)HV * K : (size_t)HV;
    double *q = malloc(sizeof(double) * K), *k = malloc(sizeof(double) * K);
    double *v = malloc(sizeof(double) * V), *u = malloc(sizeof(double) * V);
    double *S = malloc(sizeof(double) * (size_t)V * K);
    for (int b = 0; b < B; b++) {
        int slot = indices[b];
        if (slot >= G->N) *status |= ORACLE_BAD_SLOT;
        for (int hv = 0; hv < HV; hv++) {
            if (slot < 0 || slot >= G->N) {
                for (int t = 0; t < T; t++)
                    for (int r = 0; r < V; r++) o[(((size_t)b * T + t) * HV + hv) * V + r] = 0.0;
                continue;
            }
            int hk = hv / (HV / HK);
            memcpy(S, state + ((size_t)slot * HV + hv) * V * K, sizeof(double) * (size_t)V * K);
            for (int t = 0; t < T; t++) {
                size_t row = (size_t)b * T + t;
                unpack_head(G, mixed_qkv + row * row_len(G), hv, q, k, v);
                prepare_qk(K, q, k, q_scale, qk_l2norm);
                double bt = beta[row * HV + hv];
                double *ob = o + (row * HV + hv) * V;
                const double *gt = g + row * gsz + (kda ? (size_t)hv * K : (size_t)hv);
                if (kda) oracle_kda_step(K, V, S, q, k, v, gt, bt, ob, u);
                else oracle_gdn_step(K, V, S, q, k, v, gt[0], bt, ob, u);
                for (int r = 0; r < V; r++) tup_u[(row * HV + hv) * V + r] = oracle_round(u[r], ORACLE_F32);
                for (int c = 0; c < K; c++) tup_k[(row * HK + hk) * K + c] = oracle_round(k[c], ORACLE_F32);
                if (kda)
                    for (int c = 0; c < K; c++) tup_g[(row * HV + hv) * K + c] = oracle_round(gt[c], ORACLE_F32);
                else
                    tup_g[row * HV + hv] = oracle_round(gt[0], ORACLE_F32);
            }
        }
    }
    free(q); free(k); free(v); free(u); free(S);
    return 0;
}

/* Exact-order commit: for row b with source slot s = src[b] and a = accepted[b]
 * tokens (0 <= a <= T), every value head replays, in IEEE binary32,
 *   h[r][c] <- fma(k_t[c], u_t[r], fl32(h[r][c] * a_t)),   t = 0 .. a-1,
 * from h = state[s], with a_t = expf(g_t) (KDA: a_t[c] = expf(g_t[c])): the
 * decayed state is one rounded multiply and the rank-1 update one fused
 * multiply-add, as in the sequential step.  The result is stored at slot
 * dst[b] (dst == NULL: back at s).  Tuples as oracle_lossless_verify lays them
 * out, in fp32.  Rows with s < 0, a < 0 or dst[b] < 0 are skipped; a slot >= N
 * sets ORACLE_BAD_SLOT and a > T sets ORACLE_BAD_ACCEPTED (row skipped). */
int oracle_lossless_commit(const oracle_geom *G, float *state, int B, int T, const int *src,
                           const int *dst, const int *accepted, const float *tup_u, const float *tup_k,
                           const float *tup_g, unsigned *status)
{
    int K = G->K, V = G->V, HV = G->HV, HK = G->HK;
    int kda = G->gate == ORACLE_GATE_PER_K;
    float *h = malloc(sizeof(float) * (size_t)V * K);
    for (int b = 0; b < B; b++) {
        int s = src[b], d = dst ? dst[b] : s, a = accepted[b];
        if (s < 0 || d < 0 || a < 0) continue;
        if (s >= G->N || d >= G->N) { *status |= ORACLE_BAD_SLOT; continue; }
        if (a > T) { *status |= ORACLE_BAD_ACCEPTED; continue; }
        for (int hv = 0; hv < HV; hv++) {
            int hk = hv / (HV / HK);
            memcpy(h, state + ((size_t)s * HV + hv) * V * K, sizeof(float) * (size_t)V * K);
            for (int t = 0; t < a; t++) {
                size_t row = (size_t)b * T + t;
                const float *ut = tup_u + (row * HV + hv) * V;
                const float *kt = tup_k + (row * HK + hk) * K;
                for (int r = 0; r < V; r++)
                    for (int c = 0; c < K; c++) {
                        float at = kda ? expf(tup_g[(row * HV + hv) * K + c]) : expf(tup_g[row * HV + hv]);
                        float decayed = h[(size_t)r * K + c] * at;
                        h[(size_t)r * K + c] = fmaf(kt[c], ut[r], decayed);
                    }
            }
            memcpy(state + ((size_t)d * HV + hv) * V * K, h, sizeof(float) * (size_t)V * K);
        }
    }
    free(h);
    return 0;
}
