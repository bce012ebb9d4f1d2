/*
 * CPU oracle for GDN / KDA ReplaySSM decode.  TEST INFRASTRUCTURE ONLY: the
 * product library never includes this header or links this code.
 *
 * Every array is double and row-major.  Shapes (N slots, HV value heads, HK key
 * heads, K key dim, V value dim, L ring length, B batch rows):
 *   state      [N][HV][V][K]     checkpoint S0 (values held at the state type)
 *   ring_d     [N][HV][L][V]     cached corrections d
 *   ring_k     [N][HK][L][K]     cached keys, shared by the value heads of a group
 *   ring_g     [N][HV][L]        GDN log-gates   ([N][HV][L][K] for KDA)
 *   write_pos  [N]               valid ring entries = next write index
 *   mixed_qkv  [B][2*HK*K+HV*V]  q | k | v
 *   g          [B][HV]           GDN log-gate    ([B][HV][K] for KDA)
 *   beta       [B][HV]
 *   o          [B][HV][V]
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_F16 = 2, ORACLE_BF16 = 3 };
enum { ORACLE_GATE_SCALAR = 0, ORACLE_GATE_PER_K = 1 };
enum { ORACLE_BAD_SLOT = 1u, ORACLE_BAD_WRITE_POS = 2u, ORACLE_BAD_ACCEPTED = 16u };

typedef struct {
    int N, HV, HK, K, V, L;
    int gate;         /* ORACLE_GATE_SCALAR (GDN) or ORACLE_GATE_PER_K (KDA) */
    int state_dtype;  /* storage rounding of the checkpoint                  */
    int ring_dtype;   /* storage rounding of ring d and k (g is never rounded) */
} oracle_geom;

double oracle_round(double x, int dtype);
void oracle_round_array(double *x, long n, int dtype);

void oracle_gdn_step(int K, int V, double *S, const double *q, const double *k,
                     const double *v, double g, double beta, double *y, double *u);
void oracle_kda_step(int K, int V, double *S, const double *q, const double *k,
                     const double *v, const double *g, double beta, double *y, double *u);

int oracle_packed_decode(const oracle_geom *G, double *state, int B, const int *indices,
                         const double *mixed_qkv, const double *g, const double *beta,
                         double q_scale, int qk_l2norm, double *o, unsigned *status);

void oracle_replay_state(const oracle_geom *G, const double *state, const double *ring_d,
                         const double *ring_k, const double *ring_g, int slot, int hv, int p,
                         double *S);

int oracle_replay_decode(const oracle_geom *G, double *state, double *ring_d, double *ring_k,
                         double *ring_g, const int *write_pos, int B, const int *indices,
                         const unsigned char *force_flush, const double *mixed_qkv,
                         const double *g, const double *beta, double q_scale, int qk_l2norm,
                         double *o, unsigned char *flushed, unsigned *status);

int oracle_replay_advance(int N, int B, const int *indices, const unsigned char *force_flush,
                          int L, int *write_pos, unsigned *status);

int oracle_replay_fold(const oracle_geom *G, double *state, const double *ring_d,
                       const double *ring_k, const double *ring_g, const int *write_pos,
                       int n, const int *slots, unsigned *status);

/* Speculative verify window (B rows x T tokens, token t of row b at row b*T+t)
 * and the commit that moves the cursors over the accepted tokens. */
int oracle_spec_verify(const oracle_geom *G, double *state, double *ring_d, double *ring_k,
                       double *ring_g, const int *write_pos, int B, int T, const int *indices,
                       const double *mixed_qkv, const double *g, const double *beta,
                       double q_scale, int qk_l2norm, double *o, unsigned *status);

int oracle_spec_commit(int N, int L, int T, int B, const int *indices, const int *accepted,
                       int *write_pos, int *flush_slots, unsigned *status);

/* Lossless verify (no state update, fp32 (u, k, g) tuples per draft token) and
 * the exact-order commit that replays the accepted tuples in binary32.  The
 * commit's state is float [N][HV][V][K]; tuples:
 *   tup_u [B][T][HV][V], tup_k [B][T][HK][K], tup_g [B][T][HV] ([B][T][HV][K] for KDA). */
void oracle_step_f32(int K, int V, float *h, const float *q, const float *k, const float *v,
                     float g, const float *gk, float beta, float *y, float *u);

int oracle_lossless_verify(const oracle_geom *G, const double *state, int B, int T, const int *indices,
                           const double *mixed_qkv, const double *g, const double *beta,
                           double q_scale, int qk_l2norm, double *o, double *tup_u, double *tup_k,
                           double *tup_g, unsigned *status);

int oracle_lossless_commit(const oracle_geom *G, float *state, int B, int T, const int *src,
                           const int *dst, const int *accepted, const float *tup_u, const float *tup_k,
                           const float *tup_g, unsigned *status);

#ifdef __cplusplus
}
#endif
#endif
