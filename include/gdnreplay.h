/*
 * gdnreplay — Gated DeltaNet (GDN) / Kimi Delta Attention (KDA) single-token
 * decode with the ReplaySSM checkpoint + ring cache, for one GB300 (sm_103a).
 *
 * C ABI.  Every pointer in a call below is a DEVICE pointer unless its comment
 * says otherwise.  Every buffer, scratch workspace included, is owned by the
 * caller; the library allocates no device memory and never synchronises: each
 * call enqueues kernels on `stream` and returns.  Host-side argument checks run before any launch and
 * return GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED with nothing enqueued; a
 * launch failure returns GDN_ERR_CUDA.  gdn_last_error() gives the calling
 * thread's message for its last failing call.
 *
 * Problems found on the device (a slot index >= num_slots, a write_pos outside
 * [0, ring_len), a wait that ran out) are OR-ed as GDN_DEV_* bits into the
 * optional `dev_status` word (a device uint32; NULL disables reporting).  The
 * row is then treated as a padding row.  No kernel traps.
 *
 * Sources, by page title and section:
 *  [P1] sglang pull request #28451 "ReplaySSM decode": Modifications (the GDN
 *       decode equations), Design 1 (output-only reconstruction), Design 2
 *       (tensor-core reconstruction), Design 3 (per-slot write_pos and its
 *       advance rule), Design 4 (device-side flush branch), Design 5
 *       (force_flush, write_pos reset on copy-on-write), Design 7 (KDA gate).
 *  [P2] "ReplaySSM" explainer (llm.rainlin.net): section 1 (recurrence), 2.1
 *       (replay identity), 2.2 (cache layout table), 3.1 (packed mixed_qkv,
 *       ssm_state_indices, negative padding rows), 3.2 (non-flush step), 3.3
 *       (flush step), 5.2 (KDA gate cache [N, HV, L, K]).
 *  [P3] vLLM pull request #49887 "ReplaySSM: cache SSM inputs for faster Gated
 *       DeltaNet speculative decode": Core concept, Design notes.
 *  [P5] sglang pull request #42388 (lossless verify): The idea; Modifications
 *       (Verify kernel, Commit).
 *
 * Layouts (row-major, innermost last; N slots, HV value heads, HK key heads
 * with HV % HK == 0, K key dim, V value dim, L ring length, B batch rows):
 *   state      [N, HV, V, K]  fp32 checkpoint S0 ("temporal", [P2] 2.2)
 *   ring_d     [N, HV, L, V]  ring dtype: cached corrections d
 *   ring_k     [N, HK, L, K]  ring dtype: cached keys, shared by a key head's group
 *   ring_g     [N, HV, L]     fp32 GDN log-gates; [N, HV, L, K] for KDA
 *   write_pos  [N]            int32 per-slot valid count = next write index
 *   mixed_qkv  [B, 2*HK*K + HV*V] (row stride given): q | k | v, q and k in HK
 *              blocks of K, v in HV blocks of V; value head hv uses key head
 *              hv / (HV/HK)
 *   g          [B, HV] fp32 log-gate (<= 0); [B, HV, K] for KDA
 *   beta       [B, HV] fp32
 *   out        [B, HV, V] out dtype
 */
#ifndef GDNREPLAY_H
#define GDNREPLAY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer       */
    GDN_ERR_UNSUPPORTED = 2, /* valid but not built: K/V, dtype combination, L   */
    GDN_ERR_CUDA = 3         /* a launch or runtime call failed                   */
} gdn_status_t;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype_t;

/* Gate granularity ([P1] Design 7): one log-gate per value head (GDN), or one
 * per key channel of each value head (KDA). */
typedef enum { GDN_GATE_SCALAR = 0, GDN_GATE_PER_K = 1 } gdn_gate_t;

/* How the replayed state S = A S0 + sum_j w_j d_j k_j^T is evaluated.
 * TENSOR: the L-deep sum is one small GEMM on the tensor cores (tcgen05, fp32
 *         accumulation) — [P1] Design 2.  Operands: f16, bf16 or tf32 for an
 *         fp16, bf16 or fp32 ring.
 * FFMA:   every term in fp32 on the CUDA cores (slower, tighter error bound).
 * OUTPUT: a non-flush row never forms S: its readout is factored through the
 *         ring, S x = A (S0 x) + sum_j w_j d_j (k_j . x) (KDA: S0 (A o x) +
 *         sum_j d_j ((w_j o k_j) . x)), fp32 on the CUDA cores — the
 *         "output-only" reconstruction of [P1] Design 1 and [P2] 3.2; flush rows
 *         rebuild S as FFMA does.  Same results as FFMA up to rounding order. */
typedef enum { GDN_RECON_TENSOR = 0, GDN_RECON_FFMA = 1, GDN_RECON_OUTPUT = 2 } gdn_recon_t;

/* dev_status bits */
#define GDN_DEV_BAD_SLOT      1u /* ssm_state_indices[b] >= num_slots               */
#define GDN_DEV_BAD_WRITE_POS 2u /* write_pos[slot] outside [0, ring_len)           */
#define GDN_DEV_TIMEOUT       4u /* an on-chip wait gave up (row output is garbage) */
#define GDN_DEV_INTERNAL      8u /* shared memory not aligned as the kernel assumes  */
#define GDN_DEV_BAD_ACCEPTED 16u /* a spec commit's accepted count outside [0, window] */

/* One layer's geometry.  Built: k_dim == v_dim in {64, 128}; 1 <= ring_len <= 64;
 * state_dtype GDN_F32; ring_dtype GDN_F32, GDN_F16 or GDN_BF16.
 *
 * Accuracy, as max|error| / max|exact| over one launch's outputs or flushed
 * checkpoints, against the recurrence with the ring's storage rounding:
 *   fp32 ring, FFMA or OUTPUT reconstruction           1e-5
 *   fp16 ring (any reconstruction), fp32 ring TENSOR   2e-3
 *   bf16 ring                                          2e-3 + 2^-7 (about 9.8e-3)
 * The bf16 ring is OUTSIDE the 2e-3 bound the tensor-core reconstruction is
 * specified to: a correction d that lies near a bf16 rounding boundary is
 * rounded one way here and may round the other way in any other evaluation,
 * one bf16 unit (2^-7 of the entry) apart, and the replay carries that into
 * later outputs and checkpoints.  It is accepted for callers that trade that
 * accuracy for a bf16 cache; the fp16 ring holds the same bytes within 2e-3. */
typedef struct {
    int32_t num_slots;   /* N  */
    int32_t num_v_heads; /* HV */
    int32_t num_k_heads; /* HK, HV % HK == 0 */
    int32_t k_dim;       /* K  */
    int32_t v_dim;       /* V  */
    int32_t ring_len;    /* L >= 1 (L == 1: every step flushes, the ring is never used) */
    int32_t gate;        /* gdn_gate_t  */
    int32_t state_dtype; /* gdn_dtype_t */
    int32_t ring_dtype;  /* gdn_dtype_t; the g ring is always fp32 */
} gdn_layer_desc_t;

/* One layer's cache, device pointers, layouts above.  state, ring_d and ring_k
 * must be 16-byte aligned.  The rings may be NULL when ring_len == 1. */
typedef struct {
    float *state;
    void *ring_d;
    void *ring_k;
    float *ring_g;
} gdn_layer_cache_t;

/* One decode step's inputs and output, device pointers. */
typedef struct {
    const void *mixed_qkv;            /* [B, row] in qkv_dtype                         */
    int32_t qkv_dtype;                /* gdn_dtype_t                                   */
    int64_t qkv_row_stride;           /* elements between rows (>= 2*HK*K + HV*V)      */
    const float *g;                   /* [B, HV] (GDN) or [B, HV, K] (KDA)             */
    const float *beta;                /* [B, HV]                                       */
    const int32_t *ssm_state_indices; /* [B] row -> slot; negative = padding row       */
    int32_t batch;                    /* B >= 0 (0: nothing is launched)               */
    float q_scale;                    /* q <- q * q_scale (1 when pre-scaled)          */
    int32_t qk_l2norm;                /* 1: q, k <- x / sqrt(sum x^2 + 1e-6) first     */
    void *out;                        /* [B, HV, V] in out_dtype                       */
    int32_t out_dtype;                /* gdn_dtype_t                                   */
    uint32_t flags;                   /* GDN_STEP_* bits below; 0 for none             */
} gdn_step_t;

/* gdn_step_t.flags.
 * GDN_STEP_OVERLAP_PREVIOUS: the caller states that the launch issued on the
 *   same stream just before this call writes none of this call's cache (state
 *   and rings), write_pos, ssm_state_indices and force_flush, and, if that
 *   launch was itself made with programmatic dependent launch, that it lets
 *   the work after it start only after it has waited for the work before it
 *   (every kernel of this library does; a kernel launched without programmatic
 *   dependent launch is always fine).  Example: each layer of a forward but
 *   the first, when the layers' decodes follow one another on the stream.
 *   The tensor-core decode then reads its rows and cursors and starts
 *   streaming checkpoints before that launch has finished, so its own start
 *   overlaps that launch's tail; it still reads mixed_qkv, g and beta, and
 *   writes anything at all, only after that launch has completed.  If the
 *   statement is false the results are undefined.  The other recon modes and
 *   gdn_packed_decode ignore the flag.  No counterpart in the pages: a
 *   property of this library's launches. */
#define GDN_STEP_OVERLAP_PREVIOUS 1u
/* GDN_STEP_PERSISTENT_KERNEL: with GDN_RECON_TENSOR, always run the
 *   persistent tensor-core kernel.  By default a batch of at most 64
 *   (row, value head) items (a GDN layer: up to 256 items while items x
 *   ring_len <= 2048) runs the small-batch kernel instead, and a layer
 *   with ring_len 1 the CUDA-core kernel (see gdn_replayssm_decode_kernel);
 *   this flag keeps the tensor-core kernel at any batch size and ring length.
 *   Ignored by the other recon modes. */
#define GDN_STEP_PERSISTENT_KERNEL 2u
#define GDN_STEP_KNOWN_FLAGS      3u

/* Packed decode, the read + write baseline ([P1] Motivation; [P2] section 1):
 * per row b with slot s = ssm_state_indices[b] >= 0 and every value head,
 *   S~ = alpha S (KDA: S Diag(exp g)),  d = beta (v - S~ k),  S <- S~ + d k^T,
 *   out = S q,
 * with S = state[s, hv] read and written back in place.  Padding rows (s < 0)
 * get out = 0 and touch nothing.  Rows must map to distinct slots. */
GDN_API gdn_status_t gdn_packed_decode(const gdn_layer_desc_t *desc, float *state,
                               const gdn_step_t *step, uint32_t *dev_status,
                               gdn_stream_t stream);

/* ReplaySSM decode of one layer ([P1] Modifications, Design 1/2/4/5/7; [P2]
 * 3.2, 3.3).  Per row b, slot s, p = write_pos[s], value head hv:
 *   is_flush = (p == L-1) or force_flush[b];
 *   S = A S0 + sum_{j<p} w_j d_j k_j^T (KDA: S0 Diag(A) + sum d_j (w_j o k_j)^T),
 *       A and w_j from the cached log-gates (empty sums give 1);
 *   GDN: Sq = alpha S q, Sk = alpha S k;   KDA: Sq = S (a o q), Sk = S (a o k);
 *   d = beta (v - Sk);   out = Sq + d (k^T q);
 *   flush:     state[s, hv] <- alpha S + d k^T (KDA: S Diag(a) + d k^T);
 *   otherwise: ring_d[s, hv, p] <- d, ring_g[s, hv, p] <- g and, from the first
 *              value head of each group, ring_k[s, hk, p] <- k (ring dtype, RNE).
 * Only ring entries j < p are read, so stale entries need no clearing.
 * write_pos is read only: call gdn_replayssm_advance once after the last layer
 * of the forward.  force_flush ([B] uint8, nonzero = flush) may be NULL.
 * flushed_out ([B] uint8, may be NULL) receives 1 for rows that flushed.
 * Padding rows (s < 0) get out = 0, flushed_out = 0 and touch nothing.
 * Rows must map to distinct slots.  recon is a gdn_recon_t (all three built). */
GDN_API gdn_status_t gdn_replayssm_decode(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                  const int32_t *write_pos, const uint8_t *force_flush,
                                  const gdn_step_t *step, int32_t recon, uint8_t *flushed_out,
                                  uint32_t *dev_status, gdn_stream_t stream);

/* Which kernel gdn_replayssm_decode (and _decode_advance) would launch for
 * these arguments, without launching anything (host only; reads the current
 * device's SM count and shared-memory limit).  *kernel receives one of:
 *   GDN_KERNEL_PERSISTENT_TC  persistent warp-specialised tensor-core kernel,
 *                             one block per SM (TENSOR recon)
 *   GDN_KERNEL_PER_HEAD_TC    one block per (row, value head), tensor cores
 *                             (TENSOR recon the persistent kernel cannot
 *                             take, e.g. a KDA g ring not 16-byte aligned,
 *                             32768 or more value heads, 2^24 or more slots)
 *   GDN_KERNEL_CUDA_CORE      CUDA-core kernel (FFMA or OUTPUT recon; also
 *                             TENSOR recon at ring_len 1 without
 *                             GDN_STEP_PERSISTENT_KERNEL: the ring is empty
 *                             and the decode is the packed decode's
 *                             read-modify-write, [P1] Design 1)
 *   GDN_KERNEL_SMALL_BATCH    TENSOR recon of a batch with at most 64
 *                             (row, value head) items, or a GDN layer's batch
 *                             of at most 256 with items x ring_len <= 2048
 *                             (unless the step has
 *                             GDN_STEP_PERSISTENT_KERNEL): one block per (row,
 *                             value head, slice of 16 to 128 state rows), every block on its
 *                             rows' whole step, replay sum in fp32 on the CUDA
 *                             cores (so within the FFMA bound), so that a
 *                             small batch still spreads over every SM
 * Argument checks and errors as in gdn_replayssm_decode.  No counterpart in
 * the pages: a diagnostic of this library's dispatch. */
#define GDN_KERNEL_PERSISTENT_TC 0
#define GDN_KERNEL_PER_HEAD_TC   1
#define GDN_KERNEL_CUDA_CORE     2
#define GDN_KERNEL_SMALL_BATCH   3
GDN_API gdn_status_t gdn_replayssm_decode_kernel(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                                 const gdn_step_t *step, int32_t recon, int32_t *kernel);

/* gdn_replayssm_decode of the forward's last layer followed by
 * gdn_replayssm_advance for the same rows, with the same results as the two
 * calls: the cursors are read before any is advanced.  On the tensor-core path
 * both happen in one launch (every block reads the cursors first; the last
 * block to finish advances them), otherwise in two.  write_pos is read and
 * written.  workspace: a caller-owned device buffer of
 * GDN_DECODE_ADVANCE_WORKSPACE_BYTES, 4-byte aligned, zeroed once before its
 * first use; every call leaves it zero again.  Calls that share a workspace
 * must not overlap on the GPU (e.g. on two streams).  Other arguments as in
 * gdn_replayssm_decode. */
#define GDN_DECODE_ADVANCE_WORKSPACE_BYTES 4
GDN_API gdn_status_t gdn_replayssm_decode_advance(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                          int32_t *write_pos, const uint8_t *force_flush,
                                          const gdn_step_t *step, int32_t recon, uint8_t *flushed_out,
                                          uint32_t *workspace, uint32_t *dev_status,
                                          gdn_stream_t stream);

/* gdn_replayssm_decode_advance without a caller workspace, for callers that
 * cannot allocate device memory: an engine that has reserved the whole device
 * for its own state and KV pools, a plugin whose host owns every allocation,
 * code that must not trigger cudaMalloc's implicit synchronisation.  The pages
 * have no counterpart; it exists only for such callers.
 * The scratch (one completion counter, GDN_DECODE_ADVANCE_WORKSPACE_BYTES)
 * comes from a 256-byte array compiled into the library, which every GPU that
 * loads the library keeps until the process exits; a call whose scratch need
 * exceeded it would be rejected with GDN_ERR_UNSUPPORTED.  The array is zero
 * when the library's module loads into a context, and every launch leaves the
 * counter at zero again, so nothing is ever cleared.  The first call in a
 * context (that of the current device) looks the array's device address up on
 * the host (cudaGetSymbolAddress); later calls in the same context reuse it,
 * and a new context (after cudaDeviceReset, say) gets a fresh lookup.  Make
 * that first call before any stream capture.  All calls in a context share
 * the array: calls that overlap on the GPU (e.g. on two streams) race on it
 * and must not be issued.  Nothing is allocated.  Arguments and results as in
 * gdn_replayssm_decode_advance. */
GDN_API gdn_status_t gdn_replayssm_decode_advance_noalloc(const gdn_layer_desc_t *desc,
                                                  const gdn_layer_cache_t *cache, int32_t *write_pos,
                                                  const uint8_t *force_flush, const gdn_step_t *step,
                                                  int32_t recon, uint8_t *flushed_out,
                                                  uint32_t *dev_status, gdn_stream_t stream);

/* Diagnostic for gdn_replayssm_decode_advance_noalloc (the pages have no
 * counterpart): copies the first n (1 .. 64) 32-bit words of the library's
 * scratch array on the current device into host_words (HOST memory), with a
 * blocking cudaMemcpy.  Between calls the first word, the completion counter,
 * is zero.  Allocates nothing. */
GDN_API gdn_status_t gdn_noalloc_scratch_peek(uint32_t *host_words, int32_t n);

/* Cursor advance, once per forward after all layers ([P1] Design 3):
 * write_pos[s] <- (write_pos[s] == L-1 or force_flush[b]) ? 0 : write_pos[s] + 1
 * for each row b with s = ssm_state_indices[b] >= 0.  force_flush may be NULL. */
GDN_API gdn_status_t gdn_replayssm_advance(const int32_t *ssm_state_indices, int32_t batch,
                                   const uint8_t *force_flush, int32_t num_slots,
                                   int32_t ring_len, int32_t *write_pos,
                                   uint32_t *dev_status, gdn_stream_t stream);

/* Fold the ring into the checkpoint for each listed slot (every value head):
 * state[s] <- A S0 + sum_{j<write_pos[s]} w_j d_j k_j^T, in fp32 on the CUDA
 * cores.  This is the state a snapshot or a copy-on-write must see ([P1]
 * Design 5; [P2] 4.1).  write_pos is not changed: follow with
 * gdn_replayssm_reset_slots.  Negative entries of slots[n] are skipped. */
GDN_API gdn_status_t gdn_replayssm_flush(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                 const int32_t *write_pos, const int32_t *slots, int32_t n,
                                 uint32_t *dev_status, gdn_stream_t stream);

/* write_pos[slots[i]] <- 0 for each listed slot (slot allocation and
 * copy-on-write, [P1] Design 3 and 5).  Negative entries are skipped. */
GDN_API gdn_status_t gdn_replayssm_reset_slots(int32_t *write_pos, int32_t num_slots,
                                       const int32_t *slots, int32_t n,
                                       uint32_t *dev_status, gdn_stream_t stream);

/* One speculative verify step: B rows of T tokens each; token t of row b is
 * input / output row b*T + t ([P3] Core concept).  Device pointers. */
typedef struct {
    const void *mixed_qkv;            /* [B*T, row] in qkv_dtype (row layout as gdn_step_t) */
    int32_t qkv_dtype;                /* gdn_dtype_t                                         */
    int64_t qkv_row_stride;           /* elements between token rows                         */
    const float *g;                   /* [B*T, HV] (GDN) or [B*T, HV, K] (KDA)               */
    const float *beta;                /* [B*T, HV]                                           */
    const int32_t *ssm_state_indices; /* [B] row -> slot; negative = padding row             */
    int32_t batch;                    /* B >= 0                                              */
    int32_t window;                   /* T, 1 <= T <= min(ring_len - 1, 32)                   */
    float q_scale;                    /* as in gdn_step_t                                    */
    int32_t qk_l2norm;                /* as in gdn_step_t                                    */
    void *out;                        /* [B*T, HV, V] in out_dtype                           */
    int32_t out_dtype;                /* gdn_dtype_t                                         */
} gdn_spec_step_t;

/* Speculative verify window of one layer ([P3] Core concept, Design notes).
 * Row b with slot s and p = write_pos[s] (requires p + T <= L - 1) decodes its
 * T tokens from the checkpoint and the committed entries j < p: token t is the
 * non-flush decode at cursor p + t, seeing the window's earlier tokens as
 * cached entries; its output goes to out row b*T + t and its (d, k, g) to ring
 * position p + t (k once per key head).  The checkpoint and write_pos are not
 * changed: after the target model has accepted a tokens, call
 * gdn_replayssm_spec_commit.  A row whose window does not fit sets
 * GDN_DEV_BAD_WRITE_POS and is treated as padding (zeros).
 * recon = GDN_RECON_TENSOR: the checkpoint products S0 [q_t, k_t] run on the
 * tensor cores (tf32) for K = V = 128 and window <= 16, the ring and window
 * terms in fp32 on the CUDA cores; other shapes, or GDN_RECON_FFMA, use the
 * CUDA-core kernel (all fp32). */
GDN_API gdn_status_t gdn_replayssm_spec_verify(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                       const int32_t *write_pos, const gdn_spec_step_t *step, int32_t recon,
                                       uint32_t *dev_status, gdn_stream_t stream);

/* Commit after a verify window, once per forward ([P3] Core concept: a
 * rejected draft is undone by moving the cursor, nothing else):
 * write_pos[s] += accepted[b] (0 <= accepted[b] <= window); rejected drafts
 * stay in the ring past the cursor and are never read.  flush_slots[b]
 * ([B] int32) receives s when the next window would not fit
 * (write_pos[s] + window > L - 1), else -1: pass it to gdn_replayssm_flush for
 * every layer and then to gdn_replayssm_reset_slots.  Padding rows get -1. */
GDN_API gdn_status_t gdn_replayssm_spec_commit(const int32_t *ssm_state_indices, const int32_t *accepted,
                                       int32_t batch, int32_t window, int32_t num_slots,
                                       int32_t ring_len, int32_t *write_pos, int32_t *flush_slots,
                                       uint32_t *dev_status, gdn_stream_t stream);

/* Lossless speculative verify ([P5] The idea; Modifications, Verify kernel):
 * the sequential verify that updates no state and, in place of a state
 * snapshot per draft token, keeps each token's (u, k, g) in fp32 tuple buffers.
 * Row b with slot s = ssm_state_indices[b] decodes its T = window tokens (input
 * and output rows b*T + t, layouts as in gdn_spec_step_t) with the recurrence of
 * gdn_packed_decode, starting from state[s]: token t's output is bit-identical
 * to the output of the t-th of T successive gdn_packed_decode calls on the same
 * inputs.  Tuples (device, fp32, caller-owned):
 *   tup_u [B, T, HV, V]          u = beta (v - S~ k), the correction
 *   tup_k [B, T, HK, K]          the key as the update uses it (after the optional norm)
 *   tup_g [B, T, HV] (KDA [B, T, HV, K])  the log-gate
 * state is only read.  Padding rows (s < 0) get zero outputs and leave their
 * tuples alone; s >= num_slots sets GDN_DEV_BAD_SLOT and is treated the same.
 * The ring fields of desc are not used.  1 <= window <= 32. */
GDN_API gdn_status_t gdn_lossless_verify(const gdn_layer_desc_t *desc, const float *state,
                                         const gdn_spec_step_t *step, float *tup_u, float *tup_k,
                                         float *tup_g, uint32_t *dev_status, gdn_stream_t stream);

/* Exact-order commit after gdn_lossless_verify ([P5] The idea; Modifications,
 * Commit): for row b with source slot s = ssm_state_indices[b] and
 * a = accepted[b] (0 <= a <= window), every value head replays
 *   h <- fma(k_t, u_t, fl(h * exp(g_t))),   t = 0 .. a-1   (KDA: exp per key channel)
 * from h = state[s] in fp32, with the decayed state one rounded multiply and the
 * rank-1 update one fused multiply-add per element — the rounding of
 * gdn_packed_decode's update — and stores h at slot dst = dst_indices[b]
 * (dst_indices NULL: back at s).  The stored state is bit-identical to the one
 * a successive gdn_packed_decode calls leave.  A second target (a prefix-cache
 * track state at another slot) must be committed before the in-place commit of
 * the same source, in an earlier call: both replay from the pre-verify state.
 * Rows with a negative s, dst or a are skipped; s or dst >= num_slots
 * (GDN_DEV_BAD_SLOT) and a > window (GDN_DEV_BAD_ACCEPTED) are reported and
 * skipped.  Within one call the rows' destinations must be distinct and differ
 * from the other rows' sources.  Tuples as gdn_lossless_verify wrote them. */
GDN_API gdn_status_t gdn_lossless_commit(const gdn_layer_desc_t *desc, float *state,
                                         const int32_t *ssm_state_indices, const int32_t *dst_indices,
                                         const int32_t *accepted, int32_t batch, int32_t window,
                                         const float *tup_u, const float *tup_k, const float *tup_g,
                                         uint32_t *dev_status, gdn_stream_t stream);

/* Self-test of the on-chip wait bound (no counterpart in the pages).  The
 * decode kernels wait on shared-memory barriers through one bounded wait: when
 * a wait runs out (a copy or a contraction that never completes) the kernel
 * ORs GDN_DEV_TIMEOUT into dev_status and returns instead of hanging.  This
 * call launches one block that runs that same wait on a barrier no thread ever
 * arrives on, with a limit of limit_us microseconds (1 .. 100000), so it
 * always runs out: *dev_status gets GDN_DEV_TIMEOUT and the context stays
 * usable.  dev_status is a device uint32 (required). */
GDN_API gdn_status_t gdn_selftest_wait_timeout(uint32_t *dev_status, uint32_t limit_us, gdn_stream_t stream);

/* Static text for a status code (host). */
GDN_API const char *gdn_status_str(gdn_status_t status);

/* Message for the calling host thread's last failing call ("" if none). */
GDN_API const char *gdn_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GDNREPLAY_H */
