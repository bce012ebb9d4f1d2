// Internal launchers (host side) of the gdnreplay kernels; arguments are
// already validated by the C ABI layer.
#pragma once

#include <cuda_runtime.h>

#include "gdn_common.cuh"

namespace gdn {

// Packed decode (replay = false) or ReplaySSM decode with FFMA replay (replay = true).
cudaError_t launch_ffma_decode(const DecodeParams &P, int D, int gate, bool replay, cudaStream_t s);

// ReplaySSM decode whose non-flush rows read the output out through the ring
// without forming the replayed state (CUDA cores); flush rows as the FFMA replay.
cudaError_t launch_output_only_decode(const DecodeParams &P, int D, int gate, cudaStream_t s);

// ReplaySSM decode with the replay sum on the tensor cores (tcgen05) and the
// checkpoint streamed by TMA.  Writes a reason into *why on a host-side failure.
// With P.sync set, *fused tells whether the launched kernel also advanced the
// cursors (the persistent kernel does; the one-CTA-per-head fallback does not).
cudaError_t launch_tc_decode(const DecodeParams &P, int D, int gate, cudaStream_t s, const char **why,
                             bool *fused);

// Persistent warp-specialised variant of the above (one CTA per SM).  Returns
// cudaErrorNotSupported, with nothing launched, when its shared-memory layout
// does not fit the configuration.
cudaError_t launch_tcp_decode(const DecodeParams &P, int D, int gate, const CUtensorMap &map, cudaStream_t s);
// Whether launch_tcp_decode would take this launch (host-side, launches nothing).
bool tcp_decode_fits(const DecodeParams &P, int D, int gate);

// Small-batch decode (one block per (row, value head, slice of state rows),
// CUDA cores): taken by the tensor-core recon when the batch has at most
// kSlabMaxItems (row, value head) items, or, for a GDN layer, at most
// 4 kSlabMaxItems items with items x L <= 32 kSlabMaxItems, unless
// P.persistent_only (measured, HV = 32: it beats the persistent kernel up to
// B = 2 at any ring length and at B = 4 and 8 with short rings; past that its
// CUDA-core replay sum becomes the cost).
constexpr int kSlabMaxItems = 64;
bool slab_decode_takes(const DecodeParams &P, int gate);
cudaError_t launch_slab_decode(const DecodeParams &P, int D, int gate, cudaStream_t s);

cudaError_t launch_fold(const DecodeParams &P, int D, int gate, int n, cudaStream_t s);

// Tensor map of the checkpoint as [N*HV*V rows, K fp32 columns] with boxes of
// [V rows x 32 columns], 128-byte swizzled.  Writes a reason into *why on failure.
cudaError_t make_state_tmap(const DecodeParams &P, int D, CUtensorMap *map, const char **why);
// A plain (unswizzled) 2-D tensor map: `rows` rows of `inner` elements of
// `dtype` (a gdn_dtype_t), `row_bytes` apart, boxes of box_rows x box_inner.
cudaError_t make_tmap_2d(const void *base, int dtype, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_rows, CUtensorMap *map);

// Speculative verify window (P.T tokens per row) on the CUDA cores, and the
// commit that follows.
cudaError_t launch_spec_verify(const DecodeParams &P, int D, int gate, cudaStream_t s);
// The same window with the checkpoint contraction on the tensor cores.  Returns
// cudaErrorNotSupported, with nothing launched, for configurations it does not
// cover (the caller then uses the CUDA-core kernel).
cudaError_t launch_spec_tc(const DecodeParams &P, int D, int gate, cudaStream_t s, const char **why);
cudaError_t launch_spec_commit(const int32_t *idx, const int32_t *accepted, int B, int T, int N, int L,
                               int32_t *write_pos, int32_t *flush_slots, uint32_t *status, cudaStream_t s);

// Lossless verify (P.T tokens per row, no state update, fp32 (u, k, g) tuples)
// and the exact-order commit that replays accepted tuples into the state.
cudaError_t launch_lossless_verify(const DecodeParams &P, int D, int gate, float *tup_u, float *tup_k,
                                   float *tup_g, cudaStream_t s);
cudaError_t launch_lossless_commit(const DecodeParams &P, int D, int gate, const int32_t *dst_idx,
                                   const int32_t *accepted, const float *tup_u, const float *tup_k,
                                   const float *tup_g, cudaStream_t s);

cudaError_t launch_advance(const int32_t *idx, int B, const uint8_t *ff, int N, int L,
                           int32_t *write_pos, uint32_t *status, cudaStream_t s);

cudaError_t launch_reset(int32_t *write_pos, int N, const int32_t *slots, int n, uint32_t *status,
                         cudaStream_t s);

// Dynamic shared memory of one tensor-core decode CTA (bytes).
size_t tc_smem_bytes(int D, int gate, int ring_dtype, int L);

// Sets the calling thread's gdn_last_error() text (for entry points defined
// outside the C ABI file).
void set_last_error(const char *msg);

}  // namespace gdn
