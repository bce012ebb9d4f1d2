// C ABI of libgdnreplay: host-side argument checks, then one kernel launch per
// call on the caller's stream.  Nothing here allocates or synchronises.
#include <stdio.h>

#include <string>

#include "gdn_kernels.h"

namespace {

thread_local std::string g_last_error;

gdn_status_t fail(gdn_status_t st, const std::string &msg) {
  g_last_error = msg;
  return st;
}

gdn_status_t cuda_fail(cudaError_t e, const char *what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return GDN_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dtype_ok(int32_t d) { return d == GDN_F32 || d == GDN_BF16 || d == GDN_F16; }

gdn_status_t check_desc(const gdn_layer_desc_t *d) {
  if (!d) return fail(GDN_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_slots <= 0 || d->num_v_heads <= 0 || d->num_k_heads <= 0 || d->k_dim <= 0 ||
      d->v_dim <= 0 || d->ring_len <= 0)
    return fail(GDN_ERR_INVALID_ARG, "sizes must be positive");
  if (d->num_v_heads % d->num_k_heads)
    return fail(GDN_ERR_INVALID_ARG, "num_v_heads must be a multiple of num_k_heads");
  if (d->gate != GDN_GATE_SCALAR && d->gate != GDN_GATE_PER_K)
    return fail(GDN_ERR_INVALID_ARG, "gate must be GDN_GATE_SCALAR or GDN_GATE_PER_K");
  if (!dtype_ok(d->state_dtype) || !dtype_ok(d->ring_dtype))
    return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
  if (d->k_dim != d->v_dim || (d->k_dim != 64 && d->k_dim != 128))
    return fail(GDN_ERR_UNSUPPORTED, "built for k_dim == v_dim in {64, 128}");
  if (d->ring_len > 64) return fail(GDN_ERR_UNSUPPORTED, "built for ring_len <= 64");
  if (d->state_dtype != GDN_F32) return fail(GDN_ERR_UNSUPPORTED, "state must be fp32");
  const int64_t elems = (int64_t)d->num_slots * d->num_v_heads * d->v_dim;
  if (elems >= (int64_t)1 << 31) return fail(GDN_ERR_UNSUPPORTED, "N*HV*V must be < 2^31");
  return GDN_OK;
}

gdn_status_t check_step(const gdn_layer_desc_t *d, const gdn_step_t *s) {
  if (!s) return fail(GDN_ERR_INVALID_ARG, "step is NULL");
  if (s->batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch must be >= 0");
  if (s->batch == 0) return GDN_OK;
  if (!s->mixed_qkv || !s->g || !s->beta || !s->ssm_state_indices || !s->out)
    return fail(GDN_ERR_INVALID_ARG, "step has a NULL input or output pointer");
  if (!dtype_ok(s->qkv_dtype) || !dtype_ok(s->out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "unknown qkv or out dtype");
  const int64_t row = 2 * (int64_t)d->num_k_heads * d->k_dim + (int64_t)d->num_v_heads * d->v_dim;
  if (s->qkv_row_stride < row)
    return fail(GDN_ERR_INVALID_ARG, "qkv_row_stride is shorter than 2*HK*K + HV*V");
  if ((int64_t)s->batch * d->num_v_heads >= (int64_t)1 << 31)
    return fail(GDN_ERR_UNSUPPORTED, "batch * num_v_heads must be < 2^31");
  if (s->flags & ~GDN_STEP_KNOWN_FLAGS) return fail(GDN_ERR_INVALID_ARG, "unknown bits in step flags");
  return GDN_OK;
}

gdn::DecodeParams base_params(const gdn_layer_desc_t *d) {
  gdn::DecodeParams P{};
  P.N = d->num_slots;
  P.HV = d->num_v_heads;
  P.HK = d->num_k_heads;
  P.G = d->num_v_heads / d->num_k_heads;
  P.L = d->ring_len;
  P.ring_dtype = d->ring_dtype;
  return P;
}

void fill_step(gdn::DecodeParams &P, const gdn_step_t *s) {
  P.qkv = s->mixed_qkv;
  P.qkv_dtype = s->qkv_dtype;
  P.qkv_stride = s->qkv_row_stride;
  P.g = s->g;
  P.beta = s->beta;
  P.idx = s->ssm_state_indices;
  P.B = s->batch;
  P.q_scale = s->q_scale;
  P.qk_l2norm = s->qk_l2norm;
  P.out = s->out;
  P.out_dtype = s->out_dtype;
  P.overlap = (s->flags & GDN_STEP_OVERLAP_PREVIOUS) ? 1 : 0;
  P.persistent_only = (s->flags & GDN_STEP_PERSISTENT_KERNEL) ? 1 : 0;
}

gdn_status_t check_cache(const gdn_layer_desc_t *d, const gdn_layer_cache_t *c) {
  if (!c) return fail(GDN_ERR_INVALID_ARG, "cache is NULL");
  if (!c->state) return fail(GDN_ERR_INVALID_ARG, "cache.state is NULL");
  if (!aligned16(c->state)) return fail(GDN_ERR_INVALID_ARG, "cache.state must be 16-byte aligned");
  if (d->ring_len > 1) {
    if (!c->ring_d || !c->ring_k || !c->ring_g)
      return fail(GDN_ERR_INVALID_ARG, "ring pointers must be set when ring_len > 1");
    if (!aligned16(c->ring_d) || !aligned16(c->ring_k))
      return fail(GDN_ERR_INVALID_ARG, "ring_d and ring_k must be 16-byte aligned");
  }
  return GDN_OK;
}

}  // namespace

namespace gdn {
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace gdn

extern "C" {

const char *gdn_status_str(gdn_status_t s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char *gdn_last_error(void) { return g_last_error.c_str(); }

gdn_status_t gdn_packed_decode(const gdn_layer_desc_t *desc, float *state, const gdn_step_t *step,
                               uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_step(desc, step)) != GDN_OK) return st;
  if (!state) return fail(GDN_ERR_INVALID_ARG, "state is NULL");
  if (!aligned16(state)) return fail(GDN_ERR_INVALID_ARG, "state must be 16-byte aligned");
  if (step->batch == 0) return GDN_OK;
  gdn::DecodeParams P = base_params(desc);
  fill_step(P, step);
  P.state = state;
  P.status = dev_status;
  cudaError_t e = gdn::launch_ffma_decode(P, desc->k_dim, desc->gate, false, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_packed_decode launch");
}

// L = 1: there is no ring, every live row flushes, and the replay contraction
// is empty, so the decode is the packed decode ([P1] Design 1).  A tensor-core call then
// runs the CUDA-core replay kernel, which at L = 1 is the packed decode's
// read-modify-write with the replay's row checks, flush flags and status: the
// persistent tensor-core kernel would move the same bytes with its per-launch
// set-up on top.  GDN_STEP_PERSISTENT_KERNEL still forces the persistent kernel.
static bool tensor_recon_is_empty(const gdn_layer_desc_t *desc, const gdn_step_t *step) {
  return desc->ring_len == 1 && !(step->flags & GDN_STEP_PERSISTENT_KERNEL);
}

gdn_status_t gdn_replayssm_decode(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                  const int32_t *write_pos, const uint8_t *force_flush,
                                  const gdn_step_t *step, int32_t recon, uint8_t *flushed_out,
                                  uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_step(desc, step)) != GDN_OK) return st;
  if ((st = check_cache(desc, cache)) != GDN_OK) return st;
  if (!write_pos) return fail(GDN_ERR_INVALID_ARG, "write_pos is NULL");
  if (recon != GDN_RECON_TENSOR && recon != GDN_RECON_FFMA && recon != GDN_RECON_OUTPUT)
    return fail(GDN_ERR_INVALID_ARG, "recon must be GDN_RECON_TENSOR, GDN_RECON_FFMA or GDN_RECON_OUTPUT");
  if (step->batch == 0) return GDN_OK;
  gdn::DecodeParams P = base_params(desc);
  fill_step(P, step);
  P.state = cache->state;
  P.ring_d = cache->ring_d;
  P.ring_k = cache->ring_k;
  P.ring_g = cache->ring_g;
  P.write_pos = write_pos;
  P.force_flush = force_flush;
  P.flushed = flushed_out;
  P.status = dev_status;
  cudaError_t e;
  if (recon == GDN_RECON_FFMA || (recon == GDN_RECON_TENSOR && tensor_recon_is_empty(desc, step))) {
    e = gdn::launch_ffma_decode(P, desc->k_dim, desc->gate, true, (cudaStream_t)stream);
  } else if (recon == GDN_RECON_OUTPUT) {
    e = gdn::launch_output_only_decode(P, desc->k_dim, desc->gate, (cudaStream_t)stream);
  } else {
    const char *why = nullptr;
    bool fused = false;
    e = gdn::launch_tc_decode(P, desc->k_dim, desc->gate, (cudaStream_t)stream, &why, &fused);
    if (e != cudaSuccess && why) return fail(GDN_ERR_CUDA, why);
  }
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_decode launch");
}

gdn_status_t gdn_replayssm_decode_kernel(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                         const gdn_step_t *step, int32_t recon, int32_t *kernel) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_step(desc, step)) != GDN_OK) return st;
  if ((st = check_cache(desc, cache)) != GDN_OK) return st;
  if (!kernel) return fail(GDN_ERR_INVALID_ARG, "kernel is NULL");
  if (recon != GDN_RECON_TENSOR && recon != GDN_RECON_FFMA && recon != GDN_RECON_OUTPUT)
    return fail(GDN_ERR_INVALID_ARG, "recon must be GDN_RECON_TENSOR, GDN_RECON_FFMA or GDN_RECON_OUTPUT");
  if (recon != GDN_RECON_TENSOR || tensor_recon_is_empty(desc, step)) {
    *kernel = GDN_KERNEL_CUDA_CORE;
    return GDN_OK;
  }
  gdn::DecodeParams P = base_params(desc);
  fill_step(P, step);
  P.state = cache->state;
  P.ring_d = cache->ring_d;
  P.ring_k = cache->ring_k;
  P.ring_g = cache->ring_g;
  if (gdn::slab_decode_takes(P, desc->gate))
    *kernel = GDN_KERNEL_SMALL_BATCH;
  else
    *kernel = gdn::tcp_decode_fits(P, desc->k_dim, desc->gate) ? GDN_KERNEL_PERSISTENT_TC : GDN_KERNEL_PER_HEAD_TC;
  return GDN_OK;
}

gdn_status_t gdn_replayssm_decode_advance(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                          int32_t *write_pos, const uint8_t *force_flush,
                                          const gdn_step_t *step, int32_t recon, uint8_t *flushed_out,
                                          uint32_t *workspace, uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_step(desc, step)) != GDN_OK) return st;
  if ((st = check_cache(desc, cache)) != GDN_OK) return st;
  if (!write_pos) return fail(GDN_ERR_INVALID_ARG, "write_pos is NULL");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
    return fail(GDN_ERR_INVALID_ARG, "workspace must be a 4-byte aligned device pointer");
  if (recon != GDN_RECON_TENSOR && recon != GDN_RECON_FFMA && recon != GDN_RECON_OUTPUT)
    return fail(GDN_ERR_INVALID_ARG, "recon must be GDN_RECON_TENSOR, GDN_RECON_FFMA or GDN_RECON_OUTPUT");
  if (step->batch == 0) return GDN_OK;
  gdn::DecodeParams P = base_params(desc);
  fill_step(P, step);
  P.state = cache->state;
  P.ring_d = cache->ring_d;
  P.ring_k = cache->ring_k;
  P.ring_g = cache->ring_g;
  P.write_pos = write_pos;
  P.force_flush = force_flush;
  P.flushed = flushed_out;
  P.status = dev_status;
  cudaError_t e;
  bool fused = false;
  if (recon == GDN_RECON_TENSOR && tensor_recon_is_empty(desc, step)) {
    e = gdn::launch_ffma_decode(P, desc->k_dim, desc->gate, true, (cudaStream_t)stream);
    fused = true;  // L = 1: a valid cursor is 0 and stays 0 (every live row flushes), so no advance is due
  } else if (recon == GDN_RECON_FFMA) {
    e = gdn::launch_ffma_decode(P, desc->k_dim, desc->gate, true, (cudaStream_t)stream);
  } else if (recon == GDN_RECON_OUTPUT) {
    e = gdn::launch_output_only_decode(P, desc->k_dim, desc->gate, (cudaStream_t)stream);
  } else {
    P.sync = workspace;
    P.write_pos_w = write_pos;
    const char *why = nullptr;
    e = gdn::launch_tc_decode(P, desc->k_dim, desc->gate, (cudaStream_t)stream, &why, &fused);
    if (e != cudaSuccess && why) return fail(GDN_ERR_CUDA, why);
  }
  if (e != cudaSuccess) return cuda_fail(e, "gdn_replayssm_decode_advance launch");
  if (!fused) {  // the kernel that ran left the cursors alone: advance them in a second launch
    e = gdn::launch_advance(step->ssm_state_indices, step->batch, force_flush, desc->num_slots, desc->ring_len,
                            write_pos, dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_replayssm_decode_advance: advance launch");
  }
  return GDN_OK;
}

gdn_status_t gdn_replayssm_spec_verify(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                       const int32_t *write_pos, const gdn_spec_step_t *step, int32_t recon,
                                       uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_cache(desc, cache)) != GDN_OK) return st;
  if (!step) return fail(GDN_ERR_INVALID_ARG, "step is NULL");
  if (!write_pos) return fail(GDN_ERR_INVALID_ARG, "write_pos is NULL");
  if (recon != GDN_RECON_TENSOR && recon != GDN_RECON_FFMA) return fail(GDN_ERR_INVALID_ARG, "unknown recon");
  if (step->batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch must be >= 0");
  if (step->window < 1 || step->window > desc->ring_len - 1)
    return fail(GDN_ERR_INVALID_ARG, "window must be in [1, ring_len - 1]");
  if (step->window > 32) return fail(GDN_ERR_UNSUPPORTED, "built for window <= 32");
  if (step->batch == 0) return GDN_OK;
  if (!step->mixed_qkv || !step->g || !step->beta || !step->ssm_state_indices || !step->out)
    return fail(GDN_ERR_INVALID_ARG, "step has a NULL input or output pointer");
  if (!dtype_ok(step->qkv_dtype) || !dtype_ok(step->out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "unknown qkv or out dtype");
  const int64_t row = 2 * (int64_t)desc->num_k_heads * desc->k_dim + (int64_t)desc->num_v_heads * desc->v_dim;
  if (step->qkv_row_stride < row) return fail(GDN_ERR_INVALID_ARG, "qkv_row_stride is shorter than 2*HK*K + HV*V");
  if ((int64_t)step->batch * step->window * desc->num_v_heads >= (int64_t)1 << 31)
    return fail(GDN_ERR_UNSUPPORTED, "batch * window * num_v_heads must be < 2^31");
  gdn::DecodeParams P = base_params(desc);
  P.qkv = step->mixed_qkv;
  P.qkv_dtype = step->qkv_dtype;
  P.qkv_stride = step->qkv_row_stride;
  P.g = step->g;
  P.beta = step->beta;
  P.idx = step->ssm_state_indices;
  P.B = step->batch;
  P.T = step->window;
  P.q_scale = step->q_scale;
  P.qk_l2norm = step->qk_l2norm;
  P.out = step->out;
  P.out_dtype = step->out_dtype;
  P.state = cache->state;
  P.ring_d = cache->ring_d;
  P.ring_k = cache->ring_k;
  P.ring_g = cache->ring_g;
  P.write_pos = write_pos;
  P.status = dev_status;
  cudaError_t e = cudaErrorNotSupported;
  if (recon == GDN_RECON_TENSOR) {
    const char *why = nullptr;
    e = gdn::launch_spec_tc(P, desc->k_dim, desc->gate, (cudaStream_t)stream, &why);
    if (e != cudaSuccess && e != cudaErrorNotSupported)
      return cuda_fail(e, why ? why : "gdn_replayssm_spec_verify tensor-core launch");
  }
  if (e == cudaErrorNotSupported) e = gdn::launch_spec_verify(P, desc->k_dim, desc->gate, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_spec_verify launch");
}

gdn_status_t gdn_replayssm_spec_commit(const int32_t *ssm_state_indices, const int32_t *accepted,
                                       int32_t batch, int32_t window, int32_t num_slots,
                                       int32_t ring_len, int32_t *write_pos, int32_t *flush_slots,
                                       uint32_t *dev_status, gdn_stream_t stream) {
  if (batch < 0 || num_slots <= 0 || ring_len <= 1 || window < 1 || window > ring_len - 1)
    return fail(GDN_ERR_INVALID_ARG,
                "batch >= 0, num_slots > 0, ring_len > 1 and 1 <= window <= ring_len - 1 are required");
  if (batch == 0) return GDN_OK;
  if (!ssm_state_indices || !accepted || !write_pos || !flush_slots)
    return fail(GDN_ERR_INVALID_ARG, "ssm_state_indices, accepted, write_pos and flush_slots must be set");
  cudaError_t e = gdn::launch_spec_commit(ssm_state_indices, accepted, batch, window, num_slots, ring_len,
                                          write_pos, flush_slots, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_spec_commit launch");
}

gdn_status_t gdn_lossless_verify(const gdn_layer_desc_t *desc, const float *state, const gdn_spec_step_t *step,
                                 float *tup_u, float *tup_k, float *tup_g, uint32_t *dev_status,
                                 gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if (!step) return fail(GDN_ERR_INVALID_ARG, "step is NULL");
  if (step->batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch must be >= 0");
  if (step->window < 1) return fail(GDN_ERR_INVALID_ARG, "window must be >= 1");
  if (step->window > 32) return fail(GDN_ERR_UNSUPPORTED, "built for window <= 32");
  if (step->batch == 0) return GDN_OK;
  if (!state) return fail(GDN_ERR_INVALID_ARG, "state is NULL");
  if (!aligned16(state)) return fail(GDN_ERR_INVALID_ARG, "state must be 16-byte aligned");
  if (!tup_u || !tup_k || !tup_g) return fail(GDN_ERR_INVALID_ARG, "tuple buffers must be set");
  if (!step->mixed_qkv || !step->g || !step->beta || !step->ssm_state_indices || !step->out)
    return fail(GDN_ERR_INVALID_ARG, "step has a NULL input or output pointer");
  if (!dtype_ok(step->qkv_dtype) || !dtype_ok(step->out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "unknown qkv or out dtype");
  const int64_t row = 2 * (int64_t)desc->num_k_heads * desc->k_dim + (int64_t)desc->num_v_heads * desc->v_dim;
  if (step->qkv_row_stride < row) return fail(GDN_ERR_INVALID_ARG, "qkv_row_stride is shorter than 2*HK*K + HV*V");
  if ((int64_t)step->batch * step->window * desc->num_v_heads >= (int64_t)1 << 31)
    return fail(GDN_ERR_UNSUPPORTED, "batch * window * num_v_heads must be < 2^31");
  gdn::DecodeParams P = base_params(desc);
  P.qkv = step->mixed_qkv;
  P.qkv_dtype = step->qkv_dtype;
  P.qkv_stride = step->qkv_row_stride;
  P.g = step->g;
  P.beta = step->beta;
  P.idx = step->ssm_state_indices;
  P.B = step->batch;
  P.T = step->window;
  P.q_scale = step->q_scale;
  P.qk_l2norm = step->qk_l2norm;
  P.out = step->out;
  P.out_dtype = step->out_dtype;
  P.state = const_cast<float *>(state);  // read only
  P.status = dev_status;
  cudaError_t e = gdn::launch_lossless_verify(P, desc->k_dim, desc->gate, tup_u, tup_k, tup_g, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_lossless_verify launch");
}

gdn_status_t gdn_lossless_commit(const gdn_layer_desc_t *desc, float *state, const int32_t *ssm_state_indices,
                                 const int32_t *dst_indices, const int32_t *accepted, int32_t batch,
                                 int32_t window, const float *tup_u, const float *tup_k, const float *tup_g,
                                 uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if (batch < 0) return fail(GDN_ERR_INVALID_ARG, "batch must be >= 0");
  if (window < 1) return fail(GDN_ERR_INVALID_ARG, "window must be >= 1");
  if (window > 32) return fail(GDN_ERR_UNSUPPORTED, "built for window <= 32");
  if (batch == 0) return GDN_OK;
  if (!state) return fail(GDN_ERR_INVALID_ARG, "state is NULL");
  if (!aligned16(state)) return fail(GDN_ERR_INVALID_ARG, "state must be 16-byte aligned");
  if (!ssm_state_indices || !accepted || !tup_u || !tup_k || !tup_g)
    return fail(GDN_ERR_INVALID_ARG, "ssm_state_indices, accepted and the tuple buffers must be set");
  if ((int64_t)batch * window * desc->num_v_heads >= (int64_t)1 << 31)
    return fail(GDN_ERR_UNSUPPORTED, "batch * window * num_v_heads must be < 2^31");
  gdn::DecodeParams P = base_params(desc);
  P.state = state;
  P.idx = ssm_state_indices;
  P.B = batch;
  P.T = window;
  P.status = dev_status;
  cudaError_t e = gdn::launch_lossless_commit(P, desc->k_dim, desc->gate, dst_indices, accepted, tup_u, tup_k,
                                              tup_g, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_lossless_commit launch");
}

gdn_status_t gdn_replayssm_advance(const int32_t *ssm_state_indices, int32_t batch,
                                   const uint8_t *force_flush, int32_t num_slots, int32_t ring_len,
                                   int32_t *write_pos, uint32_t *dev_status, gdn_stream_t stream) {
  if (batch < 0 || num_slots <= 0 || ring_len <= 0)
    return fail(GDN_ERR_INVALID_ARG, "batch >= 0, num_slots > 0 and ring_len > 0 are required");
  if (batch == 0) return GDN_OK;
  if (!ssm_state_indices || !write_pos)
    return fail(GDN_ERR_INVALID_ARG, "ssm_state_indices and write_pos must be set");
  cudaError_t e = gdn::launch_advance(ssm_state_indices, batch, force_flush, num_slots, ring_len,
                                      write_pos, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_advance launch");
}

gdn_status_t gdn_replayssm_flush(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                 const int32_t *write_pos, const int32_t *slots, int32_t n,
                                 uint32_t *dev_status, gdn_stream_t stream) {
  gdn_status_t st = check_desc(desc);
  if (st != GDN_OK) return st;
  if ((st = check_cache(desc, cache)) != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_INVALID_ARG, "n must be >= 0");
  if (n == 0) return GDN_OK;
  if (!write_pos || !slots) return fail(GDN_ERR_INVALID_ARG, "write_pos and slots must be set");
  if ((int64_t)n * desc->num_v_heads >= (int64_t)1 << 31)
    return fail(GDN_ERR_UNSUPPORTED, "n * num_v_heads must be < 2^31");
  gdn::DecodeParams P = base_params(desc);
  P.state = cache->state;
  P.ring_d = cache->ring_d;
  P.ring_k = cache->ring_k;
  P.ring_g = cache->ring_g;
  P.write_pos = write_pos;
  P.slots = slots;
  P.status = dev_status;
  cudaError_t e = gdn::launch_fold(P, desc->k_dim, desc->gate, n, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_flush launch");
}

gdn_status_t gdn_replayssm_reset_slots(int32_t *write_pos, int32_t num_slots, const int32_t *slots,
                                       int32_t n, uint32_t *dev_status, gdn_stream_t stream) {
  if (n < 0 || num_slots <= 0) return fail(GDN_ERR_INVALID_ARG, "n >= 0 and num_slots > 0 are required");
  if (n == 0) return GDN_OK;
  if (!write_pos || !slots) return fail(GDN_ERR_INVALID_ARG, "write_pos and slots must be set");
  cudaError_t e = gdn::launch_reset(write_pos, num_slots, slots, n, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_replayssm_reset_slots launch");
}

}  // extern "C"
