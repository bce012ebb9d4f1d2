// gdn_replayssm_decode_advance for callers that cannot hand the library a
// workspace: some inference engines reserve all device memory for their own
// state and KV pools up front, some plugin hosts own every allocation, and some
// callers cannot afford cudaMalloc's implicit device-wide synchronisation.  The
// decode + advance kernel needs a little scratch memory (a completion counter),
// so this entry point takes it from a fixed array compiled into the library.
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "gdn_kernels.h"

namespace {

// Scratch for the no-allocation entry point.  Every GPU that loads the library
// keeps these 256 bytes until the process exits; all calls in a context share
// them.  A call needs GDN_DECODE_ADVANCE_WORKSPACE_BYTES of it.  The explicit
// initialiser makes the array zero whenever the module is loaded into a
// context, so the counter starts at zero without any clearing call.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / 4] = {};

// Device address of the scratch array, looked up once per context (in host
// code the array's name stands for a host-side shadow, not for device memory).
// The entry is keyed by the context's unique id, so a context created after
// cudaDeviceReset (or a non-primary context) gets its own lookup.
constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  uint32_t *ptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

gdn_status_t noalloc_fail(gdn_status_t st, const std::string &msg) {
  gdn::set_last_error(msg.c_str());
  return st;
}

// Driver calls reached through the runtime's entry-point query (the library
// does not link libcuda directly).
struct CtxQueries {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxQueries &ctx_queries() {
  static const CtxQueries q = [] {
    CtxQueries r;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult res = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      r.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &res) == cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      r.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return r;
  }();
  return q;
}

// Unique id of the calling thread's current context, or 0 when there is none
// (or the driver calls are missing).
unsigned long long current_ctx_id() {
  const CtxQueries &q = ctx_queries();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!q.get_current || !q.get_id || q.get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      q.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The current context's scratch address, or null with *st set on failure.  The
// first call in a context looks the address up (cudaGetSymbolAddress, which
// also makes the device's primary context current if none is); later calls in
// the same context reuse it.  Nothing is cleared: the array is zero when the
// module loads, and every launch that uses it leaves it zero.
uint32_t *scratch_for_current_context(gdn_status_t *st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = noalloc_fail(GDN_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = noalloc_fail(GDN_ERR_UNSUPPORTED, "device ordinal beyond the 64 this entry point keeps scratch for");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  // A thread that has not used the runtime yet may have no current context:
  // then the symbol lookup below runs first and makes the primary one current.
  unsigned long long id = current_ctx_id();
  if (id != 0 && g_scratch[dev].ptr && g_scratch[dev].ctx_id == id) return g_scratch[dev].ptr;
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    *st = noalloc_fail(GDN_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    return nullptr;
  }
  if (id == 0 && (id = current_ctx_id()) == 0) {
    *st = noalloc_fail(GDN_ERR_CUDA, "no current CUDA context after the scratch lookup");
    return nullptr;
  }
  g_scratch[dev] = ScratchEntry{id, static_cast<uint32_t *>(p)};
  return g_scratch[dev].ptr;
}

}  // namespace

extern "C" {

gdn_status_t gdn_replayssm_decode_advance_noalloc(const gdn_layer_desc_t *desc, const gdn_layer_cache_t *cache,
                                                  int32_t *write_pos, const uint8_t *force_flush,
                                                  const gdn_step_t *step, int32_t recon, uint8_t *flushed_out,
                                                  uint32_t *dev_status, gdn_stream_t stream) {
  const size_t need = GDN_DECODE_ADVANCE_WORKSPACE_BYTES;
  if (need > kNoAllocScratchBytes)
    return noalloc_fail(GDN_ERR_UNSUPPORTED, "gdn_replayssm_decode_advance_noalloc: the call needs " +
                                                 std::to_string(need) + " bytes of scratch, the library holds " +
                                                 std::to_string(kNoAllocScratchBytes));
  gdn_status_t st = GDN_OK;
  uint32_t *scratch = scratch_for_current_context(&st);
  if (!scratch) return st;
  // The counter starts every launch at zero: the array is zero when the module
  // loads, and every launch leaves it there (a block that cannot run its items
  // still counts itself before it returns).
  return gdn_replayssm_decode_advance(desc, cache, write_pos, force_flush, step, recon, flushed_out, scratch,
                                      dev_status, stream);
}

gdn_status_t gdn_noalloc_scratch_peek(uint32_t *host_words, int32_t n) {
  if (!host_words || n < 1 || (size_t)n * 4 > kNoAllocScratchBytes)
    return noalloc_fail(GDN_ERR_INVALID_ARG, "gdn_noalloc_scratch_peek: 1 <= n <= 64 host words required");
  gdn_status_t st = GDN_OK;
  uint32_t *scratch = scratch_for_current_context(&st);
  if (!scratch) return st;
  const cudaError_t e = cudaMemcpy(host_words, scratch, (size_t)n * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return noalloc_fail(GDN_ERR_CUDA, std::string("gdn_noalloc_scratch_peek: ") + cudaGetErrorString(e));
  return GDN_OK;
}

}  // extern "C"
