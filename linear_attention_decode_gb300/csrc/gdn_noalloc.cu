// gdn_replayssm_decode_advance for callers that cannot hand the library a
// workspace: some inference engines reserve all device memory for their own
// state and KV pools up front, some plugin hosts own every allocation, and some
// callers cannot afford cudaMalloc's implicit device-wide synchronisation.  The
// decode + advance kernel needs a little scratch memory (a completion counter),
// so this entry point takes it from a fixed array compiled into the library.
#include <mutex>
#include <string>

#include "gdn_kernels.h"

namespace {

// Scratch for the no-allocation entry point.  Every GPU that loads the library
// keeps these 256 bytes until the process exits; all calls on a device share
// them.  A call needs GDN_DECODE_ADVANCE_WORKSPACE_BYTES of it.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / 4];

// Device address of the scratch array, looked up once per device (in host code
// the array's name stands for a host-side shadow, not for device memory).
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint32_t *g_scratch_ptr[kMaxDevices] = {};

gdn_status_t noalloc_fail(gdn_status_t st, const std::string &msg) {
  gdn::set_last_error(msg.c_str());
  return st;
}

// The current device's scratch address, or null with *st set on failure.  The
// first call on a device looks the address up and clears the array (before
// any launch that uses it); later calls reuse both.
uint32_t *scratch_for_current_device(gdn_status_t *st) {
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
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      *st = noalloc_fail(GDN_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
      return nullptr;
    }
    e = cudaMemset(p, 0, kNoAllocScratchBytes);
    if (e != cudaSuccess) {
      *st = noalloc_fail(GDN_ERR_CUDA, std::string("clearing the scratch array: ") + cudaGetErrorString(e));
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<uint32_t *>(p);
  }
  return g_scratch_ptr[dev];
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
  uint32_t *scratch = scratch_for_current_device(&st);
  if (!scratch) return st;
  // The counter starts every launch at zero: it was cleared when the device's
  // scratch was set up, and every launch that runs to its end leaves it there.
  return gdn_replayssm_decode_advance(desc, cache, write_pos, force_flush, step, recon, flushed_out, scratch,
                                      dev_status, stream);
}

}  // extern "C"
