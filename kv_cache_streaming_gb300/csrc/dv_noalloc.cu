// Swap-out that allocates nothing: the staged swap path run through a
// built-in device buffer instead of one the caller provides.
//
// The paper has no counterpart to this entry point; it exists for callers
// that cannot allocate device memory themselves (see dv_swap_out_noalloc in
// dv.h for who they are and for the limits).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dv.h"
#include "dv_plan.h"

namespace {

// The built-in staging buffer.  Every GPU that loads libdv holds these bytes
// until the process exits.  Host code must not pass the name itself to a
// kernel (on the host it names a stand-in, not device memory): the device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_staging[DV_NOALLOC_STAGING_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the built-in buffer on the current device; resolved with
// that device current on the first call there.
dv_status staging_address(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess)
    return dv::set_error(DV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorName(err));
  if (dev < 0 || dev >= kMaxDevices)
    return dv::set_error(DV_ERR_UNSUPPORTED, "device %d is beyond the %d devices supported", dev,
                         kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_staging);
    if (err != cudaSuccess || !p) {
      cudaGetLastError();
      return dv::set_error(DV_ERR_CUDA, "cudaGetSymbolAddress of the built-in staging buffer: %s",
                           cudaGetErrorName(err));
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DV_OK;
}

}  // namespace

extern "C" dv_status dv_swap_out_noalloc(const dv_cache* cache, int32_t l0, int32_t l1,
                                         const int32_t* seq_start, const int32_t* seq_end,
                                         void* host_dst, size_t host_bytes, dv_stream stream) {
  size_t total = 0;
  dv_status st = dv_staging_bytes(cache, l0, l1, seq_start, seq_end, &total);
  if (st != DV_OK) return st;
  if (total == 0) return DV_OK;
  const size_t slab = total / (size_t)(l1 - l0);  // every layer of the ranges is the same size
  if (slab > (size_t)DV_NOALLOC_STAGING_BYTES)
    return dv::set_error(DV_ERR_BUFFER_TOO_SMALL,
                         "dv_swap_out_noalloc: one layer of these ranges needs %zu staging bytes, "
                         "more than the built-in %zu; use dv_swap_out with a staging buffer",
                         slab, (size_t)DV_NOALLOC_STAGING_BYTES);
  void* staging = nullptr;
  if ((st = staging_address(&staging)) != DV_OK) return st;
  return dv_swap_out(cache, l0, l1, seq_start, seq_end, host_dst, host_bytes, staging,
                     (size_t)DV_NOALLOC_STAGING_BYTES, stream);
}
