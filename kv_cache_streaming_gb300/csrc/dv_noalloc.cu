// Swap-out that allocates nothing: the staged swap path run through a
// built-in device buffer instead of one the caller provides.
//
// The paper has no counterpart to this entry point; it exists for callers
// that cannot allocate device memory themselves (see dv_swap_out_noalloc in
// dv.h for who they are and for the limits).
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "dv_host.h"

namespace {

// The built-in staging buffer.  Every GPU that loads libdv holds these bytes
// until the process exits.  Host code must not pass the name itself to a
// kernel (on the host it names a stand-in, not device memory): the device
// address comes from cudaGetSymbolAddress, once per CUDA context.
static __device__ __align__(256) unsigned char g_noalloc_staging[DV_NOALLOC_STAGING_BYTES];

std::mutex g_mu;
std::vector<std::pair<unsigned long long, void*>> g_addr;  // (context id, address)

// Device address of the built-in buffer in the current CUDA context, looked
// up (cudaGetSymbolAddress, with the context current) on the first call in
// that context and kept per context: a device reset or a new context gets an
// id of its own and a fresh lookup, never a stale address.
dv_status staging_address(void** out) {
  unsigned long long id = 0;
  if (!dv::context_id(&id))
    return dv::fail(DV_ERR_CUDA, "dv_swap_out_noalloc: no current CUDA context");
  std::lock_guard<std::mutex> lock(g_mu);
  for (const auto& e : g_addr)
    if (e.first == id) {
      *out = e.second;
      return DV_OK;
    }
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_staging);
  if (err != cudaSuccess || !p) {
    cudaGetLastError();
    return dv::fail(DV_ERR_CUDA, "cudaGetSymbolAddress of the built-in staging buffer: %s",
                         cudaGetErrorName(err));
  }
  try {
    g_addr.emplace_back(id, p);
  } catch (...) {
    return dv::fail(DV_ERR_INVALID_ARG, "out of host memory for the buffer address");
  }
  *out = p;
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
    return dv::fail(DV_ERR_BUFFER_TOO_SMALL,
                         "dv_swap_out_noalloc: one layer of these ranges needs %zu staging bytes, "
                         "more than the built-in %zu; use dv_swap_out with a staging buffer",
                         slab, (size_t)DV_NOALLOC_STAGING_BYTES);
  void* staging = nullptr;
  if ((st = staging_address(&staging)) != DV_OK) return st;
  return dv_swap_out(cache, l0, l1, seq_start, seq_end, host_dst, host_bytes, staging,
                     (size_t)DV_NOALLOC_STAGING_BYTES, stream);
}
