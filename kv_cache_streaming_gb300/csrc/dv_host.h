// Internal to libdv: what the ABI translation units (dv_api.cu, dv_replica.cu,
// dv_sched.cu, dv_noalloc.cu) share: error reporting, argument validation,
// pointer resolution, NVTX ranges, and the handles that more than one of them
// opens (the streamer, the fetcher and the replica).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/dv.h"
#include "dv_plan.h"

#ifndef DV_NVTX
#define DV_NVTX 1  // NVTX ranges around every ABI call that enqueues work
#endif
#if DV_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace dv {

struct Record {
  int64_t step;
  int32_t l0, l1;
  size_t offset, bytes;
  size_t ranges;  // index of this record's ranges in dv_replica::ranges (2 * batch ints)
};

}  // namespace dv

struct dv_streamer {
  void* slot[2];
  size_t slot_bytes;
  cudaStream_t pack;
  cudaStream_t copy;
  cudaEvent_t packed[2];
  cudaEvent_t freed[2];
  bool used[2];
  int next;
};

struct dv_fetcher {
  void* slot[2];
  size_t slot_bytes;
  cudaStream_t copy;
  cudaStream_t unpack;
  cudaEvent_t copied[2];
  cudaEvent_t freed[2];
  bool used[2];
  int next;
};

struct dv_replica {
  uint8_t* arena;
  size_t arena_bytes;
  size_t used;
  int32_t batch;
  std::vector<dv::Record> records;
  std::vector<int32_t> ranges;
};

namespace dv {

// A named range on the calling thread's NVTX stack for the duration of one
// ABI call, so that a timeline taken with an NVTX-aware profiler shows each
// call and the launches and copies it enqueued; without a profiler attached
// the push and pop do nothing.
struct Trace {
  explicit Trace(const char* name) {
#if DV_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~Trace() {
#if DV_NVTX
    nvtxRangePop();
#endif
  }
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;
};

// Records a message for dv_last_error() on the calling thread; returns `st`.
dv_status fail(dv_status st, const char* fmt, ...);
// fail(DV_ERR_CUDA, ...) with the error's name and text after `what`.
dv_status cuda_fail(cudaError_t err, const char* what);

// The unique id of the calling thread's current CUDA context (made current
// by the runtime if none is); false if it cannot be had.  Keys per-context
// state: a context that is destroyed and made again gets a new id.
bool context_id(unsigned long long* id);

// Makes the current device's primary context current on a thread that has
// none yet (one that has made no CUDA runtime call).
void ensure_context();

// Validates geometry and ranges (no pointer is touched) and fills `p`.
dv_status plan_ranges(const dv_cache* c, int32_t l0, int32_t l1, const int32_t* s,
                      const int32_t* e, Plan* p);

// Device-visible address of `ptr` after checking its memory kind (device
// memory; pinned, mapped host memory too when `allow_host`, which sets
// *is_host); when the driver knows the allocation, also that
// [ptr, ptr + need) lies inside it.
dv_status resolve(const void* ptr, size_t need, bool allow_host, const char* what, void** dev,
                  bool* is_host = nullptr);

// Resolves the cache's K and V bases (device memory, extent of layers < l1).
dv_status resolve_cache(const dv_cache* c, Plan* p);

// The device-visible address of pinned, mapped host memory `ptr`.
dv_status check_host(const void* ptr, const char* what, void** dev);

// Packs the planned ranges (p's cache bases resolved) into the streamer's
// next slot on its pack stream, after that slot's previous copy, then copies
// the p.bytes of the slot to `dst` (host memory) on its copy stream.
cudaError_t stream_piece(dv_streamer* h, const Plan& p, void* dst);

// Copies `bytes` from `src` (host memory) into the fetcher's next slot on its
// copy stream, after that slot's previous unpack, then runs unpack(slot) on
// its unpack stream after the copy.
template <typename Unpack>
cudaError_t fetch_piece(dv_fetcher* h, const void* src, size_t bytes, Unpack&& unpack) {
  const int i = h->next;
  cudaError_t err;
  if (h->used[i] && (err = cudaStreamWaitEvent(h->copy, h->freed[i], 0)) != cudaSuccess)
    return err;
  if ((err = cudaMemcpyAsync(h->slot[i], src, bytes, cudaMemcpyDefault, h->copy)) != cudaSuccess)
    return err;
  if ((err = cudaEventRecord(h->copied[i], h->copy)) != cudaSuccess) return err;
  if ((err = cudaStreamWaitEvent(h->unpack, h->copied[i], 0)) != cudaSuccess) return err;
  if ((err = unpack(h->slot[i])) != cudaSuccess) return err;
  if ((err = cudaEventRecord(h->freed[i], h->unpack)) != cudaSuccess) return err;
  h->used[i] = true;
  h->next = i ^ 1;
  return cudaSuccess;
}

}  // namespace dv
