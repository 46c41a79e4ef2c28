// libdv C ABI: argument validation, planning, the swap paths, the layer
// streamer and the host-side replica log.  The copy work itself is in
// dv_kernels.cu; this file only validates, plans and enqueues.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/dv.h"
#include "dv_plan.h"

#ifndef DV_NVTX
#define DV_NVTX 1  // NVTX ranges around every ABI call that enqueues work
#endif
#if DV_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace {

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

thread_local std::string g_last_error;

dv_status fail(dv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dv_status cuda_fail(cudaError_t err, const char* what) {
  return fail(DV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuMemGetAddressRange, fetched through the runtime so that the library does
// not link the driver library directly (it then loads on machines without a
// GPU driver, where only symbol checks run).
using GetRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

GetRangeFn get_range_fn() {
  static GetRangeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<GetRangeFn>(f);
  }();
  return fn;
}

// A driver entry point fetched through the runtime (nullptr if unavailable).
void* driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    f = nullptr;
  }
  return f;
}

// A library-owned stream for the copies of a pipelined staged swap, one per
// CUDA context (created on first use there, with the context current; kept
// until the process exits).  nullptr when none can be had, or when none
// exists yet and `caller` is being captured into a graph (no stream is made
// during a capture): the swap then runs in order on the caller's stream.
cudaStream_t copy_stream(cudaStream_t caller) {
  static std::mutex mu;
  static std::vector<std::pair<unsigned long long, cudaStream_t>> streams;
  unsigned long long id = 0;
  if (!dv::context_id(&id)) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : streams)
    if (e.first == id) return e.second;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cap != cudaStreamCaptureStatusNone) return nullptr;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  try {
    streams.emplace_back(id, cs);
  } catch (...) {
    cudaStreamDestroy(cs);
    return nullptr;
  }
  return cs;
}

// Events a pipelined swap orders its two streams with, created per call and
// released when the call returns (a recorded event is freed once it
// completes).
struct Events {
  cudaEvent_t e[5] = {};
  int n = 0;
  cudaError_t make() {
    for (; n < 5; ++n) {
      const cudaError_t err = cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming);
      if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
  }
  ~Events() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
  }
};

// Validates geometry and ranges (no pointer is touched) and fills `p`.
dv_status plan_ranges(const dv_cache* c, int32_t l0, int32_t l1, const int32_t* s,
                      const int32_t* e, dv::Plan* p) {
  if (!c) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (c->num_layers <= 0 || c->batch <= 0 || c->num_heads <= 0 || c->head_dim <= 0 ||
      c->max_seq <= 0)
    return fail(DV_ERR_INVALID_ARG, "cache geometry must be positive (L=%d B=%d H=%d D=%d S=%d)",
                c->num_layers, c->batch, c->num_heads, c->head_dim, c->max_seq);
  if (c->elem_bytes != 1 && c->elem_bytes != 2 && c->elem_bytes != 4)
    return fail(DV_ERR_INVALID_ARG, "elem_bytes must be 1, 2 or 4 (got %d)", c->elem_bytes);
  if (c->batch > dv::kMaxBatch)
    return fail(DV_ERR_UNSUPPORTED, "batch %d exceeds DV_MAX_BATCH %d", c->batch, dv::kMaxBatch);
  const int32_t x = 16 / c->elem_bytes;
  if (c->head_dim % x != 0)
    return fail(DV_ERR_UNSUPPORTED, "head_dim %d is not a multiple of x = %d", c->head_dim, x);
  const int64_t dense = (int64_t)c->batch * c->num_heads * c->head_dim * c->max_seq;
  const int64_t stride = c->layer_stride_elems ? c->layer_stride_elems : dense;
  if (stride < dense)
    return fail(DV_ERR_INVALID_ARG, "layer_stride_elems %lld < batch*heads*head_dim*max_seq %lld",
                (long long)stride, (long long)dense);
  if ((stride * c->elem_bytes) % 16 != 0)
    return fail(DV_ERR_MISALIGNED, "layer stride of %lld bytes is not a multiple of 16",
                (long long)(stride * c->elem_bytes));
  if (l0 < 0 || l1 > c->num_layers || l0 > l1)
    return fail(DV_ERR_RANGE, "layer range [%d,%d) outside [0,%d)", l0, l1, c->num_layers);
  if (!s || !e) return fail(DV_ERR_INVALID_ARG, "seq_start / seq_end is NULL");
  p->L = c->num_layers;
  p->B = c->batch;
  p->H = c->num_heads;
  p->D = c->head_dim;
  p->S = c->max_seq;
  p->P = c->elem_bytes;
  p->C = c->head_dim / x;
  p->layer_chunks = stride * c->elem_bytes / 16;
  p->l0 = l0;
  p->l1 = l1;
  int64_t acc = 0;
  int32_t mx = 0, mn = 0, act = 0;
  for (int32_t b = 0; b < c->batch; ++b) {
    if (s[b] < 0 || s[b] > e[b] || e[b] > c->max_seq)
      return fail(DV_ERR_RANGE, "sequence %d range [%d,%d) outside [0,%d]", b, s[b], e[b],
                  c->max_seq);
    const int32_t len = e[b] - s[b];
    p->seq_start[b] = s[b];
    p->seq_len[b] = len;
    p->tok_pre[b] = (int32_t)acc;
    acc += len;
    if (len > mx) mx = len;
    if (len > 0 && (mn == 0 || len < mn)) mn = len;
    if (len > 0) ++act;
  }
  p->tok_pre[c->batch] = (int32_t)acc;
  p->tokens = acc;
  p->max_len = mx;
  p->min_len = mn;
  p->active = act;
  p->lkv_chunks = (int64_t)p->H * acc * p->C;
  if (p->lkv_chunks >= (int64_t)1 << 31)
    return fail(DV_ERR_UNSUPPORTED, "one (layer, K|V) slab of %lld chunks exceeds 2^31",
                (long long)p->lkv_chunks);
  p->bytes = 2 * (int64_t)(l1 - l0) * p->lkv_chunks * 16;
  p->k = c->k_base;
  p->v = c->v_base;
  p->host_side = false;
  return DV_OK;
}

// Makes the current device's primary context current on a thread that has
// none yet (one that has made no CUDA runtime call): the pointer attributes of
// pinned host memory, its device-visible address above all, are answered per
// context, and a thread without one gets none.
void ensure_context() {
  unsigned long long id = 0;
  dv::context_id(&id);
}

// Device-visible address of `ptr` after checking its memory kind; when the
// driver knows the allocation, also that [ptr, ptr + need) lies inside it.
dv_status resolve(const void* ptr, size_t need, bool allow_host, const char* what, void** dev,
                  bool* is_host = nullptr) {
  if (is_host) *is_host = false;
  if (!ptr) return fail(DV_ERR_INVALID_ARG, "%s is NULL", what);
  if (!aligned16(ptr)) return fail(DV_ERR_MISALIGNED, "%s %p is not 16-byte aligned", what, ptr);
  ensure_context();
  cudaPointerAttributes a;
  cudaError_t err = cudaPointerGetAttributes(&a, ptr);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fail(DV_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes failed (%s)", what,
                cudaGetErrorName(err));
  }
  int cur = -1;
  if ((err = cudaGetDevice(&cur)) != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != cur)
        return fail(DV_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", what,
                    a.device, cur);
      *dev = const_cast<void*>(ptr);
      break;
    case cudaMemoryTypeManaged:
      *dev = const_cast<void*>(ptr);
      break;
    case cudaMemoryTypeHost:
      if (!allow_host)
        return fail(DV_ERR_INVALID_ARG, "%s must be device memory (got pinned host memory)", what);
      if (!a.devicePointer)
        return fail(DV_ERR_INVALID_ARG, "%s: pinned host memory not mapped for the device", what);
      *dev = a.devicePointer;
      if (is_host) *is_host = true;
      break;
    default:
      return fail(DV_ERR_INVALID_ARG, "%s is not CUDA-registered memory (pageable host memory "
                  "must be pinned first)", what);
  }
  CUdeviceptr base = 0;
  size_t size = 0;
  const GetRangeFn range = get_range_fn();
  if (range && range(&base, &size, reinterpret_cast<CUdeviceptr>(*dev)) == CUDA_SUCCESS) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(*dev);
    if (p0 + need > (uintptr_t)base + size)
      return fail(DV_ERR_BUFFER_TOO_SMALL,
                  "%s: %zu bytes needed from %p but its allocation ends %zu bytes after it", what,
                  need, ptr, (size_t)((uintptr_t)base + size - p0));
  }
  return DV_OK;
}

// Resolves the cache's K and V bases (device memory, extent of layers < l1).
dv_status resolve_cache(const dv_cache* c, dv::Plan* p) {
  if (p->l1 == p->l0) return DV_OK;
  const int64_t dense = (int64_t)p->B * p->H * p->D * p->S;
  const size_t need = (size_t)(((int64_t)(p->l1 - 1) * p->layer_chunks * 16) + dense * p->P);
  void* k = nullptr;
  void* v = nullptr;
  dv_status st = resolve(p->k, need, false, "cache.k_base", &k);
  if (st != DV_OK) return st;
  st = resolve(p->v, need, false, "cache.v_base", &v);
  if (st != DV_OK) return st;
  p->k = k;
  p->v = v;
  return DV_OK;
}

dv_status check_variant(const dv::Plan& p, int32_t variant) {
  if (variant < dv::kAuto || variant > dv::kToken)
    return fail(DV_ERR_INVALID_ARG, "unknown variant %d", variant);
  if (variant == dv::kTile && !dv::tile_supported(p))
    return fail(DV_ERR_UNSUPPORTED, "tile kernel handles at most 64 chunks per token (got %d)",
                p.C);
  if (variant == dv::kToken && !dv::token_supported(p))
    return fail(DV_ERR_UNSUPPORTED, "token kernel needs every non-empty range to be equally long");
  return DV_OK;
}

dv_status do_pack(const dv_cache* c, int32_t l0, int32_t l1, const int32_t* s, const int32_t* e,
                  void* dst, size_t dst_bytes, cudaStream_t stream, int32_t variant) {
  dv::Plan p;
  dv_status st = plan_ranges(c, l0, l1, s, e, &p);
  if (st != DV_OK) return st;
  if ((st = check_variant(p, variant)) != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if (dst_bytes < (size_t)p.bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "pack needs %lld bytes, dst has %zu", (long long)p.bytes,
                dst_bytes);
  if ((st = resolve_cache(c, &p)) != DV_OK) return st;
  void* d = nullptr;
  if ((st = resolve(dst, (size_t)p.bytes, true, "dst", &d, &p.host_side)) != DV_OK) return st;
  const cudaError_t err = dv::launch_pack(p, d, stream, variant);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "pack launch");
}

dv_status do_unpack(const dv_cache* c, int32_t l0, int32_t l1, const int32_t* s,
                    const int32_t* e, const void* src, size_t src_bytes, cudaStream_t stream,
                    int32_t variant) {
  dv::Plan p;
  dv_status st = plan_ranges(c, l0, l1, s, e, &p);
  if (st != DV_OK) return st;
  if ((st = check_variant(p, variant)) != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if (src_bytes < (size_t)p.bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "unpack needs %lld bytes, src has %zu",
                (long long)p.bytes, src_bytes);
  if ((st = resolve_cache(c, &p)) != DV_OK) return st;
  void* d = nullptr;
  if ((st = resolve(src, (size_t)p.bytes, true, "src", &d, &p.host_side)) != DV_OK) return st;
  const cudaError_t err = dv::launch_unpack(p, d, stream, variant);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "unpack launch");
}

// Memory kind check for the host side of a swap (pinned host memory).
dv_status check_host(const void* ptr, const char* what, void** dev) {
  if (!ptr) return fail(DV_ERR_INVALID_ARG, "%s is NULL", what);
  if (!aligned16(ptr)) return fail(DV_ERR_MISALIGNED, "%s %p is not 16-byte aligned", what, ptr);
  ensure_context();
  cudaPointerAttributes a;
  const cudaError_t err = cudaPointerGetAttributes(&a, ptr);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fail(DV_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes failed", what);
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer)
    return fail(DV_ERR_INVALID_ARG, "%s must be pinned, mapped host memory", what);
  *dev = a.devicePointer;
  return DV_OK;
}

enum class Dir { kOut, kIn };

dv_status do_swap(Dir dir, const dv_cache* c, int32_t l0, int32_t l1, const int32_t* s,
                  const int32_t* e, void* host, size_t host_bytes, void* staging,
                  size_t staging_bytes, cudaStream_t stream) {
  dv::Plan p;
  dv_status st = plan_ranges(c, l0, l1, s, e, &p);
  if (st != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if (host_bytes < (size_t)p.bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "swap needs %lld host bytes, buffer has %zu",
                (long long)p.bytes, host_bytes);
  if ((st = resolve_cache(c, &p)) != DV_OK) return st;
  void* host_dev = nullptr;
  if ((st = check_host(host, dir == Dir::kOut ? "host_dst" : "host_src", &host_dev)) != DV_OK)
    return st;
  cudaError_t err;
  if (!staging) {  // fused: the kernel touches host memory directly
    p.host_side = true;
    err = dir == Dir::kOut ? dv::launch_pack(p, host_dev, stream, dv::kAuto)
                           : dv::launch_unpack(p, host_dev, stream, dv::kAuto);
    return err == cudaSuccess ? DV_OK : cuda_fail(err, "fused swap launch");
  }
  const int64_t slab = dv::layer_slab_bytes(p);
  if (staging_bytes < (size_t)slab)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "staging of %zu bytes holds less than one layer slab "
                "(%lld bytes)", staging_bytes, (long long)slab);
  const int64_t fit = (int64_t)(staging_bytes / (size_t)slab);
  const int32_t nl = l1 - l0;
  uint8_t* hp = static_cast<uint8_t*>(host);
  // Pipelined: the staging buffer in two halves, the copies on the library's
  // copy stream, so that the pack (unpack) of one group of layers overlaps
  // the copy of the other.  Needs room for a layer in each half.
  cudaStream_t cs = fit >= 2 && nl >= 2 ? copy_stream(stream) : nullptr;
  Events ev;
  if (cs && ev.make() != cudaSuccess) {
    cudaGetLastError();
    cs = nullptr;
  }
  if (cs) {
    const int32_t group = (int32_t)(fit / 2 < (int64_t)nl ? fit / 2 : (int64_t)nl);
    const size_t half = (size_t)group * (size_t)slab;
    void* stg = nullptr;
    if ((st = resolve(staging, 2 * half, false, "staging", &stg)) != DV_OK) return st;
    uint8_t* sp = static_cast<uint8_t*>(stg);
    cudaEvent_t start = ev.e[0], a[2] = {ev.e[1], ev.e[2]}, b[2] = {ev.e[3], ev.e[4]};
    if (dir == Dir::kIn) {  // copies into staging wait for the caller's earlier work
      if ((err = cudaEventRecord(start, stream)) != cudaSuccess ||
          (err = cudaStreamWaitEvent(cs, start, 0)) != cudaSuccess)
        return cuda_fail(err, "swap-in: order the copy stream");
    }
    int g = 0;
    for (int32_t la = l0; la < l1; la += group, ++g) {
      const int32_t lb = la + group < l1 ? la + group : l1;
      const int h = g & 1;
      dv::Plan q = p;
      dv::restrict_layers(q, la, lb);
      uint8_t* hchunk = hp + (int64_t)(la - l0) * slab;
      uint8_t* half_h = sp + h * half;
      if (dir == Dir::kOut) {  // a[h]: packed into half h;  b[h]: half h copied out
        if (g >= 2 && (err = cudaStreamWaitEvent(stream, b[h], 0)) != cudaSuccess)
          return cuda_fail(err, "swap-out: wait for a free half");
        if ((err = dv::launch_pack(q, half_h, stream, dv::kAuto)) != cudaSuccess)
          return cuda_fail(err, "swap-out pack launch");
        if ((err = cudaEventRecord(a[h], stream)) != cudaSuccess ||
            (err = cudaStreamWaitEvent(cs, a[h], 0)) != cudaSuccess)
          return cuda_fail(err, "swap-out: order the copy");
        if ((err = cudaMemcpyAsync(hchunk, half_h, (size_t)q.bytes, cudaMemcpyDeviceToHost,
                                   cs)) != cudaSuccess)
          return cuda_fail(err, "swap-out copy");
        if ((err = cudaEventRecord(b[h], cs)) != cudaSuccess)
          return cuda_fail(err, "swap-out: record the copy");
      } else {  // a[h]: half h copied in;  b[h]: half h unpacked
        if (g >= 2 && (err = cudaStreamWaitEvent(cs, b[h], 0)) != cudaSuccess)
          return cuda_fail(err, "swap-in: wait for a free half");
        if ((err = cudaMemcpyAsync(half_h, hchunk, (size_t)q.bytes, cudaMemcpyHostToDevice,
                                   cs)) != cudaSuccess)
          return cuda_fail(err, "swap-in copy");
        if ((err = cudaEventRecord(a[h], cs)) != cudaSuccess ||
            (err = cudaStreamWaitEvent(stream, a[h], 0)) != cudaSuccess)
          return cuda_fail(err, "swap-in: order the unpack");
        if ((err = dv::launch_unpack(q, half_h, stream, dv::kAuto)) != cudaSuccess)
          return cuda_fail(err, "swap-in unpack launch");
        if ((err = cudaEventRecord(b[h], stream)) != cudaSuccess)
          return cuda_fail(err, "swap-in: record the unpack");
      }
    }
    if (dir == Dir::kOut) {  // the swap is done, in the caller's stream, when both copies are
      for (int h = 0; h < 2 && h < g; ++h)
        if ((err = cudaStreamWaitEvent(stream, b[h], 0)) != cudaSuccess)
          return cuda_fail(err, "swap-out: join the copy stream");
    }
    return DV_OK;
  }
  const int32_t group = (int32_t)(fit < (int64_t)nl ? fit : (int64_t)nl);
  void* stg = nullptr;
  if ((st = resolve(staging, (size_t)(group * slab), false, "staging", &stg)) != DV_OK) return st;
  for (int32_t la = l0; la < l1; la += group) {
    const int32_t lb = la + group < l1 ? la + group : l1;
    dv::Plan q = p;
    dv::restrict_layers(q, la, lb);
    uint8_t* hchunk = hp + (int64_t)(la - l0) * slab;
    if (dir == Dir::kOut) {
      if ((err = dv::launch_pack(q, stg, stream, dv::kAuto)) != cudaSuccess)
        return cuda_fail(err, "swap-out pack launch");
      if ((err = cudaMemcpyAsync(hchunk, stg, (size_t)q.bytes, cudaMemcpyDeviceToHost, stream)) !=
          cudaSuccess)
        return cuda_fail(err, "swap-out copy");
    } else {
      if ((err = cudaMemcpyAsync(stg, hchunk, (size_t)q.bytes, cudaMemcpyHostToDevice, stream)) !=
          cudaSuccess)
        return cuda_fail(err, "swap-in copy");
      if ((err = dv::launch_unpack(q, stg, stream, dv::kAuto)) != cudaSuccess)
        return cuda_fail(err, "swap-in unpack launch");
    }
  }
  return DV_OK;
}

}  // namespace

namespace dv {
bool context_id(unsigned long long* id) {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static const GetCurrentFn get_current =
      reinterpret_cast<GetCurrentFn>(driver_fn("cuCtxGetCurrent"));
  static const GetIdFn get_id = reinterpret_cast<GetIdFn>(driver_fn("cuCtxGetId"));
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  if (!ctx) {  // setting the current device again makes its primary context current
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  }
  return get_id(ctx, id) == CUDA_SUCCESS;
}

dv_status set_error(dv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
}  // namespace dv

// ---- streamer ----------------------------------------------------------------

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

// ---- replica -----------------------------------------------------------------

namespace {
struct Record {
  int64_t step;
  int32_t l0, l1;
  size_t offset, bytes;
  size_t ranges;  // index of this record's ranges in dv_replica::ranges (2 * batch ints)
};
}  // namespace

struct dv_replica {
  uint8_t* arena;
  size_t arena_bytes;
  size_t used;
  int32_t batch;
  std::vector<Record> records;
  std::vector<int32_t> ranges;
};

namespace {

// One record of a log: its layers, its ranges (batch starts, then batch ends)
// and where its staging bytes lie relative to the log's first byte.
struct LogRec {
  int32_t l0, l1;
  const int32_t* ranges;
  size_t offset, bytes;
  int64_t step;
};

// The non-empty records of a log, validated against a cache, and how they go:
//  - alone: long ranges (the tile kernel's, normally a snapshot), or larger
//    than a piece, unpacked by themselves;
//  - run[i] > 1: records i .. i + run[i] - 1 are a run of one-token records
//    (run_length) at least dv::run_min_records long, unpacked by the run
//    kernel;
//  - the others, consecutive and disjoint, by the record kernel.
struct LogPlan {
  std::vector<LogRec> todo;
  std::vector<dv::RecordRanges> recs;
  std::vector<char> alone;
  std::vector<int> run;
  dv::Plan base;  // the cache: geometry, resolved K / V, layers [0, the last record's l1)
  size_t total = 0;

  // How many records from i on one record-kernel launch takes: consecutive
  // records neither alone nor the start of a run, whose writes are disjoint,
  // that fit the parameters and (piece > 0) piece bytes together.
  int batch_at(int i, size_t piece) const {
    int n = 0;
    while (i + n < (int)todo.size() && !alone[i + n] && (n == 0 || run[i + n] <= 1)) ++n;
    const int k = dv::records_per_launch(base, recs.data() + i, n);
    size_t bytes = 0;
    for (int j = 0; j < k; ++j) {
      if (piece && bytes + todo[i + j].bytes > piece) return j;
      bytes += todo[i + j].bytes;
    }
    return k;
  }

  // Records per run-kernel launch from a run starting at i (piece > 0: as many
  // as piece bytes hold).
  int run_piece(int i, size_t piece) const {
    int64_t k = dv::run_max_records(base, recs[i]);
    if (piece) {
      const int64_t fit = (int64_t)(piece / todo[i].bytes);
      if (fit < k) k = fit;
    }
    return k < 1 ? 1 : (int)k;
  }
};

// Validates every record of `all` against `cache` before anything is
// enqueued and plans the log.  piece > 0: the bytes one copy can carry; a
// record larger than that goes by itself in groups of layers, so one of its
// layer slabs must fit.
dv_status plan_log(const dv_cache* cache, const std::vector<LogRec>& all, size_t piece,
                   LogPlan* lp) {
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  const int32_t B = cache->batch;
  int32_t l_end = 0;
  try {
    dv::Plan q;
    for (const LogRec& rec : all) {
      const int32_t* s = rec.ranges;
      const dv_status st = plan_ranges(cache, rec.l0, rec.l1, s, s + B, &q);
      if (st != DV_OK) return st;
      if ((size_t)q.bytes != rec.bytes)
        return fail(DV_ERR_INVALID_ARG, "record of step %lld does not match this cache geometry",
                    (long long)rec.step);
      if (rec.bytes == 0) continue;
      const bool by_itself = dv::auto_kind(q) == dv::kTile || (piece && rec.bytes > piece);
      if (by_itself && piece && piece < (size_t)dv::layer_slab_bytes(q))
        return fail(DV_ERR_BUFFER_TOO_SMALL, "a staging piece of %zu bytes holds less than one "
                    "layer slab (%lld bytes) of the record of step %lld", piece,
                    (long long)dv::layer_slab_bytes(q), (long long)rec.step);
      lp->todo.push_back(rec);
      lp->recs.push_back(dv::RecordRanges{rec.l0, rec.l1, s, s + B});
      lp->alone.push_back(by_itself);
      if (rec.l1 > l_end) l_end = rec.l1;
      lp->total += rec.bytes;
    }
  } catch (...) {
    return fail(DV_ERR_INVALID_ARG, "out of host memory for the restore plan");
  }
  if (lp->todo.empty()) return DV_OK;
  std::vector<int32_t> zero((size_t)B, 0);
  dv_status st = plan_ranges(cache, 0, l_end, zero.data(), zero.data(), &lp->base);
  if (st != DV_OK) return st;
  if ((st = resolve_cache(cache, &lp->base)) != DV_OK) return st;
  // Runs of one-token records, greedily from the front, among the records
  // that do not go alone and lie back to back.
  const int n = (int)lp->todo.size();
  const int min_run = dv::run_min_records(lp->base);
  lp->run.assign((size_t)n, 1);
  for (int i = 0; i < n;) {
    if (lp->alone[i]) {
      ++i;
      continue;
    }
    int m = i + 1;
    while (m < n && !lp->alone[m] &&
           lp->todo[m].offset == lp->todo[m - 1].offset + lp->todo[m - 1].bytes)
      ++m;
    const int len = dv::run_length(lp->base, lp->recs.data() + i, m - i);
    if (len >= min_run) {
      lp->run[i] = len;
      i += len;
    } else {
      ++i;
    }
  }
  return DV_OK;
}

// The records of `r` with from <= step < upto (no upper limit when upto < 0),
// planned for `cache`.
dv_status plan_restore(const dv_replica* r, const dv_cache* cache, int64_t from, int64_t upto,
                       size_t piece, LogPlan* lp) {
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (cache->batch != r->batch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d differs from the replica's %d", cache->batch,
                r->batch);
  std::vector<LogRec> all;
  try {
    for (const Record& rec : r->records) {
      if (upto >= 0 && rec.step >= upto) break;
      if (rec.step < from) continue;
      all.push_back(LogRec{rec.l0, rec.l1, r->ranges.data() + rec.ranges, rec.offset, rec.bytes,
                           rec.step});
    }
  } catch (...) {
    return fail(DV_ERR_INVALID_ARG, "out of host memory for the restore plan");
  }
  return plan_log(cache, all, piece, lp);
}

// Enqueues the unpack of every planned record straight from `src` (the
// device-visible address of the log's first byte; host memory when
// `host_side`), on `stream`.
dv_status unpack_log_direct(const dv_cache* cache, LogPlan& lp, const uint8_t* src,
                            bool host_side, cudaStream_t stream) {
  lp.base.host_side = host_side;
  const int n = (int)lp.todo.size();
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n;) {
    const LogRec& first = lp.todo[i];
    if (lp.alone[i]) {
      dv::Plan q;
      const dv_status st = plan_ranges(cache, first.l0, first.l1, first.ranges,
                                       first.ranges + cache->batch, &q);
      if (st != DV_OK) return st;
      q.k = lp.base.k;
      q.v = lp.base.v;
      q.host_side = host_side;
      if ((err = dv::launch_unpack(q, src + first.offset, stream, dv::kAuto)) != cudaSuccess)
        return cuda_fail(err, "log unpack launch");
      ++i;
    } else if (lp.run[i] > 1) {
      const int len = lp.run[i];
      for (int j = 0; j < len;) {
        const int k = std::min(lp.run_piece(i + j, 0), len - j);
        if ((err = dv::launch_unpack_run(lp.base, lp.recs[i + j], k,
                                         src + lp.todo[i + j].offset, stream)) != cudaSuccess)
          return cuda_fail(err, "run unpack launch");
        j += k;
      }
      i += len;
    } else {
      const int k = lp.batch_at(i, 0);
      if ((err = dv::launch_unpack_records(lp.base, lp.recs.data() + i, k, src + first.offset,
                                           stream)) != cudaSuccess)
        return cuda_fail(err, "record unpack launch");
      i += k;
    }
  }
  return DV_OK;
}

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

}  // namespace

extern "C" {

int32_t dv_abi_version(void) { return DV_ABI_VERSION; }

const char* dv_status_string(dv_status st) {
  switch (st) {
    case DV_OK: return "DV_OK";
    case DV_ERR_INVALID_ARG: return "DV_ERR_INVALID_ARG";
    case DV_ERR_RANGE: return "DV_ERR_RANGE";
    case DV_ERR_BUFFER_TOO_SMALL: return "DV_ERR_BUFFER_TOO_SMALL";
    case DV_ERR_MISALIGNED: return "DV_ERR_MISALIGNED";
    case DV_ERR_CUDA: return "DV_ERR_CUDA";
    case DV_ERR_TIMEOUT: return "DV_ERR_TIMEOUT";
    case DV_ERR_UNSUPPORTED: return "DV_ERR_UNSUPPORTED";
  }
  return "DV_ERR_UNKNOWN";
}

const char* dv_last_error(void) { return g_last_error.c_str(); }

dv_status dv_debug_fault(uint64_t* fault) {
  if (!fault) return fail(DV_ERR_INVALID_ARG, "fault is NULL");
  *fault = 0;
  if (!dv::checked_build())
    return fail(DV_ERR_UNSUPPORTED, "this libdv was built without device-side bounds checks");
  const cudaError_t err = dv::read_fault(fault);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "reading the fault record");
}

dv_status dv_allocation_extent(const void* ptr, size_t* bytes_after) {
  if (!ptr || !bytes_after) return fail(DV_ERR_INVALID_ARG, "ptr / bytes_after is NULL");
  CUdeviceptr base = 0;
  size_t size = 0;
  const GetRangeFn range = get_range_fn();
  if (!range || range(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS)
    return fail(DV_ERR_UNSUPPORTED, "the driver does not know an allocation at %p", ptr);
  *bytes_after = (size_t)((uintptr_t)base + size - reinterpret_cast<uintptr_t>(ptr));
  return DV_OK;
}

dv_status dv_staging_bytes(const dv_cache* cache, int32_t l0, int32_t l1,
                           const int32_t* seq_start, const int32_t* seq_end, size_t* bytes) {
  if (!bytes) return fail(DV_ERR_INVALID_ARG, "bytes is NULL");
  dv::Plan p;
  p.bytes = 0;
  const dv_status st = plan_ranges(cache, l0, l1, seq_start, seq_end, &p);
  if (st != DV_OK) return st;
  *bytes = (size_t)p.bytes;
  return DV_OK;
}

dv_status dv_kv_pack(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                     const int32_t* seq_end, void* dst, size_t dst_bytes, dv_stream stream) {
  const Trace trace("dv_kv_pack");
  return do_pack(cache, l0, l1, seq_start, seq_end, dst, dst_bytes, stream, dv::kAuto);
}

dv_status dv_kv_unpack(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                       const int32_t* seq_end, const void* src, size_t src_bytes,
                       dv_stream stream) {
  const Trace trace("dv_kv_unpack");
  return do_unpack(cache, l0, l1, seq_start, seq_end, src, src_bytes, stream, dv::kAuto);
}

dv_status dv_kv_pack_variant(const dv_cache* cache, int32_t l0, int32_t l1,
                             const int32_t* seq_start, const int32_t* seq_end, void* dst,
                             size_t dst_bytes, dv_stream stream, int32_t variant) {
  const Trace trace("dv_kv_pack_variant");
  return do_pack(cache, l0, l1, seq_start, seq_end, dst, dst_bytes, stream, variant);
}

dv_status dv_kv_unpack_variant(const dv_cache* cache, int32_t l0, int32_t l1,
                               const int32_t* seq_start, const int32_t* seq_end,
                               const void* src, size_t src_bytes, dv_stream stream,
                               int32_t variant) {
  const Trace trace("dv_kv_unpack_variant");
  return do_unpack(cache, l0, l1, seq_start, seq_end, src, src_bytes, stream, variant);
}

dv_status dv_naive_gather(const dv_cache* cache, int32_t l0, int32_t l1,
                          const int32_t* seq_start, const int32_t* seq_end, void* dst,
                          size_t dst_bytes, dv_stream stream, int64_t* num_copies) {
  const Trace trace("dv_naive_gather");
  if (num_copies) *num_copies = 0;
  dv::Plan p;
  dv_status st = plan_ranges(cache, l0, l1, seq_start, seq_end, &p);
  if (st != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if (dst_bytes < (size_t)p.bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "gather needs %lld bytes, dst has %zu",
                (long long)p.bytes, dst_bytes);
  if ((st = resolve_cache(cache, &p)) != DV_OK) return st;
  void* d = nullptr;
  if ((st = resolve(dst, (size_t)p.bytes, true, "dst", &d)) != DV_OK) return st;
  const int64_t row = (int64_t)p.D * p.P;  // bytes of one token of one head
  const int64_t S16 = (int64_t)p.S * 16;
  const uint8_t* kb = static_cast<const uint8_t*>(p.k);
  const uint8_t* vb = static_cast<const uint8_t*>(p.v);
  uint8_t* out = static_cast<uint8_t*>(dst);
  int64_t off = 0, calls = 0;
  cudaError_t err = cudaSuccess;
  for (int64_t l = l0; l < l1 && err == cudaSuccess; ++l)
    for (int kv = 0; kv < 2 && err == cudaSuccess; ++kv)
      for (int64_t b = 0; b < p.B && err == cudaSuccess; ++b) {
        const int64_t len = p.seq_len[b];
        for (int64_t h = 0; h < p.H && len > 0 && err == cudaSuccess; ++h) {
          const int64_t bh = b * p.H + h;
          if (kv == 1) {  // one contiguous run
            const uint8_t* src = vb + (l * p.layer_chunks * 16) + (bh * p.S + p.seq_start[b]) * row;
            err = cudaMemcpyAsync(out + off, src, (size_t)(len * row), cudaMemcpyDefault, stream);
            ++calls;
          } else if (len < p.C) {  // per token: C chunks S*16 bytes apart -> C contiguous
            for (int64_t t = 0; t < len && err == cudaSuccess; ++t) {
              const uint8_t* src =
                  kb + (l * p.layer_chunks + bh * p.C * p.S + p.seq_start[b] + t) * 16;
              err = cudaMemcpy2DAsync(out + off + t * row, 16, src, (size_t)S16, 16, (size_t)p.C,
                                      cudaMemcpyDefault, stream);
              ++calls;
            }
          } else {  // per chunk row: len contiguous chunks -> every C-th chunk
            for (int64_t c = 0; c < p.C && err == cudaSuccess; ++c) {
              const uint8_t* src =
                  kb + (l * p.layer_chunks + (bh * p.C + c) * p.S + p.seq_start[b]) * 16;
              err = cudaMemcpy2DAsync(out + off + c * 16, (size_t)row, src, 16, 16, (size_t)len,
                                      cudaMemcpyDefault, stream);
              ++calls;
            }
          }
          off += len * row;
        }
      }
  if (num_copies) *num_copies = calls;
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "naive gather copy");
}

dv_status dv_swap_out(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                      const int32_t* seq_end, void* host_dst, size_t host_bytes, void* staging,
                      size_t staging_bytes, dv_stream stream) {
  const Trace trace("dv_swap_out");
  return do_swap(Dir::kOut, cache, l0, l1, seq_start, seq_end, host_dst, host_bytes, staging,
                 staging_bytes, stream);
}

dv_status dv_swap_in(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                     const int32_t* seq_end, const void* host_src, size_t host_bytes,
                     void* staging, size_t staging_bytes, dv_stream stream) {
  const Trace trace("dv_swap_in");
  return do_swap(Dir::kIn, cache, l0, l1, seq_start, seq_end, const_cast<void*>(host_src),
                 host_bytes, staging, staging_bytes, stream);
}

dv_status dv_streamer_create(dv_streamer** out, void* slot0, void* slot1, size_t slot_bytes,
                             dv_stream pack_stream, dv_stream copy_stream) {
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  void* d0 = nullptr;
  void* d1 = nullptr;
  dv_status st = resolve(slot0, slot_bytes, false, "slot0", &d0);
  if (st != DV_OK) return st;
  if ((st = resolve(slot1, slot_bytes, false, "slot1", &d1)) != DV_OK) return st;
  if (slot0 == slot1) return fail(DV_ERR_INVALID_ARG, "slot0 and slot1 must differ");
  dv_streamer* h = new (std::nothrow) dv_streamer();
  if (!h) return fail(DV_ERR_INVALID_ARG, "out of host memory for the streamer handle");
  h->slot[0] = d0;
  h->slot[1] = d1;
  h->slot_bytes = slot_bytes;
  h->pack = pack_stream;
  h->copy = copy_stream;
  h->used[0] = h->used[1] = false;
  h->next = 0;
  int made = 0;
  cudaError_t err = cudaSuccess;
  cudaEvent_t* evs[4] = {&h->packed[0], &h->packed[1], &h->freed[0], &h->freed[1]};
  for (; made < 4; ++made)
    if ((err = cudaEventCreateWithFlags(evs[made], cudaEventDisableTiming)) != cudaSuccess) break;
  if (made < 4) {
    for (int i = 0; i < made; ++i) cudaEventDestroy(*evs[i]);
    delete h;
    return cuda_fail(err, "cudaEventCreateWithFlags");
  }
  *out = h;
  return DV_OK;
}

dv_status dv_stream_layer(dv_streamer* h, const dv_cache* cache, int32_t layer,
                          const int32_t* seq_start, const int32_t* seq_end, void* host_dst,
                          size_t host_dst_bytes, int32_t l0) {
  const Trace trace("dv_stream_layer");
  if (!h) return fail(DV_ERR_INVALID_ARG, "streamer is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (l0 < 0 || layer < l0)
    return fail(DV_ERR_RANGE, "layer %d is before the streamed range start %d", layer, l0);
  dv::Plan p;
  dv_status st = plan_ranges(cache, layer, layer + 1, seq_start, seq_end, &p);
  if (st != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if ((size_t)p.bytes > h->slot_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "layer slab of %lld bytes exceeds slot of %zu",
                (long long)p.bytes, h->slot_bytes);
  const size_t off = (size_t)(layer - l0) * (size_t)p.bytes;
  if (!host_dst) return fail(DV_ERR_INVALID_ARG, "host_dst is NULL");
  if (off + (size_t)p.bytes > host_dst_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "layer %d lands at bytes [%zu,%zu) of a %zu-byte buffer",
                layer, off, off + (size_t)p.bytes, host_dst_bytes);
  if ((st = resolve_cache(cache, &p)) != DV_OK) return st;
  {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host_dst) != cudaSuccess ||
        a.type == cudaMemoryTypeUnregistered) {
      cudaGetLastError();
      return fail(DV_ERR_INVALID_ARG, "host_dst must be pinned host or device memory");
    }
  }
  const int i = h->next;
  cudaError_t err;
  if (h->used[i] && (err = cudaStreamWaitEvent(h->pack, h->freed[i], 0)) != cudaSuccess)
    return cuda_fail(err, "cudaStreamWaitEvent(slot free)");
  if ((err = dv::launch_pack(p, h->slot[i], h->pack, dv::kAuto)) != cudaSuccess)
    return cuda_fail(err, "stream_layer pack launch");
  if ((err = cudaEventRecord(h->packed[i], h->pack)) != cudaSuccess)
    return cuda_fail(err, "cudaEventRecord(packed)");
  if ((err = cudaStreamWaitEvent(h->copy, h->packed[i], 0)) != cudaSuccess)
    return cuda_fail(err, "cudaStreamWaitEvent(packed)");
  if ((err = cudaMemcpyAsync(static_cast<uint8_t*>(host_dst) + off, h->slot[i], (size_t)p.bytes,
                             cudaMemcpyDefault, h->copy)) != cudaSuccess)
    return cuda_fail(err, "stream_layer copy");
  if ((err = cudaEventRecord(h->freed[i], h->copy)) != cudaSuccess)
    return cuda_fail(err, "cudaEventRecord(freed)");
  h->used[i] = true;
  h->next = i ^ 1;
  return DV_OK;
}

dv_status dv_streamer_wait(dv_streamer* h) {
  if (!h) return fail(DV_ERR_INVALID_ARG, "streamer is NULL");
  for (int i = 0; i < 2; ++i) {
    if (!h->used[i]) continue;
    const cudaError_t err = cudaEventSynchronize(h->freed[i]);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventSynchronize");
  }
  return DV_OK;
}

void dv_streamer_destroy(dv_streamer* h) {
  if (!h) return;
  cudaEventDestroy(h->packed[0]);
  cudaEventDestroy(h->packed[1]);
  cudaEventDestroy(h->freed[0]);
  cudaEventDestroy(h->freed[1]);
  delete h;
}

dv_status dv_fetcher_create(dv_fetcher** out, void* slot0, void* slot1, size_t slot_bytes,
                            dv_stream copy_stream, dv_stream unpack_stream) {
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  void* d0 = nullptr;
  void* d1 = nullptr;
  dv_status st = resolve(slot0, slot_bytes, false, "slot0", &d0);
  if (st != DV_OK) return st;
  if ((st = resolve(slot1, slot_bytes, false, "slot1", &d1)) != DV_OK) return st;
  if (slot0 == slot1) return fail(DV_ERR_INVALID_ARG, "slot0 and slot1 must differ");
  dv_fetcher* h = new (std::nothrow) dv_fetcher();
  if (!h) return fail(DV_ERR_INVALID_ARG, "out of host memory for the fetcher handle");
  h->slot[0] = d0;
  h->slot[1] = d1;
  h->slot_bytes = slot_bytes;
  h->copy = copy_stream;
  h->unpack = unpack_stream;
  h->used[0] = h->used[1] = false;
  h->next = 0;
  int made = 0;
  cudaError_t err = cudaSuccess;
  cudaEvent_t* evs[4] = {&h->copied[0], &h->copied[1], &h->freed[0], &h->freed[1]};
  for (; made < 4; ++made)
    if ((err = cudaEventCreateWithFlags(evs[made], cudaEventDisableTiming)) != cudaSuccess) break;
  if (made < 4) {
    for (int i = 0; i < made; ++i) cudaEventDestroy(*evs[i]);
    delete h;
    return cuda_fail(err, "cudaEventCreateWithFlags");
  }
  *out = h;
  return DV_OK;
}

dv_status dv_fetch_layer(dv_fetcher* h, const dv_cache* cache, int32_t layer,
                         const int32_t* seq_start, const int32_t* seq_end, const void* host_src,
                         size_t host_src_bytes, int32_t l0) {
  const Trace trace("dv_fetch_layer");
  if (!h) return fail(DV_ERR_INVALID_ARG, "fetcher is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (l0 < 0 || layer < l0)
    return fail(DV_ERR_RANGE, "layer %d is before the streamed range start %d", layer, l0);
  dv::Plan p;
  dv_status st = plan_ranges(cache, layer, layer + 1, seq_start, seq_end, &p);
  if (st != DV_OK) return st;
  if (p.bytes == 0) return DV_OK;
  if ((size_t)p.bytes > h->slot_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "layer slab of %lld bytes exceeds slot of %zu",
                (long long)p.bytes, h->slot_bytes);
  const size_t off = (size_t)(layer - l0) * (size_t)p.bytes;
  if (!host_src) return fail(DV_ERR_INVALID_ARG, "host_src is NULL");
  if (off + (size_t)p.bytes > host_src_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "layer %d lies at bytes [%zu,%zu) of a %zu-byte buffer",
                layer, off, off + (size_t)p.bytes, host_src_bytes);
  if ((st = resolve_cache(cache, &p)) != DV_OK) return st;
  {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host_src) != cudaSuccess ||
        a.type == cudaMemoryTypeUnregistered) {
      cudaGetLastError();
      return fail(DV_ERR_INVALID_ARG, "host_src must be pinned host or device memory");
    }
  }
  const cudaError_t err =
      fetch_piece(h, static_cast<const uint8_t*>(host_src) + off, (size_t)p.bytes,
                  [&](void* slot) { return dv::launch_unpack(p, slot, h->unpack, dv::kAuto); });
  if (err != cudaSuccess) return cuda_fail(err, "fetch_layer");
  return DV_OK;
}

dv_status dv_fetcher_wait(dv_fetcher* h) {
  if (!h) return fail(DV_ERR_INVALID_ARG, "fetcher is NULL");
  for (int i = 0; i < 2; ++i) {
    if (!h->used[i]) continue;
    const cudaError_t err = cudaEventSynchronize(h->freed[i]);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventSynchronize");
  }
  return DV_OK;
}

void dv_fetcher_destroy(dv_fetcher* h) {
  if (!h) return;
  cudaEventDestroy(h->copied[0]);
  cudaEventDestroy(h->copied[1]);
  cudaEventDestroy(h->freed[0]);
  cudaEventDestroy(h->freed[1]);
  delete h;
}

dv_status dv_replica_create(dv_replica** out, void* host_arena, size_t arena_bytes,
                            int32_t batch) {
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (batch <= 0 || batch > dv::kMaxBatch)
    return fail(DV_ERR_INVALID_ARG, "batch %d outside [1, %d]", batch, dv::kMaxBatch);
  void* dev = nullptr;
  dv_status st = check_host(host_arena, "host_arena", &dev);
  if (st != DV_OK) return st;
  dv_replica* r = new (std::nothrow) dv_replica();
  if (!r) return fail(DV_ERR_INVALID_ARG, "out of host memory for the replica handle");
  r->arena = static_cast<uint8_t*>(host_arena);
  r->arena_bytes = arena_bytes;
  r->used = 0;
  r->batch = batch;
  *out = r;
  return DV_OK;
}

dv_status dv_replica_append(dv_replica* r, const dv_cache* cache, int32_t l0, int32_t l1,
                            const int32_t* seq_start, const int32_t* seq_end, int64_t step,
                            void* staging, size_t staging_bytes, dv_stream stream) {
  const Trace trace("dv_replica_append");
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (cache->batch != r->batch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d differs from the replica's %d", cache->batch,
                r->batch);
  if (!r->records.empty() && step < r->records.back().step)
    return fail(DV_ERR_INVALID_ARG, "step %lld is before the last record's %lld",
                (long long)step, (long long)r->records.back().step);
  size_t bytes = 0;
  dv_status st = dv_staging_bytes(cache, l0, l1, seq_start, seq_end, &bytes);
  if (st != DV_OK) return st;
  const size_t off = r->used;  // records are multiples of 16 bytes
  if (off + bytes > r->arena_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "replica arena full: %zu + %zu > %zu bytes", off, bytes,
                r->arena_bytes);
  if (bytes > 0) {
    st = dv_swap_out(cache, l0, l1, seq_start, seq_end, r->arena + off, bytes, staging,
                     staging_bytes, stream);
    if (st != DV_OK) return st;
  }
  Record rec{step, l0, l1, off, bytes, r->ranges.size()};
  try {
    r->ranges.insert(r->ranges.end(), seq_start, seq_start + r->batch);
    r->ranges.insert(r->ranges.end(), seq_end, seq_end + r->batch);
    r->records.push_back(rec);
  } catch (...) {
    r->ranges.resize(rec.ranges);
    return fail(DV_ERR_INVALID_ARG, "out of host memory for the replica index");
  }
  r->used = off + bytes;
  return DV_OK;
}

dv_status dv_replica_restore(const dv_replica* r, const dv_cache* cache, int64_t upto_step,
                             void* staging, size_t staging_bytes, dv_stream stream) {
  const Trace trace("dv_replica_restore");
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (cache->batch != r->batch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d differs from the replica's %d", cache->batch,
                r->batch);
  // Validate every record against this cache before enqueuing anything.
  for (const Record& rec : r->records) {
    if (upto_step >= 0 && rec.step >= upto_step) break;
    size_t bytes = 0;
    const int32_t* s = r->ranges.data() + rec.ranges;
    const dv_status st = dv_staging_bytes(cache, rec.l0, rec.l1, s, s + r->batch, &bytes);
    if (st != DV_OK) return st;
    if (bytes != rec.bytes)
      return fail(DV_ERR_INVALID_ARG, "record of step %lld does not match this cache geometry",
                  (long long)rec.step);
  }
  for (const Record& rec : r->records) {
    if (upto_step >= 0 && rec.step >= upto_step) break;
    if (rec.bytes == 0) continue;
    const int32_t* s = r->ranges.data() + rec.ranges;
    const dv_status st = dv_swap_in(cache, rec.l0, rec.l1, s, s + r->batch, r->arena + rec.offset,
                                    rec.bytes, staging, staging_bytes, stream);
    if (st != DV_OK) return st;
  }
  return DV_OK;
}

dv_status dv_replica_restore_batched(const dv_replica* r, const dv_cache* cache,
                                    int64_t upto_step, void* staging, size_t staging_bytes,
                                    dv_stream stream) {
  const Trace trace("dv_replica_restore_batched");
  LogPlan lp;
  dv_status st = plan_restore(r, cache, INT64_MIN, upto_step, staging ? staging_bytes : 0, &lp);
  if (st != DV_OK) return st;
  const int n = (int)lp.todo.size();
  if (n == 0) return DV_OK;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (!staging) {  // fused: every kernel reads the arena over the host link
    void* arena_dev = nullptr;
    if ((st = check_host(r->arena, "replica arena", &arena_dev)) != DV_OK) return st;
    return unpack_log_direct(cache, lp, static_cast<const uint8_t*>(arena_dev), true, cs);
  }
  void* stg = nullptr;
  const size_t need = lp.total < staging_bytes ? lp.total : staging_bytes;
  if ((st = resolve(staging, need, false, "staging", &stg)) != DV_OK) return st;
  uint8_t* sp = static_cast<uint8_t*>(stg);
  cudaError_t err;
  for (int i = 0; i < n;) {
    const LogRec& first = lp.todo[i];
    if (lp.alone[i]) {
      const int32_t* s = first.ranges;
      st = dv_swap_in(cache, first.l0, first.l1, s, s + r->batch, r->arena + first.offset,
                      first.bytes, staging, staging_bytes, stream);
      if (st != DV_OK) return st;
      ++i;
      continue;
    }
    if (lp.run[i] > 1) {  // a run, in pieces of as many records as staging holds
      const int len = lp.run[i];
      for (int j = 0; j < len;) {
        const int k = std::min(lp.run_piece(i + j, staging_bytes), len - j);
        const LogRec& f = lp.todo[i + j];
        if ((err = cudaMemcpyAsync(sp, r->arena + f.offset, (size_t)k * f.bytes,
                                   cudaMemcpyHostToDevice, cs)) != cudaSuccess)
          return cuda_fail(err, "restore copy");
        if ((err = dv::launch_unpack_run(lp.base, lp.recs[i + j], k, sp, cs)) != cudaSuccess)
          return cuda_fail(err, "run restore launch");
        j += k;
      }
      i += len;
      continue;
    }
    const int k = lp.batch_at(i, staging_bytes);
    size_t bytes = 0;
    for (int j = 0; j < k; ++j) bytes += lp.todo[i + j].bytes;
    if ((err = cudaMemcpyAsync(sp, r->arena + first.offset, bytes, cudaMemcpyHostToDevice, cs)) !=
        cudaSuccess)
      return cuda_fail(err, "restore copy");
    if ((err = dv::launch_unpack_records(lp.base, lp.recs.data() + i, k, sp, cs)) != cudaSuccess)
      return cuda_fail(err, "batched restore launch");
    i += k;
  }
  return DV_OK;
}

dv_status dv_replica_restore_fetched(const dv_replica* r, const dv_cache* cache,
                                    int64_t upto_step, dv_fetcher* h) {
  const Trace trace("dv_replica_restore_fetched");
  return dv_replica_restore_fetched_steps(r, cache, INT64_MIN, upto_step, h);
}

dv_status dv_replica_restore_fetched_steps(const dv_replica* r, const dv_cache* cache,
                                          int64_t from_step, int64_t upto_step, dv_fetcher* h) {
  const Trace trace("dv_replica_restore_fetched_steps");
  if (!h) return fail(DV_ERR_INVALID_ARG, "fetcher is NULL");
  LogPlan lp;
  dv_status st = plan_restore(r, cache, from_step, upto_step, h->slot_bytes, &lp);
  if (st != DV_OK) return st;
  const int n = (int)lp.todo.size();
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n;) {
    const LogRec& first = lp.todo[i];
    if (lp.alone[i]) {
      // Whole layers at a time, as many as a slot holds.
      const int32_t* s = first.ranges;
      dv::Plan q;
      if ((st = plan_ranges(cache, first.l0, first.l1, s, s + r->batch, &q)) != DV_OK) return st;
      q.k = lp.base.k;
      q.v = lp.base.v;
      const int64_t slab = dv::layer_slab_bytes(q);
      const int64_t fit = (int64_t)(h->slot_bytes / (size_t)slab);
      const int32_t group = (int32_t)(fit < (int64_t)(q.l1 - q.l0) ? fit : (int64_t)(q.l1 - q.l0));
      for (int32_t la = first.l0; la < first.l1; la += group) {
        const int32_t lb = la + group < first.l1 ? la + group : first.l1;
        dv::Plan g = q;
        dv::restrict_layers(g, la, lb);
        const uint8_t* src = r->arena + first.offset + (size_t)(la - first.l0) * (size_t)slab;
        err = fetch_piece(h, src, (size_t)g.bytes, [&](void* slot) {
          return dv::launch_unpack(g, slot, h->unpack, dv::kAuto);
        });
        if (err != cudaSuccess) return cuda_fail(err, "fetched restore (layers)");
      }
      ++i;
      continue;
    }
    if (lp.run[i] > 1) {  // a run, in pieces of as many records as a slot holds
      const int len = lp.run[i];
      for (int j = 0; j < len;) {
        const int k = std::min(lp.run_piece(i + j, h->slot_bytes), len - j);
        const LogRec& f = lp.todo[i + j];
        const dv::RecordRanges& fr = lp.recs[i + j];
        err = fetch_piece(h, r->arena + f.offset, (size_t)k * f.bytes, [&](void* slot) {
          return dv::launch_unpack_run(lp.base, fr, k, slot, h->unpack);
        });
        if (err != cudaSuccess) return cuda_fail(err, "fetched restore (run)");
        j += k;
      }
      i += len;
      continue;
    }
    const int k = lp.batch_at(i, h->slot_bytes);
    size_t bytes = 0;
    for (int j = 0; j < k; ++j) bytes += lp.todo[i + j].bytes;
    err = fetch_piece(h, r->arena + first.offset, bytes, [&](void* slot) {
      return dv::launch_unpack_records(lp.base, lp.recs.data() + i, k, slot, h->unpack);
    });
    if (err != cudaSuccess) return cuda_fail(err, "fetched restore (records)");
    i += k;
  }
  return DV_OK;
}

dv_status dv_kv_unpack_records(const dv_cache* cache, int32_t num_records,
                               const int32_t* layers, const int32_t* ranges, const void* src,
                               size_t src_bytes, dv_stream stream) {
  const Trace trace("dv_kv_unpack_records");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (num_records < 0) return fail(DV_ERR_INVALID_ARG, "num_records %d < 0", num_records);
  if (num_records > 0 && (!layers || !ranges))
    return fail(DV_ERR_INVALID_ARG, "layers / ranges is NULL");
  if (cache->batch <= 0 || cache->batch > dv::kMaxBatch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d outside [1, %d]", cache->batch,
                dv::kMaxBatch);
  std::vector<LogRec> all;
  size_t off = 0;
  try {
    all.reserve((size_t)num_records);
    for (int32_t i = 0; i < num_records; ++i) {
      const int32_t* rg = ranges + (size_t)i * 2 * cache->batch;
      size_t bytes = 0;
      const dv_status st = dv_staging_bytes(cache, layers[2 * i], layers[2 * i + 1], rg,
                                            rg + cache->batch, &bytes);
      if (st != DV_OK) return st;
      all.push_back(LogRec{layers[2 * i], layers[2 * i + 1], rg, off, bytes, (int64_t)i});
      off += bytes;
    }
  } catch (...) {
    return fail(DV_ERR_INVALID_ARG, "out of host memory for the record plan");
  }
  if (off == 0) return DV_OK;
  if (src_bytes < off)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "the records need %zu bytes, src has %zu", off,
                src_bytes);
  LogPlan lp;
  dv_status st = plan_log(cache, all, 0, &lp);
  if (st != DV_OK) return st;
  void* d = nullptr;
  bool host_side = false;
  if ((st = resolve(src, off, true, "src", &d, &host_side)) != DV_OK) return st;
  return unpack_log_direct(cache, lp, static_cast<const uint8_t*>(d), host_side,
                           static_cast<cudaStream_t>(stream));
}

dv_status dv_replica_truncate(dv_replica* r, int64_t step) {
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  size_t keep = 0;
  while (keep < r->records.size() && r->records[keep].step < step) ++keep;
  if (keep < r->records.size()) {
    r->used = r->records[keep].offset;
    r->ranges.resize(r->records[keep].ranges);
    r->records.resize(keep);
  }
  return DV_OK;
}

dv_status dv_replica_info(const dv_replica* r, int64_t* num_records, size_t* bytes_used) {
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (num_records) *num_records = (int64_t)r->records.size();
  if (bytes_used) *bytes_used = r->used;
  return DV_OK;
}

void dv_replica_destroy(dv_replica* r) { delete r; }

// ---- microbatch swapping through two device caches (Fig 9) -------------------

struct dv_swapper {
  dv_cache slot[2];
  dv_fetcher* fetcher;
  cudaStream_t compute;
  cudaStream_t swap;
  const dv_replica* holds[2];  // microbatch swapped in to each cache (or on its way)
  const dv_replica* cur;       // the acquired microbatch, NULL between steps
  int current;                 // its cache
  int last;                    // the cache of the last acquire, -1 before the first
  cudaEvent_t ready[2];        // after a cache's swap-in (fetcher's unpack stream)
  cudaEvent_t computed[2];     // after a step's compute (compute stream)
  cudaEvent_t freed[2];        // after a cache's last swap-out (swap stream)
  bool ready_set[2], freed_set[2];
};

namespace {

// Swaps `mb` in to cache i on the fetcher's streams, after that cache's
// previous step and swap-out.
dv_status swap_in_slot(dv_swapper* sw, int i, const dv_replica* mb) {
  dv_fetcher* f = sw->fetcher;
  cudaError_t err;
  if (sw->freed_set[i]) {
    if ((err = cudaStreamWaitEvent(f->copy, sw->freed[i], 0)) != cudaSuccess ||
        (err = cudaStreamWaitEvent(f->unpack, sw->freed[i], 0)) != cudaSuccess)
      return cuda_fail(err, "swapper: wait for the cache's swap-out");
  }
  const dv_status st = dv_replica_restore_fetched(mb, &sw->slot[i], -1, f);
  if (st != DV_OK) return st;
  if ((err = cudaEventRecord(sw->ready[i], f->unpack)) != cudaSuccess)
    return cuda_fail(err, "swapper: record the swap-in");
  sw->ready_set[i] = true;
  sw->holds[i] = mb;
  return DV_OK;
}

bool same_geometry(const dv_cache& a, const dv_cache& b) {
  return a.num_layers == b.num_layers && a.batch == b.batch && a.num_heads == b.num_heads &&
         a.head_dim == b.head_dim && a.max_seq == b.max_seq && a.elem_bytes == b.elem_bytes &&
         a.layer_stride_elems == b.layer_stride_elems;
}

}  // namespace

dv_status dv_swapper_create(dv_swapper** out, const dv_cache* slot0, const dv_cache* slot1,
                            dv_fetcher* fetcher, dv_stream compute_stream, dv_stream swap_stream) {
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!slot0 || !slot1 || !fetcher)
    return fail(DV_ERR_INVALID_ARG, "slot0 / slot1 / fetcher is NULL");
  if (!same_geometry(*slot0, *slot1))
    return fail(DV_ERR_INVALID_ARG, "the two caches must have the same geometry");
  if (slot0->k_base == slot1->k_base || slot0->v_base == slot1->v_base)
    return fail(DV_ERR_INVALID_ARG, "the two caches must not share memory");
  std::vector<int32_t> zero((size_t)(slot0->batch > 0 ? slot0->batch : 1), 0);
  for (const dv_cache* c : {slot0, slot1}) {
    dv::Plan p;
    dv_status st = plan_ranges(c, 0, c->num_layers, zero.data(), zero.data(), &p);
    if (st != DV_OK) return st;
    if ((st = resolve_cache(c, &p)) != DV_OK) return st;
  }
  dv_swapper* sw = new (std::nothrow) dv_swapper();
  if (!sw) return fail(DV_ERR_INVALID_ARG, "out of host memory for the swapper handle");
  sw->slot[0] = *slot0;
  sw->slot[1] = *slot1;
  sw->fetcher = fetcher;
  sw->compute = compute_stream;
  sw->swap = swap_stream;
  sw->holds[0] = sw->holds[1] = nullptr;
  sw->cur = nullptr;
  sw->current = -1;
  sw->last = -1;
  sw->ready_set[0] = sw->ready_set[1] = sw->freed_set[0] = sw->freed_set[1] = false;
  cudaEvent_t* evs[6] = {&sw->ready[0], &sw->ready[1], &sw->computed[0], &sw->computed[1],
                         &sw->freed[0], &sw->freed[1]};
  int made = 0;
  cudaError_t err = cudaSuccess;
  for (; made < 6; ++made)
    if ((err = cudaEventCreateWithFlags(evs[made], cudaEventDisableTiming)) != cudaSuccess) break;
  if (made < 6) {
    for (int i = 0; i < made; ++i) cudaEventDestroy(*evs[i]);
    delete sw;
    return cuda_fail(err, "cudaEventCreateWithFlags");
  }
  *out = sw;
  return DV_OK;
}

dv_status dv_swapper_acquire(dv_swapper* sw, const dv_replica* mb, int32_t* slot) {
  const Trace trace("dv_swapper_acquire");
  if (!sw || !mb || !slot) return fail(DV_ERR_INVALID_ARG, "swapper / microbatch / slot is NULL");
  if (sw->cur) return fail(DV_ERR_INVALID_ARG, "the current microbatch has not been released");
  if (mb->batch != sw->slot[0].batch)
    return fail(DV_ERR_INVALID_ARG, "microbatch batch %d differs from the caches' %d", mb->batch,
                sw->slot[0].batch);
  int i = sw->holds[0] == mb ? 0 : sw->holds[1] == mb ? 1 : -1;
  if (i < 0) {  // not swapped in: now, into the cache the last step did not use
    i = sw->last < 0 ? 0 : 1 - sw->last;
    const dv_status st = swap_in_slot(sw, i, mb);
    if (st != DV_OK) return st;
  }
  if (sw->ready_set[i]) {
    const cudaError_t err = cudaStreamWaitEvent(sw->compute, sw->ready[i], 0);
    if (err != cudaSuccess) return cuda_fail(err, "swapper: wait for the swap-in");
  }
  sw->cur = mb;
  sw->current = i;
  sw->last = i;
  *slot = i;
  return DV_OK;
}

dv_status dv_swapper_prefetch(dv_swapper* sw, const dv_replica* mb) {
  const Trace trace("dv_swapper_prefetch");
  if (!sw || !mb) return fail(DV_ERR_INVALID_ARG, "swapper / microbatch is NULL");
  if (mb->batch != sw->slot[0].batch)
    return fail(DV_ERR_INVALID_ARG, "microbatch batch %d differs from the caches' %d", mb->batch,
                sw->slot[0].batch);
  if (sw->holds[0] == mb || sw->holds[1] == mb) return DV_OK;  // already there
  const int j = sw->last < 0 ? 0 : 1 - sw->last;
  return swap_in_slot(sw, j, mb);
}

dv_status dv_swapper_release(dv_swapper* sw, dv_replica* mb, int32_t l0, int32_t l1,
                             const int32_t* seq_start, const int32_t* seq_end, int64_t step) {
  const Trace trace("dv_swapper_release");
  if (!sw || !mb) return fail(DV_ERR_INVALID_ARG, "swapper / microbatch is NULL");
  if (sw->cur != mb) return fail(DV_ERR_INVALID_ARG, "this microbatch is not the acquired one");
  const int i = sw->current;
  size_t bytes = 0;
  dv_status st = dv_staging_bytes(&sw->slot[i], l0, l1, seq_start, seq_end, &bytes);
  if (st != DV_OK) return st;
  if (!mb->records.empty() && step < mb->records.back().step)
    return fail(DV_ERR_INVALID_ARG, "step %lld is before the last record's %lld",
                (long long)step, (long long)mb->records.back().step);
  if (mb->used + bytes > mb->arena_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "replica arena full: %zu + %zu > %zu bytes", mb->used,
                bytes, mb->arena_bytes);
  cudaError_t err;
  if ((err = cudaEventRecord(sw->computed[i], sw->compute)) != cudaSuccess ||
      (err = cudaStreamWaitEvent(sw->swap, sw->computed[i], 0)) != cudaSuccess)
    return cuda_fail(err, "swapper: order the swap-out after the step");
  if ((st = dv_replica_append(mb, &sw->slot[i], l0, l1, seq_start, seq_end, step, nullptr, 0,
                              sw->swap)) != DV_OK)
    return st;
  if ((err = cudaEventRecord(sw->freed[i], sw->swap)) != cudaSuccess)
    return cuda_fail(err, "swapper: record the swap-out");
  sw->freed_set[i] = true;
  sw->cur = nullptr;
  return DV_OK;
}

dv_status dv_swapper_wait(dv_swapper* sw) {
  if (!sw) return fail(DV_ERR_INVALID_ARG, "swapper is NULL");
  for (int i = 0; i < 2; ++i) {
    cudaError_t err = cudaSuccess;
    if (sw->ready_set[i] && (err = cudaEventSynchronize(sw->ready[i])) != cudaSuccess)
      return cuda_fail(err, "cudaEventSynchronize");
    if (sw->freed_set[i] && (err = cudaEventSynchronize(sw->freed[i])) != cudaSuccess)
      return cuda_fail(err, "cudaEventSynchronize");
  }
  return DV_OK;
}

void dv_swapper_destroy(dv_swapper* sw) {
  if (!sw) return;
  for (cudaEvent_t e : {sw->ready[0], sw->ready[1], sw->computed[0], sw->computed[1],
                        sw->freed[0], sw->freed[1]})
    cudaEventDestroy(e);
  delete sw;
}

// ---- decode deltas streamed beside the compute (Fig 7c) ------------------------

struct dv_delta_streamer {
  dv_replica* replica;
  cudaStream_t compute;
  cudaStream_t side;
  void* staging;
  size_t staging_bytes;
  cudaEvent_t written;   // after a step's writes (compute stream)
  cudaEvent_t streamed;  // after the last append (side stream)
  bool any;
};

dv_status dv_delta_streamer_create(dv_delta_streamer** out, dv_replica* replica,
                                   dv_stream compute_stream, dv_stream side_stream,
                                   void* staging, size_t staging_bytes) {
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!replica) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (compute_stream == side_stream)
    return fail(DV_ERR_INVALID_ARG, "the side stream must differ from the compute stream");
  if (staging) {
    void* d = nullptr;
    const dv_status st = resolve(staging, staging_bytes, false, "staging", &d);
    if (st != DV_OK) return st;
  }
  dv_delta_streamer* ds = new (std::nothrow) dv_delta_streamer();
  if (!ds) return fail(DV_ERR_INVALID_ARG, "out of host memory for the delta streamer handle");
  ds->replica = replica;
  ds->compute = compute_stream;
  ds->side = side_stream;
  ds->staging = staging;
  ds->staging_bytes = staging ? staging_bytes : 0;
  ds->any = false;
  cudaError_t err = cudaEventCreateWithFlags(&ds->written, cudaEventDisableTiming);
  if (err == cudaSuccess) {
    err = cudaEventCreateWithFlags(&ds->streamed, cudaEventDisableTiming);
    if (err != cudaSuccess) cudaEventDestroy(ds->written);
  }
  if (err != cudaSuccess) {
    delete ds;
    return cuda_fail(err, "cudaEventCreateWithFlags");
  }
  *out = ds;
  return DV_OK;
}

dv_status dv_delta_stream(dv_delta_streamer* ds, const dv_cache* cache, int32_t l0, int32_t l1,
                          const int32_t* seq_start, const int32_t* seq_end, int64_t step) {
  const Trace trace("dv_delta_stream");
  if (!ds) return fail(DV_ERR_INVALID_ARG, "delta streamer is NULL");
  dv_replica* r = ds->replica;
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (cache->batch != r->batch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d differs from the replica's %d", cache->batch,
                r->batch);
  size_t bytes = 0;
  dv_status st = dv_staging_bytes(cache, l0, l1, seq_start, seq_end, &bytes);
  if (st != DV_OK) return st;
  if (!r->records.empty() && step < r->records.back().step)
    return fail(DV_ERR_INVALID_ARG, "step %lld is before the last record's %lld",
                (long long)step, (long long)r->records.back().step);
  if (r->used + bytes > r->arena_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "replica arena full: %zu + %zu > %zu bytes", r->used,
                bytes, r->arena_bytes);
  if (ds->staging && bytes > 0) {
    dv::Plan p;
    if ((st = plan_ranges(cache, l0, l1, seq_start, seq_end, &p)) != DV_OK) return st;
    if ((size_t)dv::layer_slab_bytes(p) > ds->staging_bytes)
      return fail(DV_ERR_BUFFER_TOO_SMALL, "staging of %zu bytes holds less than one layer slab "
                  "(%lld bytes)", ds->staging_bytes, (long long)dv::layer_slab_bytes(p));
  }
  cudaError_t err;
  if ((err = cudaEventRecord(ds->written, ds->compute)) != cudaSuccess ||
      (err = cudaStreamWaitEvent(ds->side, ds->written, 0)) != cudaSuccess)
    return cuda_fail(err, "delta stream: order the append after the step");
  if ((st = dv_replica_append(r, cache, l0, l1, seq_start, seq_end, step, ds->staging,
                              ds->staging_bytes, ds->side)) != DV_OK)
    return st;
  if ((err = cudaEventRecord(ds->streamed, ds->side)) != cudaSuccess)
    return cuda_fail(err, "delta stream: record the append");
  ds->any = true;
  return DV_OK;
}

dv_status dv_delta_streamer_join(dv_delta_streamer* ds) {
  if (!ds) return fail(DV_ERR_INVALID_ARG, "delta streamer is NULL");
  if (!ds->any) return DV_OK;
  const cudaError_t err = cudaStreamWaitEvent(ds->compute, ds->streamed, 0);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "delta stream: join");
}

dv_status dv_delta_streamer_wait(dv_delta_streamer* ds) {
  if (!ds) return fail(DV_ERR_INVALID_ARG, "delta streamer is NULL");
  if (!ds->any) return DV_OK;
  const cudaError_t err = cudaEventSynchronize(ds->streamed);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "cudaEventSynchronize");
}

void dv_delta_streamer_destroy(dv_delta_streamer* ds) {
  if (!ds) return;
  cudaEventDestroy(ds->written);
  cudaEventDestroy(ds->streamed);
  delete ds;
}

}  // extern "C"
