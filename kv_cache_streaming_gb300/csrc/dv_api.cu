// libdv C ABI, part 1: status and errors, argument validation and pointer
// resolution (shared with the other parts through dv_host.h), pack and unpack,
// the swap paths, and the layer streamer and fetcher.  The copy work itself is
// in dv_kernels.cu; this file only validates, plans and enqueues.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "dv_host.h"

namespace {

thread_local std::string g_last_error;

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

}  // namespace

namespace dv {

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

// Makes the current device's primary context current on a thread that has
// none yet (one that has made no CUDA runtime call): the pointer attributes of
// pinned host memory, its device-visible address above all, are answered per
// context, and a thread without one gets none.
void ensure_context() {
  unsigned long long id = 0;
  dv::context_id(&id);
}

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

// Device-visible address of `ptr` after checking its memory kind; when the
// driver knows the allocation, also that [ptr, ptr + need) lies inside it.
dv_status resolve(const void* ptr, size_t need, bool allow_host, const char* what, void** dev,
                  bool* is_host) {
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

}  // namespace dv

using dv::check_host;
using dv::cuda_fail;
using dv::fail;
using dv::fetch_piece;
using dv::plan_ranges;
using dv::resolve;
using dv::resolve_cache;
using dv::Trace;

namespace {

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

cudaError_t stream_piece(dv_streamer* h, const Plan& p, void* dst) {
  const int i = h->next;
  cudaError_t err;
  if (h->used[i] && (err = cudaStreamWaitEvent(h->pack, h->freed[i], 0)) != cudaSuccess)
    return err;
  if ((err = launch_pack(p, h->slot[i], h->pack, kAuto)) != cudaSuccess) return err;
  if ((err = cudaEventRecord(h->packed[i], h->pack)) != cudaSuccess) return err;
  if ((err = cudaStreamWaitEvent(h->copy, h->packed[i], 0)) != cudaSuccess) return err;
  if ((err = cudaMemcpyAsync(dst, h->slot[i], (size_t)p.bytes, cudaMemcpyDefault, h->copy)) !=
      cudaSuccess)
    return err;
  if ((err = cudaEventRecord(h->freed[i], h->copy)) != cudaSuccess) return err;
  h->used[i] = true;
  h->next = i ^ 1;
  return cudaSuccess;
}

}  // namespace dv

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
    dv::ensure_context();
    if (cudaPointerGetAttributes(&a, host_dst) != cudaSuccess ||
        a.type == cudaMemoryTypeUnregistered) {
      cudaGetLastError();
      return fail(DV_ERR_INVALID_ARG, "host_dst must be pinned host or device memory");
    }
  }
  const cudaError_t err = dv::stream_piece(h, p, static_cast<uint8_t*>(host_dst) + off);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "stream_layer");
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
    dv::ensure_context();
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
}  // extern "C"
