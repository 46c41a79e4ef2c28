// libdv C ABI, part 4: pinned host memory for replicas and swap buffers.
//
// The host side of every transfer (§3 "Microbatch swapping", "Fault detection
// and recovery": the replica lives in CPU memory) is pinned memory the copy
// engines and the kernels reach over the host link.  On a GB300 host with
// 64 KiB base pages, passes over tens of GB of pinned memory backed by base
// pages periodically run at about half the link rate; the same memory backed
// by transparent huge pages runs every pass at the full rate.  This allocator
// maps anonymous memory, asks for huge pages on its huge-page-aligned part,
// and registers it with CUDA as pinned, mapped, portable memory.
#include <cuda_runtime.h>
#include <sys/mman.h>
#include <unistd.h>

#include <cstdio>
#include <mutex>
#include <new>
#include <vector>

#include "dv_host.h"

using dv::cuda_fail;
using dv::fail;

namespace {

struct Mapping {
  void* ptr;     // the address handed out (huge-page aligned)
  size_t bytes;  // the length mapped at ptr
};

std::mutex g_mu;
std::vector<Mapping> g_maps;

// The transparent huge page size the kernel uses for anonymous memory (2 MiB
// when it cannot be read).
size_t huge_page_bytes() {
  static const size_t hp = [] {
    size_t v = 0;
    if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
      unsigned long long x = 0;
      if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
      std::fclose(f);
    }
    return v ? v : (size_t)2 << 20;
  }();
  return hp;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

dv_status dv_host_alloc(size_t bytes, void** out) {
  const dv::Trace trace("dv_host_alloc");
  if (!out) return fail(DV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (bytes == 0) return fail(DV_ERR_INVALID_ARG, "bytes is 0");
  const long ps = sysconf(_SC_PAGESIZE);
  const size_t page = ps > 0 ? (size_t)ps : 4096;
  const size_t hp = huge_page_bytes();
  const size_t len = round_up(bytes, page);
  if (len < bytes || len + hp < len) return fail(DV_ERR_INVALID_ARG, "bytes %zu too large", bytes);
  // Map one huge page more than needed and trim, so that the start is
  // huge-page aligned and every whole huge page of the range can be one.
  void* raw = mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED)
    return fail(DV_ERR_INVALID_ARG, "out of host memory (mmap of %zu bytes failed)", len + hp);
  const uintptr_t r = reinterpret_cast<uintptr_t>(raw);
  const uintptr_t a = round_up(r, hp);
  if (a > r) munmap(raw, a - r);
  const size_t tail = (r + len + hp) - (a + len);
  if (tail) munmap(reinterpret_cast<void*>(a + len), tail);
  void* p = reinterpret_cast<void*>(a);
  if (len >= hp) madvise(p, len / hp * hp, MADV_HUGEPAGE);  // advice only: may be ignored
  dv::ensure_context();
  const cudaError_t err =
      cudaHostRegister(p, len, cudaHostRegisterPortable | cudaHostRegisterMapped);
  if (err != cudaSuccess) {
    munmap(p, len);
    return cuda_fail(err, "cudaHostRegister");
  }
  try {
    std::lock_guard<std::mutex> lock(g_mu);
    g_maps.push_back({p, len});
  } catch (...) {
    cudaHostUnregister(p);
    munmap(p, len);
    return fail(DV_ERR_INVALID_ARG, "out of host memory for the allocation table");
  }
  *out = p;
  return DV_OK;
}

dv_status dv_host_free(void* ptr) {
  if (!ptr) return DV_OK;
  Mapping m{nullptr, 0};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (size_t i = 0; i < g_maps.size(); ++i) {
      if (g_maps[i].ptr == ptr) {
        m = g_maps[i];
        g_maps[i] = g_maps.back();
        g_maps.pop_back();
        break;
      }
    }
  }
  if (!m.ptr) return fail(DV_ERR_INVALID_ARG, "%p was not returned by dv_host_alloc", ptr);
  const cudaError_t err = cudaHostUnregister(m.ptr);
  munmap(m.ptr, m.bytes);
  return err == cudaSuccess ? DV_OK : cuda_fail(err, "cudaHostUnregister");
}

}  // extern "C"
