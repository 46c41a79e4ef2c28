// Pack / unpack kernels of the KV-cache buffered copy, for sm_103a.
//
// "DejaVu: KV-Cache Streaming for Fast, Fault-Tolerant Generative LLM
// Serving", §3 "Buffered copies" (Fig 6, Fig 7a) and Table 1 gather/scatter:
// the small non-contiguous K/V slices of a max-length cache are gathered into
// one contiguous buffer, and such a buffer is scattered back.
//
// Everything moves in 16-byte chunks (uint4): a chunk is x = 16/P elements of
// one K row (the x-interleaved layout keeps x elements of d contiguous) or of
// one V row.  Bytes are copied as bit patterns and never pass through
// floating point.
//
// Two kernels, one data path each way:
//  * flat_kernel: thread per staging chunk, in staging order, so stores (pack)
//    or loads (unpack) of the staging side are fully coalesced.  Its cache-side
//    accesses for K are one chunk per token row: right for one-token decode
//    deltas, where no two chunks of a K row are adjacent anyway.
//  * tile_kernel: one CTA per tile of up to TB tokens of one (layer, K|V,
//    sequence, head).  A V tile is one contiguous run.  A K tile is C rows of
//    TB contiguous chunks in the cache but TB rows of C chunks in staging; it
//    is transposed through shared memory so that both the cache side (512
//    contiguous bytes per warp along a row) and the staging side are
//    coalesced.  The shared-memory row pitch is odd (C | 1 chunks) so that the
//    column-wise accesses of 8 consecutive tokens fall in 8 distinct 16-byte
//    bank groups.
// Neither kernel waits on anything but __syncthreads.
#include <atomic>
#include <cstdint>

#include "dv_plan.h"

namespace dv {
namespace {

template <int MAXB>
struct KParams {
  uint4* k;                // K of layer 0 (pack: read; unpack: written)
  uint4* v;                // V of layer 0
  uint4* stg;              // staging (pack: written; unpack: read)
  int64_t layer_chunks;    // layer stride
  int64_t lkv_chunks;      // chunks per (layer, K|V) slab of staging
  int64_t total;           // flat: chunks; tile: tiles
  int32_t l0, B, H, C, S;
  int32_t tiles_per_lkv;   // tile kernel: tiles per (layer, K|V) slab
  int32_t seq_start[MAXB];
  int32_t seq_len[MAXB];
  int32_t tok_pre[MAXB + 1];
  int32_t tile_pre[MAXB + 1];  // tile kernel: H * sum of ceil(len / TB)
};

constexpr int kFlatUnroll = 4;
constexpr int kTileUnroll = 2;
constexpr int kMaxTileC = 64;  // generic tile kernel: at most 64 chunks per token

template <int LOG2C>
struct TileShape {
  // 512 chunks (8 KiB) per tile when C is a power of two we specialise.
  static constexpr int LOG2TB = LOG2C >= 0 ? 9 - LOG2C : 5;
  static constexpr int TB = 1 << LOG2TB;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// Largest b in [0, B) with pre[b] <= key (pre ascending).  With key inside
// [pre[b], pre[b+1]) of a non-empty b, that is b itself.
template <typename Arr>
__device__ __forceinline__ int find_seq(const Arr& pre, int B, int32_t key) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= key) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <bool PACK, int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads)
flat_kernel(const __grid_constant__ KParams<MAXB> p) {
  __shared__ int32_t s_rec_pre[MAXB + 1];  // first token record of each sequence
  __shared__ int32_t s_len[MAXB];
  __shared__ int32_t s_start[MAXB];
  for (int i = threadIdx.x; i <= p.B; i += kThreads) {
    s_rec_pre[i] = p.H * p.tok_pre[i];
    if (i < p.B) {
      s_len[i] = p.seq_len[i];
      s_start[i] = p.seq_start[i];
    }
  }
  __syncthreads();
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  const int64_t step = (int64_t)gridDim.x * (kThreads * kFlatUnroll);
  for (int64_t base = (int64_t)blockIdx.x * (kThreads * kFlatUnroll) + threadIdx.x;
       base < p.total; base += step) {
    uint4 val[kFlatUnroll];
    uint4* cptr[kFlatUnroll];
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = base + u * kThreads;
      cptr[u] = nullptr;
      if (g < p.total) {
        const int64_t lkv = g / p.lkv_chunks;
        const int32_t r = (int32_t)(g - lkv * p.lkv_chunks);
        const int32_t rec = LOG2C >= 0 ? (r >> LOG2C) : r / C;  // (b, h, t) record
        const int32_t c = r - rec * C;
        const int b = find_seq(s_rec_pre, p.B, rec);
        const int32_t rr = rec - s_rec_pre[b];
        const int32_t len = s_len[b];
        const int32_t h = rr / len;
        const int64_t t = s_start[b] + (rr - h * len);
        const int64_t l = p.l0 + (lkv >> 1);
        const int64_t bh = (int64_t)b * p.H + h;
        cptr[u] = (lkv & 1) == 0 ? p.k + l * p.layer_chunks + ((bh * C + c) * p.S + t)
                                 : p.v + l * p.layer_chunks + ((bh * p.S + t) * C + c);
        val[u] = PACK ? ld_stream(cptr[u]) : ld_stream(p.stg + g);
      }
    }
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = base + u * kThreads;
      if (g < p.total) {
        if (PACK) p.stg[g] = val[u];
        else *cptr[u] = val[u];
      }
    }
  }
}

// Contiguous run of `cnt` chunks between the cache and staging.
template <bool PACK>
__device__ __forceinline__ void copy_run(uint4* cache, uint4* stg, int cnt) {
  for (int q0 = threadIdx.x; q0 < cnt; q0 += kThreads * kTileUnroll) {
    uint4 val[kTileUnroll];
#pragma unroll
    for (int u = 0; u < kTileUnroll; ++u) {
      const int q = q0 + u * kThreads;
      if (q < cnt) val[u] = PACK ? ld_stream(cache + q) : ld_stream(stg + q);
    }
#pragma unroll
    for (int u = 0; u < kTileUnroll; ++u) {
      const int q = q0 + u * kThreads;
      if (q < cnt) {
        if (PACK) stg[q] = val[u];
        else cache[q] = val[u];
      }
    }
  }
}

template <bool PACK, int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads)
tile_kernel(const __grid_constant__ KParams<MAXB> p) {
  extern __shared__ uint4 smem[];  // TB rows of (C | 1) chunks
  constexpr int TB = TileShape<LOG2C>::TB;
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  const int32_t SROW = C | 1;
  const int32_t TC = TB * C;  // chunk slots of a full tile
  for (int64_t tile = blockIdx.x; tile < p.total; tile += gridDim.x) {
    // Uniform across the CTA: which (layer, K|V, sequence, head, token block).
    const int64_t lkv = tile / p.tiles_per_lkv;
    const int32_t r = (int32_t)(tile - lkv * p.tiles_per_lkv);
    const int b = find_seq(p.tile_pre, p.B, r);
    const int32_t len = p.seq_len[b];
    const int32_t nblk = (len + TB - 1) >> LOG2TB;
    const int32_t rr = r - p.tile_pre[b];
    const int32_t h = rr / nblk;
    const int32_t t0 = (rr - h * nblk) << LOG2TB;
    const int32_t n = min(TB, len - t0);  // tokens in this tile
    const int32_t cnt = n * C;            // chunks in this tile
    const int64_t l = p.l0 + (lkv >> 1);
    const int64_t bh = (int64_t)b * p.H + h;
    uint4* stg = p.stg + lkv * p.lkv_chunks +
                 ((int64_t)p.H * p.tok_pre[b] + (int64_t)h * len + t0) * C;
    if (lkv & 1) {
      uint4* cv = p.v + l * p.layer_chunks + (bh * p.S + p.seq_start[b] + t0) * C;
      copy_run<PACK>(cv, stg, cnt);
      continue;
    }
    // K: row c of this tile starts at ck + c * S.
    uint4* ck = p.k + l * p.layer_chunks + bh * C * p.S + p.seq_start[b] + t0;
    if (PACK) {
      for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
        uint4 val[kTileUnroll];
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u) {
          const int q = q0 + u * kThreads;
          const int c = q >> LOG2TB, t = q & (TB - 1);
          if (q < TC && t < n) val[u] = ld_stream(ck + (int64_t)c * p.S + t);
        }
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u) {
          const int q = q0 + u * kThreads;
          const int c = q >> LOG2TB, t = q & (TB - 1);
          if (q < TC && t < n) smem[t * SROW + c] = val[u];
        }
      }
      __syncthreads();
      for (int q = threadIdx.x; q < cnt; q += kThreads) {
        const int t = LOG2C >= 0 ? q >> LOG2C : q / C;
        const int c = q - t * C;
        stg[q] = smem[t * SROW + c];
      }
      __syncthreads();
    } else {
      for (int q0 = threadIdx.x; q0 < cnt; q0 += kThreads * kTileUnroll) {
        uint4 val[kTileUnroll];
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u) {
          const int q = q0 + u * kThreads;
          if (q < cnt) val[u] = ld_stream(stg + q);
        }
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u) {
          const int q = q0 + u * kThreads;
          if (q < cnt) {
            const int t = LOG2C >= 0 ? q >> LOG2C : q / C;
            const int c = q - t * C;
            smem[t * SROW + c] = val[u];
          }
        }
      }
      __syncthreads();
      for (int q = threadIdx.x; q < TC; q += kThreads) {
        const int c = q >> LOG2TB, t = q & (TB - 1);
        if (t < n) ck[(int64_t)c * p.S + t] = smem[t * SROW + c];
      }
      __syncthreads();
    }
  }
}

// ---- host side -------------------------------------------------------------

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) dev = 0;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = 1;
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Resident CTAs per SM of `kernel` with `smem` dynamic bytes, cached per
// (kernel instantiation, smem size).
template <typename Kernel>
int blocks_per_sm(Kernel kernel, size_t smem, std::atomic<int64_t>& cache) {
  const int64_t c = cache.load(std::memory_order_relaxed);
  if (c > 0 && (c >> 20) == (int64_t)smem) return (int)(c & 0xFFFFF);
  int v = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, kThreads, smem) != cudaSuccess ||
      v <= 0) {
    cudaGetLastError();
    v = 1;
  }
  cache.store(((int64_t)smem << 20) | v, std::memory_order_relaxed);
  return v;
}

template <int MAXB>
void fill_params(KParams<MAXB>& kp, const Plan& p, void* stg) {
  kp.k = static_cast<uint4*>(p.k);
  kp.v = static_cast<uint4*>(p.v);
  kp.stg = static_cast<uint4*>(stg);
  kp.layer_chunks = p.layer_chunks;
  kp.lkv_chunks = p.lkv_chunks;
  kp.l0 = p.l0;
  kp.B = p.B;
  kp.H = p.H;
  kp.C = p.C;
  kp.S = p.S;
  for (int b = 0; b < p.B; ++b) {
    kp.seq_start[b] = p.seq_start[b];
    kp.seq_len[b] = p.seq_len[b];
    kp.tok_pre[b] = p.tok_pre[b];
  }
  kp.tok_pre[p.B] = p.tok_pre[p.B];
}

template <bool PACK, int MAXB, int LOG2C>
cudaError_t run_flat(const Plan& p, void* stg, cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  KParams<MAXB> kp;
  fill_params(kp, p, stg);
  kp.total = 2 * (int64_t)(p.l1 - p.l0) * p.lkv_chunks;
  kp.tiles_per_lkv = 0;
  const auto kernel = flat_kernel<PACK, MAXB, LOG2C>;
  const int64_t want = (kp.total + kThreads * kFlatUnroll - 1) / (kThreads * kFlatUnroll);
  const int64_t cap = (int64_t)sm_count() * blocks_per_sm(kernel, 0, occ_cache);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  kernel<<<grid, kThreads, 0, stream>>>(kp);
  return cudaGetLastError();
}

template <bool PACK, int MAXB, int LOG2C>
cudaError_t run_tile(const Plan& p, void* stg, cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  constexpr int TB = TileShape<LOG2C>::TB;
  KParams<MAXB> kp;
  fill_params(kp, p, stg);
  int32_t acc = 0;
  for (int b = 0; b < p.B; ++b) {
    kp.tile_pre[b] = acc;
    acc += p.H * ((p.seq_len[b] + TB - 1) / TB);
  }
  kp.tile_pre[p.B] = acc;
  kp.tiles_per_lkv = acc;
  kp.total = 2 * (int64_t)(p.l1 - p.l0) * acc;
  const size_t smem = (size_t)TB * (p.C | 1) * sizeof(uint4);
  const auto kernel = tile_kernel<PACK, MAXB, LOG2C>;
  const int64_t cap = (int64_t)sm_count() * blocks_per_sm(kernel, smem, occ_cache);
  const unsigned grid = (unsigned)(kp.total < cap ? kp.total : cap);
  kernel<<<grid, kThreads, smem, stream>>>(kp);
  return cudaGetLastError();
}

template <bool PACK, int MAXB>
cudaError_t dispatch_c(const Plan& p, void* stg, cudaStream_t stream, bool tile) {
  if (tile) {
    if (p.C == 8) return run_tile<PACK, MAXB, 3>(p, stg, stream);
    if (p.C == 16) return run_tile<PACK, MAXB, 4>(p, stg, stream);
    return run_tile<PACK, MAXB, -1>(p, stg, stream);
  }
  if (p.C == 8) return run_flat<PACK, MAXB, 3>(p, stg, stream);
  if (p.C == 16) return run_flat<PACK, MAXB, 4>(p, stg, stream);
  return run_flat<PACK, MAXB, -1>(p, stg, stream);
}

template <bool PACK>
cudaError_t launch(const Plan& p, void* stg, cudaStream_t stream, int variant) {
  if (p.bytes == 0) return cudaSuccess;
  const bool tile = variant == kTile || (variant == kAuto && auto_uses_tile(p));
  if (p.B <= kSmallBatch) return dispatch_c<PACK, kSmallBatch>(p, stg, stream, tile);
  return dispatch_c<PACK, kMaxBatch>(p, stg, stream, tile);
}

}  // namespace

bool tile_supported(const Plan& p) { return p.C <= kMaxTileC; }

bool auto_uses_tile(const Plan& p) {
  if (!tile_supported(p) || p.active == 0) return false;
  return p.tokens >= (int64_t)16 * p.active;  // mean range length >= 16 tokens
}

cudaError_t launch_pack(const Plan& p, void* stg, cudaStream_t stream, int variant) {
  return launch<true>(p, stg, stream, variant);
}

cudaError_t launch_unpack(const Plan& p, const void* stg, cudaStream_t stream, int variant) {
  return launch<false>(p, const_cast<void*>(stg), stream, variant);
}

}  // namespace dv
