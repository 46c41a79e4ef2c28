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
// Seven kernels, the first four with a pack and an unpack form:
//  * tile_kernel (long ranges): one CTA of 256 threads moves one tile, up to TB
//    tokens of one (layer, K|V, sequence, head); TB * C = 1024 chunks (16 KiB)
//    when C is 8 or 16, four in flight per thread.  A V tile is one contiguous
//    run.  A K tile is C rows of TB contiguous chunks in the cache but TB rows
//    of C chunks in staging; it is transposed through shared memory so that
//    the cache side (512 contiguous bytes per warp instruction along a row)
//    and the staging side are both coalesced.  The shared-memory row pitch is
//    odd (C | 1 chunks), so the column-wise accesses of 8 consecutive tokens
//    fall in 8 distinct 16-byte bank groups.  The grid is persistent (SMs x
//    resident CTAs) and strides over the tiles in staging order, so at any
//    moment the whole GPU works on neighbouring tiles.  Two occupancy forms:
//    4 CTAs per SM (more registers) for launches of many rounds of tiles, 5
//    for smaller ones (kBigLaunchRounds).
//  * group_kernel (grouped tiles, C = 8 or 16): the tile kernel's shape for
//    ranges of at most half the token block, G = TB / NT heads of one
//    sequence to a tile (NT = the range length rounded up to a power of two),
//    so that short ranges fill the tile; a launch with both long and short
//    ranges runs the tile kernel over the long ones, then this one.
//  * token_kernel (every non-empty range of one common length: one-token
//    decode deltas, multi-token deltas): one chunk per thread, its run and
//    token found with multiply-high divisions by host constants; no shared
//    memory, no barrier.  A one-token K record is C isolated 16-byte chunks
//    (S * 16 bytes apart) by the layout itself.
//  * flat_kernel (ragged short ranges): each warp moves windows of 128
//    consecutive staging chunks; the window head's slab and sequence are
//    found once (binary search over the prefix table passed by value), and
//    each lane splits its own offset into head, token and chunk with the
//    sequence's multiply-high constant (a window that crosses a sequence
//    looks each chunk up on its own); no shared memory, no barrier.
//  * run_unpack_kernel / run_group_kernel (batched restore of runs of
//    one-token log records, the decode deltas of consecutive steps): the
//    tile kernel's unpack with one token per record, tiles of one head (long
//    runs) or of several heads side by side (short runs).
//  * record_unpack_kernel (batched restore of other log records): the flat
//    kernel's unpack with one more level, a record table in the parameters.
// All launches use programmatic dependent launch: a kernel waits for the grids
// it depends on (griddepcontrol.wait) before touching memory, then lets the
// next launch in the stream be scheduled.  Nothing waits on anything else
// but __syncthreads.  A launch whose staging side is host memory keeps to a
// small grid (see host_ctas) and leaves the rest of the GPU to other work.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <vector>

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
  int64_t k_lim, v_lim, stg_lim;  // checked builds: extents (chunks) the host validated
  int32_t l0, B, H, C, S;
  int32_t tiles_per_lkv;   // tile kernel: tiles per (layer, K|V) slab
  uint64_t m_tpl;          // ceil(2^64 / tiles_per_lkv) (0 when it is 1)
  uint64_t m_lkv;          // flat kernel: ceil(2^64 / lkv_chunks) (0 when it is 1)
  int32_t seq_start[MAXB];
  int32_t seq_len[MAXB];
  int32_t tok_pre[MAXB + 1];
  int32_t tile_pre[MAXB + 1];  // tile kernel: H * sum of ceil(len / TB)
  uint32_t m_len[MAXB];        // flat kernel: ceil(2^32 / seq_len[b]), 0 for length 1
  uint8_t log2nt[MAXB];        // grouped tile kernel: log2 of token slots per head (LOG2TB: plain tiles)
};

#ifndef DV_TILE_CPT
#define DV_TILE_CPT 4  // 16-byte chunks each thread moves per tile
#endif
#ifndef DV_TILE_MIN_BLOCKS
#define DV_TILE_MIN_BLOCKS 5  // resident CTAs per SM the tile kernel is compiled for
#endif
#ifndef DV_TILE_MIN_BLOCKS_BIG
#define DV_TILE_MIN_BLOCKS_BIG 4  // ... for launches of many rounds of tiles (64 registers)
#endif
// Launches of at least this many rounds of a 4-CTA-per-SM grid take the
// 64-register form: 2-3% faster on gigabyte launches (snapshot pack 0.950
// against 0.925 of the copy peak), 2.5% slower on 51 MB ones, level at 150 MB.
constexpr int kBigLaunchRounds = 16;
#ifndef DV_FLAT_MIN_BLOCKS
#define DV_FLAT_MIN_BLOCKS 4  // resident CTAs per SM the flat kernel is compiled for
                              // (5 spills: 20-40% slower on 16..64-token unpacks)
#endif
#ifndef DV_GROUP_MIN_BLOCKS_PACK
#define DV_GROUP_MIN_BLOCKS_PACK 4    // resident CTAs per SM of the grouped tile kernel's pack:
                                      // 64 registers, 4-10% faster than 5 CTAs at 48
#endif
#ifndef DV_GROUP_MIN_BLOCKS_UNPACK
#define DV_GROUP_MIN_BLOCKS_UNPACK 5  // ... and of its unpack (at 4: up to 6% slower)
#endif
#ifndef DV_LOOKUP_HOST_SCALE
#define DV_LOOKUP_HOST_SCALE 2  // flat / record kernels on host memory: CTAs per tile-kernel CTA
#endif

#ifndef DV_PDL
#define DV_PDL 1  // programmatic dependent launch
#endif

constexpr int kFlatUnroll = 4;
constexpr int kTileUnroll = DV_TILE_CPT;
constexpr int kMaxTileC = 64;  // generic tile kernel: at most 64 chunks per token

template <int LOG2C>
struct TileShape {
  // kThreads * DV_TILE_CPT chunks per tile when C is a power of two we
  // specialise (16 KiB for 4 chunks per thread); 32 tokens otherwise.
  static constexpr int LOG2CH =
      DV_TILE_CPT == 8 ? 11 : DV_TILE_CPT == 4 ? 10 : DV_TILE_CPT == 2 ? 9 : 8;
  static constexpr int LOG2TB = LOG2C >= 0 ? LOG2CH - LOG2C : 5;
  static constexpr int TB = 1 << LOG2TB;
};

// Programmatic dependent launch: wait until the grids this launch depends on
// have completed and their memory is visible, then let the next launch in the
// stream be scheduled while this one runs (it still waits for this grid to
// finish before it touches memory).  No-ops when launched without PDL.
__device__ __forceinline__ void pdl_enter() {
#if DV_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// A 16-byte load cached in L2 only, whose miss fetches a 64-byte segment from
// DRAM rather than the default whole 128-byte line (the PTX prefetch-size
// qualifier).  Volatile so that it stays after griddepcontrol.wait.
__device__ __forceinline__ uint4 ld_seg64(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.cg.L2::64B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

#ifndef DV_CHECKED
#define DV_CHECKED 0  // 1: every global access is checked against the host-validated extents
#endif

#if DV_CHECKED
// First access outside its buffer since the last read: bit 63 set, bits 56..62
// the site, bits 0..55 the chunk index relative to the buffer.  The access is
// skipped; nothing traps.
__device__ unsigned long long g_dv_fault;

__device__ __forceinline__ bool in_bounds(const uint4* ptr, const uint4* base, int64_t lim,
                                          int site) {
  const int64_t i = ptr - base;
  if (i >= 0 && i < lim) return true;
  const unsigned long long code = (1ull << 63) | ((unsigned long long)(site & 0x7f) << 56) |
                                  ((unsigned long long)i & 0x00FFFFFFFFFFFFFFull);
  atomicCAS(&g_dv_fault, 0ull, code);
  return false;
}
#define DV_OK_K(ptr, site) in_bounds((ptr), p.k, p.k_lim, (site))
#define DV_OK_V(ptr, site) in_bounds((ptr), p.v, p.v_lim, (site))
#define DV_OK_S(ptr, site) in_bounds((ptr), p.stg, p.stg_lim, (site))
#else
#define DV_OK_K(ptr, site) true
#define DV_OK_V(ptr, site) true
#define DV_OK_S(ptr, site) true
#endif

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

// floor(n / d) for n < 2^31, with m = ceil(2^32 / d): n*m / 2^32 lies in
// [n/d, n/d + 1/2), so its floor is the quotient or one more.
__device__ __forceinline__ uint32_t div_by(uint32_t n, uint32_t d, uint64_t m) {
  uint32_t q = (uint32_t)(((uint64_t)n * m) >> 32);
  if ((uint64_t)q * d > n) --q;
  return q;
}

// floor(n / d) for 0 <= n < 2^63 and 1 <= d < 2^32, with m = ceil(2^64 / d)
// (m = 0 stands for d = 1): n*m / 2^64 lies in [n/d, n/d + 1/2).
__device__ __forceinline__ uint64_t div64_by(uint64_t n, uint64_t d, uint64_t m) {
  if (m == 0) return n;
  uint64_t q = __umul64hi(n, m);
  if (q * d > n) --q;
  return q;
}

constexpr int kWin = 32 * kFlatUnroll;  // chunks of one warp's window

// Address of the cache chunk of staging chunk g < total: the (layer, K|V)
// slab, the sequence (the last one whose run starts at or before the chunk's
// token-head; a non-empty one, as in find_seq), head, token and chunk, each
// from the kernel parameters alone.
template <int MAXB, int LOG2C>
__device__ __forceinline__ uint4* flat_addr(const KParams<MAXB>& p, int64_t g) {
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  const int64_t lkv = (int64_t)div64_by((uint64_t)g, (uint64_t)p.lkv_chunks, p.m_lkv);
  const int32_t r = (int32_t)(g - lkv * p.lkv_chunks);
  const int32_t rec = LOG2C >= 0 ? (r >> LOG2C) : r / C;
  const int32_t c = r - rec * C;
  int b = 0;
#pragma unroll
  for (int half = MAXB / 2; half > 0; half >>= 1)
    if (b + half < p.B && p.H * p.tok_pre[b + half] <= rec) b += half;
  const int32_t rr = rec - p.H * p.tok_pre[b];
  const int32_t len = p.seq_len[b];
  const int32_t h = p.m_len[b] ? (int32_t)div_by((uint32_t)rr, (uint32_t)len, p.m_len[b]) : rr;
  const int64_t t = p.seq_start[b] + (rr - h * len);
  const int64_t l = p.l0 + (lkv >> 1);
  const int64_t bh = (int64_t)b * p.H + h;
  uint4* ptr = (lkv & 1) == 0 ? p.k + l * p.layer_chunks + ((bh * C + c) * p.S + t)
                              : p.v + l * p.layer_chunks + ((bh * p.S + t) * C + c);
  return ((lkv & 1) == 0 ? DV_OK_K(ptr, 1) : DV_OK_V(ptr, 2)) ? ptr : nullptr;
}

// Addresses of the chunks w0 + u * 32 + lane (u < kFlatUnroll) of one warp's
// window of kWin consecutive staging chunks; nullptr where there is none.
// The window head's (layer, K|V) slab and sequence are looked up once for
// the warp; when the whole window lies inside that sequence's block of the
// slab, each lane only splits its own offset into head, token and chunk.
// Otherwise each chunk is looked up on its own.  Reads only the kernel
// parameters, so it may run before griddepcontrol.wait.
template <int MAXB, int LOG2C>
__device__ __forceinline__ void flat_window(const KParams<MAXB>& p, int64_t w0, int lane,
                                            uint4* (&cptr)[kFlatUnroll]) {
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
#pragma unroll
  for (int u = 0; u < kFlatUnroll; ++u) cptr[u] = nullptr;
  if (w0 >= p.total) return;
  const int64_t lkv = (int64_t)div64_by((uint64_t)w0, (uint64_t)p.lkv_chunks, p.m_lkv);
  const int32_t r0 = (int32_t)(w0 - lkv * p.lkv_chunks);
  const int32_t rec0 = LOG2C >= 0 ? (r0 >> LOG2C) : r0 / C;
  int b = 0;
#pragma unroll
  for (int half = MAXB / 2; half > 0; half >>= 1)
    if (b + half < p.B && p.H * p.tok_pre[b + half] <= rec0) b += half;
  const int32_t lo = p.H * p.tok_pre[b] * C;      // sequence b's block in the slab
  const int32_t hi = p.H * p.tok_pre[b + 1] * C;
  if (r0 <= hi - kWin) {  // (r0 + kWin could pass INT32_MAX in a slab near 2^31 chunks)
    const int32_t len = p.seq_len[b];
    const uint32_t m = p.m_len[b];
    const bool is_k = (lkv & 1) == 0;
    uint4* const slab = (is_k ? p.k : p.v) + (p.l0 + (lkv >> 1)) * p.layer_chunks;
    const int64_t bh0 = (int64_t)b * p.H;
    const int64_t s0 = p.seq_start[b];
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = w0 + u * 32 + lane;
      if (g >= p.total || !DV_OK_S(p.stg + g, 3)) continue;
      const int32_t q = r0 - lo + u * 32 + lane;  // chunk in the sequence's block
      const int32_t tokc = LOG2C >= 0 ? (q >> LOG2C) : q / C;
      const int32_t c = q - tokc * C;
      const int32_t h = m ? (int32_t)div_by((uint32_t)tokc, (uint32_t)len, m) : tokc;
      const int64_t t = s0 + (tokc - h * len);
      const int64_t bh = bh0 + h;
      uint4* ptr = is_k ? slab + ((bh * C + c) * p.S + t) : slab + ((bh * p.S + t) * C + c);
      if (is_k ? DV_OK_K(ptr, 1) : DV_OK_V(ptr, 2)) cptr[u] = ptr;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = w0 + u * 32 + lane;
      if (g < p.total && DV_OK_S(p.stg + g, 3)) cptr[u] = flat_addr<MAXB, LOG2C>(p, g);
    }
  }
}

// One unpack round whose staging loads (chunks g0 + u * USTRIDE) are issued
// before their addresses are known: `cptr` is looked up (when `lookup`, by
// find(key, cptr)) while the loads are in flight.
template <int USTRIDE, typename Params, typename Lookup>
__device__ __forceinline__ void unpack_round(const Params& p, int64_t g0, int64_t key,
                                             uint4* (&cptr)[kFlatUnroll], bool lookup,
                                             Lookup&& find) {
  uint4 val[kFlatUnroll];
#pragma unroll
  for (int u = 0; u < kFlatUnroll; ++u) {
    const int64_t g = g0 + u * USTRIDE;
    if (g < p.total && DV_OK_S(p.stg + g, 3)) val[u] = ld_stream(p.stg + g);
  }
  if (lookup) find(key, cptr);
#pragma unroll
  for (int u = 0; u < kFlatUnroll; ++u)
    if (cptr[u]) *cptr[u] = val[u];
}

// Each warp moves a window of kWin consecutive staging chunks per round (its
// lanes kFlatUnroll chunks each, 32 apart, so every warp instruction covers
// 512 contiguous staging bytes).  The first round's addresses are looked up
// before the wait for the preceding grid.  Pack: each later round's
// addresses are looked up while the previous round's loads are in flight.
// Unpack reads staging in order: each round's staging loads go first, and
// its lookups run while they are in flight.
template <bool PACK, int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads, DV_FLAT_MIN_BLOCKS)
flat_kernel(const __grid_constant__ KParams<MAXB> p) {
  const int lane = threadIdx.x & 31;
  const int64_t step = (int64_t)gridDim.x * (kThreads * kFlatUnroll);
  int64_t w0 = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kWin;
  uint4* cptr[kFlatUnroll];
  flat_window<MAXB, LOG2C>(p, w0, lane, cptr);
  pdl_enter();
  if (PACK) {
    for (; w0 < p.total; w0 += step) {
      uint4 val[kFlatUnroll];
#pragma unroll
      for (int u = 0; u < kFlatUnroll; ++u)
        if (cptr[u]) val[u] = ld_stream(cptr[u]);
      uint4* next[kFlatUnroll];
      flat_window<MAXB, LOG2C>(p, w0 + step, lane, next);
#pragma unroll
      for (int u = 0; u < kFlatUnroll; ++u) {
        if (cptr[u]) p.stg[w0 + u * 32 + lane] = val[u];
        cptr[u] = next[u];
      }
    }
  } else {
    const auto find = [&p, lane](int64_t w, uint4* (&c)[kFlatUnroll]) {
      flat_window<MAXB, LOG2C>(p, w, lane, c);
    };
    if (w0 < p.total) unpack_round<32>(p, w0 + lane, w0, cptr, false, find);
    for (w0 += step; w0 < p.total; w0 += step)
      unpack_round<32>(p, w0 + lane, w0, cptr, true, find);
  }
}

// ---- one-token ranges (decode deltas) ----------------------------------------

template <int MAXB>
struct TokParams {
  uint4* k;
  uint4* v;
  uint4* stg;
  int64_t layer_chunks;
  int64_t k_lim, v_lim, stg_lim;  // checked builds: extents (chunks) the host validated
  uint32_t total;         // staging chunks
  uint32_t AH;            // active sequences x heads: runs per (layer, K|V)
  uint32_t n;             // tokens of every non-empty range
  uint64_t m_AH, m_H, m_n;  // ceil(2^32 / d) for d = AH, H, n
  int32_t l0, H, C, S;
  int32_t act_b[MAXB];    // sequence of the a-th non-empty range
  int32_t act_t[MAXB];    // its one token
};

// Address of the cache chunk of staging chunk g (nullptr if there is none)
// and whether it is a K chunk; parameters only, so it may run before
// griddepcontrol.wait.
template <int MAXB, int LOG2C>
__device__ __forceinline__ uint4* token_lookup(const TokParams<MAXB>& p, uint32_t g,
                                               bool& is_k) {
  is_k = false;
  if (g >= p.total || !DV_OK_S(p.stg + g, 13)) return nullptr;
  const uint32_t C = LOG2C >= 0 ? (1u << LOG2C) : (uint32_t)p.C;
  const uint32_t rec = LOG2C >= 0 ? (g >> LOG2C) : g / C;
  const uint32_t c = g - rec * C;
  const uint32_t run = div_by(rec, p.n, p.m_n);
  const uint32_t j = rec - run * p.n;
  const uint32_t lkv = div_by(run, p.AH, p.m_AH);
  const uint32_t rem = run - lkv * p.AH;
  const uint32_t a = div_by(rem, (uint32_t)p.H, p.m_H);
  const uint32_t h = rem - a * p.H;
  const int64_t b = p.act_b[a];
  const int64_t t = p.act_t[a] + j;
  const int64_t l = p.l0 + (lkv >> 1);
  const int64_t bh = b * p.H + h;
  is_k = (lkv & 1) == 0;
  uint4* ptr = is_k ? p.k + l * p.layer_chunks + ((bh * C + c) * p.S + t)
                    : p.v + l * p.layer_chunks + ((bh * p.S + t) * C + c);
  return (is_k ? DV_OK_K(ptr, 11) : DV_OK_V(ptr, 12)) ? ptr : nullptr;
}

// Every non-empty range holds the same n tokens (n = 1: decode deltas):
// staging chunk g is chunk c of token j of run (layer, K|V, a-th non-empty
// sequence, head).  One chunk per thread, no shared memory, no barrier: the
// shortest chain from launch to the copy.  The first address is computed
// before the wait for the preceding grid, so only the copy is left after it.
//
// A K chunk of a one-token range is alone in its 128-byte line (the rest of
// the line holds the next tokens of its K row).  By default a miss brings the
// whole line in from DRAM; the pack asks for a 64-byte segment instead
// (measured on the full BLOOM-stage delta, 25.7 MB: 28.0 -> 24.4 us, DRAM
// reads 144 -> 80 bytes per K chunk), and reads it at normal L2 priority, so
// that the decode deltas of the next steps still find the segment in L2 when
// nothing evicted it in between.  V rows are read as a stream.
template <bool PACK, int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads)
token_kernel(const __grid_constant__ TokParams<MAXB> p) {
  const uint32_t stride = gridDim.x * kThreads;
  uint32_t g = blockIdx.x * kThreads + threadIdx.x;
  bool is_k;
  uint4* ptr = token_lookup<MAXB, LOG2C>(p, g, is_k);
  pdl_enter();
  for (; g < p.total; g += stride) {
    if (ptr) {
      if (PACK) p.stg[g] = is_k ? ld_seg64(ptr) : ld_stream(ptr);
      else *ptr = ld_stream(p.stg + g);
    }
    ptr = token_lookup<MAXB, LOG2C>(p, g + stride, is_k);
  }
}

// ---- batched unpack of log records (replica restore) -------------------------

constexpr int kRecMax = 128;     // records one launch takes at most (a power of two)
constexpr int kRecWords = 7000;  // int32 words of range tables one launch carries

// Records whose staging bytes lie back to back in `stg` (device memory or
// mapped host memory), each with its own layer range and token ranges.
struct RecParams {
  uint4* k;
  uint4* v;
  uint4* stg;              // the records' bytes, back to back (read only)
  int64_t layer_chunks;
  int64_t total;           // chunks of all records
  int64_t k_lim, v_lim, stg_lim;  // checked builds: extents (chunks) the host validated
  int32_t B, H, C, S;
  int32_t nrec;
  int64_t rec_pre[kRecMax + 1];  // first chunk of record r in stg
  int64_t rec_lkv[kRecMax];      // chunks of one (layer, K|V) slab of record r: H * T_r * C
  uint64_t rec_m[kRecMax];       // ceil(2^64 / rec_lkv[r]) (0 when it is 1)
  int32_t rec_l0[kRecMax];
  int32_t rec_tab[kRecMax];      // first word of record r's table in `words`
  int32_t words[kRecWords];      // per record: seq_start[B], tok_pre[B + 1], m_len[B]
};
static_assert(sizeof(RecParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// Address of the cache chunk of launch chunk g < total: the record (the last
// one starting at or before g), its (layer, K|V) slab, the sequence (the last
// one of the record whose run starts at or before the chunk's token-head; a
// non-empty one, as in find_seq), head, token and chunk, from the kernel
// parameters alone.  The searches are fixed-depth and free of branches.
template <int LOG2C>
__device__ __forceinline__ uint4* record_addr(const RecParams& p, int64_t g) {
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  int r = 0;
#pragma unroll
  for (int half = kRecMax / 2; half > 0; half >>= 1)
    if (r + half < p.nrec && p.rec_pre[r + half] <= g) r += half;
  const int64_t q = g - p.rec_pre[r];
  const int64_t lkv = (int64_t)div64_by((uint64_t)q, (uint64_t)p.rec_lkv[r], p.rec_m[r]);
  const int32_t w = (int32_t)(q - lkv * p.rec_lkv[r]);
  const int32_t rec = LOG2C >= 0 ? (w >> LOG2C) : w / C;
  const int32_t c = w - rec * C;
  const int32_t tab = p.rec_tab[r];
  const int32_t pre = tab + p.B;  // tok_pre of the record
  int b = 0;
#pragma unroll
  for (int half = kMaxBatch / 2; half > 0; half >>= 1)
    if (b + half < p.B && p.H * p.words[pre + b + half] <= rec) b += half;
  const int32_t rr = rec - p.H * p.words[pre + b];
  const int32_t len = p.words[pre + b + 1] - p.words[pre + b];
  const uint32_t m = (uint32_t)p.words[pre + p.B + 1 + b];
  const int32_t h = m ? (int32_t)div_by((uint32_t)rr, (uint32_t)len, m) : rr;
  const int64_t t = p.words[tab + b] + (rr - h * len);
  const int64_t l = p.rec_l0[r] + (lkv >> 1);
  const int64_t bh = (int64_t)b * p.H + h;
  uint4* ptr = (lkv & 1) == 0 ? p.k + l * p.layer_chunks + ((bh * C + c) * p.S + t)
                              : p.v + l * p.layer_chunks + ((bh * p.S + t) * C + c);
  return ((lkv & 1) == 0 ? DV_OK_K(ptr, 31) : DV_OK_V(ptr, 32)) ? ptr : nullptr;
}

// Addresses of the chunks w0 + u * 32 + lane (u < kFlatUnroll) of one warp's
// window of the launch, as flat_window finds them, with the record looked up
// first: once for the window head, and when the whole window lies inside
// one sequence's block of one slab of that record, each lane only splits its
// own offset; otherwise each chunk is looked up on its own.  Parameters
// only, so it may run before griddepcontrol.wait.
template <int LOG2C>
__device__ __forceinline__ void record_window(const RecParams& p, int64_t w0, int lane,
                                              uint4* (&cptr)[kFlatUnroll]) {
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
#pragma unroll
  for (int u = 0; u < kFlatUnroll; ++u) cptr[u] = nullptr;
  if (w0 >= p.total) return;
  int r = 0;
#pragma unroll
  for (int half = kRecMax / 2; half > 0; half >>= 1)
    if (r + half < p.nrec && p.rec_pre[r + half] <= w0) r += half;
  const int64_t q0 = w0 - p.rec_pre[r];
  const int64_t lkv = (int64_t)div64_by((uint64_t)q0, (uint64_t)p.rec_lkv[r], p.rec_m[r]);
  const int32_t r0 = (int32_t)(q0 - lkv * p.rec_lkv[r]);
  const int32_t rec0 = LOG2C >= 0 ? (r0 >> LOG2C) : r0 / C;
  const int32_t tab = p.rec_tab[r];
  const int32_t pre = tab + p.B;
  int b = 0;
#pragma unroll
  for (int half = kMaxBatch / 2; half > 0; half >>= 1)
    if (b + half < p.B && p.H * p.words[pre + b + half] <= rec0) b += half;
  const int32_t lo = p.H * p.words[pre + b] * C;  // sequence b's block in the slab
  const int32_t hi = p.H * p.words[pre + b + 1] * C;
  if (r0 <= hi - kWin) {  // (r0 + kWin could pass INT32_MAX in a slab near 2^31 chunks)
    const int32_t len = p.words[pre + b + 1] - p.words[pre + b];
    const uint32_t m = (uint32_t)p.words[pre + p.B + 1 + b];
    const bool is_k = (lkv & 1) == 0;
    uint4* const slab = (is_k ? p.k : p.v) + (p.rec_l0[r] + (lkv >> 1)) * p.layer_chunks;
    const int64_t bh0 = (int64_t)b * p.H;
    const int64_t s0 = p.words[tab + b];
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = w0 + u * 32 + lane;
      if (g >= p.total || !DV_OK_S(p.stg + g, 33)) continue;
      const int32_t q = r0 - lo + u * 32 + lane;  // chunk in the sequence's block
      const int32_t tokc = LOG2C >= 0 ? (q >> LOG2C) : q / C;
      const int32_t c = q - tokc * C;
      const int32_t h = m ? (int32_t)div_by((uint32_t)tokc, (uint32_t)len, m) : tokc;
      const int64_t t = s0 + (tokc - h * len);
      const int64_t bh = bh0 + h;
      uint4* ptr = is_k ? slab + ((bh * C + c) * p.S + t) : slab + ((bh * p.S + t) * C + c);
      if (is_k ? DV_OK_K(ptr, 31) : DV_OK_V(ptr, 32)) cptr[u] = ptr;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kFlatUnroll; ++u) {
      const int64_t g = w0 + u * 32 + lane;
      if (g < p.total && DV_OK_S(p.stg + g, 33)) cptr[u] = record_addr<LOG2C>(p, g);
    }
  }
}

// The flat kernel's unpack with one more level: chunk g of the launch belongs
// to the record whose first chunk is the last one at or below g, and inside
// that record it is addressed exactly as the flat kernel addresses a staging
// chunk (staging order [layer][K|V][sequence][head][token][chunk]).  Records
// of one launch write disjoint parts of the cache (the host splits launches
// where they would not), so their order inside a launch does not matter.
// Each warp moves windows of kWin consecutive chunks, as the flat kernel
// does.  The source is read in order (often from host memory, a long round
// trip): each round's loads go first and its lookups run while they are in
// flight.
template <int LOG2C>
__global__ void __launch_bounds__(kThreads, DV_FLAT_MIN_BLOCKS)
record_unpack_kernel(const __grid_constant__ RecParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t step = (int64_t)gridDim.x * (kThreads * kFlatUnroll);
  int64_t w0 = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kWin;
  uint4* cptr[kFlatUnroll];
  record_window<LOG2C>(p, w0, lane, cptr);
  pdl_enter();
  const auto find = [&p, lane](int64_t w, uint4* (&c)[kFlatUnroll]) {
    record_window<LOG2C>(p, w, lane, c);
  };
  if (w0 < p.total) unpack_round<32>(p, w0 + lane, w0, cptr, false, find);
  for (w0 += step; w0 < p.total; w0 += step) unpack_round<32>(p, w0 + lane, w0, cptr, true, find);
}

// Staging index of chunk q of a tile, q = t * C + c (token t, chunk c).  The
// tile kernel's staging tokens are contiguous (index q); a run of log records
// holds one token per record, so consecutive tokens are `rs` chunks apart.
template <bool STRIDED, int LOG2C>
__device__ __forceinline__ int64_t stg_index(int q, int32_t C, int64_t rs) {
  if (!STRIDED) return q;
  const int t = LOG2C >= 0 ? q >> LOG2C : q / C;
  return (int64_t)t * rs + (q - t * C);
}

// Run of `cnt` chunks between a contiguous span of the V cache and staging
// (contiguous too, or tokens of C chunks `rs` apart when STRIDED).
template <bool PACK, bool STRIDED, int LOG2C, typename Params>
__device__ __forceinline__ void copy_run(const Params& p, uint4* cache, uint4* stg, int cnt,
                                         int32_t C, int64_t rs) {
  for (int q0 = threadIdx.x; q0 < cnt; q0 += kThreads * kTileUnroll) {
    uint4 val[kTileUnroll];
    bool ok[kTileUnroll];
#pragma unroll
    for (int u = 0; u < kTileUnroll; ++u) {
      const int q = q0 + u * kThreads;
      const int64_t sq = stg_index<STRIDED, LOG2C>(q, C, rs);
      ok[u] = q < cnt && DV_OK_V(cache + q, 21) && DV_OK_S(stg + sq, 22);
      if (ok[u]) val[u] = PACK ? ld_stream(cache + q) : ld_stream(stg + sq);
    }
#pragma unroll
    for (int u = 0; u < kTileUnroll; ++u) {
      const int q = q0 + u * kThreads;
      if (ok[u]) {
        if (PACK) stg[stg_index<STRIDED, LOG2C>(q, C, rs)] = val[u];
        else cache[q] = val[u];
      }
    }
  }
}

// One tile, uniform across the CTA: its staging chunks, the cache chunk its
// first token starts at (V: the start of the contiguous run; K: row 0, row c
// at + c * S), its token count, whether it is a V tile, and (strided tiles)
// the staging chunks from one token to the next.
struct TileJob {
  uint4* stg;
  uint4* cache;
  int64_t rs;
  int32_t n;
  bool is_v;
};

template <int LOG2TB, int MAXB>
__device__ __forceinline__ TileJob decode_tile(const KParams<MAXB>& p, int64_t tile, int32_t C) {
  constexpr int TB = 1 << LOG2TB;
  const int64_t lkv = (int64_t)div64_by((uint64_t)tile, (uint64_t)p.tiles_per_lkv, p.m_tpl);
  const int32_t r = (int32_t)(tile - lkv * p.tiles_per_lkv);
  const int b = find_seq(p.tile_pre, p.B, r);
  const int32_t len = p.seq_len[b];
  const int32_t nblk = (len + TB - 1) >> LOG2TB;
  const int32_t rr = r - p.tile_pre[b];
  const int32_t h = rr / nblk;
  const int32_t t0 = (rr - h * nblk) << LOG2TB;
  const int64_t l = p.l0 + (lkv >> 1);
  const int64_t bh = (int64_t)b * p.H + h;
  TileJob j;
  j.n = min(TB, len - t0);
  j.rs = C;
  j.stg = p.stg + lkv * p.lkv_chunks + ((int64_t)p.H * p.tok_pre[b] + (int64_t)h * len + t0) * C;
  j.is_v = (lkv & 1) != 0;
  j.cache = j.is_v ? p.v + l * p.layer_chunks + (bh * p.S + p.seq_start[b] + t0) * C
                   : p.k + l * p.layer_chunks + bh * C * p.S + p.seq_start[b] + t0;
  return j;
}

// Moves one tile (see tile_kernel).  STRIDED: the tile's tokens lie job.rs
// chunks apart in staging (a run of log records) instead of back to back.
template <bool PACK, bool STRIDED, int LOG2C, typename Params>
__device__ __forceinline__ void copy_tile(const Params& p, const TileJob& job, uint4* smem) {
  constexpr int TB = TileShape<LOG2C>::TB;
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  const int32_t SROW = C | 1;
  const int32_t TC = TB * C;  // chunk slots of a full tile
  uint4* const stg = job.stg;
  const int64_t rs = job.rs;
  const int32_t n = job.n;
  const int32_t cnt = n * C;            // chunks in this tile
  if (job.is_v) {
    copy_run<PACK, STRIDED, LOG2C>(p, job.cache, stg, cnt, C, rs);
  } else if (PACK) {
    // K: row c of this tile starts at ck + c * S.
    uint4* ck = job.cache;
    for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int c = q >> LOG2TB, t = q & (TB - 1);
        if (q < TC && t < n && DV_OK_K(ck + (int64_t)c * p.S + t, 31))
          val[u] = ld_stream(ck + (int64_t)c * p.S + t);
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
      const int64_t sq = stg_index<STRIDED, LOG2C>(q, C, rs);
      if (DV_OK_S(stg + sq, 32)) stg[sq] = smem[t * SROW + c];
    }
    __syncthreads();
  } else {
    uint4* ck = job.cache;
    for (int q0 = threadIdx.x; q0 < cnt; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int64_t sq = stg_index<STRIDED, LOG2C>(q, C, rs);
        if (q < cnt && DV_OK_S(stg + sq, 33)) val[u] = ld_stream(stg + sq);
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
      if (t < n && DV_OK_K(ck + (int64_t)c * p.S + t, 34))
        ck[(int64_t)c * p.S + t] = smem[t * SROW + c];
    }
    __syncthreads();
  }
}

template <bool PACK, int MAXB, int LOG2C, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
tile_kernel(const __grid_constant__ KParams<MAXB> p) {
  extern __shared__ uint4 smem[];  // TB rows of (C | 1) chunks
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  int64_t tile = blockIdx.x;
  if (tile >= p.total) return;
  // The first tile is decoded before the wait for the preceding grid (that
  // reads only the kernel parameters), so its loads start right after it.
  const TileJob first = decode_tile<LOG2TB>(p, tile, C);
  pdl_enter();
  copy_tile<PACK, false, LOG2C>(p, first, smem);
  for (tile += gridDim.x; tile < p.total; tile += gridDim.x)
    copy_tile<PACK, false, LOG2C>(p, decode_tile<LOG2TB>(p, tile, C), smem);
}

// ---- grouped tiles: short ranges in the tile kernel's shape -------------------

// A tile of several heads of one sequence whose range is at most half the
// token block: G = TB / NT consecutive heads with NT = 2^log2nt >= n token
// slots each (n the range's length).  In staging the heads' blocks lie back to
// back, one span of heads * n * C chunks.  In the cache, K is heads * C rows of
// n chunks, S apart (head h's rows continue head h - 1's: row r of the tile is
// row r % C of head r / C), and V one run of n * C chunks per head, S * C
// apart.
struct GroupJob {
  uint4* stg;
  uint4* cache;    // K: row 0 of the first head at the range start; V: its first token row
  int32_t n;       // tokens of each head
  int32_t heads;   // heads in the tile (G; fewer in the sequence's last tile)
  int32_t log2nt;  // NT = 2^log2nt token slots per head
  bool is_v;
};

// Moves one grouped tile.  Its TB * C slots are G heads x NT tokens x C
// chunks; slot (g, t, c) is live when g < heads and t < n.  Staging and V are
// walked in token order (g, t, c): head g's block is n * C chunks from
// g * n * C in staging and from g * S * C in V.  K goes through shared memory
// ([t][r], odd pitch; r = g * C + c), its cache side walked in row order
// (r, t) so that consecutive lanes move a row's consecutive tokens.  No
// division: every index is a shift or a mask.
template <bool PACK, int LOG2C, typename Params>
__device__ __forceinline__ void copy_group(const Params& p, const GroupJob& j, uint4* smem) {
  constexpr int C = 1 << LOG2C;
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  constexpr int TC = (1 << LOG2TB) * C;  // chunk slots of a tile
  const int log2nt = j.log2nt;
  const int ntm = (1 << log2nt) - 1;
  const int log2hc = log2nt + LOG2C;     // slots of one head
  const int hcm = (1 << log2hc) - 1;
  const int RP = (1 << (LOG2TB - log2nt + LOG2C)) | 1;  // row pitch: G * C rows, odd
  const int n = j.n;
  const int heads = j.heads;
  const int rows = heads << LOG2C;
  uint4* const stg = j.stg;
  uint4* const cache = j.cache;
  const int64_t S = p.S;
  const int64_t vstride = S << LOG2C;   // V chunks from one head's first token row to the next's
  // staging index of slot (g, t, c), or -1 when the slot is not live
  const auto slot_stg = [&](int q) -> int {
    const int g = q >> log2hc, t = (q >> LOG2C) & ntm;
    return (g < heads && t < n) ? (g * n + t) * C + (q & (C - 1)) : -1;
  };
  if (j.is_v) {
    for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
      int sq[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        sq[u] = slot_stg(q);
        uint4* const cp = cache + (q >> log2hc) * vstride + (q & hcm);
        if (sq[u] >= 0 && !(DV_OK_V(cp, 51) && DV_OK_S(stg + sq[u], 52))) sq[u] = -1;
        if (sq[u] >= 0) val[u] = PACK ? ld_stream(cp) : ld_stream(stg + sq[u]);
      }
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        if (sq[u] < 0) continue;
        if (PACK) stg[sq[u]] = val[u];
        else cache[(q >> log2hc) * vstride + (q & hcm)] = val[u];
      }
    }
  } else if (PACK) {
    for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int t = q & ntm, r = q >> log2nt;
        if (t < n && r < rows && DV_OK_K(cache + (int64_t)r * S + t, 53))
          val[u] = ld_stream(cache + (int64_t)r * S + t);
      }
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int t = q & ntm, r = q >> log2nt;
        if (t < n && r < rows) smem[t * RP + r] = val[u];
      }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < TC; q += kThreads) {
      const int s = slot_stg(q);
      const int r = ((q >> log2hc) << LOG2C) + (q & (C - 1));
      if (s >= 0 && DV_OK_S(stg + s, 54)) stg[s] = smem[((q >> LOG2C) & ntm) * RP + r];
    }
    __syncthreads();
  } else {
    for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
      int sq[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        sq[u] = slot_stg(q0 + u * kThreads);
        if (sq[u] >= 0 && !DV_OK_S(stg + sq[u], 55)) sq[u] = -1;
        if (sq[u] >= 0) val[u] = ld_stream(stg + sq[u]);
      }
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        if (sq[u] < 0) continue;
        const int r = ((q >> log2hc) << LOG2C) + (q & (C - 1));
        smem[((q >> LOG2C) & ntm) * RP + r] = val[u];
      }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < TC; q += kThreads) {
      const int t = q & ntm, r = q >> log2nt;
      if (t < n && r < rows && DV_OK_K(cache + (int64_t)r * S + t, 56))
        cache[(int64_t)r * S + t] = smem[t * RP + r];
    }
    __syncthreads();
  }
}

// Grouped tiles of the sequences whose range is at most half the token block
// (log2nt[b] < LOG2TB; the other sequences have no tiles here and go to the
// tile kernel in a launch of their own).  Tiles in staging order: (layer,
// K|V), sequence, head group.  C = 8 or 16.
template <bool PACK, int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads,
                                  PACK ? DV_GROUP_MIN_BLOCKS_PACK : DV_GROUP_MIN_BLOCKS_UNPACK)
group_kernel(const __grid_constant__ KParams<MAXB> p) {
  extern __shared__ uint4 smem[];  // TB rows of (C | 1) chunks
  constexpr int C = 1 << LOG2C;
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  int64_t tile = blockIdx.x;
  if (tile >= p.total) return;
  pdl_enter();
  for (; tile < p.total; tile += gridDim.x) {
    const int64_t lkv = (int64_t)div64_by((uint64_t)tile, (uint64_t)p.tiles_per_lkv, p.m_tpl);
    const int32_t r = (int32_t)(tile - lkv * p.tiles_per_lkv);
    const int b = find_seq(p.tile_pre, p.B, r);
    const int32_t len = p.seq_len[b];
    const int lg = p.log2nt[b];
    const int32_t h0 = (r - p.tile_pre[b]) << (LOG2TB - lg);
    const int64_t l = p.l0 + (lkv >> 1);
    const int64_t bh0 = (int64_t)b * p.H + h0;
    GroupJob j;
    j.n = len;
    j.heads = min(1 << (LOG2TB - lg), p.H - h0);
    j.log2nt = lg;
    j.is_v = (lkv & 1) != 0;
    j.stg = p.stg + lkv * p.lkv_chunks + ((int64_t)p.H * p.tok_pre[b] + (int64_t)h0 * len) * C;
    j.cache = j.is_v ? p.v + l * p.layer_chunks + (bh0 * p.S + p.seq_start[b]) * C
                     : p.k + l * p.layer_chunks + bh0 * C * p.S + p.seq_start[b];
    copy_group<PACK, LOG2C>(p, j, smem);
  }
}

// ---- runs of one-token log records (replica restore) -------------------------

// n consecutive log records over the same layers [l0, l0 + nl) and the same
// A non-empty sequences, each record one token per sequence, one token further
// on than the record before: record j holds token act_p[a] + j of sequence
// act_b[a].  The records lie back to back in `stg`, rec_chunks apart, each in
// staging order [layer][K|V][a][head][chunk].
template <int MAXB>
struct RunParams {
  uint4* k;
  uint4* v;
  uint4* stg;
  int64_t layer_chunks;
  int64_t rec_chunks;      // chunks of one record: staging stride from token j to j + 1
  int64_t total;           // tiles
  int64_t k_lim, v_lim, stg_lim;  // checked builds: extents (chunks) the host validated
  int32_t l0, H, C, S;
  int32_t n;               // records of the run
  int32_t ah;              // A * H: tiles of one token block of one (layer, K|V)
  int64_t tiles_per_lkv;   // A * H * ceil(n / TB)  (< 2^31)
  uint64_t m_tpl;          // ceil(2^64 / tiles_per_lkv) (0 when it is 1)
  uint64_t m_ah;           // ceil(2^32 / ah)
  uint64_t m_H;            // ceil(2^32 / H)
  int32_t log2nt;          // grouped tiles: NT = 2^log2nt >= n token slots per head
  int32_t groups;          // grouped tiles: G = TB / NT heads per tile
  int32_t act_b[MAXB];
  int32_t act_p[MAXB];
};

// Tile `tile` of a run: (layer, K|V) slab, token block, then (sequence, head),
// so that the CTAs working side by side read neighbouring C-chunk segments of
// the same TB records.  Its tokens are j0 .. j0 + n - 1 of the run, that is
// cache tokens act_p[a] + j0 ..; token j of the tile is at staging chunk
// j * rec_chunks of the tile's base.
template <int LOG2TB, int MAXB>
__device__ __forceinline__ TileJob decode_run_tile(const RunParams<MAXB>& p, int64_t tile,
                                                   int32_t C) {
  constexpr int TB = 1 << LOG2TB;
  const int64_t lkv = (int64_t)div64_by((uint64_t)tile, (uint64_t)p.tiles_per_lkv, p.m_tpl);
  const uint32_t r = (uint32_t)(tile - lkv * p.tiles_per_lkv);
  const uint32_t jb = div_by(r, (uint32_t)p.ah, p.m_ah);
  const uint32_t ah = r - jb * (uint32_t)p.ah;
  const uint32_t a = div_by(ah, (uint32_t)p.H, p.m_H);
  const uint32_t h = ah - a * (uint32_t)p.H;
  const int32_t j0 = (int32_t)(jb << LOG2TB);
  const int64_t l = p.l0 + (lkv >> 1);
  const int64_t bh = (int64_t)p.act_b[a] * p.H + h;
  const int64_t t0 = (int64_t)p.act_p[a] + j0;
  TileJob j;
  j.n = min(TB, p.n - j0);
  j.rs = p.rec_chunks;
  j.stg = p.stg + (int64_t)j0 * p.rec_chunks + (lkv * p.ah + ah) * C;
  j.is_v = (lkv & 1) != 0;
  j.cache = j.is_v ? p.v + l * p.layer_chunks + (bh * p.S + t0) * C
                   : p.k + l * p.layer_chunks + bh * C * p.S + t0;
  return j;
}

// Unpacks a run of one-token records as the tile kernel unpacks long ranges:
// per (layer, K|V, sequence, head) and block of TB consecutive records, the
// TB tokens' C-chunk rows are read from the TB records (full 32-byte sectors),
// and K goes out as C rows of TB consecutive chunks through the shared-memory
// transpose.  A restore of one record at a time, or of records in staging
// order, writes each K chunk alone into a half-filled sector; here the tokens
// that share a K sector or line are written together.
template <int MAXB, int LOG2C, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
run_unpack_kernel(const __grid_constant__ RunParams<MAXB> p) {
  extern __shared__ uint4 smem[];  // TB rows of (C | 1) chunks
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  const int32_t C = LOG2C >= 0 ? (1 << LOG2C) : p.C;
  int64_t tile = blockIdx.x;
  if (tile >= p.total) return;
  const TileJob first = decode_run_tile<LOG2TB>(p, tile, C);
  pdl_enter();
  copy_tile<false, true, LOG2C>(p, first, smem);
  for (tile += gridDim.x; tile < p.total; tile += gridDim.x)
    copy_tile<false, true, LOG2C>(p, decode_run_tile<LOG2TB>(p, tile, C), smem);
}

// Cache chunk of chunk c of token t of the g-th (sequence, head) of a grouped
// tile starting at (sequence, head) index ah0 (K: row c of its block; V: its
// token row), or nullptr past the last (sequence, head).
template <int MAXB, int LOG2C>
__device__ __forceinline__ uint4* group_addr(const RunParams<MAXB>& p, bool is_v, int64_t l,
                                             uint32_t ah0, int g, int t, int c) {
  constexpr int32_t C = 1 << LOG2C;
  const uint32_t ah = ah0 + (uint32_t)g;
  if (ah >= (uint32_t)p.ah) return nullptr;
  const uint32_t a = div_by(ah, (uint32_t)p.H, p.m_H);
  const int64_t bh = (int64_t)p.act_b[a] * p.H + (ah - a * (uint32_t)p.H);
  const int64_t tt = (int64_t)p.act_p[a] + t;
  uint4* ptr = is_v ? p.v + l * p.layer_chunks + (bh * p.S + tt) * C + c
                    : p.k + l * p.layer_chunks + (bh * C + c) * p.S + tt;
  return (is_v ? DV_OK_V(ptr, 42) : DV_OK_K(ptr, 41)) ? ptr : nullptr;
}

// Unpacks a run shorter than half the token block (n <= NT = 2^log2nt <=
// TB / 2) in grouped tiles: a tile is one (layer, K|V) and G = TB / NT
// consecutive (sequence, head) pairs, each with its n tokens, so that a tile
// holds as many chunk slots as a full run tile and every thread has work.
// Token t of the tile reads G * C contiguous chunks of record t (the G heads
// lie side by side in it).  V goes straight from staging to its token rows; K
// goes through shared memory ([g][t][c], odd pitch) and out as G * C rows of
// n consecutive chunks.
template <int MAXB, int LOG2C>
__global__ void __launch_bounds__(kThreads, DV_TILE_MIN_BLOCKS)
run_group_kernel(const __grid_constant__ RunParams<MAXB> p) {
  extern __shared__ uint4 smem[];  // TB rows of (C | 1) chunks
  constexpr int C = 1 << LOG2C;
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  constexpr int TC = (1 << LOG2TB) * C;  // chunk slots of a tile
  constexpr int SROW = C | 1;
  const int log2nt = p.log2nt;
  const int log2gc = LOG2TB - log2nt + LOG2C;  // chunks of one token across the G heads
  const int n = p.n;
  int64_t tile = blockIdx.x;
  if (tile >= p.total) return;
  pdl_enter();
  for (; tile < p.total; tile += gridDim.x) {
    const int64_t lkv = (int64_t)div64_by((uint64_t)tile, (uint64_t)p.tiles_per_lkv, p.m_tpl);
    const uint32_t ah0 = (uint32_t)(tile - lkv * p.tiles_per_lkv) * (uint32_t)p.groups;
    const int64_t l = p.l0 + (lkv >> 1);
    const bool is_v = (lkv & 1) != 0;
    const uint4* sbase = p.stg + (lkv * p.ah + ah0) * C;
    // slots in record order: q = (t, g, c), t slowest
    for (int q0 = threadIdx.x; q0 < TC; q0 += kThreads * kTileUnroll) {
      uint4 val[kTileUnroll];
      bool ok[kTileUnroll];
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int t = q >> log2gc;
        const int gc = q & ((1 << log2gc) - 1);
        const uint4* sp = sbase + (int64_t)t * p.rec_chunks + gc;
        ok[u] = t < n && ah0 + (uint32_t)(gc >> LOG2C) < (uint32_t)p.ah && DV_OK_S(sp, 43);
        if (ok[u]) val[u] = ld_stream(sp);
      }
#pragma unroll
      for (int u = 0; u < kTileUnroll; ++u) {
        const int q = q0 + u * kThreads;
        if (!ok[u]) continue;
        const int t = q >> log2gc;
        const int g = (q >> LOG2C) & ((1 << (log2gc - LOG2C)) - 1);
        const int c = q & (C - 1);
        if (is_v) {
          uint4* cp = group_addr<MAXB, LOG2C>(p, true, l, ah0, g, t, c);
          if (cp) *cp = val[u];
        } else {
          smem[((g << log2nt) + t) * SROW + c] = val[u];
        }
      }
    }
    if (!is_v) {
      __syncthreads();
      // slots in cache order: q = (g, c, t), t fastest: each K row's n tokens
      for (int q = threadIdx.x; q < TC; q += kThreads) {
        const int t = q & ((1 << log2nt) - 1);
        const int row = q >> log2nt;
        const int g = row >> LOG2C;
        const int c = row & (C - 1);
        if (t >= n) continue;
        uint4* cp = group_addr<MAXB, LOG2C>(p, false, l, ah0, g, t, c);
        if (cp) *cp = smem[((g << log2nt) + t) * SROW + c];
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

// Launches `kernel` with programmatic stream serialisation allowed (when
// DV_PDL), so that it is scheduled while the previous kernel in the stream
// drains; the kernel's pdl_enter() keeps the ordering.
template <typename Params>
cudaError_t launch_kernel(void (*kernel)(Params), unsigned grid, size_t smem,
                          cudaStream_t stream, const Params& kp) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = DV_PDL ? 1 : 0;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, kp);
  return err != cudaSuccess ? err : cudaGetLastError();
}

inline uint64_t div_magic(uint32_t d) { return ((1ull << 32) + d - 1) / d; }

// Grid cap for a transfer whose staging side is (mapped) host memory: it is
// bound by the host link, so it keeps to a few CTAs and leaves the rest of
// the GPU to other work.  32 CTAs of 256 threads carry the full link (193 /
// 211 GB/s each way on the GB300 measured) and let a concurrent compute
// kernel run nearly unslowed; the whole GPU would serialise it.  The
// environment variable DV_HOST_CTAS, read once, overrides the count (0: no
// cap) for hosts with a faster link.
int64_t host_ctas() {
  static const int64_t v = [] {
    const char* e = std::getenv("DV_HOST_CTAS");
    if (!e || !*e) return (int64_t)32;
    const long x = std::strtol(e, nullptr, 10);
    return (int64_t)(x > 0 ? x : 0);
  }();
  return v;
}

// `per_cta` scales the count for kernels whose CTAs keep fewer bytes in flight
// than a tile CTA's 16 KiB (the token kernel keeps 4 KiB: 4x the CTAs) or
// spend longer between loads on address lookups (flat and record kernels:
// 2x; at 1x they carried 70-85% of the link).
inline int64_t host_cap(const Plan& p, int64_t cap, int64_t per_cta = 1) {
  const int64_t h = host_ctas() * per_cta;
  return (h > 0 && p.host_side && cap > h) ? h : cap;
}

// ceil(2^64 / d) for d >= 2; 0 for d <= 1 (div64_by then returns n).
inline uint64_t div64_magic(uint64_t d) {
  if (d <= 1) return 0;
  return (uint64_t)((((unsigned __int128)1 << 64) + d - 1) / d);
}

// Chunks of K (and of V) the host validated from the base pointer: layers
// [0, l1) at the layer stride, the last one dense.
inline int64_t cache_limit(const Plan& p) {
  const int64_t dense = (int64_t)p.B * p.H * p.D * p.S * p.P / 16;
  return p.l1 > 0 ? (int64_t)(p.l1 - 1) * p.layer_chunks + dense : 0;
}

template <int MAXB>
void fill_params(KParams<MAXB>& kp, const Plan& p, void* stg) {
  kp.k_lim = kp.v_lim = cache_limit(p);
  kp.stg_lim = p.bytes / 16;
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
  kp.m_lkv = div64_magic((uint64_t)p.lkv_chunks);  // the flat kernel divides by lkv_chunks
  for (int b = 0; b < p.B; ++b)
    kp.m_len[b] = p.seq_len[b] > 1 ? (uint32_t)div_magic((uint32_t)p.seq_len[b]) : 0u;
  const auto kernel = flat_kernel<PACK, MAXB, LOG2C>;
  const int64_t want = (kp.total + kThreads * kFlatUnroll - 1) / (kThreads * kFlatUnroll);
  const int64_t cap = host_cap(p, (int64_t)sm_count() * blocks_per_sm(kernel, 0, occ_cache),
                               DV_LOOKUP_HOST_SCALE);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  return launch_kernel(kernel, grid, 0, stream, kp);
}

// Whether sequence b's range goes in grouped tiles: non-empty and at most half
// the token block, with C = 8 or 16.
template <int LOG2C>
bool grouped_seq(const Plan& p, int b) {
  return LOG2C >= 0 && p.seq_len[b] > 0 && 2 * p.seq_len[b] <= TileShape<LOG2C>::TB;
}

// The grouped tiles of a launch (group_kernel): sequences whose range is at
// most half the token block, G = TB / NT heads per tile, NT the range length
// rounded up to a power of two.
template <bool PACK, int MAXB, int LOG2C>
cudaError_t run_group(const Plan& p, void* stg, cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  constexpr int LOG2TB = TileShape<LOG2C>::LOG2TB;
  constexpr int TB = 1 << LOG2TB;
  KParams<MAXB> kp;
  fill_params(kp, p, stg);
  int32_t acc = 0;
  for (int b = 0; b < p.B; ++b) {
    kp.tile_pre[b] = acc;
    kp.log2nt[b] = (uint8_t)LOG2TB;
    if (!grouped_seq<LOG2C>(p, b)) continue;
    int lg = 0;
    while ((1 << lg) < p.seq_len[b]) ++lg;
    kp.log2nt[b] = (uint8_t)lg;
    const int32_t G = TB >> lg;  // heads per tile
    acc += (p.H + G - 1) / G;
  }
  kp.tile_pre[p.B] = acc;
  kp.tiles_per_lkv = acc;
  const int64_t tiles = 2 * (int64_t)(p.l1 - p.l0) * acc;
  kp.total = tiles;
  kp.m_tpl = div64_magic((uint64_t)kp.tiles_per_lkv);
  const size_t smem = (size_t)TB * (p.C | 1) * sizeof(uint4);
  const auto kernel = group_kernel<PACK, MAXB, LOG2C>;
  // On host memory, twice the tile kernel's CTAs: a grouped tile is 50-100% live,
  // and at 1x its transfers carried 90-93% of the link (2..32-token ranges, batch
  // 32), at 2x 99-100%.
  const int64_t cap =
      host_cap(p, (int64_t)sm_count() * blocks_per_sm(kernel, smem, occ_cache), 2);
  const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
  return launch_kernel(kernel, grid, smem, stream, kp);
}

// The tile kernel's launch over the sequences with long ranges, then (C = 8
// or 16) the grouped tiles of the short ones in a second launch.
template <bool PACK, int MAXB, int LOG2C>
cudaError_t run_tile(const Plan& p, void* stg, cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  static std::atomic<int64_t> occ_big{0};
  constexpr int TB = TileShape<LOG2C>::TB;
  KParams<MAXB> kp;
  fill_params(kp, p, stg);
  bool grouped = false;
  int32_t acc = 0;
  for (int b = 0; b < p.B; ++b) {
    kp.tile_pre[b] = acc;
    if (grouped_seq<LOG2C>(p, b)) {
      grouped = true;  // no tiles here
      continue;
    }
    acc += p.H * ((p.seq_len[b] + TB - 1) / TB);
  }
  kp.tile_pre[p.B] = acc;
  if (acc > 0) {
    kp.tiles_per_lkv = acc;
    const int64_t tiles = 2 * (int64_t)(p.l1 - p.l0) * acc;
    kp.total = tiles;
    kp.m_tpl = div64_magic((uint64_t)kp.tiles_per_lkv);
    const size_t smem = (size_t)TB * (p.C | 1) * sizeof(uint4);
    const bool big = !p.host_side && tiles >= (int64_t)kBigLaunchRounds *
                                                 DV_TILE_MIN_BLOCKS_BIG * sm_count();
    const auto kernel = big ? tile_kernel<PACK, MAXB, LOG2C, DV_TILE_MIN_BLOCKS_BIG>
                            : tile_kernel<PACK, MAXB, LOG2C, DV_TILE_MIN_BLOCKS>;
    const int64_t cap = host_cap(
        p, (int64_t)sm_count() * blocks_per_sm(kernel, smem, big ? occ_big : occ_cache));
    const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
    const cudaError_t err = launch_kernel(kernel, grid, smem, stream, kp);
    if (err != cudaSuccess) return err;
  }
  if constexpr (LOG2C >= 0) {
    if (grouped) return run_group<PACK, MAXB, LOG2C>(p, stg, stream);
  }
  return cudaSuccess;
}

template <bool PACK, int MAXB, int LOG2C>
cudaError_t run_token(const Plan& p, void* stg, cudaStream_t stream) {
  TokParams<MAXB> kp;
  kp.k = static_cast<uint4*>(p.k);
  kp.v = static_cast<uint4*>(p.v);
  kp.stg = static_cast<uint4*>(stg);
  kp.layer_chunks = p.layer_chunks;
  kp.k_lim = kp.v_lim = cache_limit(p);
  kp.stg_lim = p.bytes / 16;
  int32_t a = 0;
  for (int32_t b = 0; b < p.B; ++b) {
    if (p.seq_len[b] == 0) continue;
    kp.act_b[a] = b;
    kp.act_t[a] = p.seq_start[b];
    ++a;
  }
  kp.AH = (uint32_t)(a * p.H);
  kp.n = (uint32_t)p.max_len;
  kp.m_AH = div_magic(kp.AH);
  kp.m_H = div_magic((uint32_t)p.H);
  kp.m_n = div_magic(kp.n);
  kp.total = (uint32_t)(2 * (int64_t)(p.l1 - p.l0) * kp.AH * kp.n * p.C);
  kp.l0 = p.l0;
  kp.H = p.H;
  kp.C = p.C;
  kp.S = p.S;
  const auto kernel = token_kernel<PACK, MAXB, LOG2C>;
  const unsigned want = (kp.total + kThreads - 1) / kThreads;
  const unsigned cap = (unsigned)host_cap(p, (int64_t)sm_count() * 8, 4);
  return launch_kernel(kernel, want < cap ? want : cap, 0, stream, kp);
}

template <bool PACK, int MAXB>
cudaError_t dispatch_c(const Plan& p, void* stg, cudaStream_t stream, int kind) {
  if (kind == kToken) {
    if (p.C == 8) return run_token<PACK, MAXB, 3>(p, stg, stream);
    if (p.C == 16) return run_token<PACK, MAXB, 4>(p, stg, stream);
    return run_token<PACK, MAXB, -1>(p, stg, stream);
  }
  const bool tile = kind == kTile;
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
  int kind = variant;
  if (variant == kAuto) kind = auto_kind(p, PACK);
  if (p.B <= kSmallBatch) return dispatch_c<PACK, kSmallBatch>(p, stg, stream, kind);
  return dispatch_c<PACK, kMaxBatch>(p, stg, stream, kind);
}

template <int LOG2C>
cudaError_t run_records(const Plan& cache, const RecordRanges* recs, int n, const void* src,
                        cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  static thread_local RecParams kp;  // 32 KB: kept off the stack
  const int32_t B = cache.B;
  if (n > kRecMax || (int64_t)n * (3 * B + 1) > kRecWords) return cudaErrorInvalidValue;
  kp.k = static_cast<uint4*>(cache.k);
  kp.v = static_cast<uint4*>(cache.v);
  kp.stg = static_cast<uint4*>(const_cast<void*>(src));
  kp.layer_chunks = cache.layer_chunks;
  kp.k_lim = kp.v_lim = cache_limit(cache);
  kp.B = B;
  kp.H = cache.H;
  kp.C = cache.C;
  kp.S = cache.S;
  kp.nrec = n;
  int64_t chunk = 0;
  int32_t word = 0;
  for (int r = 0; r < n; ++r) {
    const RecordRanges& rec = recs[r];
    kp.rec_pre[r] = chunk;
    kp.rec_tab[r] = word;
    kp.rec_l0[r] = rec.l0;
    int32_t* start = kp.words + word;
    int32_t* pre = start + B;
    int32_t* mlen = pre + B + 1;
    int64_t tokens = 0;
    for (int32_t b = 0; b < B; ++b) {
      const int32_t len = rec.end[b] > rec.start[b] ? rec.end[b] - rec.start[b] : 0;
      start[b] = rec.start[b];
      pre[b] = (int32_t)tokens;
      mlen[b] = len > 1 ? (int32_t)(uint32_t)div_magic((uint32_t)len) : 0;
      tokens += len;
    }
    pre[B] = (int32_t)tokens;
    const int64_t lkv = (int64_t)cache.H * tokens * cache.C;
    kp.rec_lkv[r] = lkv;
    kp.rec_m[r] = div64_magic((uint64_t)lkv);
    chunk += 2 * (int64_t)(rec.l1 - rec.l0) * lkv;
    word += 3 * B + 1;
  }
  kp.rec_pre[n] = chunk;
  kp.total = chunk;
  kp.stg_lim = chunk;
  if (chunk == 0) return cudaSuccess;
  const auto kernel = record_unpack_kernel<LOG2C>;
  const int64_t want = (chunk + kThreads * kFlatUnroll - 1) / (kThreads * kFlatUnroll);
  const int64_t cap = host_cap(cache, (int64_t)sm_count() * blocks_per_sm(kernel, 0, occ_cache),
                               DV_LOOKUP_HOST_SCALE);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  return launch_kernel(kernel, grid, 0, stream, kp);
}

template <int MAXB, int LOG2C>
cudaError_t run_run(const Plan& cache, const RecordRanges& first, int n, const void* src,
                    cudaStream_t stream) {
  static std::atomic<int64_t> occ_cache{0};
  static std::atomic<int64_t> occ_big{0};
  constexpr int TB = TileShape<LOG2C>::TB;
  RunParams<MAXB> kp;
  kp.k = static_cast<uint4*>(cache.k);
  kp.v = static_cast<uint4*>(cache.v);
  kp.stg = static_cast<uint4*>(const_cast<void*>(src));
  kp.layer_chunks = cache.layer_chunks;
  kp.k_lim = kp.v_lim = cache_limit(cache);
  int32_t a = 0;
  for (int32_t b = 0; b < cache.B; ++b) {
    if (first.end[b] <= first.start[b]) continue;
    kp.act_b[a] = b;
    kp.act_p[a] = first.start[b];
    ++a;
  }
  const int64_t ah = (int64_t)a * cache.H;
  const int64_t nblk = ((int64_t)n + TB - 1) / TB;
  const int32_t nl = first.l1 - first.l0;
  if (a == 0 || n <= 0 || nl <= 0) return cudaSuccess;
  if (ah * nblk >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  kp.l0 = first.l0;
  kp.H = cache.H;
  kp.C = cache.C;
  kp.S = cache.S;
  kp.n = n;
  kp.ah = (int32_t)ah;
  kp.rec_chunks = 2 * (int64_t)nl * ah * cache.C;
  kp.m_ah = div_magic((uint32_t)ah);
  kp.m_H = div_magic((uint32_t)cache.H);
  kp.stg_lim = (int64_t)n * kp.rec_chunks;
  kp.log2nt = 0;
  kp.groups = 1;
  const size_t smem = (size_t)TB * (cache.C | 1) * sizeof(uint4);
  if constexpr (LOG2C >= 0) {
  if (2 * n <= TB) {  // a short run: grouped tiles
    int lg = 0;
    while ((1 << lg) < n) ++lg;
    kp.log2nt = lg;
    kp.groups = TB >> lg;
    kp.tiles_per_lkv = (ah + kp.groups - 1) / kp.groups;
    kp.total = 2 * (int64_t)nl * kp.tiles_per_lkv;
    kp.m_tpl = div64_magic((uint64_t)kp.tiles_per_lkv);
    const auto gkernel = run_group_kernel<MAXB, LOG2C>;
    static std::atomic<int64_t> occ_group{0};
    const int64_t fill = ((int64_t(1) << lg) + n - 1) / n;  // <= 2: NT / n
    const int64_t gcap = host_cap(
        cache, (int64_t)sm_count() * blocks_per_sm(gkernel, smem, occ_group), fill);
    const unsigned ggrid = (unsigned)(kp.total < gcap ? kp.total : gcap);
    return launch_kernel(gkernel, ggrid, smem, stream, kp);
  }
  }
  kp.tiles_per_lkv = ah * nblk;
  kp.total = 2 * (int64_t)nl * kp.tiles_per_lkv;
  kp.m_tpl = div64_magic((uint64_t)kp.tiles_per_lkv);
  const bool big = !cache.host_side && kp.total >= (int64_t)kBigLaunchRounds *
                                                       DV_TILE_MIN_BLOCKS_BIG * sm_count();
  const auto kernel = big ? run_unpack_kernel<MAXB, LOG2C, DV_TILE_MIN_BLOCKS_BIG>
                          : run_unpack_kernel<MAXB, LOG2C, DV_TILE_MIN_BLOCKS>;
  // From host memory, a run shorter than the token block leaves each tile
  // (and so each CTA's bytes in flight over the link) that much emptier than
  // a full one: scale the CTA cap up to match, at most 8x.
  const int64_t fill = n < TB ? (TB + n - 1) / n : 1;
  const int64_t cap = host_cap(
      cache, (int64_t)sm_count() * blocks_per_sm(kernel, smem, big ? occ_big : occ_cache),
      fill < 8 ? fill : 8);
  const unsigned grid = (unsigned)(kp.total < cap ? kp.total : cap);
  return launch_kernel(kernel, grid, smem, stream, kp);
}

// Whether record k writes a part of the cache that one of recs[0, k) writes:
// their layer ranges meet and, for some sequence, so do their token ranges.
// `lo` / `hi` hold the hull of the token ranges of recs[0, k) per sequence.
bool overlaps_earlier(const RecordRanges* recs, int k, int32_t B, const int32_t* lo,
                      const int32_t* hi) {
  const RecordRanges& x = recs[k];
  for (int32_t b = 0; b < B; ++b) {
    const int32_t s = x.start[b], e = x.end[b];
    if (s >= e || s >= hi[b] || e <= lo[b]) continue;
    for (int j = 0; j < k; ++j) {
      const RecordRanges& y = recs[j];
      if (y.l0 >= x.l1 || x.l0 >= y.l1) continue;
      if (y.start[b] < y.end[b] && y.start[b] < e && s < y.end[b]) return true;
    }
  }
  return false;
}

}  // namespace

bool tile_supported(const Plan& p) { return p.C <= kMaxTileC; }

bool token_supported(const Plan& p) {
  return p.active > 0 && p.min_len == p.max_len &&
         2 * (int64_t)(p.l1 - p.l0) * p.H * p.tokens * p.C < ((int64_t)1 << 31);
}

// Whether the lower crossovers of grouped tiles apply: C = 8 or 16, and a
// transfer of at least 4 MiB (below that a launch costs about its start, and
// the token or flat kernel's single launch is the cheaper one: a 150 KB
// unpack took 1.9 us in grouped tiles against 1.3 in the token kernel).
static bool grouped_pays(const Plan& p) {
  return (p.C == 8 || p.C == 16) && p.bytes >= ((int64_t)4 << 20);
}

int auto_kind(const Plan& p, bool pack) {
  // Equal-length ranges: the token kernel up to about 640 chunks per run
  // (measured on GB300: between 64 and 96 tokens at head_dim 64, between 32
  // and 48 at 128 in fp16), the tile kernel beyond.  With grouped tiles (C = 8
  // or 16) the unpack takes the tile kernel from 128 chunks per run (8 tokens
  // at head_dim 128, 16 at 64; one-token deltas stay with the token kernel):
  // its K stores cover each row's tokens together, 7-26% faster at batch 32
  // (at head_dim 64 from 4 tokens, 32 chunks); the pack at head_dim 128 from
  // 512 chunks.  Ragged ranges: the flat kernel
  // below the tile kernel's crossover (auto_uses_tile).
  if (token_supported(p)) {
    if (!tile_supported(p)) return kToken;
    const int64_t run = (int64_t)p.max_len * p.C;  // chunks per (layer, K|V, sequence, head)
    if (grouped_pays(p) && !pack && p.max_len > 1)
      return run >= (p.C == 8 ? 32 : 128) ? kTile : kToken;
    return run >= (grouped_pays(p) && pack && p.C == 16 ? 512 : 640) ? kTile : kToken;
  }
  return auto_uses_tile(p, pack) ? kTile : kFlat;
}

bool auto_uses_tile(const Plan& p, bool pack) {
  if (!tile_supported(p) || p.active == 0) return false;
  // Tiles pay once a (layer, K|V, sequence, head) run holds about 512 chunks
  // (8 KiB) on average, for pack and unpack alike (measured on GB300 with
  // ragged ranges over all layers: the flat kernel wins at 292 chunks per run
  // for head_dim 128 and at 477 for 64 in fp16, the tile kernel at 648 and 712
  // for 128 and at 770 for 64).  With grouped tiles (C = 8 or 16; ranges of at
  // most half the token block go several heads to a tile) the tile variant
  // wins from about 64 chunks per run for the unpack and for the pack at
  // head_dim 128 (4-13% on 4..16- to 16..32-token ranges, batch 8 and 32), at
  // any length for the unpack at head_dim 64 (1..8-token ranges: 6-16%), and
  // for the pack at head_dim 64 from about 300.
  int64_t per_run = 512;
  if (grouped_pays(p) && p.C == 16) per_run = 64;
  if (grouped_pays(p) && p.C == 8) per_run = pack ? 300 : 0;  // the unpack at head_dim 64: any
  return p.tokens * p.C >= per_run * p.active;
}

bool checked_build() { return DV_CHECKED != 0; }

cudaError_t read_fault(uint64_t* out) {
#if DV_CHECKED
  unsigned long long v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_dv_fault, sizeof(v));
  if (err != cudaSuccess) return err;
  const unsigned long long zero = 0;
  err = cudaMemcpyToSymbol(g_dv_fault, &zero, sizeof(zero));
  *out = v;
  return err;
#else
  *out = 0;
  return cudaSuccess;
#endif
}

cudaError_t launch_pack(const Plan& p, void* stg, cudaStream_t stream, int variant) {
  return launch<true>(p, stg, stream, variant);
}

cudaError_t launch_unpack(const Plan& p, const void* stg, cudaStream_t stream, int variant) {
  return launch<false>(p, const_cast<void*>(stg), stream, variant);
}

int records_per_launch(const Plan& cache, const RecordRanges* recs, int n) {
  if (n <= 0) return 0;
  const int32_t B = cache.B;
  int limit = kRecWords / (3 * B + 1);
  if (limit > kRecMax) limit = kRecMax;
  if (limit > n) limit = n;
  std::vector<int32_t> lo(B, INT32_MAX), hi(B, INT32_MIN);
  int k = 0;
  for (; k < limit; ++k) {
    if (k > 0 && overlaps_earlier(recs, k, B, lo.data(), hi.data())) break;
    for (int32_t b = 0; b < B; ++b) {
      if (recs[k].start[b] >= recs[k].end[b]) continue;
      if (recs[k].start[b] < lo[b]) lo[b] = recs[k].start[b];
      if (recs[k].end[b] > hi[b]) hi[b] = recs[k].end[b];
    }
  }
  return k;
}

int run_length(const Plan& cache, const RecordRanges* recs, int n) {
  if (n <= 0 || !tile_supported(cache)) return n > 0 ? 1 : 0;
  const RecordRanges& f = recs[0];
  const int32_t B = cache.B;
  bool any = false;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t len = f.end[b] - f.start[b];
    if (len > 1) return 1;
    any = any || len == 1;
  }
  if (!any) return 1;
  int k = 1;
  for (; k < n; ++k) {
    const RecordRanges& x = recs[k];
    if (x.l0 != f.l0 || x.l1 != f.l1) break;
    bool same = true;
    for (int32_t b = 0; b < B && same; ++b) {
      const bool act = f.end[b] > f.start[b];
      if (act) same = x.start[b] == f.start[b] + k && x.end[b] == x.start[b] + 1;
      else same = x.end[b] <= x.start[b];
    }
    if (!same) break;
  }
  return k;
}

int run_min_records(const Plan& cache) {
  // C = 8 and 16 (head_dim 64 / 128 in 2-byte elements): runs up to half the
  // token block go in grouped tiles (run_group_kernel), so any run of two
  // records or more pays.  Other C have no grouped tiles; there a run's tiles
  // cost about the same whatever their depth, and it pays from a quarter of
  // the token block (measured with 2-byte elements before grouped tiles: the
  // record kernel won at 16 records and the run kernel at 32 for TB = 128, at
  // 8 and at 16 for TB = 64).
  if (cache.C == 8 || cache.C == 16) return 2;
  return TileShape<-1>::TB / 4 > 2 ? TileShape<-1>::TB / 4 : 2;
}

int run_max_records(const Plan& cache, const RecordRanges& first) {
  int64_t a = 0;
  for (int32_t b = 0; b < cache.B; ++b) a += first.end[b] > first.start[b];
  const int64_t ah = a * cache.H;
  if (ah == 0) return INT32_MAX;
  const int64_t tb = cache.C == 8 ? TileShape<3>::TB : cache.C == 16 ? TileShape<4>::TB
                                                                      : TileShape<-1>::TB;
  const int64_t blocks = (((int64_t)1 << 31) - 1) / ah;  // tiles of one slab stay below 2^31
  const int64_t m = blocks * tb;
  return m < INT32_MAX ? (int)m : INT32_MAX;
}

cudaError_t launch_unpack_run(const Plan& cache, const RecordRanges& first, int n,
                              const void* src, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (!tile_supported(cache)) return cudaErrorInvalidValue;
  if (cache.B <= kSmallBatch) {
    if (cache.C == 8) return run_run<kSmallBatch, 3>(cache, first, n, src, stream);
    if (cache.C == 16) return run_run<kSmallBatch, 4>(cache, first, n, src, stream);
    return run_run<kSmallBatch, -1>(cache, first, n, src, stream);
  }
  if (cache.C == 8) return run_run<kMaxBatch, 3>(cache, first, n, src, stream);
  if (cache.C == 16) return run_run<kMaxBatch, 4>(cache, first, n, src, stream);
  return run_run<kMaxBatch, -1>(cache, first, n, src, stream);
}

cudaError_t launch_unpack_records(const Plan& cache, const RecordRanges* recs, int n,
                                  const void* src, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (cache.C == 8) return run_records<3>(cache, recs, n, src, stream);
  if (cache.C == 16) return run_records<4>(cache, recs, n, src, stream);
  return run_records<-1>(cache, recs, n, src, stream);
}

}  // namespace dv
