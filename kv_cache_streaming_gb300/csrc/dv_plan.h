// Internal to libdv: a validated copy plan and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dv.h"

namespace dv {

constexpr int kMaxBatch = 1024;   // == DV_MAX_BATCH
constexpr int kSmallBatch = 32;   // kernels with 32-entry range tables
constexpr int kThreads = 256;     // threads per CTA of every copy kernel

// Everything a pack / unpack launch needs, validated on the host.  Sizes in
// 16-byte chunks: one chunk is x = 16 / P consecutive elements of a K row or
// of a V row, the unit every kernel moves.
struct Plan {
  int32_t L, B, H, D, S, P;
  int32_t C;                 // chunks per token of one head: D * P / 16
  int64_t layer_chunks;      // layer stride of K and V
  int32_t l0, l1;
  int32_t seq_start[kMaxBatch];
  int32_t seq_len[kMaxBatch];
  int32_t tok_pre[kMaxBatch + 1];  // tok_pre[b] = sum of seq_len[0..b)
  int64_t tokens;            // T = tok_pre[B]
  int32_t max_len;
  int32_t min_len;           // shortest non-empty range (0 when all are empty)
  int32_t active;            // sequences with a non-empty range
  int64_t lkv_chunks;        // chunks of one (layer, K|V) slab: H * T * C
  int64_t bytes;             // staging bytes: 2 * (l1 - l0) * lkv_chunks * 16
  void* k;                   // device-visible K / V bases
  void* v;
  bool host_side;            // the staging bytes are in (mapped) host memory
};

// Re-targets `p` to the layer sub-range [la, lb) (inside [p.l0, p.l1)).
inline void restrict_layers(Plan& p, int32_t la, int32_t lb) {
  p.l0 = la;
  p.l1 = lb;
  p.bytes = 2 * (int64_t)(lb - la) * p.lkv_chunks * 16;
}

// Bytes of one layer's slab of the staging buffer.
inline int64_t layer_slab_bytes(const Plan& p) { return 2 * p.lkv_chunks * 16; }

enum Variant { kAuto = 0, kFlat = 1, kTile = 2, kToken = 3 };

// Kernel choice of kAuto for a pack (pack = true) or an unpack.
int auto_kind(const Plan& p, bool pack);
// For ragged ranges: whether the tile kernel beats the flat kernel.
bool auto_uses_tile(const Plan& p, bool pack);
// Whether the tile kernel handles this geometry (C <= 64).
bool tile_supported(const Plan& p);
// Whether the token kernel handles these ranges (every non-empty range the
// same length; fewer than 2^31 staging chunks).
bool token_supported(const Plan& p);

// `stg` is the device-visible address of the staging bytes (device memory or
// mapped pinned host memory).  Both return cudaSuccess without launching
// when the plan moves nothing.
cudaError_t launch_pack(const Plan& p, void* stg, cudaStream_t stream, int variant);
cudaError_t launch_unpack(const Plan& p, const void* stg, cudaStream_t stream, int variant);

// One record of a log: layers [l0, l1) and per-sequence token ranges
// [start[b], end[b]) (B entries each, validated), whose staging bytes follow
// the previous record's in the source buffer.
struct RecordRanges {
  int32_t l0, l1;
  const int32_t* start;
  const int32_t* end;
};

// How many of recs[0, n), from the first, one launch_unpack_records call
// takes: consecutive records whose writes to the cache are pairwise disjoint
// and whose range tables fit in the kernel parameters (at least 1 for n > 0).
int records_per_launch(const Plan& cache, const RecordRanges* recs, int n);

// Unpacks recs[0, n) (n at most records_per_launch) from `src` into the cache
// of `cache` (its k, v, geometry, l1 covering every record, host_side) in one
// launch.
cudaError_t launch_unpack_records(const Plan& cache, const RecordRanges* recs, int n,
                                  const void* src, cudaStream_t stream);

// How many of recs[0, n), from the first, form a run that one
// launch_unpack_run call can take: records over the same layers and the same
// non-empty sequences, each one token per sequence, the token of record k
// being k after the first record's (1 when recs[0] is not such a record, or
// the geometry is beyond the tile kernel).  The records must lie back to back
// in the source.
int run_length(const Plan& cache, const RecordRanges* recs, int n);
// The fewest records of a run worth a launch_unpack_run (a quarter of the tile
// kernel's token block); shorter runs go to the record kernel.
int run_min_records(const Plan& cache);
// The most records of a run one launch_unpack_run call takes (its tile count
// stays below 2^31).
int run_max_records(const Plan& cache, const RecordRanges& first);
// Unpacks n records of a run that starts with `first` (n at most run_length
// and run_max_records) from `src` in one launch: the tile kernel's unpack,
// each tile TB consecutive records of one (layer, K|V, sequence, head).
cudaError_t launch_unpack_run(const Plan& cache, const RecordRanges& first, int n,
                              const void* src, cudaStream_t stream);

// Whether this library was built with device-side bounds checks, and the
// first out-of-bounds access they recorded since the last call (0 if none;
// the record is cleared).  Synchronous.
bool checked_build();
cudaError_t read_fault(uint64_t* out);

}  // namespace dv
