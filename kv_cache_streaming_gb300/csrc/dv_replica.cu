// libdv C ABI, part 2: the host replica of decode deltas (a log of records in
// a pinned host arena) and its restores: record by record, batched (the log
// planned into runs and record batches), and pipelined through a fetcher; and
// the unpack of a caller's own record list.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "dv_host.h"

using dv::check_host;
using dv::cuda_fail;
using dv::fail;
using dv::fetch_piece;
using dv::plan_ranges;
using dv::Record;
using dv::resolve;
using dv::resolve_cache;
using dv::Trace;

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
//  - alone: records of at least kAloneMinBytes that the unpack gives the tile
//    kernel (normally a snapshot), or larger than a piece, unpacked by
//    themselves;
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

constexpr size_t kAloneMinBytes = (size_t)4 << 20;  // smallest record unpacked by itself

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
      // A record the unpack would give the tile kernel goes by itself, unless it
      // is small enough for its own launch to cost more than its share of a
      // record-kernel launch (64 ragged 0.16 MB records: 203 us alone, 68 us
      // batched; from 6 MB on the same either way).
      const bool tile = dv::auto_kind(q, false) == dv::kTile && rec.bytes >= kAloneMinBytes;
      const bool by_itself = tile || (piece && rec.bytes > piece);
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

// The checks every append makes before it plans anything.
dv_status check_append(const dv_replica* r, const dv_cache* cache, int64_t step) {
  if (!r) return fail(DV_ERR_INVALID_ARG, "replica is NULL");
  if (!cache) return fail(DV_ERR_INVALID_ARG, "cache is NULL");
  if (cache->batch != r->batch)
    return fail(DV_ERR_INVALID_ARG, "cache batch %d differs from the replica's %d", cache->batch,
                r->batch);
  if (!r->records.empty() && step < r->records.back().step)
    return fail(DV_ERR_INVALID_ARG, "step %lld is before the last record's %lld",
                (long long)step, (long long)r->records.back().step);
  return DV_OK;
}

// Adds the record of an append whose bytes were enqueued to r->arena + off.
dv_status add_record(dv_replica* r, int64_t step, int32_t l0, int32_t l1, size_t off,
                     size_t bytes, const int32_t* seq_start, const int32_t* seq_end) {
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

}  // namespace

extern "C" {

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
  dv_status st = check_append(r, cache, step);
  if (st != DV_OK) return st;
  size_t bytes = 0;
  if ((st = dv_staging_bytes(cache, l0, l1, seq_start, seq_end, &bytes)) != DV_OK) return st;
  const size_t off = r->used;  // records are multiples of 16 bytes
  if (off + bytes > r->arena_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "replica arena full: %zu + %zu > %zu bytes", off, bytes,
                r->arena_bytes);
  if (bytes > 0) {
    st = dv_swap_out(cache, l0, l1, seq_start, seq_end, r->arena + off, bytes, staging,
                     staging_bytes, stream);
    if (st != DV_OK) return st;
  }
  return add_record(r, step, l0, l1, off, bytes, seq_start, seq_end);
}

dv_status dv_replica_append_streamed(dv_replica* r, dv_streamer* streamer, const dv_cache* cache,
                                     int32_t l0, int32_t l1, const int32_t* seq_start,
                                     const int32_t* seq_end, int64_t step) {
  const Trace trace("dv_replica_append_streamed");
  dv_status st = check_append(r, cache, step);
  if (st != DV_OK) return st;
  if (!streamer) return fail(DV_ERR_INVALID_ARG, "streamer is NULL");
  dv::Plan p;
  if ((st = plan_ranges(cache, l0, l1, seq_start, seq_end, &p)) != DV_OK) return st;
  const size_t bytes = (size_t)p.bytes;
  const size_t off = r->used;
  if (off + bytes > r->arena_bytes)
    return fail(DV_ERR_BUFFER_TOO_SMALL, "replica arena full: %zu + %zu > %zu bytes", off, bytes,
                r->arena_bytes);
  if (bytes > 0) {
    // Whole layers per slot: the record goes in groups of layers, each group
    // a contiguous part of its staging bytes.
    const size_t slab = (size_t)dv::layer_slab_bytes(p);
    if (slab > streamer->slot_bytes)
      return fail(DV_ERR_BUFFER_TOO_SMALL, "a layer slab of %zu bytes exceeds the slots of %zu",
                  slab, streamer->slot_bytes);
    if ((st = resolve_cache(cache, &p)) != DV_OK) return st;
    const int32_t per = (int32_t)std::min<size_t>((size_t)(l1 - l0), streamer->slot_bytes / slab);
    for (int32_t la = l0; la < l1; la += per) {
      dv::Plan q = p;
      dv::restrict_layers(q, la, std::min(l1, la + per));
      const cudaError_t err = dv::stream_piece(streamer, q, r->arena + off + (la - l0) * slab);
      if (err != cudaSuccess) return cuda_fail(err, "append_streamed");
    }
  }
  return add_record(r, step, l0, l1, off, bytes, seq_start, seq_end);
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

}  // extern "C"
