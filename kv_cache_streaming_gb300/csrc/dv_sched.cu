// libdv C ABI, part 3: the two schedulers over the replica: microbatch
// swapping through two device caches (the swapper) and decode deltas streamed
// beside the compute (the delta streamer).
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "dv_host.h"

using dv::cuda_fail;
using dv::fail;
using dv::plan_ranges;
using dv::resolve;
using dv::resolve_cache;
using dv::Trace;

extern "C" {

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
