/*
 * dv.h — C ABI of libdv, the KV-cache buffered copy for one GB300 GPU.
 *
 * The operations follow "DejaVu: KV-Cache Streaming for Fast, Fault-Tolerant
 * Generative LLM Serving" (Strati et al., ICML 2024):
 *
 *   dv_kv_pack       Table 1 "gather" and §3 "Buffered copies" (Fig 7a): the
 *                    many small, non-contiguous K/V slices of a cache that is
 *                    preallocated at the maximum sequence length (Fig 6) are
 *                    gathered into one contiguous buffer in GPU memory.
 *   dv_kv_unpack     Table 1 "scatter" / stream_in: the inverse, a contiguous
 *                    buffer split back into the same slices.
 *   dv_swap_out/in   §3 "Microbatch swapping" (Fig 9): the used part of a
 *                    microbatch's cache moved to pinned host memory and back;
 *                    Table 1 flush/fetch are the contiguous copies inside.
 *   dv_stream_layer  §3 "Layer-by-layer prompt cache streaming" (Fig 7b): the
 *                    pack of layer l+1 overlaps the device-to-host copy of
 *                    layer l, on two streams ordered by events.
 *   dv_fetch_layer   the receiving side of that stream (Table 1 stream_in).
 *   dv_replica_*     §3 "Fault detection and recovery" (Fig 10) on one GPU:
 *                    per-step decode deltas (§3 "Token computation and
 *                    streaming parallelization", Fig 7c) appended to a
 *                    host-side replica, and the restore of a cache from it;
 *                    dv_replica_append_streamed appends through a layer
 *                    streamer's two slots (Fig 7b streaming into Fig 10).
 *   dv_kv_unpack_records  the scatter of a whole log of records at once.
 *   dv_swapper_*     §3 "Microbatch swapping" (Fig 9): N microbatches
 *                    through two device caches, the next swapped in while
 *                    one computes, each step's update swapped out after it.
 *   dv_delta_*       §3 "Token computation and streaming parallelization"
 *                    (Fig 7c): each step's delta streamed on a side stream
 *                    while the next step computes.
 *   dv_host_alloc    pinned, mapped host memory on huge pages for replica
 *                    arenas and swap buffers (the host side of every
 *                    transfer above).
 *
 * Cache layout (the FasterTransformer-style layout the pages build on).  Per
 * layer, with x = 16 / elem_bytes elements per 16-byte chunk:
 *   K: [batch][num_heads][head_dim / x][max_seq][x]   (x-interleaved keys)
 *   V: [batch][num_heads][max_seq][head_dim]
 * Layer l starts at element l * layer_stride_elems of k_base (and v_base).
 *
 * Staging (packed) order, the same for every call:
 *   [layer l0..l1)[K, then V][sequence b][head h][token t in [s_b, e_b)][d]
 * with d in logical order (0..head_dim-1).  The size is
 *   2 * (l1 - l0) * num_heads * head_dim * elem_bytes * sum_b (e_b - s_b)
 * bytes; for a full cache (all layers, all ranges [0, max_seq)) this is the
 * capacity formula 2*B*S*H*D*P*N of the KV-cache capacity page.  Each
 * layer's slab is contiguous, so packing layers one at a time lays down the
 * same bytes as one pack of all of them.
 *
 * Conventions shared by every call:
 *  - Ranges: seq_start / seq_end are HOST arrays of `batch` int32 values,
 *    read during the call only; 0 <= s_b <= e_b <= max_seq; an empty range is
 *    legal (a finished sequence).  Layer range: 0 <= l0 <= l1 <= num_layers.
 *  - Ownership: the caller allocates every buffer.  The library allocates no
 *    device or host memory except its small handles (streamer, fetcher,
 *    replica, swapper, delta streamer), one copy stream per CUDA context for
 *    staged swaps, and the pinned host memory dv_host_alloc returns when
 *    asked (dv_swap_out_noalloc's buffer is static device memory).
 *  - Memory kinds: k_base / v_base and `staging` are device memory of the
 *    current device.  A pack destination or unpack source may be device
 *    memory or pinned (page-locked, mapped) host memory; for host memory the
 *    kernel reads or writes it directly over the host link (zero copy) with a
 *    small grid (32 CTAs by default for the tile kernel, 64 for the kernels
 *    that look up every chunk's address, 128 for the one-chunk-per-thread
 *    token kernel; the environment variable DV_HOST_CTAS overrides the base
 *    32, 0 for none), enough for the link, so that other kernels keep the
 *    rest of the GPU.
 *  - Alignment: k_base, v_base, buffers and layer_stride_elems * elem_bytes
 *    must be multiples of 16 bytes (DV_ERR_MISALIGNED); head_dim must be a
 *    multiple of x (DV_ERR_UNSUPPORTED).  batch <= DV_MAX_BATCH.
 *  - Asynchrony: every call validates all arguments first and enqueues
 *    nothing when it fails.  On success the work is enqueued on the given
 *    stream(s) and the call returns; buffers must stay alive and unmodified
 *    until the stream reaches that point.  A launch failure returns
 *    DV_ERR_CUDA.  No call blocks except dv_streamer_wait, dv_fetcher_wait
 *    and the synchronous helpers marked as such.
 *  - Tracing: every call that enqueues work pushes an NVTX range named
 *    after the call for its duration (nested when one call makes another),
 *    so NVTX-aware profilers show each call with the launches and copies it
 *    enqueued; without such a profiler the ranges cost nothing.
 *  - Errors: every call returns a dv_status; dv_last_error() gives a
 *    message for the calling thread's most recent failure.
 *  - Threads: calls on distinct handles may run concurrently; a streamer,
 *    fetcher or replica handle must not be used by two threads at once.
 */
#ifndef DV_H_
#define DV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DV_ABI_VERSION 1
#define DV_MAX_BATCH 1024

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default
 * stream. */
typedef struct CUstream_st* dv_stream;

typedef enum {
  DV_OK = 0,
  DV_ERR_INVALID_ARG = 1,      /* null pointer, bad geometry, wrong memory kind */
  DV_ERR_RANGE = 2,            /* a layer or token range outside the cache */
  DV_ERR_BUFFER_TOO_SMALL = 3, /* destination / source / staging too small */
  DV_ERR_MISALIGNED = 4,       /* a pointer or stride not 16-byte aligned */
  DV_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
  DV_ERR_TIMEOUT = 6,          /* reserved for bounded waits */
  DV_ERR_UNSUPPORTED = 7       /* a geometry the library does not handle */
} dv_status;

/* Cache geometry and base pointers; owned by the caller. */
typedef struct {
  int32_t num_layers;         /* resident layers N */
  int32_t batch;              /* sequences B */
  int32_t num_heads;          /* H */
  int32_t head_dim;           /* D */
  int32_t max_seq;            /* S, token slots per sequence */
  int32_t elem_bytes;         /* P: 1, 2 (fp16 / bf16) or 4 */
  int64_t layer_stride_elems; /* 0 = batch*num_heads*head_dim*max_seq */
  void* k_base;               /* device pointer, K of layer 0 */
  void* v_base;               /* device pointer, V of layer 0 */
} dv_cache;

/* Kernel choice for dv_kv_pack_variant / dv_kv_unpack_variant (testing and
 * tuning; the plain calls use DV_VARIANT_AUTO). */
typedef enum {
  DV_VARIANT_AUTO = 0, /* equal-length ranges (e.g. one-token decode deltas): the
                          token kernel below 640 16-byte chunks per head and range
                          (80 tokens at head_dim 64, fp16), the tile kernel above;
                          ragged ranges: the flat kernel below a mean of 512 chunks,
                          the tile kernel above.  With grouped tiles (8 or 16 chunks
                          per token: head_dim 64 / 128 in 2-byte elements), for
                          transfers of at least 4 MiB, the tile kernel from fewer
                          chunks: the unpack of ragged ranges at any
                          length (8 chunks per token) or from 64 (16), of equal ranges
                          of more than one token from 32 (8) or 128 (16); the pack of
                          ragged ranges from 300 (8) or 64 (16), of equal ranges from
                          512 (16) */
  DV_VARIANT_FLAT = 1, /* staging order, each warp a window of 128 chunks */
  DV_VARIANT_TILE = 2, /* token tiles; K transposed through shared memory; at 8 or
                          16 chunks per token, ranges of at most half the token block
                          go several heads to a tile (a second launch) */
  DV_VARIANT_TOKEN = 3 /* every non-empty range equally long: one chunk per thread */
} dv_variant;

int32_t dv_abi_version(void);
const char* dv_status_string(dv_status status);
/* Message for the calling thread's most recent failed call ("" if none). */
const char* dv_last_error(void);

/* Debugging.  A checked build of the library (built with DV_CHECKED=1, file
 * libdv_checked.so) checks every global access of its kernels against the
 * extents the host validated; an access outside them is skipped and the
 * first one is recorded (nothing traps).  dv_debug_fault waits for the device,
 * returns that record in *fault (0: none; else bit 63 set, bits 56..62 the
 * kernel site, bits 0..55 the chunk index relative to the buffer) and clears
 * it.  In the regular build it returns DV_ERR_UNSUPPORTED. */
dv_status dv_debug_fault(uint64_t* fault);

/* Bytes from `ptr` to the end of the CUDA allocation that holds it, as the
 * driver reports it; every call checks the buffers it is given against this
 * extent when the driver knows it.  DV_ERR_UNSUPPORTED when the driver cannot
 * tell (then calls rely on the sizes the caller passes). */
dv_status dv_allocation_extent(const void* ptr, size_t* bytes_after);

/* ---- pinned host memory (the host side of swaps and replicas) ---------- */

/* Allocates `bytes` of host memory and registers it with CUDA as pinned,
 * mapped and portable memory (cudaHostRegister), for use wherever a call
 * takes pinned host memory: a replica's arena, a swap's host buffer, a
 * streamer's destination.  The memory is anonymous and zeroed, its start is
 * aligned to the kernel's transparent-huge-page size, and the huge-page-
 * aligned part of it is marked for huge pages (madvise; the kernel may
 * decline).  Why: on a GB300 host with 64 KiB base pages, copy-engine passes
 * over tens of GB of pinned memory made of base pages periodically run at
 * about half the link rate, where the same passes over huge pages run at the
 * full rate every time.  Synchronous; safe from any thread.  Needs a CUDA
 * device (the registration makes the current device's primary context
 * current if the thread has none).  Errors: DV_ERR_INVALID_ARG (out is NULL,
 * bytes is 0, no host memory), DV_ERR_CUDA (the registration failed; nothing
 * stays allocated).  No counterpart on the pages: they state only that the
 * host copies live in pinned CPU memory. */
dv_status dv_host_alloc(size_t bytes, void** out);

/* Unregisters and unmaps memory from dv_host_alloc (NULL: nothing to do);
 * synchronous.
 * The caller ensures that no enqueued work still reads or writes it.
 * DV_ERR_INVALID_ARG for a pointer dv_host_alloc did not return (or already
 * freed); DV_ERR_CUDA if the unregistration fails (the memory is unmapped
 * all the same). */
dv_status dv_host_free(void* ptr);

/* Bytes the staging buffer of (l0, l1, ranges) takes (see the size formula
 * above).  Host only; enqueues nothing.  Pointers in `cache` are not read. */
dv_status dv_staging_bytes(const dv_cache* cache, int32_t l0, int32_t l1,
                           const int32_t* seq_start, const int32_t* seq_end, size_t* bytes);

/* Gather (Table 1; Fig 7a).  Writes the staging bytes of (l0, l1, ranges)
 * to `dst` (device memory, or pinned host memory written directly).
 * DV_ERR_BUFFER_TOO_SMALL if dst_bytes is less than dv_staging_bytes.
 * dst may be NULL when that size is 0. */
dv_status dv_kv_pack(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                     const int32_t* seq_end, void* dst, size_t dst_bytes, dv_stream stream);

/* Scatter (Table 1).  Reads staging bytes from `src` (device memory or
 * pinned host memory) and writes exactly the selected K/V slices; every other
 * byte of the cache is left as it was. */
dv_status dv_kv_unpack(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                       const int32_t* seq_end, const void* src, size_t src_bytes,
                       dv_stream stream);

dv_status dv_kv_pack_variant(const dv_cache* cache, int32_t l0, int32_t l1,
                             const int32_t* seq_start, const int32_t* seq_end, void* dst,
                             size_t dst_bytes, dv_stream stream, int32_t variant);
dv_status dv_kv_unpack_variant(const dv_cache* cache, int32_t l0, int32_t l1,
                               const int32_t* seq_start, const int32_t* seq_end,
                               const void* src, size_t src_bytes, dv_stream stream,
                               int32_t variant);

/* Scatter of a log (Table 1 scatter, applied to many records at once; the
 * restore side of §3 "Microbatch swapping", Fig 9, and of the replication log
 * of "Fault detection and recovery", Fig 10): `src` holds num_records
 * staging buffers back to back, record i being the staging bytes of layers
 * [layers[2i], layers[2i+1]) and of the ranges at ranges + 2*batch*i
 * (batch starts, then batch ends, host memory, read during the call).  The
 * result is that of dv_kv_unpack of each record in order (a later record wins
 * where two write the same slice).  src: device memory or pinned, mapped host
 * memory of src_bytes (at least the records' total).  Records long enough for
 * the tile kernel are unpacked by themselves; runs of one-token records (the
 * decode deltas of consecutive steps over the same sequences: record k one
 * token further on than the one before; two records or more at head_dim 64
 * and 128 in 2-byte elements, a quarter of the token block otherwise) are
 * unpacked together, each K row's consecutive tokens written as one span; the
 * other records go in as few record-batched launches as the kernel parameters
 * allow.  Validates every
 * record before enqueuing anything. */
dv_status dv_kv_unpack_records(const dv_cache* cache, int32_t num_records,
                               const int32_t* layers, const int32_t* ranges, const void* src,
                               size_t src_bytes, dv_stream stream);

/* The naive transfer the pages measure buffered copies against (§5.1, Fig 11:
 * "many cudaMemcpy calls" for the small non-contiguous regions): the same bytes
 * as dv_kv_pack written to `dst` (device or pinned host memory) with one
 * cudaMemcpyAsync per contiguous V run and one cudaMemcpy2DAsync per K token
 * (when a range holds fewer tokens than C = head_dim*elem_bytes/16) or per K
 * chunk row (otherwise), and no kernel.  It exists to be timed against
 * dv_kv_pack plus one copy; *num_copies (may be NULL) receives the number of
 * copy calls it enqueued. */
dv_status dv_naive_gather(const dv_cache* cache, int32_t l0, int32_t l1,
                          const int32_t* seq_start, const int32_t* seq_end, void* dst,
                          size_t dst_bytes, dv_stream stream, int64_t* num_copies);

/* Swap-out (§3 microbatch swapping, Fig 9; Table 1 flush).  Leaves the
 * staging bytes of (l0, l1, ranges) in `host_dst` (pinned host memory,
 * host_bytes at least dv_staging_bytes).
 *  - staging == NULL: fused path, the pack kernel stores straight into
 *    host_dst over the host link (one launch, no device buffer).
 *  - staging != NULL: staged path, groups of whole layers are packed into
 *    `staging` (device, staging_bytes >= one layer's slab) and copied to
 *    the host with cudaMemcpyAsync.  When staging holds two layer slabs or
 *    more, it is used in two halves: the pack of one group (on `stream`)
 *    overlaps the copy of the other, which runs on a copy stream the library
 *    owns (one per CUDA context, made on the first such call there: make it
 *    outside a stream capture), ordered by events; the work is complete in
 *    `stream`'s order when it returns.  With room for one slab only,
 *    everything runs in order on `stream`.
 *  Should a launch or copy fail partway (DV_ERR_CUDA), the groups before it
 *  stay enqueued; validation failures enqueue nothing. */
dv_status dv_swap_out(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                      const int32_t* seq_end, void* host_dst, size_t host_bytes, void* staging,
                      size_t staging_bytes, dv_stream stream);

/* Swap-in (§3 microbatch swapping; Table 1 fetch + scatter).  The inverse of
 * dv_swap_out: host_src holds staging bytes; staging == NULL unpacks straight
 * from host memory, otherwise layer groups go host -> staging -> cache, in
 * two halves as for dv_swap_out (the copy of one group, on the library's copy
 * stream after the work enqueued on `stream` so far, overlaps the unpack of
 * the other on `stream`). */
dv_status dv_swap_in(const dv_cache* cache, int32_t l0, int32_t l1, const int32_t* seq_start,
                     const int32_t* seq_end, const void* host_src, size_t host_bytes,
                     void* staging, size_t staging_bytes, dv_stream stream);

/* ---- swap-out without allocation ------------------------------------------ */

/* Size of the device buffer built into libdv for dv_swap_out_noalloc. */
#define DV_NOALLOC_STAGING_BYTES 67108864 /* 64 MiB */

/* The paper has no counterpart to this call.  It is dv_swap_out on the
 * staged path, but the staging buffer is built into the library, so the
 * caller allocates nothing on the device.  It is meant for callers that
 * cannot call cudaMalloc: a host that embeds libdv but owns no device
 * allocator (it only receives the cache and host pointers from elsewhere), a
 * serving process whose device memory is owned entirely by another allocator
 * (a framework's caching allocator holding the whole budget, where an extra
 * cudaMalloc fails or fragments it), or a latency-critical loop that must not
 * take the device-wide synchronisation cudaMalloc can cause.
 *
 * Limits and behaviour:
 *  - The buffer is DV_NOALLOC_STAGING_BYTES (64 MiB) of device memory that
 *    every GPU loading libdv holds until the process exits.  Layers are
 *    packed into it in groups and copied to host_dst, as on dv_swap_out's
 *    staged path (in two halves when each holds a layer), so the whole swap
 *    may be larger; one layer of the ranges
 *    larger than 64 MiB is refused with DV_ERR_BUFFER_TOO_SMALL before
 *    anything is enqueued.
 *  - The first call in a CUDA context looks up the buffer's device address
 *    there (cudaGetSymbolAddress, with the context current) and keeps it for
 *    that context; a device reset or another context gets a lookup of its
 *    own.  Make the first call in each context before any stream capture
 *    (the staged path may also create its copy stream then).
 *  - All calls share the one buffer, which keeps the last call's bytes
 *    (nothing in it needs to start at zero: each group is packed in full
 *    before it is copied).  Calls whose work overlaps on the GPU (on
 *    different streams, or from different threads without ordering) race on
 *    it and corrupt each other's output: order them on one stream.
 *  - Arguments, validation and errors are those of dv_swap_out. */
dv_status dv_swap_out_noalloc(const dv_cache* cache, int32_t l0, int32_t l1,
                              const int32_t* seq_start, const int32_t* seq_end, void* host_dst,
                              size_t host_bytes, dv_stream stream);

/* ---- layer-by-layer streaming (§3, Fig 7b) ------------------------------ */

/* Owns two events per slot; borrows the slots and streams. */
typedef struct dv_streamer dv_streamer;

/* slot0 / slot1: device buffers of slot_bytes each (16-byte aligned), used
 * alternately.  Packs run on pack_stream, copies on copy_stream (two
 * different streams overlap the pack of layer l+1 with the copy of layer l;
 * one stream serialises them). */
dv_status dv_streamer_create(dv_streamer** out, void* slot0, void* slot1, size_t slot_bytes,
                             dv_stream pack_stream, dv_stream copy_stream);

/* Packs layer `layer` of the ranges into the next slot on the pack stream
 * (after the slot's previous copy has finished) and copies it, on the copy
 * stream, to host_dst + (layer - l0) * slab, where slab is this layer's
 * staging size: host_dst is the base of the buffer of the whole layer range
 * [l0, ...) streamed with the same ranges, so the layers land in the order
 * of one dv_kv_pack over that range.  host_dst_bytes is that buffer's size. */
dv_status dv_stream_layer(dv_streamer* streamer, const dv_cache* cache, int32_t layer,
                          const int32_t* seq_start, const int32_t* seq_end, void* host_dst,
                          size_t host_dst_bytes, int32_t l0);

/* Blocks the calling thread until every copy issued so far has finished. */
dv_status dv_streamer_wait(dv_streamer* streamer);

/* Releases the handle (its events are released once pending work ends). */
void dv_streamer_destroy(dv_streamer* streamer);

/* ---- layer-by-layer receive (§3, Fig 7b, the receiving side; Table 1
 * stream_in) ------------------------------------------------------------- */

/* The mirror image of dv_streamer: layer slabs come in from host memory
 * through two device slots and are unpacked into a cache as they arrive.
 * Owns two events per slot; borrows the slots and streams. */
typedef struct dv_fetcher dv_fetcher;

/* slot0 / slot1: device buffers of slot_bytes each (16-byte aligned), used
 * alternately.  Host-to-device copies run on copy_stream, unpacks on
 * unpack_stream (two different streams overlap the copy of layer l+1 with
 * the unpack of layer l; one stream serialises them). */
dv_status dv_fetcher_create(dv_fetcher** out, void* slot0, void* slot1, size_t slot_bytes,
                            dv_stream copy_stream, dv_stream unpack_stream);

/* Copies the slab of layer `layer` from host_src + (layer - l0) * slab, where
 * slab is this layer's staging size (the layout dv_stream_layer and one
 * dv_kv_pack over [l0, ...) produce with the same ranges), into the next
 * slot on the copy stream (after that slot's previous unpack has finished),
 * then unpacks it into `cache` on the unpack stream.  host_src: pinned host
 * memory (or device memory) of host_src_bytes.  The caller orders the copy
 * stream after whatever wrote host_src and the unpack stream after whatever
 * last used the cache's slices; an event recorded on the unpack stream after
 * the call marks the layer as present.  Errors as dv_stream_layer. */
dv_status dv_fetch_layer(dv_fetcher* fetcher, const dv_cache* cache, int32_t layer,
                         const int32_t* seq_start, const int32_t* seq_end, const void* host_src,
                         size_t host_src_bytes, int32_t l0);

/* Blocks the calling thread until every unpack issued so far has finished. */
dv_status dv_fetcher_wait(dv_fetcher* fetcher);

/* Releases the handle (its events are released once pending work ends). */
void dv_fetcher_destroy(dv_fetcher* fetcher);

/* ---- host-side replica of a cache (§3 state replication, Fig 10) -------- */

/* A log of records in a caller-owned pinned host arena.  Each record holds
 * the staging bytes of (l0, l1, ranges) and is tagged with a step number;
 * the first record is normally a snapshot of the used prefixes and the rest
 * one-token decode deltas. */
typedef struct dv_replica dv_replica;

dv_status dv_replica_create(dv_replica** out, void* host_arena, size_t arena_bytes,
                            int32_t batch);

/* Appends the staging bytes of (l0, l1, ranges) of `cache` as a record
 * tagged `step` (steps must not decrease), by dv_swap_out (fused when
 * staging is NULL).  DV_ERR_BUFFER_TOO_SMALL when the arena is full. */
dv_status dv_replica_append(dv_replica* replica, const dv_cache* cache, int32_t l0, int32_t l1,
                            const int32_t* seq_start, const int32_t* seq_end, int64_t step,
                            void* staging, size_t staging_bytes, dv_stream stream);

/* The append of dv_replica_append through a layer streamer (§3 "Layer-by-
 * layer prompt cache streaming", Fig 7b, streaming into the replica of Fig
 * 10): the record's staging bytes are packed into the streamer's next slot on
 * its pack stream, after that slot's previous copy, and copied into the arena
 * on its copy stream.  A record larger than a slot goes in groups of whole
 * layers, one group per slot, the slots taken in turn.  Unlike the staged
 * dv_replica_append, no stream waits for the copy: the pack of the next
 * record (or group) runs while the previous one is being copied.  The caller
 * orders the pack stream after the writes to the record's ranges; an event
 * recorded on the copy stream after the call marks the record in host
 * memory.  DV_ERR_BUFFER_TOO_SMALL, before anything is enqueued, when the
 * arena is full or when one layer of the record is larger than a slot;
 * otherwise the errors of dv_replica_append.  If a CUDA call fails part-way,
 * the record is not added (bytes already copied past the last record are
 * overwritten by the next append). */
dv_status dv_replica_append_streamed(dv_replica* replica, dv_streamer* streamer,
                                     const dv_cache* cache, int32_t l0, int32_t l1,
                                     const int32_t* seq_start, const int32_t* seq_end,
                                     int64_t step);

/* Unpacks every record with step < upto_step (all records if upto_step < 0),
 * in append order, into `cache` by dv_swap_in.  The cache must have the
 * geometry of the appended records. */
dv_status dv_replica_restore(const dv_replica* replica, const dv_cache* cache, int64_t upto_step,
                             void* staging, size_t staging_bytes, dv_stream stream);

/* The restore of dv_replica_restore with the records batched: every record
 * whose ranges are long enough for the tile kernel (normally the snapshot) is
 * unpacked by itself, as by dv_swap_in; the others (the decode deltas) go
 * into as few launches of one record-batched unpack kernel as its kernel
 * parameters allow (up to 128 records per launch; at batch 32, 72 records).
 * This is the restore of the pages' delta-only swapping: swap-in = snapshot +
 * every delta (§3 "Microbatch swapping", Fig 9, with the replication log of
 * "Fault detection and recovery", Fig 10), with one launch for the deltas
 * instead of one per step.  A launch takes consecutive records whose writes
 * to the cache are disjoint; where a record overwrites what an earlier record
 * of the run wrote, a new launch starts, so the result equals dv_replica_restore
 * (append order) for any log.  staging == NULL: the kernel reads the records
 * straight from the arena (mapped pinned memory).  Otherwise each launch's
 * records go to `staging` with one host-to-device copy first (consecutive
 * records up to staging_bytes; a record larger than staging_bytes is restored
 * by itself through dv_swap_in's layer groups).  Validates every record before
 * enqueuing anything; same errors as dv_replica_restore. */
dv_status dv_replica_restore_batched(const dv_replica* replica, const dv_cache* cache,
                                     int64_t upto_step, void* staging, size_t staging_bytes,
                                     dv_stream stream);

/* The restore of dv_replica_restore_batched with the host-to-device copies
 * pipelined through a fetcher (see dv_fetcher_create): the log is cut into
 * pieces of at most the fetcher's slot size (a record long enough for the
 * tile kernel, or larger than a slot, into groups of whole layers; the other
 * records into runs that one record-batched launch takes), and each piece is
 * copied into the fetcher's next free slot on its copy stream and unpacked on
 * its unpack stream, so the copy of piece i+1 overlaps the unpack of piece
 * i.  Same result as dv_replica_restore (append order).  The caller orders
 * the fetcher's streams after earlier work on the cache; an event recorded on
 * the unpack stream after the call marks the end of the restore.
 * DV_ERR_BUFFER_TOO_SMALL (before anything is enqueued) when a record that
 * goes by itself has a layer slab larger than a slot; otherwise the errors of
 * dv_replica_restore. */
dv_status dv_replica_restore_fetched(const dv_replica* replica, const dv_cache* cache,
                                     int64_t upto_step, dv_fetcher* fetcher);

/* The restore of dv_replica_restore_fetched limited to the records with
 * from_step <= step < upto_step (no upper limit when upto_step < 0), in append
 * order: a cache that already holds the earlier records catches up with the
 * later ones.  This keeps a standby cache current while the log grows, or lets
 * a restore start before the last record is appended (the caller orders the
 * fetcher's copy stream after the appends it restores).  No counterpart on
 * the pages beyond the recovery of Fig 10, which it performs in parts. */
dv_status dv_replica_restore_fetched_steps(const dv_replica* replica, const dv_cache* cache,
                                          int64_t from_step, int64_t upto_step,
                                          dv_fetcher* fetcher);

/* Drops every record with step >= step (the acknowledged prefix is kept);
 * their arena bytes are reused by the next appends.  Host-side only: copies
 * of dropped records still in flight are not waited for, so an append that
 * reuses their bytes must be ordered after them (the same stream, the same
 * streamer, or an event). */
dv_status dv_replica_truncate(dv_replica* replica, int64_t step);

dv_status dv_replica_info(const dv_replica* replica, int64_t* num_records, size_t* bytes_used);

void dv_replica_destroy(dv_replica* replica);

/* ---- microbatch swapping through two device caches (§3 "Microbatch
 * swapping", Fig 9) -------------------------------------------------------- */

/* N microbatches share two device caches of one geometry (the pages' 2*M of
 * GPU memory for a stage).  Each microbatch lives in host memory as a replica
 * (dv_replica: a snapshot of its prompt cache, then one record per decode
 * step).  While microbatch x computes in one cache, the next one, (x+1) % N,
 * is swapped in to the other cache, and the update of x's step is swapped
 * out after its compute: swap-in = the replica restored through a fetcher
 * (dv_replica_restore_fetched, on the fetcher's copy and unpack streams),
 * swap-out = the step's delta appended to the replica (dv_replica_append,
 * fused, on the swap stream).  A swap-in writes the microbatch's recorded
 * slices only; the rest of the cache keeps what an earlier microbatch left.
 *
 * Use, per step of microbatch x:  dv_swapper_acquire(x) -> the cache to
 * compute in;  dv_swapper_prefetch(next);  the step's kernels on the compute
 * stream;  dv_swapper_release(x, the slices the step wrote, step).  No call
 * blocks the host.  The caller orders earlier work on the two caches before
 * the first call.  A microbatch is known by its replica handle: destroy the
 * swapper before a replica it has seen, and do not truncate or append to a
 * replica outside the swapper while it sits in a cache (the cache would no
 * longer match it).  Borrows the caches, the fetcher and the streams; owns six
 * events.  Not for two threads at once. */
typedef struct dv_swapper dv_swapper;

dv_status dv_swapper_create(dv_swapper** out, const dv_cache* slot0, const dv_cache* slot1,
                            dv_fetcher* fetcher, dv_stream compute_stream, dv_stream swap_stream);

/* Makes microbatch `mb` resident for its next step.  If it was prefetched (or
 * is still in a cache from its last step), the compute stream waits for that
 * swap-in; otherwise it is swapped in now to the cache the previous step did
 * not use, and the compute stream waits for that.  *slot receives the cache
 * (0 or 1) that holds it.  DV_ERR_INVALID_ARG while another microbatch is
 * acquired and not released. */
dv_status dv_swapper_acquire(dv_swapper* sw, const dv_replica* mb, int32_t* slot);

/* Swaps microbatch `mb` in to the cache the current step does not use, on
 * the fetcher's streams, as soon as that cache's last step and swap-out are
 * done (no host wait).  A no-op when `mb` is already in a cache. */
dv_status dv_swapper_prefetch(dv_swapper* sw, const dv_replica* mb);

/* Ends the acquired microbatch's step: after everything enqueued so far on
 * the compute stream, the slices of (l0, l1, ranges) of its cache (the
 * token the step wrote) are appended to its replica as the record of `step`,
 * on the swap stream; the cache is free for a prefetch once that append has
 * read it.  Errors of dv_replica_append, checked before anything is
 * enqueued. */
dv_status dv_swapper_release(dv_swapper* sw, dv_replica* mb, int32_t l0, int32_t l1,
                             const int32_t* seq_start, const int32_t* seq_end, int64_t step);

/* Blocks the calling thread until every swap issued so far has finished. */
dv_status dv_swapper_wait(dv_swapper* sw);

void dv_swapper_destroy(dv_swapper* sw);

/* ---- decode deltas streamed beside the compute (§3 "Token computation and
 * streaming parallelization", Fig 7c) -------------------------------------- */

/* Streams each decode step's delta to a host replica on a side stream while
 * the compute stream goes on with the next step: the pages stream step i's
 * cache while step i+1 computes, with the GPU side on its own CUDA stream.
 * staging: NULL (the pack stores straight into the replica's pinned arena) or
 * a device buffer of at least one layer slab of a delta.  Borrows the replica,
 * the streams and the staging buffer; owns two events.  The calls can be
 * captured in a CUDA graph on the compute stream (the side stream joins and
 * leaves the capture through the events; call dv_delta_streamer_join before
 * the capture ends). */
typedef struct dv_delta_streamer dv_delta_streamer;

dv_status dv_delta_streamer_create(dv_delta_streamer** out, dv_replica* replica,
                                   dv_stream compute_stream, dv_stream side_stream,
                                   void* staging, size_t staging_bytes);

/* After everything enqueued so far on the compute stream (the step's writes),
 * the slices of (l0, l1, ranges) of `cache` are appended to the replica as the
 * record of `step`, on the side stream; the compute stream does not wait.
 * Errors of dv_replica_append, checked before anything is enqueued. */
dv_status dv_delta_stream(dv_delta_streamer* ds, const dv_cache* cache, int32_t l0, int32_t l1,
                          const int32_t* seq_start, const int32_t* seq_end, int64_t step);

/* Makes the compute stream wait for every delta streamed so far (before it
 * overwrites or frees streamed slices, or ends a graph capture). */
dv_status dv_delta_streamer_join(dv_delta_streamer* ds);

/* Blocks the calling thread until every delta streamed so far is in the
 * replica. */
dv_status dv_delta_streamer_wait(dv_delta_streamer* ds);

void dv_delta_streamer_destroy(dv_delta_streamer* ds);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* DV_H_ */
