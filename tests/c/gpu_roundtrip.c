/* A C program using libdv with cudaMalloc'd buffers: fills a cache with
 * known bytes, packs a ragged range set into device staging, packs it again
 * straight into pinned host memory, unpacks the staging into a zeroed cache,
 * and checks (1) both packs agree, (2) every byte of the selected slices came
 * back and every other byte stayed zero, (3) the first staging record is the
 * K row of token s_0 of (layer 0, sequence 0, head 0) read through the layout.
 * Then the same bytes go out layer by layer through a streamer and come back
 * through a fetcher, and a replica (snapshot + one decode token) is restored
 * record-batched and pipelined through the fetcher, and unpacked from the
 * mapped arena by dv_kv_unpack_records.  Decode deltas are streamed on a side
 * stream (dv_delta_streamer), and the two replicas go through two caches
 * (dv_swapper).  Exit status 0 when every check holds. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dv.h"

#define L 3
#define B 4
#define H 2
#define D 64
#define S 40
#define P 2
#define X (16 / P)

static int failures = 0;
#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

/* Number of bytes of the device cache (yk, yv) that differ from hk / hv on
 * tokens [lo_b, hi_b) of every sequence and from zero elsewhere. */
static int check_cache(const void* yk, const void* yv, const uint16_t* hk, const uint16_t* hv,
                       const int32_t* lo, const int32_t* hi, size_t n) {
  uint16_t* gk = (uint16_t*)malloc(n * P);
  uint16_t* gv = (uint16_t*)malloc(n * P);
  cudaMemcpy(gk, yk, n * P, cudaMemcpyDeviceToHost);
  cudaMemcpy(gv, yv, n * P, cudaMemcpyDeviceToHost);
  int bad = 0;
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int t = 0; t < S; ++t)
          for (int d = 0; d < D; ++d) {
            const size_t ki = (size_t)l * B * H * D * S +
                              ((((size_t)b * H + h) * (D / X) + d / X) * S + t) * X + d % X;
            const size_t vi = (size_t)l * B * H * D * S + (((size_t)b * H + h) * S + t) * D + d;
            const int sel = t >= lo[b] && t < hi[b];
            if (gk[ki] != (sel ? hk[ki] : 0) || gv[vi] != (sel ? hv[vi] : 0)) ++bad;
          }
  free(gk);
  free(gv);
  return bad;
}

int main(void) {
  const size_t n = (size_t)L * B * H * D * S; /* elements per tensor */
  uint16_t* hk = (uint16_t*)malloc(n * P);
  uint16_t* hv = (uint16_t*)malloc(n * P);
  for (size_t i = 0; i < n; ++i) {
    hk[i] = (uint16_t)(i * 2654435761u >> 7);
    hv[i] = (uint16_t)(i * 40503u + 17u);
  }
  void *dk, *dv, *zk, *zv, *stg;
  int32_t s[B] = {0, 5, 17, 40}, e[B] = {33, 6, 40, 40}; /* the last range is empty */
  dv_cache c = {L, B, H, D, S, P, 0, NULL, NULL};
  size_t bytes = 0;
  CHECK(dv_staging_bytes(&c, 0, L, s, e, &bytes) == DV_OK);
  CHECK(cudaMalloc(&dk, n * P) == cudaSuccess && cudaMalloc(&dv, n * P) == cudaSuccess);
  CHECK(cudaMalloc(&zk, n * P) == cudaSuccess && cudaMalloc(&zv, n * P) == cudaSuccess);
  CHECK(cudaMalloc(&stg, bytes) == cudaSuccess);
  uint8_t* host = NULL;
  CHECK(cudaHostAlloc((void**)&host, bytes, cudaHostAllocDefault) == cudaSuccess);
  cudaMemcpy(dk, hk, n * P, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, hv, n * P, cudaMemcpyHostToDevice);
  cudaMemset(zk, 0, n * P);
  cudaMemset(zv, 0, n * P);
  c.k_base = dk;
  c.v_base = dv;
  CHECK(dv_kv_pack(&c, 0, L, s, e, stg, bytes, NULL) == DV_OK);
  CHECK(dv_kv_pack(&c, 0, L, s, e, host, bytes, NULL) == DV_OK);
  dv_cache z = c;
  z.k_base = zk;
  z.v_base = zv;
  CHECK(dv_kv_unpack(&z, 0, L, s, e, stg, bytes, NULL) == DV_OK);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  uint8_t* hs = (uint8_t*)malloc(bytes);
  cudaMemcpy(hs, stg, bytes, cudaMemcpyDeviceToHost);
  CHECK(memcmp(hs, host, bytes) == 0);
  /* record 0: K of (layer 0, sequence 0, head 0, token s_0), d = 0..D-1 */
  const uint16_t* rec = (const uint16_t*)hs;
  for (int d = 0; d < D; ++d)
    CHECK(rec[d] == hk[((size_t)(d / X) * S + s[0]) * X + d % X]);
  uint16_t* bk = (uint16_t*)malloc(n * P);
  uint16_t* bv = (uint16_t*)malloc(n * P);
  cudaMemcpy(bk, zk, n * P, cudaMemcpyDeviceToHost);
  cudaMemcpy(bv, zv, n * P, cudaMemcpyDeviceToHost);
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h)
        for (int t = 0; t < S; ++t)
          for (int d = 0; d < D; ++d) {
            const size_t ki = (size_t)l * B * H * D * S +
                              ((((size_t)b * H + h) * (D / X) + d / X) * S + t) * X + d % X;
            const size_t vi = (size_t)l * B * H * D * S + (((size_t)b * H + h) * S + t) * D + d;
            const int sel = t >= s[b] && t < e[b];
            if (bk[ki] != (sel ? hk[ki] : 0) || bv[vi] != (sel ? hv[vi] : 0)) ++failures;
          }

  /* Layer by layer from C: the streamer copies each layer's slab out to pinned
   * host memory, the fetcher copies it back into another zeroed cache; the
   * bytes out equal one pack, the cache back equals the unpack above. */
  void *slot[4], *yk, *yv;
  const size_t slab = bytes / L;
  for (int i = 0; i < 4; ++i) CHECK(cudaMalloc(&slot[i], slab) == cudaSuccess);
  CHECK(cudaMalloc(&yk, n * P) == cudaSuccess && cudaMalloc(&yv, n * P) == cudaSuccess);
  cudaMemset(yk, 0, n * P);
  cudaMemset(yv, 0, n * P);
  /* The host side from dv_host_alloc: pinned, mapped, on huge pages where the
   * kernel gives them. */
  uint8_t* out = NULL;
  CHECK(dv_host_alloc(bytes, (void**)&out) == DV_OK && out != NULL);
  CHECK(((uintptr_t)out & 15) == 0);
  cudaStream_t ps, cs, fc, fu;
  cudaStreamCreate(&ps);
  cudaStreamCreate(&cs);
  cudaStreamCreate(&fc);
  cudaStreamCreate(&fu);
  cudaEvent_t out_done;
  cudaEventCreateWithFlags(&out_done, cudaEventDisableTiming);
  dv_streamer* st = NULL;
  dv_fetcher* ft = NULL;
  CHECK(dv_streamer_create(&st, slot[0], slot[1], slab, ps, cs) == DV_OK);
  CHECK(dv_fetcher_create(&ft, slot[2], slot[3], slab, fc, fu) == DV_OK);
  dv_cache y = c;
  y.k_base = yk;
  y.v_base = yv;
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  for (int l = 0; l < L; ++l) {
    CHECK(dv_stream_layer(st, &c, l, s, e, out, bytes, 0) == DV_OK);
    cudaEventRecord(out_done, cs);         /* layer l is in host memory ... */
    cudaStreamWaitEvent(fc, out_done, 0);  /* ... before it is fetched */
    CHECK(dv_fetch_layer(ft, &y, l, s, e, out, bytes, 0) == DV_OK);
  }
  CHECK(dv_streamer_wait(st) == DV_OK && dv_fetcher_wait(ft) == DV_OK);
  CHECK(memcmp(out, host, bytes) == 0);
  uint16_t* yk_h = (uint16_t*)malloc(n * P);
  uint16_t* yv_h = (uint16_t*)malloc(n * P);
  cudaMemcpy(yk_h, yk, n * P, cudaMemcpyDeviceToHost);
  cudaMemcpy(yv_h, yv, n * P, cudaMemcpyDeviceToHost);
  CHECK(memcmp(yk_h, bk, n * P) == 0 && memcmp(yv_h, bv, n * P) == 0);

  /* A replica of the ranges (snapshot) and one decode token after each range
   * (where it fits), restored record-batched and pipelined through the
   * fetcher into zeroed caches: both give the selected slices of [s, e + 1).
   * Then the same log appended again through the streamer (one layer per
   * slot: the snapshot in L groups), byte for byte the same arena, restored
   * record-batched. */
  int32_t e1[B];
  for (int b = 0; b < B; ++b) e1[b] = e[b] < S ? e[b] + 1 : e[b];
  size_t delta = 0;
  CHECK(dv_staging_bytes(&c, 0, L, e, e1, &delta) == DV_OK);
  uint8_t* arena = NULL;
  CHECK(cudaHostAlloc((void**)&arena, bytes + delta, cudaHostAllocMapped) == cudaSuccess);
  dv_replica* rep = NULL;
  CHECK(dv_replica_create(&rep, arena, bytes + delta, B) == DV_OK);
  CHECK(dv_replica_append(rep, &c, 0, L, s, e, 0, NULL, 0, NULL) == DV_OK);
  CHECK(dv_replica_append(rep, &c, 0, L, e, e1, 1, NULL, 0, NULL) == DV_OK);
  for (int mode = 0; mode < 3; ++mode) {
    if (mode == 2) {
      CHECK(cudaDeviceSynchronize() == cudaSuccess);
      uint8_t* first = (uint8_t*)malloc(bytes + delta);
      memcpy(first, arena, bytes + delta);
      memset(arena, 0, bytes + delta);
      CHECK(dv_replica_truncate(rep, 0) == DV_OK);
      CHECK(dv_replica_append_streamed(rep, st, &c, 0, L, s, e, 0) == DV_OK);
      CHECK(dv_replica_append_streamed(rep, st, &c, 0, L, e, e1, 1) == DV_OK);
      CHECK(dv_streamer_wait(st) == DV_OK);
      CHECK(memcmp(first, arena, bytes + delta) == 0);
      free(first);
    }
    cudaMemset(yk, 0, n * P);
    cudaMemset(yv, 0, n * P);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    if (mode != 1) {
      CHECK(dv_replica_restore_batched(rep, &y, -1, NULL, 0, NULL) == DV_OK);
    } else {
      CHECK(dv_replica_restore_fetched(rep, &y, -1, ft) == DV_OK);
      CHECK(dv_fetcher_wait(ft) == DV_OK);
    }
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    cudaMemcpy(yk_h, yk, n * P, cudaMemcpyDeviceToHost);
    cudaMemcpy(yv_h, yv, n * P, cudaMemcpyDeviceToHost);
    int bad = 0;
    for (int l = 0; l < L; ++l)
      for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
          for (int t = 0; t < S; ++t)
            for (int d = 0; d < D; ++d) {
              const size_t ki = (size_t)l * B * H * D * S +
                                ((((size_t)b * H + h) * (D / X) + d / X) * S + t) * X + d % X;
              const size_t vi = (size_t)l * B * H * D * S + (((size_t)b * H + h) * S + t) * D + d;
              const int sel = t >= s[b] && t < e1[b];
              if (yk_h[ki] != (sel ? hk[ki] : 0) || yv_h[vi] != (sel ? hv[vi] : 0)) ++bad;
            }
    CHECK(bad == 0);
  }

  /* The same log unpacked by dv_kv_unpack_records straight from the mapped
   * arena (its device-visible address), records back to back. */
  {
    int32_t layers[4] = {0, L, 0, L};
    int32_t ranges[4 * B];
    memcpy(ranges, s, sizeof s);
    memcpy(ranges + B, e, sizeof e);
    memcpy(ranges + 2 * B, e, sizeof e);
    memcpy(ranges + 3 * B, e1, sizeof e1);
    void* arena_dev = NULL;
    CHECK(cudaHostGetDevicePointer(&arena_dev, arena, 0) == cudaSuccess);
    cudaMemset(yk, 0, n * P);
    cudaMemset(yv, 0, n * P);
    CHECK(dv_kv_unpack_records(&y, 2, layers, ranges, arena_dev, bytes + delta, NULL) == DV_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(check_cache(yk, yv, hk, hv, s, e1, n) == 0);
  }

  /* Decode deltas streamed on a side stream (dv_delta_streamer) after a
   * snapshot of [s, e): two more tokens; the replica then restores to
   * [s, e + 2) (where the tokens fit). */
  {
    int32_t lo[B], hi[B];
    for (int b = 0; b < B; ++b) hi[b] = e[b];
    const size_t cap = bytes + 2 * delta;
    uint8_t* ar2 = NULL;
    CHECK(cudaHostAlloc((void**)&ar2, cap, cudaHostAllocMapped) == cudaSuccess);
    dv_replica* r2 = NULL;
    CHECK(dv_replica_create(&r2, ar2, cap, B) == DV_OK);
    CHECK(dv_replica_append(r2, &c, 0, L, s, e, 0, NULL, 0, ps) == DV_OK);
    dv_delta_streamer* ds = NULL;
    CHECK(dv_delta_streamer_create(&ds, r2, ps, cs, NULL, 0) == DV_OK);
    for (int k = 0; k < 2; ++k) {
      for (int b = 0; b < B; ++b) {
        lo[b] = hi[b];
        hi[b] = hi[b] < S ? hi[b] + 1 : hi[b];
      }
      CHECK(dv_delta_stream(ds, &c, 0, L, lo, hi, 1 + k) == DV_OK);
    }
    CHECK(dv_delta_streamer_join(ds) == DV_OK && dv_delta_streamer_wait(ds) == DV_OK);
    cudaMemset(yk, 0, n * P);
    cudaMemset(yv, 0, n * P);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(dv_replica_restore_batched(r2, &y, -1, NULL, 0, NULL) == DV_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(check_cache(yk, yv, hk, hv, s, hi, n) == 0);

    /* Two microbatches (rep: [s, e + 1), r2: [s, e + 2)) through two caches
     * (dv_swapper): each acquire hands out a cache holding its replica. */
    void *wk, *wv;
    CHECK(cudaMalloc(&wk, n * P) == cudaSuccess && cudaMalloc(&wv, n * P) == cudaSuccess);
    cudaMemset(wk, 0, n * P);
    cudaMemset(wv, 0, n * P);
    cudaMemset(yk, 0, n * P);
    cudaMemset(yv, 0, n * P);
    dv_cache w = c;
    w.k_base = wk;
    w.v_base = wv;
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    dv_swapper* sw = NULL;
    CHECK(dv_swapper_create(&sw, &y, &w, ft, ps, cs) == DV_OK);
    int32_t none[B];
    memcpy(none, e, sizeof e);
    dv_replica* mb[2] = {rep, r2};
    const int32_t* want_hi[2] = {e1, hi};
    for (int i = 0; i < 4; ++i) {
      int32_t slot = -1;
      CHECK(dv_swapper_acquire(sw, mb[i % 2], &slot) == DV_OK);
      CHECK(dv_swapper_prefetch(sw, mb[(i + 1) % 2]) == DV_OK);
      CHECK(cudaStreamSynchronize(ps) == cudaSuccess);
      CHECK(check_cache(slot == 0 ? yk : wk, slot == 0 ? yv : wv, hk, hv, s, want_hi[i % 2], n) ==
            0);
      CHECK(dv_swapper_release(sw, mb[i % 2], 0, L, none, none, 10 + i) == DV_OK);
    }
    CHECK(dv_swapper_wait(sw) == DV_OK);
    dv_swapper_destroy(sw);
    dv_delta_streamer_destroy(ds);
    dv_replica_destroy(r2);
  }

  dv_replica_destroy(rep);
  dv_fetcher_destroy(ft);
  dv_streamer_destroy(st);
  cudaEventDestroy(out_done);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  CHECK(dv_host_free(out) == DV_OK);
  CHECK(dv_host_free(out) == DV_ERR_INVALID_ARG); /* already freed */
  if (failures == 0) printf("gpu_roundtrip: all checks passed\n");
  return failures == 0 ? 0 : 1;
}
