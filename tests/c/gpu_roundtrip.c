/* A C program using libdv with cudaMalloc'd buffers: fills a cache with
 * known bytes, packs a ragged range set into device staging, packs it again
 * straight into pinned host memory, unpacks the staging into a zeroed cache,
 * and checks (1) both packs agree, (2) every byte of the selected slices came
 * back and every other byte stayed zero, (3) the first staging record is the
 * K row of token s_0 of (layer 0, sequence 0, head 0) read through the layout.
 * Exit status 0 when every check holds. */
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
  if (failures == 0) printf("gpu_roundtrip: all checks passed\n");
  return failures == 0 ? 0 : 1;
}
