/* Calls libdv from plain C with no GPU work: staging sizes (the capacity
 * formula 2*B*S*H*D*P*N for a full cache), and the validation errors that are
 * decided on the host.  Exit status 0 when every check holds. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dv.h"

static int failures = 0;
#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

int main(void) {
  CHECK(dv_abi_version() == DV_ABI_VERSION);
  int32_t s[8], e[8];
  for (int b = 0; b < 8; ++b) {
    s[b] = 0;
    e[b] = 1024;
  }
  dv_cache c;
  memset(&c, 0, sizeof(c));
  c.num_layers = 48;
  c.batch = 8;
  c.num_heads = 25;
  c.head_dim = 64;
  c.max_seq = 1024;
  c.elem_bytes = 2;
  c.k_base = (void*)0x1000;
  c.v_base = (void*)0x2000;
  size_t bytes = 0;
  CHECK(dv_staging_bytes(&c, 0, 48, s, e, &bytes) == DV_OK);
  CHECK(bytes == (size_t)2 * 8 * 1024 * 25 * 64 * 2 * 48);
  e[3] = 1025; /* past max_seq */
  CHECK(dv_staging_bytes(&c, 0, 48, s, e, &bytes) == DV_ERR_RANGE);
  CHECK(strlen(dv_last_error()) > 0);
  e[3] = 1024;
  CHECK(dv_staging_bytes(&c, 0, 49, s, e, &bytes) == DV_ERR_RANGE);
  c.head_dim = 60; /* not a multiple of x = 8 */
  CHECK(dv_staging_bytes(&c, 0, 48, s, e, &bytes) == DV_ERR_UNSUPPORTED);
  c.head_dim = 64;
  CHECK(dv_kv_pack(&c, 0, 48, s, e, (void*)0x3000, 16, NULL) == DV_ERR_BUFFER_TOO_SMALL);
  CHECK(dv_kv_pack(NULL, 0, 48, s, e, (void*)0x3000, 16, NULL) == DV_ERR_INVALID_ARG);
  CHECK(strcmp(dv_status_string(DV_ERR_MISALIGNED), "DV_ERR_MISALIGNED") == 0);
  /* NULL handles are refused before anything reaches the GPU */
  CHECK(dv_stream_layer(NULL, &c, 0, s, e, (void*)0x3000, 16, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_fetch_layer(NULL, &c, 0, s, e, (const void*)0x3000, 16, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_streamer_wait(NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_fetcher_wait(NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_streamer_create(NULL, NULL, NULL, 0, NULL, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_fetcher_create(NULL, NULL, NULL, 0, NULL, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_restore(NULL, &c, -1, NULL, 0, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_restore_batched(NULL, &c, -1, NULL, 0, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_restore_fetched(NULL, &c, -1, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_truncate(NULL, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_restore_fetched_steps(NULL, &c, 0, -1, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_replica_append_streamed(NULL, NULL, &c, 0, 48, s, e, 0) == DV_ERR_INVALID_ARG);
  /* host memory: bad arguments and unknown pointers are refused without CUDA */
  void* hp = (void*)0x1;
  CHECK(dv_host_alloc(0, &hp) == DV_ERR_INVALID_ARG && hp == NULL);
  CHECK(dv_host_alloc(16, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_host_free((void*)0x10000) == DV_ERR_INVALID_ARG);
  CHECK(dv_host_free(NULL) == DV_OK);
  /* the log scatter: tables, counts and ranges are checked on the host */
  int32_t layers[2] = {0, 48}, ranges[16];
  memcpy(ranges, s, sizeof s);
  memcpy(ranges + 8, e, sizeof e);
  CHECK(dv_kv_unpack_records(NULL, 1, layers, ranges, (void*)0x3000, 16, NULL) ==
        DV_ERR_INVALID_ARG);
  CHECK(dv_kv_unpack_records(&c, -1, layers, ranges, (void*)0x3000, 16, NULL) ==
        DV_ERR_INVALID_ARG);
  CHECK(dv_kv_unpack_records(&c, 1, NULL, ranges, (void*)0x3000, 16, NULL) ==
        DV_ERR_INVALID_ARG);
  CHECK(dv_kv_unpack_records(&c, 1, layers, ranges, (void*)0x3000, 16, NULL) ==
        DV_ERR_BUFFER_TOO_SMALL);
  ranges[8] = 1025; /* a range past max_seq */
  CHECK(dv_kv_unpack_records(&c, 1, layers, ranges, (void*)0x3000, 1u << 30, NULL) ==
        DV_ERR_RANGE);
  CHECK(dv_kv_unpack_records(&c, 0, NULL, NULL, NULL, 0, NULL) == DV_OK);
  /* the swapper and the delta streamer refuse NULL handles and arguments */
  int32_t slot = 0;
  CHECK(dv_swapper_create(NULL, &c, &c, NULL, NULL, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_swapper_acquire(NULL, NULL, &slot) == DV_ERR_INVALID_ARG);
  CHECK(dv_swapper_prefetch(NULL, NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_swapper_release(NULL, NULL, 0, 48, s, e, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_swapper_wait(NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_delta_streamer_create(NULL, NULL, NULL, NULL, NULL, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_delta_stream(NULL, &c, 0, 48, s, e, 0) == DV_ERR_INVALID_ARG);
  CHECK(dv_delta_streamer_join(NULL) == DV_ERR_INVALID_ARG);
  CHECK(dv_delta_streamer_wait(NULL) == DV_ERR_INVALID_ARG);
  dv_swapper_destroy(NULL);
  dv_delta_streamer_destroy(NULL);
  dv_streamer_destroy(NULL);
  dv_fetcher_destroy(NULL);
  dv_replica_destroy(NULL);
  if (failures == 0) printf("abi_host: all checks passed\n");
  return failures == 0 ? 0 : 1;
}
