/*
 * Oracle of the KV-cache buffered copy (DejaVuLib gather / scatter).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this file.  The copy
 * library never links it and shares no code with it.
 *
 * What it computes ("DejaVu: KV-Cache Streaming for Fast, Fault-Tolerant
 * Generative LLM Serving", §3 DejaVuLib implementation, Fig 6 and Fig 7a;
 * Table 1 scatter/gather): the many small non-contiguous slices of a cache
 * preallocated at the maximum sequence length are gathered into one
 * contiguous buffer (pack), and a contiguous buffer is split back into the
 * same slices (unpack).
 *
 * Cache layout (per layer, layers at a stride of `layer_stride` elements):
 *   K: [B][H][D/x][S][x]   (x = 16 / elem_bytes, the x-interleaved key layout)
 *   V: [B][H][S][D]
 * Staging order (the pages say only "contiguous buffer"; reading chosen so
 * that each layer's slab is contiguous for layer-by-layer streaming, Fig 7b):
 *   [layer l0..l1)[K then V][sequence b][head h][token t in [s_b,e_b)][d]
 * with d in logical order.  Elements are copied as raw bytes (bit patterns),
 * never through floating point.
 *
 * parity: pinned (hand-written golden vectors, an independent numpy reading of
 * the layout, brute force over every range on tiny caches, the size formula
 * 2*B*S*H*D*P*N of the KV-cache capacity page, round-trip invariants).
 */
#include <stdint.h>
#include <string.h>

/* Element index of K(l,b,h,t,d) in the x-interleaved layout. */
static int64_t k_index(int64_t layer_stride, int64_t B, int64_t H, int64_t D, int64_t S,
                       int64_t x, int64_t l, int64_t b, int64_t h, int64_t t, int64_t d) {
  (void)B;
  return l * layer_stride + (((b * H + h) * (D / x) + d / x) * S + t) * x + d % x;
}

/* Element index of V(l,b,h,t,d) in the row-major layout. */
static int64_t v_index(int64_t layer_stride, int64_t B, int64_t H, int64_t D, int64_t S,
                       int64_t l, int64_t b, int64_t h, int64_t t, int64_t d) {
  (void)B;
  return l * layer_stride + ((b * H + h) * S + t) * D + d;
}

/* 0 if the geometry and ranges are usable, else a nonzero code. */
int oracle_check(int32_t L, int32_t B, int32_t H, int32_t D, int32_t S, int32_t P,
                 int64_t layer_stride, int32_t l0, int32_t l1,
                 const int32_t* seq_start, const int32_t* seq_end) {
  if (L <= 0 || B <= 0 || H <= 0 || D <= 0 || S <= 0) return 1;
  if (P != 1 && P != 2 && P != 4) return 1;
  if (D % (16 / P) != 0) return 1;
  if (layer_stride < (int64_t)B * H * D * S) return 1;
  if (l0 < 0 || l1 > L || l0 > l1) return 2;
  for (int32_t b = 0; b < B; ++b)
    if (seq_start[b] < 0 || seq_start[b] > seq_end[b] || seq_end[b] > S) return 2;
  return 0;
}

/* Elements in the staging buffer: 2 * (l1-l0) * H * D * sum_b (e_b - s_b). */
int64_t oracle_staging_elems(int32_t B, int32_t H, int32_t D, int32_t l0, int32_t l1,
                             const int32_t* seq_start, const int32_t* seq_end) {
  int64_t tokens = 0;
  for (int32_t b = 0; b < B; ++b) tokens += seq_end[b] - seq_start[b];
  return 2 * (int64_t)(l1 - l0) * H * D * tokens;
}

/* Gather: staging <- selected slices of K and V.  Returns the number of
 * elements written, or -1 on a bad argument. */
int64_t oracle_pack(const uint8_t* k, const uint8_t* v, int32_t L, int32_t B, int32_t H,
                    int32_t D, int32_t S, int32_t P, int64_t layer_stride, int32_t l0, int32_t l1,
                    const int32_t* seq_start, const int32_t* seq_end, uint8_t* staging) {
  if (oracle_check(L, B, H, D, S, P, layer_stride, l0, l1, seq_start, seq_end)) return -1;
  const int64_t x = 16 / P;
  int64_t off = 0;
  for (int64_t l = l0; l < l1; ++l)
    for (int kv = 0; kv < 2; ++kv)
      for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
          for (int64_t t = seq_start[b]; t < seq_end[b]; ++t)
            for (int64_t d = 0; d < D; ++d) {
              const uint8_t* src =
                  kv == 0 ? k + P * k_index(layer_stride, B, H, D, S, x, l, b, h, t, d)
                          : v + P * v_index(layer_stride, B, H, D, S, l, b, h, t, d);
              memcpy(staging + P * off, src, (size_t)P);
              ++off;
            }
  return off;
}

/* Scatter: selected slices of K and V <- staging; nothing else is written.
 * Returns the number of elements read, or -1 on a bad argument. */
int64_t oracle_unpack(uint8_t* k, uint8_t* v, int32_t L, int32_t B, int32_t H, int32_t D,
                      int32_t S, int32_t P, int64_t layer_stride, int32_t l0, int32_t l1,
                      const int32_t* seq_start, const int32_t* seq_end, const uint8_t* staging) {
  if (oracle_check(L, B, H, D, S, P, layer_stride, l0, l1, seq_start, seq_end)) return -1;
  const int64_t x = 16 / P;
  int64_t off = 0;
  for (int64_t l = l0; l < l1; ++l)
    for (int kv = 0; kv < 2; ++kv)
      for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
          for (int64_t t = seq_start[b]; t < seq_end[b]; ++t)
            for (int64_t d = 0; d < D; ++d) {
              uint8_t* dst =
                  kv == 0 ? k + P * k_index(layer_stride, B, H, D, S, x, l, b, h, t, d)
                          : v + P * v_index(layer_stride, B, H, D, S, l, b, h, t, d);
              memcpy(dst, staging + P * off, (size_t)P);
              ++off;
            }
  return off;
}

/* For each staging offset offs[i] (ascending), the element index inside the
 * K (kv_out[i] = 0) or V (kv_out[i] = 1) allocation of the cache element that
 * the staging buffer holds there; for sampled checks of caches too large to
 * pack on the host.  Walks the same nest as oracle_pack, one (layer, K/V,
 * sequence, head) run at a time.  Returns the number of offsets resolved (n,
 * unless an offset is past the end of the staging buffer or out of order),
 * or -1 on a bad argument. */
int64_t oracle_source_of(int32_t L, int32_t B, int32_t H, int32_t D, int32_t S, int32_t P,
                         int64_t layer_stride, int32_t l0, int32_t l1,
                         const int32_t* seq_start, const int32_t* seq_end,
                         const int64_t* offs, int64_t n, int64_t* idx_out, int32_t* kv_out) {
  if (oracle_check(L, B, H, D, S, P, layer_stride, l0, l1, seq_start, seq_end)) return -1;
  const int64_t x = 16 / P;
  int64_t i = 0;
  int64_t run0 = 0; /* staging offset of the current run's first element */
  for (int64_t l = l0; l < l1 && i < n; ++l)
    for (int kv = 0; kv < 2 && i < n; ++kv)
      for (int64_t b = 0; b < B && i < n; ++b)
        for (int64_t h = 0; h < H && i < n; ++h) {
          const int64_t run = (int64_t)(seq_end[b] - seq_start[b]) * D;
          while (i < n && offs[i] >= run0 && offs[i] < run0 + run) {
            const int64_t r = offs[i] - run0;
            const int64_t t = seq_start[b] + r / D, d = r % D;
            kv_out[i] = kv;
            idx_out[i] = kv == 0 ? k_index(layer_stride, B, H, D, S, x, l, b, h, t, d)
                                 : v_index(layer_stride, B, H, D, S, l, b, h, t, d);
            ++i;
          }
          if (i < n && offs[i] < run0) return i; /* out of order */
          run0 += run;
        }
  return i;
}
