// GPU implementation of the seeded cache fill (test and benchmark input
// generation only; not part of the copy library).
//
// Definition (the same one synth/__init__.py implements in numpy): word n of
// a tensor, bytes 8n..8n+7 little-endian, is output n (0-based) of a
// SplitMix64 generator (Steele, Lea & Flood, OOPSLA 2014; finaliser of
// Vigna's public splitmix64.c) whose state starts at `base`.  For the
// floating-point kinds, an element whose exponent field is all ones gets its
// lowest exponent bit cleared so that no element is Inf or NaN.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// kind: 0 raw, 1 fp16, 2 bf16, 3 fp32
__device__ __forceinline__ uint64_t make_finite(uint64_t w, int kind) {
  if (kind == 1 || kind == 2) {
    const uint64_t emask = kind == 1 ? 0x7C00ull : 0x7F80ull;
    const uint64_t ebit = kind == 1 ? 0x0400ull : 0x0080ull;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t m = emask << (16 * j);
      if ((w & m) == m) w &= ~(ebit << (16 * j));
    }
  } else if (kind == 3) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint64_t m = 0x7F800000ull << (32 * j);
      if ((w & m) == m) w &= ~(0x00800000ull << (32 * j));
    }
  }
  return w;
}

__global__ void fill_words_kernel(uint64_t* __restrict__ dst, uint64_t nwords,
                                  uint64_t base, int kind) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x * 2;
  for (uint64_t w = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2; w < nwords;
       w += stride) {
    const uint64_t a = make_finite(mix64(base + (w + 1) * kGamma), kind);
    if (w + 1 < nwords) {
      const uint64_t b = make_finite(mix64(base + (w + 2) * kGamma), kind);
      *reinterpret_cast<ulonglong2*>(dst + w) = make_ulonglong2(a, b);
    } else {
      dst[w] = a;
    }
  }
}

}  // namespace

extern "C" {

// Fills `nbytes` (a multiple of 16) at device address `dst` (16-byte
// aligned) with words n = 0.. of SplitMix64 started at `base`.
// Returns 0 on success, 1 on a bad argument, 2 on a CUDA error.
int synth_fill(void* dst, uint64_t nbytes, uint64_t base, int kind, cudaStream_t stream) {
  if (!dst || (nbytes % 16) || (reinterpret_cast<uintptr_t>(dst) % 16) || kind < 0 || kind > 3)
    return 1;
  if (nbytes == 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 2;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 2;
  const uint64_t nwords = nbytes / 8;
  const int threads = 256;
  uint64_t blocks = (nwords / 2 + threads - 1) / threads;
  const uint64_t cap = (uint64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  fill_words_kernel<<<(unsigned)blocks, threads, 0, stream>>>(static_cast<uint64_t*>(dst), nwords,
                                                                base, kind);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
