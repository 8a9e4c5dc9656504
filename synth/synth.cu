// Device side of the seeded input generator (see synth/__init__.py for the definition).
// Holds no arithmetic of the verify pass: it writes bytes whose values follow the stated
// distributions, bit-identical to the numpy implementation for every element index.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * kGolden + stream);
}

// dst[j] = byte (start + j) % 8 of word (start + j) / 8.
__global__ void fill_bytes_kernel(uint8_t* __restrict__ dst, uint64_t n, uint64_t key, uint64_t start) {
  const uint64_t w_first = start / 8;
  const uint64_t w_last = (start + n + 7) / 8;  // exclusive
  const uint64_t nw = w_last - w_first;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < nw;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t w = w_first + i;
    const uint64_t v = mix64(key + (w + 1) * kGolden);
    const uint64_t b0 = w * 8;  // global byte index of byte 0 of this word
    if (b0 >= start && b0 + 8 <= start + n && ((uintptr_t)(dst + (b0 - start)) & 7) == 0) {
      *reinterpret_cast<uint64_t*>(dst + (b0 - start)) = v;  // little-endian byte order
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint64_t b = b0 + j;
        if (b >= start && b < start + n) dst[b - start] = (uint8_t)(v >> (8 * j));
      }
    }
  }
}

// dst[i] = codes[#{t : thr[t] <= (word(start + i) >> 32)}]; thr ascending, n_thr <= 256.
__global__ void fill_threshold_kernel(uint8_t* __restrict__ dst, uint64_t n, uint64_t key, uint64_t start,
                                      const uint64_t* __restrict__ thr, int n_thr,
                                      const uint8_t* __restrict__ codes) {
  __shared__ uint64_t s_thr[256];
  __shared__ uint8_t s_codes[257];
  for (int i = threadIdx.x; i < n_thr; i += blockDim.x) s_thr[i] = thr[i];
  for (int i = threadIdx.x; i <= n_thr; i += blockDim.x) s_codes[i] = codes[i];
  __syncthreads();
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t r = mix64(key + (start + i + 1) * kGolden) >> 32;
    int lo = 0, hi = n_thr;  // first index with thr > r
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_thr[mid] <= r) lo = mid + 1;
      else hi = mid;
    }
    dst[i] = s_codes[lo];
  }
}

int grid_for(uint64_t items) {
  uint64_t b = (items + 255) / 256;
  if (b > 152ull * 64) b = 152ull * 64;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

extern "C" int vps_fill_bytes(void* dst, uint64_t n, uint64_t seed, uint64_t stream, uint64_t start,
                              void* cuda_stream) {
  if (n == 0) return 0;
  if (!dst) return 1;
  fill_bytes_kernel<<<grid_for(n / 8 + 2), 256, 0, (cudaStream_t)cuda_stream>>>(
      (uint8_t*)dst, n, stream_key(seed, stream), start);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

extern "C" int vps_fill_threshold_codes(void* dst, uint64_t n, uint64_t seed, uint64_t stream, uint64_t start,
                                        const void* thr, int n_thr, const void* codes, void* cuda_stream) {
  if (n == 0) return 0;
  if (!dst || !thr || !codes || n_thr < 1 || n_thr > 256) return 1;
  fill_threshold_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      (uint8_t*)dst, n, stream_key(seed, stream), start, (const uint64_t*)thr, n_thr, (const uint8_t*)codes);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}
