// Device-side fill of synthetic byte tensors, identical to synth/__init__.py:
//   base   = mix64(seed << 32 | tensor << 24 | expert)
//   word_i = mix64(base + (i + 1) * GAMMA) >> 32
//   code_i = first c with word_i < table[c]
// mix64 / GAMMA: SplitMix64 (Steele, Lea and Flood, OOPSLA 2014).
// Test-input infrastructure; not part of libfme.so.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_codes(uint8_t* out, long long n_experts, long long per_expert, unsigned seed, int tensor,
                           const unsigned long long* table, int expert0) {
  __shared__ unsigned long long T[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) T[i] = table[i];
  __syncthreads();
  const long long total = n_experts * per_expert;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total; idx += stride) {
    const long long e = idx / per_expert;
    const unsigned long long i = static_cast<unsigned long long>(idx - e * per_expert);
    const uint64_t key = (static_cast<uint64_t>(seed) << 32) | (static_cast<uint64_t>(tensor & 0xFF) << 24) |
                         (static_cast<uint64_t>(e + expert0) & 0xFFFFFFull);
    const uint64_t base = mix64(key);
    const uint64_t w = mix64(base + (i + 1ull) * 0x9E3779B97F4A7C15ull) >> 32;
    int lo = 0, hi = 256;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (T[mid] <= w) lo = mid + 1; else hi = mid;
    }
    out[idx] = static_cast<uint8_t>(lo);
  }
}

}  // namespace

extern "C" int fme_synth_fill_codes(uint8_t* out, long long n_experts, long long per_expert, unsigned seed,
                                    int tensor, const unsigned long long* table, int expert0, void* stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  fill_codes<<<sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n_experts, per_expert, seed, tensor,
                                                                     table, expert0);
  return static_cast<int>(cudaGetLastError());
}
