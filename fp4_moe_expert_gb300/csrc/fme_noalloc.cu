// fme_moe_routed_fp8_noalloc: the routed FP8 layer for callers that cannot
// allocate device memory.
//
// Some callers of this library run where cudaMalloc is off limits: code
// inside a memory pool owned by someone else, plug-ins whose host application
// forbids device allocations after start-up, or capture-time paths where an
// allocation would be recorded or would fail. They cannot provide the
// workspace fme_moe_routed_fp8 needs. This entry point uses scratch that
// lives in this file instead: a fixed device array that every GPU which
// loads the library holds until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fme.h"
#include "fme_internal.h"

namespace {

// Largest workspace the variant can serve: 16 MiB. That covers, e.g., the
// DeepSeek-V3 shape (H = 7168, I = 2048, 256 experts, top_k 8) up to M = 32
// tokens. Larger requests are rejected with FME_EUNSUPPORTED.
constexpr size_t kScratchBytes = size_t(16) << 20;

// The scratch itself. In host code `g_scratch` only names a host-side
// stand-in, never the device memory: host code must take the device address
// from cudaGetSymbolAddress (below) and pass that to the kernel.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

// Device address of g_scratch, looked up once per device with that device
// current. Returns nullptr and records the reason on failure.
void* scratch_address(int dev) {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess) {
      fme::set_last_error(FME_ECUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(err));
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int fme_moe_routed_fp8_noalloc(const void* x, const void* logits, int logits_dtype,
                                          const float* bias, const uint8_t* w13, const float* s13,
                                          const uint8_t* w2, const float* s2, int M, int H, int I, int E,
                                          int top_k, float limit, float scale, int ue8m0, void* out,
                                          int32_t* ids, float* weights, void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fme::set_last_error(FME_ECUDA, "cudaGetDevice failed");
  const size_t need = fme_moe_routed_fp8_workspace(M, H, I, E, top_k);
  if (need == 0)
    return fme::set_last_error(FME_EINVAL, "bad sizes M=%d H=%d I=%d E=%d top_k=%d", M, H, I, E, top_k);
  if (need > kScratchBytes)
    return fme::set_last_error(FME_EUNSUPPORTED,
                               "needs %zu bytes of scratch; the no-allocation variant holds %zu (16 MiB): "
                               "use fme_moe_routed_fp8 with a caller workspace",
                               need, kScratchBytes);
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return FME_ECUDA;
  // The array keeps whatever the previous call left; start from a zeroed
  // error word and zeroed counters (the rest is written before it is read).
  const cudaError_t err =
      cudaMemsetAsync(scratch, 0, fme::layer_fp8_zero_bytes(M, H, I, E, top_k, false),
                      static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return fme::set_last_error(FME_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(err));
  return fme_moe_routed_fp8(x, logits, logits_dtype, bias, w13, s13, w2, s2, M, H, I, E, top_k, limit, scale,
                            ue8m0, out, ids, weights, scratch, kScratchBytes, stream);
}
