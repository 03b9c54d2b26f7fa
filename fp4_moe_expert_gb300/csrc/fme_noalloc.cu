// fme_moe_routed_fp8_noalloc: the routed FP8 layer for callers that cannot
// allocate device memory, and fme_moe_routed_fp8_noalloc_error, which reads
// that variant's device error word.
//
// Some callers of this library run where cudaMalloc is off limits: code
// inside a memory pool owned by someone else, plug-ins whose host application
// forbids device allocations after start-up, or capture-time paths where an
// allocation would be recorded or would fail. They cannot provide the
// workspace fme_moe_routed_fp8 needs. This entry point uses scratch that
// lives in this file instead: a fixed device array that a GPU holds from the
// moment this file's module is loaded there (lazily, by default: the first
// call on that GPU) until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fme.h"
#include "fme_internal.h"

namespace {

// Largest workspace the variant can serve: 64 MiB. That covers, e.g., the
// DeepSeek-V3 shape (H = 7168, I = 2048, 256 experts, top_k 8) up to M = 63
// tokens and the Latent-MoE shape (H = 3584, 896 experts, top_k 16) up to
// M = 32. Larger requests are rejected with FME_EUNSUPPORTED.
constexpr size_t kScratchBytes = size_t(64) << 20;

// The scratch itself. In host code `g_scratch` only names a host-side
// stand-in, never the device memory: host code must take the device address
// from cudaGetSymbolAddress (below) and pass that to the kernel. The routed
// kernel's workspace layout puts its error word in the first 4 bytes.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

// Identity of the calling thread's current CUDA context (0 when none is
// current yet), from the driver's unique context id: it changes when the
// primary context is destroyed (cudaDeviceReset) and created again.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  if (ctx == nullptr) return true;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch for the current device, looked up with that
// device current and cached per device together with the context it was
// taken in; a new context (after cudaDeviceReset) triggers a new lookup.
// Returns nullptr and records the reason on failure.
void* scratch_address(int dev) {
  struct Slot {
    unsigned long long ctx_id;
    void* ptr;
  };
  static std::mutex mu;
  static Slot slots[64] = {};
  if (dev < 0 || dev >= 64) {
    fme::set_last_error(FME_EUNSUPPORTED, "device %d outside [0, 64)", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    fme::set_last_error(FME_ECUDA, "cannot query the current CUDA context");
    return nullptr;
  }
  if (slots[dev].ptr != nullptr && id != 0 && slots[dev].ctx_id == id) return slots[dev].ptr;
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_scratch);  // creates the context when none is current
  if (err != cudaSuccess) {
    fme::set_last_error(FME_ECUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(err));
    return nullptr;
  }
  if (!current_context_id(&id) || id == 0) {
    fme::set_last_error(FME_ECUDA, "no current CUDA context after the scratch lookup");
    return nullptr;
  }
  slots[dev].ctx_id = id;
  slots[dev].ptr = p;
  return p;
}

}  // namespace

extern "C" int fme_moe_routed_fp8_noalloc(const void* x, const void* logits, int logits_dtype,
                                          const float* bias, const uint8_t* w13, const float* s13,
                                          const uint8_t* w2, const float* s2, int M, int H, int I, int E,
                                          int top_k, float limit, float scale, int ue8m0, void* out,
                                          int32_t* ids, float* weights, void* stream) {
  // Every argument is checked before the shared array is touched, so a
  // rejected call leaves it as it was.
  const int st = fme::check_routed_fp8_args(x, logits, logits_dtype, bias, w13, s13, w2, s2, M, H, I, E, top_k,
                                            limit, scale, out, ids, weights, nullptr);
  if (st != FME_OK) return st;
  const size_t need = fme_moe_routed_fp8_workspace(M, H, I, E, top_k);
  if (need == 0)
    return fme::set_last_error(FME_EINVAL, "bad sizes M=%d H=%d I=%d E=%d top_k=%d", M, H, I, E, top_k);
  if (need > kScratchBytes)
    return fme::set_last_error(FME_EUNSUPPORTED,
                               "needs %zu bytes of scratch; the no-allocation variant holds %zu (64 MiB): "
                               "use fme_moe_routed_fp8 with a caller workspace",
                               need, kScratchBytes);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fme::set_last_error(FME_ECUDA, "cudaGetDevice failed");
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return FME_ECUDA;
  // The array keeps whatever the previous call left. The counters must start
  // at zero (the rest is written before it is read); the error word (its
  // first 4 bytes) is left alone, so a device-side error stays visible to
  // fme_moe_routed_fp8_noalloc_error until read there, across later calls.
  const size_t zero = fme::layer_fp8_zero_bytes(M, H, I, E, top_k, false);
  const cudaError_t err = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + 4, 0, zero - 4,
                                          static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return fme::set_last_error(FME_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(err));
  return fme_moe_routed_fp8(x, logits, logits_dtype, bias, w13, s13, w2, s2, M, H, I, E, top_k, limit, scale,
                            ue8m0, out, ids, weights, scratch, kScratchBytes, stream);
}

extern "C" int fme_moe_routed_fp8_noalloc_error(int* code, void* stream) {
  if (code == nullptr) return fme::set_last_error(FME_EINVAL, "null argument");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fme::set_last_error(FME_ECUDA, "cudaGetDevice failed");
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return FME_ECUDA;
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  if (err == cudaSuccess && word != 0u) err = cudaMemsetAsync(scratch, 0, sizeof(word), st);
  if (err != cudaSuccess)
    return fme::set_last_error(FME_ECUDA, "reading the error word: %s", cudaGetErrorString(err));
  *code = static_cast<int>(word);
  if (word != 0u) return fme::set_last_error(FME_ETIMEOUT, "device error word 0x%x", word);
  return FME_OK;
}
