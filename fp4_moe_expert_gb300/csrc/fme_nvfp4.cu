// NVFP4 slot MoE (placeholder until the kernel lands).
#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {
size_t nvfp4_workspace_bytes(int M, int H, int N, int L, int top_k) { return 256; }
int routed_nvfp4(const void*, const int32_t*, const float*, const uint8_t*, const uint8_t*, const uint8_t*,
                 const uint8_t*, int, int, int, int, int, int, float, void*, void*, size_t, cudaStream_t) {
  return set_last_error(FME_EUNSUPPORTED, "nvfp4 path not built yet");
}
}  // namespace fme
