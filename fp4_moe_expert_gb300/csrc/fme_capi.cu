// extern "C" entry points of libfme.so: argument checks, status codes and the
// small helpers (workspace clear / error word, UE8M0 scale unpacking).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <set>
#include <utility>

#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

static thread_local char g_last_error[512] = "";

int set_last_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int device_sm_count(int dev) {
  static int cache[64] = {0};
  if (dev < 0 || dev >= 64) return -1;
  if (cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  cache[dev] = n;
  return n;
}

bool ensure_smem_attr(int dev, const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, kernel})) return true;
  const cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (err != cudaSuccess) {
    set_last_error(FME_ECUDA, "cudaFuncSetAttribute(max dynamic smem = %zu): %s", bytes, cudaGetErrorString(err));
    return false;
  }
  done.insert({dev, kernel});
  return true;
}

unsigned long long wait_timeout_ns() {
  const char* env = std::getenv("FME_WAIT_TIMEOUT_MS");
  long long ms = 1000;
  if (env != nullptr) {
    const long long v = std::atoll(env);
    if (v > 0) ms = v;
  }
  return static_cast<unsigned long long>(ms) * 1000000ull;
}

// ---------------------------------------------------------------- UE8M0 unpack
// "shared_expert" block_scales: byte g % 4 of column g // 4 of row r holds the
// exponent of K group g; the FP32 scale of row block i is exponent << 23.
__global__ void ue8m0_unpack_kernel(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch) {
  const int groups = k / 128;
  const int cols = k / 512;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (n / 128) * groups) return;
  const int i = idx / groups, g = idx % groups;
  auto exponent = [&](int row) {
    const uint32_t w = static_cast<uint32_t>(__ldg(packed + static_cast<size_t>(row) * cols + g / 4));
    return (w >> (8 * (g % 4))) & 0xFFu;
  };
  const uint32_t e = exponent(128 * i);
  dst[idx] = __uint_as_float(e << 23);
  if (check) {
    for (int r = 1; r < 128; ++r)
      if (exponent(128 * i + r) != e) {
        atomicExch(mismatch, 1);
        break;
      }
  }
}

int ue8m0_unpack(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch, cudaStream_t st) {
  const int total = (n / 128) * (k / 128);
  const int threads = 128;
  ue8m0_unpack_kernel<<<(total + threads - 1) / threads, threads, 0, st>>>(packed, n, k, dst, check, mismatch);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "ue8m0 unpack launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

// Bounded-wait self-test: waits, each with the kernels' own primitives and a
// time limit, on a global flag nothing sets and on an mbarrier nothing
// arrives at; both must give up, set their error bits and return.
__global__ void selftest_wait_kernel(uint32_t* word, const uint32_t* flag, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(flag) == 0u) {
      if (globaltimer_ns() - t0 > timeout_ns) {
        atomicOr(word, kErrCrossWait);
        break;
      }
      __nanosleep(256);
    }
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, timeout_ns, nullptr)) atomicOr(word, kErrRingWait);
  }
}

}  // namespace fme

using namespace fme;

static bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

#define FME_REQUIRE(cond, status, ...)                   \
  do {                                                   \
    if (!(cond)) return set_last_error(status, __VA_ARGS__); \
  } while (0)

static int check_fp8_shapes(int M, int H, int I, int E, int top_k, float limit) {
  FME_REQUIRE(M >= 1 && M <= kMaxTokens, FME_EUNSUPPORTED, "M=%d outside [1, %d]", M, kMaxTokens);
  FME_REQUIRE(H >= 128 && H % 128 == 0 && I >= 128 && I % 128 == 0, FME_EINVAL,
              "H=%d and I=%d must be positive multiples of 128", H, I);
  FME_REQUIRE(H <= kMaxHidden && I <= kMaxHidden, FME_EUNSUPPORTED, "H=%d or I=%d above %d", H, I, kMaxHidden);
  FME_REQUIRE(E >= 1 && E <= kMaxExperts, FME_EUNSUPPORTED, "E=%d outside [1, %d]", E, kMaxExperts);
  FME_REQUIRE(top_k >= 1 && top_k <= E && top_k <= kMaxTopK, FME_EINVAL, "top_k=%d outside [1, min(E=%d, %d)]",
              top_k, E, kMaxTopK);
  FME_REQUIRE(limit > 0.0f, FME_EINVAL, "limit must be > 0 (got %g)", static_cast<double>(limit));
  return FME_OK;
}

namespace fme {
int check_routed_fp8_args(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                          const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
                          float limit, float scale, const void* out, const int32_t* ids, const float* weights,
                          const void* workspace) {
  FME_REQUIRE(x && logits && bias && w13 && s13 && w2 && s2 && out && ids && weights, FME_EINVAL,
              "null pointer argument");
  const int st = check_fp8_shapes(M, H, I, E, top_k, limit);
  if (st != FME_OK) return st;
  FME_REQUIRE(logits_dtype == FME_F32 || logits_dtype == FME_BF16, FME_EINVAL, "logits_dtype=%d", logits_dtype);
  FME_REQUIRE(std::isfinite(scale), FME_EINVAL, "scale must be finite");
  FME_REQUIRE(!misaligned(x) && !misaligned(logits) && !misaligned(bias) && !misaligned(w13) && !misaligned(s13) &&
                  !misaligned(w2) && !misaligned(s2) && !misaligned(out) && !misaligned(ids) &&
                  !misaligned(weights) && !misaligned(workspace),
              FME_EALIGN, "every pointer must be 16-byte aligned");
  return FME_OK;
}
}  // namespace fme

extern "C" {

const char* fme_last_error(void) { return g_last_error; }

int fme_version(void) { return 100; }

int fme_sm_count(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return device_sm_count(dev);
}

size_t fme_moe_routed_fp8_workspace(int M, int H, int I, int E, int top_k) {
  if (check_fp8_shapes(M, H, I, E, top_k, 1.0f) != FME_OK) return 0;
  return layer_fp8_workspace_bytes(M, H, I, E, top_k, false);
}


int fme_moe_routed_fp8(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                       const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
                       float limit, float scale, int ue8m0, void* out, int32_t* ids, float* weights,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_routed_fp8_args(x, logits, logits_dtype, bias, w13, s13, w2, s2, M, H, I, E, top_k, limit,
                                       scale, out, ids, weights, workspace);
  if (st != FME_OK) return st;
  RoutedFp8 r;
  r.x = x;
  r.logits = logits;
  r.logits_dtype = logits_dtype;
  r.bias = bias;
  r.w13 = w13;
  r.s13 = s13;
  r.w2 = w2;
  r.s2 = s2;
  r.E = E;
  r.top_k = top_k;
  r.limit = limit;
  r.scale = scale;
  r.ue8m0 = ue8m0;
  r.out = out;
  r.ids = ids;
  r.weights = weights;
  return layer_fp8(r, SharedFp8(), M, H, I, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}


int fme_moe_routed_fp8_mx(const uint8_t* xq, const uint8_t* xscales, const void* logits, int logits_dtype,
                          const float* bias, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                          int M, int H, int I, int E, int top_k, float limit, float scale, int ue8m0, void* out,
                          int32_t* ids, float* weights, void* workspace, size_t workspace_bytes, void* stream) {
  FME_REQUIRE(xq && xscales && logits && bias && w13 && s13 && w2 && s2 && out && ids && weights, FME_EINVAL,
              "null pointer argument");
  const int st = check_fp8_shapes(M, H, I, E, top_k, limit);
  if (st != FME_OK) return st;
  FME_REQUIRE(logits_dtype == FME_F32 || logits_dtype == FME_BF16, FME_EINVAL, "logits_dtype=%d", logits_dtype);
  FME_REQUIRE(std::isfinite(scale), FME_EINVAL, "scale must be finite");
  FME_REQUIRE(!misaligned(xq) && !misaligned(logits) && !misaligned(bias) && !misaligned(w13) && !misaligned(s13) &&
                  !misaligned(w2) && !misaligned(s2) && !misaligned(out) && !misaligned(ids) &&
                  !misaligned(weights) && !misaligned(workspace),
              FME_EALIGN, "every pointer except xscales must be 16-byte aligned");
  RoutedFp8 r;
  r.xq = xq;
  r.xsc = xscales;
  r.logits = logits;
  r.logits_dtype = logits_dtype;
  r.bias = bias;
  r.w13 = w13;
  r.s13 = s13;
  r.w2 = w2;
  r.s2 = s2;
  r.E = E;
  r.top_k = top_k;
  r.limit = limit;
  r.scale = scale;
  r.ue8m0 = ue8m0;
  r.out = out;
  r.ids = ids;
  r.weights = weights;
  return layer_fp8(r, SharedFp8(), M, H, I, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t fme_shared_expert_fp8_workspace(int M, int H, int I) {
  if (check_fp8_shapes(M, H, I, 1, 1, 1.0f) != FME_OK) return 0;
  return layer_fp8_workspace_bytes(M, H, I, 0, 0, true);
}

int fme_shared_expert_fp8(const void* x, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2,
                          int M, int H, int I, float limit, int ue8m0, void* gate_up, void* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  FME_REQUIRE(x && w13 && s13 && w2 && s2 && out, FME_EINVAL, "null pointer argument");
  const int st = check_fp8_shapes(M, H, I, 1, 1, limit);
  if (st != FME_OK) return st;
  FME_REQUIRE(!misaligned(x) && !misaligned(w13) && !misaligned(s13) && !misaligned(w2) && !misaligned(s2) &&
                  !misaligned(out) && !misaligned(gate_up) && !misaligned(workspace),
              FME_EALIGN, "every pointer must be 16-byte aligned");
  SharedFp8 sh;
  sh.x = x;
  sh.w13 = w13;
  sh.s13 = s13;
  sh.w2 = w2;
  sh.s2 = s2;
  sh.limit = limit;
  sh.ue8m0 = ue8m0;
  sh.gate_up = gate_up;
  sh.out = out;
  return layer_fp8(RoutedFp8(), sh, M, H, I, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t fme_moe_layer_fp8_workspace(int M, int H, int I, int E, int top_k) {
  if (check_fp8_shapes(M, H, I, E, top_k, 1.0f) != FME_OK) return 0;
  return layer_fp8_workspace_bytes(M, H, I, E, top_k, true);
}

int fme_moe_layer_fp8(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                      const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
                      float limit, float scale, int ue8m0, const uint8_t* shared_w13, const float* shared_s13,
                      const uint8_t* shared_w2, const float* shared_s2, float shared_limit, int shared_ue8m0,
                      void* out, int32_t* ids, float* weights, void* shared_out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  FME_REQUIRE(x && logits && bias && w13 && s13 && w2 && s2 && out && ids && weights && shared_w13 && shared_s13 &&
                  shared_w2 && shared_s2 && shared_out,
              FME_EINVAL, "null pointer argument");
  int st = check_fp8_shapes(M, H, I, E, top_k, limit);
  if (st != FME_OK) return st;
  FME_REQUIRE(shared_limit > 0.0f, FME_EINVAL, "shared_limit must be > 0 (got %g)", static_cast<double>(shared_limit));
  FME_REQUIRE(logits_dtype == FME_F32 || logits_dtype == FME_BF16, FME_EINVAL, "logits_dtype=%d", logits_dtype);
  FME_REQUIRE(std::isfinite(scale), FME_EINVAL, "scale must be finite");
  FME_REQUIRE(!misaligned(x) && !misaligned(logits) && !misaligned(bias) && !misaligned(w13) && !misaligned(s13) &&
                  !misaligned(w2) && !misaligned(s2) && !misaligned(out) && !misaligned(ids) &&
                  !misaligned(weights) && !misaligned(shared_w13) && !misaligned(shared_s13) &&
                  !misaligned(shared_w2) && !misaligned(shared_s2) && !misaligned(shared_out) &&
                  !misaligned(workspace),
              FME_EALIGN, "every pointer must be 16-byte aligned");
  RoutedFp8 r;
  r.x = x;
  r.logits = logits;
  r.logits_dtype = logits_dtype;
  r.bias = bias;
  r.w13 = w13;
  r.s13 = s13;
  r.w2 = w2;
  r.s2 = s2;
  r.E = E;
  r.top_k = top_k;
  r.limit = limit;
  r.scale = scale;
  r.ue8m0 = ue8m0;
  r.out = out;
  r.ids = ids;
  r.weights = weights;
  SharedFp8 sh;
  sh.x = x;
  sh.w13 = shared_w13;
  sh.s13 = shared_s13;
  sh.w2 = shared_w2;
  sh.s2 = shared_s2;
  sh.limit = shared_limit;
  sh.ue8m0 = shared_ue8m0;
  sh.out = shared_out;
  return layer_fp8(r, sh, M, H, I, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int fme_ue8m0_unpack(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch, void* stream) {
  FME_REQUIRE(packed && dst && (!check || mismatch), FME_EINVAL, "null pointer argument");
  FME_REQUIRE(n >= 128 && n % 128 == 0 && k >= 512 && k % 512 == 0, FME_EINVAL,
              "n=%d must be a multiple of 128 and k=%d of 512", n, k);
  FME_REQUIRE(!misaligned(packed) && !misaligned(dst), FME_EALIGN, "pointers must be 16-byte aligned");
  return ue8m0_unpack(packed, n, k, dst, check, mismatch, static_cast<cudaStream_t>(stream));
}

int fme_moe_finalize(const void* out, const float* weights, const void* shared_out, int M, int H, int top_k,
                     void* y, void* stream) {
  FME_REQUIRE(out && weights && y, FME_EINVAL, "null pointer argument");
  FME_REQUIRE(M >= 1 && M <= (1 << 20), FME_EINVAL, "M=%d outside [1, 2^20]", M);
  FME_REQUIRE(H >= 8 && H % 8 == 0 && H <= (1 << 20), FME_EINVAL, "H=%d must be a positive multiple of 8", H);
  FME_REQUIRE(top_k >= 1 && top_k <= kMaxTopK, FME_EINVAL, "top_k=%d outside [1, %d]", top_k, kMaxTopK);
  FME_REQUIRE(!misaligned(out) && !misaligned(y) && (shared_out == nullptr || !misaligned(shared_out)) &&
                  reinterpret_cast<uintptr_t>(weights) % 4 == 0,
              FME_EALIGN, "out, shared_out and y must be 16-byte aligned, weights 4-byte aligned");
  return finalize(out, weights, shared_out, M, H, top_k, y, static_cast<cudaStream_t>(stream));
}

int fme_moe_layer_nvfp4(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                        const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int E,
                        int e0, int top_k, float scale, float limit, void* y, int32_t* ids, float* weights,
                        void* workspace, size_t workspace_bytes, void* stream) {
  FME_REQUIRE(x && logits && bias && w13 && s13 && w2 && s2 && y && ids && weights, FME_EINVAL,
              "null pointer argument");
  FME_REQUIRE(M >= 1 && M <= kMaxTokens, FME_EUNSUPPORTED, "M=%d outside [1, %d]", M, kMaxTokens);
  FME_REQUIRE(H >= 128 && H % 128 == 0 && N >= 128 && N % 128 == 0, FME_EINVAL,
              "H=%d and N=%d must be positive multiples of 128", H, N);
  FME_REQUIRE(H <= 8192 && N <= 8192, FME_EUNSUPPORTED, "H=%d or N=%d above 8192", H, N);
  FME_REQUIRE(E >= 1 && E <= kMaxExperts, FME_EUNSUPPORTED, "E=%d outside [1, %d]", E, kMaxExperts);
  FME_REQUIRE(L >= 1 && e0 >= 0 && e0 + L <= E, FME_EINVAL, "local range [%d, %d) outside [0, %d)", e0, e0 + L, E);
  FME_REQUIRE(top_k >= 1 && top_k <= kMaxTopK && top_k <= E, FME_EINVAL, "top_k=%d outside [1, min(%d, E)]", top_k,
              kMaxTopK);
  FME_REQUIRE(logits_dtype == FME_F32 || logits_dtype == FME_BF16, FME_EINVAL, "logits_dtype=%d", logits_dtype);
  FME_REQUIRE(std::isfinite(scale), FME_EINVAL, "scale must be finite");
  FME_REQUIRE(limit > 0.0f, FME_EINVAL, "limit must be > 0");
  FME_REQUIRE(!misaligned(x) && !misaligned(logits) && !misaligned(bias) && !misaligned(w13) && !misaligned(s13) &&
                  !misaligned(w2) && !misaligned(s2) && !misaligned(y) && !misaligned(ids) && !misaligned(weights) &&
                  !misaligned(workspace),
              FME_EALIGN, "every pointer must be 16-byte aligned");
  Nvfp4Routing r;
  r.logits = logits;
  r.logits_dtype = logits_dtype;
  r.bias = bias;
  r.E = E;
  r.scale = scale;
  r.ids = ids;
  r.weights = weights;
  return routed_nvfp4(x, nullptr, nullptr, w13, s13, w2, s2, M, H, N, L, e0, top_k, limit, y, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream), &r);
}

int fme_mxfp8_quantize(const void* x, int T, int H, uint8_t* q, uint8_t* scales, void* stream) {
  FME_REQUIRE(x && q && scales, FME_EINVAL, "null pointer argument");
  FME_REQUIRE(T >= 1 && T <= (1 << 20), FME_EINVAL, "T=%d outside [1, 2^20]", T);
  FME_REQUIRE(H >= 32 && H % 32 == 0 && H <= (1 << 20), FME_EINVAL, "H=%d must be a positive multiple of 32", H);
  FME_REQUIRE(!misaligned(x) && !misaligned(q), FME_EALIGN, "x and q must be 16-byte aligned");
  return mxfp8_quantize(x, T, H, q, scales, static_cast<cudaStream_t>(stream));
}

int fme_combine_rmsnorm(const void* partials, int T, int N, int H, const void* gamma, float eps, void* latent,
                        void* normed, void* stream) {
  FME_REQUIRE(partials && gamma && latent && normed, FME_EINVAL, "null pointer argument");
  FME_REQUIRE(T >= 1 && T <= (1 << 20), FME_EINVAL, "T=%d outside [1, 2^20]", T);
  FME_REQUIRE(N >= 1 && N <= 1024, FME_EINVAL, "N=%d outside [1, 1024]", N);
  FME_REQUIRE(H >= 8 && H % 8 == 0 && H <= 8192, FME_EINVAL, "H=%d must be a multiple of 8 in [8, 8192]", H);
  FME_REQUIRE(eps >= 0.0f && std::isfinite(eps), FME_EINVAL, "eps must be finite and >= 0");
  FME_REQUIRE(!misaligned(partials) && !misaligned(gamma) && !misaligned(latent) && !misaligned(normed), FME_EALIGN,
              "every pointer must be 16-byte aligned");
  return combine_rmsnorm(partials, T, N, H, gamma, eps, latent, normed, static_cast<cudaStream_t>(stream));
}

size_t fme_moe_routed_nvfp4_workspace(int M, int H, int N, int L, int top_k) {
  if (M < 1 || M > kMaxTokens || H < 128 || H % 128 || N < 128 || N % 128 || L < 1 || L > kMaxExperts ||
      top_k < 1 || top_k > kMaxTopK || H > 8192 || N > 8192)
    return 0;
  return nvfp4_workspace_bytes(M, H, N, L, top_k);
}

int fme_moe_routed_nvfp4(const void* x, const int32_t* topk_ids, const float* topk_weights, const uint8_t* w13,
                         const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L,
                         int e0, int top_k, float limit, void* y, void* workspace, size_t workspace_bytes,
                         void* stream) {
  FME_REQUIRE(x && topk_ids && topk_weights && w13 && s13 && w2 && s2 && y, FME_EINVAL, "null pointer argument");
  FME_REQUIRE(M >= 1 && M <= kMaxTokens, FME_EUNSUPPORTED, "M=%d outside [1, %d]", M, kMaxTokens);
  FME_REQUIRE(H >= 128 && H % 128 == 0 && N >= 128 && N % 128 == 0, FME_EINVAL,
              "H=%d and N=%d must be positive multiples of 128", H, N);
  FME_REQUIRE(H <= 8192 && N <= 8192, FME_EUNSUPPORTED, "H=%d or N=%d above 8192", H, N);
  FME_REQUIRE(L >= 1 && L <= kMaxExperts, FME_EUNSUPPORTED, "L=%d outside [1, %d]", L, kMaxExperts);
  FME_REQUIRE(top_k >= 1 && top_k <= kMaxTopK, FME_EINVAL, "top_k=%d outside [1, %d]", top_k, kMaxTopK);
  FME_REQUIRE(limit > 0.0f, FME_EINVAL, "limit must be > 0");
  FME_REQUIRE(!misaligned(x) && !misaligned(topk_ids) && !misaligned(topk_weights) && !misaligned(w13) &&
                  !misaligned(s13) && !misaligned(w2) && !misaligned(s2) && !misaligned(y) &&
                  !misaligned(workspace),
              FME_EALIGN, "every pointer must be 16-byte aligned");
  return routed_nvfp4(x, topk_ids, topk_weights, w13, s13, w2, s2, M, H, N, L, e0, top_k, limit, y, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

int fme_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int timeout_ms, void* stream) {
  FME_REQUIRE(workspace != nullptr && workspace_bytes >= 512, FME_EWORKSPACE, "workspace of 512 bytes needed");
  FME_REQUIRE(timeout_ms > 0 && timeout_ms <= 10000, FME_EINVAL, "timeout_ms=%d outside [1, 10000]", timeout_ms);
  FME_REQUIRE(!misaligned(workspace), FME_EALIGN, "workspace must be 16-byte aligned");
  uint32_t* word = static_cast<uint32_t*>(workspace);
  const uint32_t* flag = reinterpret_cast<const uint32_t*>(static_cast<uint8_t*>(workspace) + 256);
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      word, flag, static_cast<unsigned long long>(timeout_ms) * 1000000ull);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "selftest launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

int fme_workspace_clear(void* workspace, size_t workspace_bytes, void* stream) {
  FME_REQUIRE(workspace != nullptr, FME_EINVAL, "null workspace");
  const cudaError_t err = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(err));
  return FME_OK;
}

int fme_workspace_error(void* workspace, int* code, void* stream) {
  FME_REQUIRE(workspace != nullptr && code != nullptr, FME_EINVAL, "null argument");
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (err == cudaSuccess) err = cudaStreamSynchronize(st);
  if (err == cudaSuccess && word != 0u) err = cudaMemsetAsync(workspace, 0, sizeof(word), st);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "reading the error word: %s", cudaGetErrorString(err));
  *code = static_cast<int>(word);
  if (word != 0u) return set_last_error(FME_ETIMEOUT, "device error word 0x%x", word);
  return FME_OK;
}

}  // extern "C"
