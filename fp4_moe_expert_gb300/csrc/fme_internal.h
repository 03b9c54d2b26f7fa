// Host-side helpers shared by the translation units of libfme.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fme.h"

namespace fme {

// Records a printf-style reason for fme_last_error() and returns `status`.
int set_last_error(int status, const char* fmt, ...);

// SM count of a device (queried once per device).
int device_sm_count(int dev);

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize once per (device, kernel).
bool ensure_smem_attr(int dev, const void* kernel, size_t bytes);

// Wall-time limit of every device-side wait, in ns (FME_WAIT_TIMEOUT_MS env
// override, default 1000 ms).
unsigned long long wait_timeout_ns();

size_t nvfp4_workspace_bytes(int M, int H, int N, int L, int top_k);

// The routed experts of one FP8 layer call (E == 0: none).
struct RoutedFp8 {
  const void* x = nullptr;
  const uint8_t* xq = nullptr;   // MXFP8 input instead of x: E4M3 [M, H] and E8M0 [M, H/32]
  const uint8_t* xsc = nullptr;
  const void* logits = nullptr;
  int logits_dtype = 0;
  const float* bias = nullptr;
  const uint8_t* w13 = nullptr;
  const float* s13 = nullptr;
  const uint8_t* w2 = nullptr;
  const float* s2 = nullptr;
  int E = 0, top_k = 0;
  float limit = 0.0f, scale = 1.0f;
  int ue8m0 = 0;
  void* out = nullptr;
  int32_t* ids = nullptr;
  float* weights = nullptr;
};

// The shared expert of one FP8 layer call (w13 == nullptr: none).
struct SharedFp8 {
  const void* x = nullptr;
  const uint8_t* w13 = nullptr;
  const float* s13 = nullptr;
  const uint8_t* w2 = nullptr;
  const float* s2 = nullptr;
  float limit = 0.0f;
  int ue8m0 = 0;
  void* gate_up = nullptr;
  void* out = nullptr;
};

// Host-side checks of a routed FP8 call (pointers, shapes, dtype, scale,
// 16-byte alignment): FME_OK or the status fme_moe_routed_fp8 returns.
int check_routed_fp8_args(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
                          const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
                          float limit, float scale, const void* out, const int32_t* ids, const float* weights,
                          const void* workspace);

// One launch of the tcgen05 kernel over the routed experts and/or the shared
// expert of M tokens (arguments already validated).
int layer_fp8(const RoutedFp8& r, const SharedFp8& sh, int M, int H, int I, void* workspace, size_t workspace_bytes,
              cudaStream_t st);
// Workspace bytes of a layer_fp8 call (E routed experts, 0 for the shared
// expert alone with top_k 0), and its leading bytes (error word and counters)
// that must be zero when a call starts.
size_t layer_fp8_workspace_bytes(int M, int H, int I, int E, int top_k, bool shared);
size_t layer_fp8_zero_bytes(int M, int H, int I, int E, int top_k, bool shared);

// y[t] = bf16(sum_r w[t, r] * out[t * top_k + r] (+ shared_out[t])) (arguments validated).
int finalize(const void* out, const float* weights, const void* shared_out, int M, int H, int top_k, void* y,
             cudaStream_t st);

// MXFP8 of x [T, H] BF16 -> q [T, H] E4M3 and scales [T, H/32] E8M0 (arguments validated).
int mxfp8_quantize(const void* x, int T, int H, uint8_t* q, uint8_t* scales, cudaStream_t st);
// partials [T, N, H] BF16 -> latent [T, H] = bf16(rank-order FP32 sum), normed [T, H] = RMSNorm(latent) * gamma.
int combine_rmsnorm(const void* partials, int T, int N, int H, const void* gamma, float eps, void* latent,
                    void* normed, cudaStream_t st);

// Routing fused into the NVFP4 call: picks from logits + bias over E experts
// (the routed FP8 rule), written to ids / weights [M, top_k].
struct Nvfp4Routing {
  const void* logits = nullptr;
  int logits_dtype = 0;
  const float* bias = nullptr;
  int E = 0;
  float scale = 1.0f;
  int32_t* ids = nullptr;
  float* weights = nullptr;
};

// ids / weights: the caller's picks, or nullptr with `route` given.
int routed_nvfp4(const void* x, const int32_t* ids, const float* weights, const uint8_t* w13, const uint8_t* s13,
                 const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int e0, int top_k, float limit,
                 void* y, void* workspace, size_t workspace_bytes, cudaStream_t st,
                 const Nvfp4Routing* route = nullptr);

int ue8m0_unpack(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch, cudaStream_t st);

}  // namespace fme
