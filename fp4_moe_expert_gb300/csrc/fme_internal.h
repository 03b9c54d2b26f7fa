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

size_t fp8_workspace_bytes(int M, int routes, int H, int I, int E);
// Leading workspace bytes (error word and counters) that must be zero when a call starts.
size_t fp8_workspace_zero_bytes(int M, int routes, int H, int I, int E);
size_t nvfp4_workspace_bytes(int M, int H, int N, int L, int top_k);

int routed_fp8(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
               const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
               float limit, float scale, int ue8m0, void* out, int32_t* ids, float* weights, void* workspace,
               size_t workspace_bytes, cudaStream_t st);

int shared_fp8(const void* x, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2, int M,
               int H, int I, float limit, int ue8m0, void* gate_up, void* out, void* workspace,
               size_t workspace_bytes, cudaStream_t st);

int routed_nvfp4(const void* x, const int32_t* ids, const float* weights, const uint8_t* w13, const uint8_t* s13,
                 const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int e0, int top_k, float limit,
                 void* y, void* workspace, size_t workspace_bytes, cudaStream_t st);

int ue8m0_unpack(const int32_t* packed, int n, int k, float* dst, int check, int* mismatch, cudaStream_t st);

}  // namespace fme
