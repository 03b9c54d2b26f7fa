// Pieces shared by the FP8 and NVFP4 kernels: launch geometry, the smem weight
// ring, warp transpose-reduction and per-device launch setup.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fme_ptx.cuh"

namespace fme {

constexpr int kComputeThreads = 256;               // 8 warps, all computing
constexpr int kComputeWarps = kComputeThreads / 32;
constexpr int kThreads = kComputeThreads;          // thread 0 also issues the copies
constexpr int kStages = 3;                         // weight ring depth
constexpr int kStageBytes = 64 * 1024;             // one work item's weight rows
constexpr int kRowsPerGroup = 8;                   // rows a thread group owns per item
constexpr int kTokChunk = 4;                       // tokens per pass over an item
constexpr int kMaxSlicesPerThread = 2;             // 16-byte K slices per thread
constexpr int kMaxTokens = 64;                     // token bit masks are uint64
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kFp8MaxCtas = 160;                 // grid cap of the FP8 kernel (partial slots)

// Device error bits (workspace error word).
constexpr uint32_t kErrRingWait = 1u;  // a ring stage never landed
constexpr uint32_t kErrCrossWait = 2u;
constexpr uint32_t kErrDrain = 4u;
constexpr uint32_t kErrRoute = 8u;  // an output row outside its tensor (write skipped)

// Thread layout of one GEMM phase: `rg` groups of `tpr` threads; a thread owns
// K slices s = t + tpr * i (16 bytes each) and the group owns 8 rows of an item.
struct PhaseGeom {
  int tpr;    // threads per row group (32..256, power of two)
  int rg;     // row groups (kComputeThreads / tpr)
  int nspt;   // K slices per thread (1..kMaxSlicesPerThread)
  int ns;     // K slices per row (K / 16)
};

// Sums V values per lane over a warp: afterwards every lane holds the warp sum
// of value index lane / (32 / V) in v[0]. V in {1, 2, 4, ..., 32}.
template <int V>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
#pragma unroll
  for (int step = V / 2, off = 16; step >= 1; step >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < step; ++k) {
      const float send = upper ? v[k] : v[k + step];
      const float keep = upper ? v[k + step] : v[k];
      v[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (int off = 16 / V; off >= 1; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  return s;
}

}  // namespace fme
