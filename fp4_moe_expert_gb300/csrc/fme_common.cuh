// Pieces shared by the kernels: size limits, device error bits and the
// routing rule.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fme_ptx.cuh"

namespace fme {

constexpr int kMaxHidden = 8192;                   // H and I bound of the FP8 entry points
constexpr int kMaxTokens = 64;                     // token bit masks are uint64
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kFp8MaxCtas = 160;                 // grid cap of the FP8 kernel (partial slots)

// Device error bits (workspace error word).
constexpr uint32_t kErrRingWait = 1u;  // a ring stage never landed
constexpr uint32_t kErrCrossWait = 2u;
constexpr uint32_t kErrDrain = 4u;
constexpr uint32_t kErrRoute = 8u;  // an output row outside its tensor (write skipped)

// ---------------------------------------------------------------- routing
// One warp routes token t ("mega_moe" _MegaKernel.top_k_pick): sigmoid scores
// (accurate expf, IEEE divide), keys score + bias as monotone uint32, top_k
// rounds of warp max key then lowest expert among equals, weights
// score / (float sum in pick order) * scale. Lane l holds experts l + 32 j in
// registers; every load is issued before any sigmoid. Lane r < top_k gets
// rank r's expert and weight.
template <int J>
__device__ void route_topk(const void* logits, bool logits_f32, const float* bias, int E, int top_k, float scale,
                           int t, int lane, int& my_e, float& my_w) {
  float lg[J], bs[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = lane + 32 * j;
    lg[j] = 0.0f;
    bs[j] = 0.0f;
    if (e < E) {
      if (logits_f32)
        lg[j] = __ldg(static_cast<const float*>(logits) + static_cast<size_t>(t) * E + e);
      else
        lg[j] = __bfloat162float(static_cast<const __nv_bfloat16*>(logits)[static_cast<size_t>(t) * E + e]);
      bs[j] = __ldg(bias + e);
    }
  }
  uint32_t ky[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const float sgm = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-lg[j])));
    lg[j] = sgm;  // score
    ky[j] = (lane + 32 * j < E) ? ordered_key(__fadd_rn(sgm, bs[j])) : 0u;
  }
  float total = 0.0f, mine = 0.0f;
  int mine_e = 0;
  for (int r = 0; r < top_k; ++r) {
    uint32_t best = 0u;
#pragma unroll
    for (int j = 0; j < J; ++j) best = max(best, ky[j]);
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
    uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
    for (int j = J - 1; j >= 0; --j)
      if (ky[j] == top) cand = static_cast<uint32_t>(lane + 32 * j);
    const int win = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
    float sv = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (lane + 32 * j == win) {
        sv = lg[j];
        ky[j] = 0u;
      }
    const float s = __shfl_sync(0xFFFFFFFFu, sv, win & 31);
    total = __fadd_rn(total, s);
    if (lane == r) {
      mine = s;
      mine_e = win;
    }
  }
  my_e = mine_e;
  my_w = __fmul_rn(__fdiv_rn(mine, total), scale);
}

// The same picks and weights as route_topk, bit for bit, with the keys and
// scores of one token in shared memory (2 * E words at `scratch`) instead of
// registers: short code for any E <= kMaxExperts, for kernels where one warp
// routes one token and the code size of the register version costs more
// than its speed saves.
inline __device__ void route_topk_smem(const void* logits, bool logits_f32, const float* bias, int E, int top_k,
                                float scale, int t, int lane, uint32_t* scratch, int& my_e, float& my_w) {
  uint32_t* key = scratch;
  float* score = reinterpret_cast<float*>(scratch + E);
  // Eight experts per lane per pass, every load of a pass issued first.
#pragma unroll 1
  for (int e0 = lane; e0 < E; e0 += 256) {
    float l[8], b[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = e0 + 32 * q;
      l[q] = 0.0f;
      b[q] = 0.0f;
      if (e < E) {
        l[q] = logits_f32 ? __ldg(static_cast<const float*>(logits) + static_cast<size_t>(t) * E + e)
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(logits)[static_cast<size_t>(t) * E + e]);
        b[q] = __ldg(bias + e);
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = e0 + 32 * q;
      if (e < E) {
        const float sgm = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l[q])));
        score[e] = sgm;
        key[e] = ordered_key(__fadd_rn(sgm, b[q]));
      }
    }
  }
  __syncwarp();
  float total = 0.0f, mine = 0.0f;
  int mine_e = 0;
#pragma unroll 1
  for (int r = 0; r < top_k; ++r) {
    uint32_t best = 0u;
    int bi = -1;
#pragma unroll 4
    for (int e = lane; e < E; e += 32) {
      const uint32_t k = key[e];
      if (k > best) {
        best = k;
        bi = e;
      }
    }
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
    const uint32_t cand = (best == top && bi >= 0) ? static_cast<uint32_t>(bi) : 0xFFFFFFFFu;
    const int win = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
    const float sv = score[win];
    __syncwarp();
    if (lane == (win & 31)) key[win] = 0u;
    __syncwarp();
    total = __fadd_rn(total, sv);
    if (lane == r) {
      mine = sv;
      mine_e = win;
    }
  }
  my_e = mine_e;
  my_w = __fmul_rn(__fdiv_rn(mine, total), scale);
}

}  // namespace fme
