// Local finalize of the routed layer: y[t] = bf16(sum over r ascending of
// w[t, r] * out[t * k + r] (+ shared_out[t])), each product and each sum one
// FP32 rounding, one BF16 rounding at the end.
//
// "vllm.models.glm5next.nvidia.specialized_decode.mega_moe" writes the
// unweighted expert rows (row t * top_k + r) and the routing weights for a
// finalize step to combine; "vllm.models.kimi_k3.nvidia.specialized_decode.
// cutedsl.moe.ep.comm" (EpCombine) states the combine: the routing-weighted
// sum, an FP32 sum in a fixed order, rounded once to BF16.
//
// HBM / L2 bound and tiny (M * (k + 2) * H * 2 bytes): one thread per 8
// columns (16 bytes) of one token, coalesced along H; launched with
// programmatic stream serialization so its launch overlaps the routed
// kernel's tail, and it waits (griddepcontrol) before reading that kernel's
// rows.
#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

constexpr int kFinThreads = 256;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const __nv_bfloat16* __restrict__ out,
                                                                const float* __restrict__ w,
                                                                const __nv_bfloat16* __restrict__ shared_out,
                                                                int M, int H, int k, __nv_bfloat16* __restrict__ y) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int chunks = H / 8;
  const int i = blockIdx.x * kFinThreads + threadIdx.x;
  if (i >= M * chunks) return;
  const int t = i / chunks, c = i - t * chunks;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  for (int r = 0; r < k; ++r) {
    const float wt = __ldg(w + static_cast<size_t>(t) * k + r);
    const uint4 o = __ldcg(reinterpret_cast<const uint4*>(out + (static_cast<size_t>(t) * k + r) * H) + c);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = __fadd_rn(acc[2 * j], __fmul_rn(wt, __uint_as_float(ow[j] << 16)));
      acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __fmul_rn(wt, __uint_as_float(ow[j] & 0xFFFF0000u)));
    }
  }
  if (shared_out != nullptr) {
    const uint4 s = __ldcg(reinterpret_cast<const uint4*>(shared_out + static_cast<size_t>(t) * H) + c);
    const uint32_t sw[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(sw[j] << 16));
      acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(sw[j] & 0xFFFF0000u));
    }
  }
  uint4 res;
  uint32_t* rw = reinterpret_cast<uint32_t*>(&res);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j + 1]));
    rw[j] = lo | (hi << 16);
  }
  reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H)[c] = res;
}

int finalize(const void* out, const float* weights, const void* shared_out, int M, int H, int top_k, void* y,
             cudaStream_t st) {
  const long long items = static_cast<long long>(M) * (H / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((items + kFinThreads - 1) / kFinThreads));
  cfg.blockDim = dim3(kFinThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err =
      cudaLaunchKernelEx(&cfg, finalize_kernel, static_cast<const __nv_bfloat16*>(out), weights,
                         static_cast<const __nv_bfloat16*>(shared_out), M, H, top_k, static_cast<__nv_bfloat16*>(y));
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "finalize kernel launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

}  // namespace fme
