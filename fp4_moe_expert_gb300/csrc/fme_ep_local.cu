// Single-GPU forms of the expert-parallel dispatch quantiser and of the
// combine's reduction with RMSNorm ("vllm.models.kimi_k3.nvidia.
// specialized_decode.cutedsl.moe.ep.comm": EpDispatch, EpCombine, rms_rstd).
//
// MXFP8: two threads per 32-value block, 16 values each (two 16-byte loads of
// BF16, one 16-byte store of E4M3); the block's amax by one shuffle; shared
// exponent floor(log2(amax)) - 8 from the FP32 exponent field, clamped to
// [-127, 127] (zero and subnormal amax: -127); values times 2^-exponent
// (exact), E4M3 round-to-nearest-even with saturation; the E8M0 byte is
// exponent + 127.
//
// Combine + RMSNorm: one CTA per token; FP32 sum of the N partials in rank
// order, one BF16 rounding (the latent); FP32 sum of squares of the BF16
// latent; rstd = rsqrt(sum / H + eps) (IEEE divide, approximate rsqrt, as the
// page); out = bf16((x * rstd) * w).
#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

constexpr int kMxThreads = 256;
constexpr int kCombThreads = 256;
constexpr int kCombMaxChunks = 4;  // 8-column chunks per thread: H <= 8192

__global__ void __launch_bounds__(kMxThreads) mxfp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, int T,
                                                                     int H, uint8_t* __restrict__ q,
                                                                     uint8_t* __restrict__ sc) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int halves = H / 16;  // two per 32-value block
  const int i = blockIdx.x * kMxThreads + threadIdx.x;
  // Whole warps stay in the loop so the pair shuffle always has its partner.
  const bool live = i < T * halves;
  const int t = live ? i / halves : 0, hcol = live ? i - t * halves : 0;
  float v[16];
  float amax = 0.0f;
  if (live) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + 16 * hcol);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (!live) return;
  const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  const int e = ef == 0 ? -127 : max(-127, min(127, ef - 127 - 8));
  const float rescale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, -e in [-119, 127]
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out[k] = f32x2_to_e4m3x2(__fmul_rn(v[4 * k], rescale), __fmul_rn(v[4 * k + 1], rescale)) |
             (f32x2_to_e4m3x2(__fmul_rn(v[4 * k + 2], rescale), __fmul_rn(v[4 * k + 3], rescale)) << 16);
  *reinterpret_cast<uint4*>(q + static_cast<size_t>(t) * H + 16 * hcol) = make_uint4(out[0], out[1], out[2], out[3]);
  if ((hcol & 1) == 0) sc[static_cast<size_t>(t) * (H / 32) + hcol / 2] = static_cast<uint8_t>(e + 127);
}

__global__ void __launch_bounds__(kCombThreads) combine_rmsnorm_kernel(const __nv_bfloat16* __restrict__ partials,
                                                                       int N, int H,
                                                                       const __nv_bfloat16* __restrict__ gamma,
                                                                       float eps, __nv_bfloat16* __restrict__ latent,
                                                                       __nv_bfloat16* __restrict__ normed) {
  __shared__ float part[kCombThreads / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x, tid = threadIdx.x;
  const int chunks = H / 8;
  float x[kCombMaxChunks][8];
  float total = 0.0f;
#pragma unroll
  for (int j = 0; j < kCombMaxChunks; ++j) {
    const int ch = tid + j * kCombThreads;
    if (ch < chunks) {
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
      // Unrolled so that several ranks' loads are in flight; the sums stay in rank order.
#pragma unroll 8
      for (int d = 0; d < N; ++d) {
        const uint4 p = __ldcg(reinterpret_cast<const uint4*>(partials + (static_cast<size_t>(t) * N + d) * H) + ch);
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] = __fadd_rn(acc[2 * k], __uint_as_float(w[k] << 16));
          acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], __uint_as_float(w[k] & 0xFFFF0000u));
        }
      }
      uint32_t lw[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat16 lo = __float2bfloat16_rn(acc[2 * k]), hi = __float2bfloat16_rn(acc[2 * k + 1]);
        x[j][2 * k] = __bfloat162float(lo);
        x[j][2 * k + 1] = __bfloat162float(hi);
        lw[k] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
        total = __fadd_rn(total, __fadd_rn(__fmul_rn(x[j][2 * k], x[j][2 * k]), __fmul_rn(x[j][2 * k + 1], x[j][2 * k + 1])));
      }
      reinterpret_cast<uint4*>(latent + static_cast<size_t>(t) * H)[ch] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) total = __fadd_rn(total, __shfl_xor_sync(0xFFFFFFFFu, total, off));
  if ((tid & 31) == 0) part[tid >> 5] = total;
  __syncthreads();
  total = 0.0f;
#pragma unroll
  for (int w = 0; w < kCombThreads / 32; ++w) total = __fadd_rn(total, part[w]);
  const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(total, static_cast<float>(H)), eps));
#pragma unroll
  for (int j = 0; j < kCombMaxChunks; ++j) {
    const int ch = tid + j * kCombThreads;
    if (ch < chunks) {
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(gamma) + ch);
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      uint32_t ow[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = __fmul_rn(__fmul_rn(x[j][2 * k], rstd), __uint_as_float(gw[k] << 16));
        const float b = __fmul_rn(__fmul_rn(x[j][2 * k + 1], rstd), __uint_as_float(gw[k] & 0xFFFF0000u));
        ow[k] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
      }
      reinterpret_cast<uint4*>(normed + static_cast<size_t>(t) * H)[ch] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  }
}

static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int mxfp8_quantize(const void* x, int T, int H, uint8_t* q, uint8_t* scales, cudaStream_t st) {
  const long long threads = static_cast<long long>(T) * (H / 16);
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(static_cast<unsigned>((threads + kMxThreads - 1) / kMxThreads)), dim3(kMxThreads), st, attr);
  const cudaError_t err =
      cudaLaunchKernelEx(&cfg, mxfp8_quantize_kernel, static_cast<const __nv_bfloat16*>(x), T, H, q, scales);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "mxfp8 quantize launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

int combine_rmsnorm(const void* partials, int T, int N, int H, const void* gamma, float eps, void* latent,
                    void* normed, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(T)), dim3(kCombThreads), st, attr);
  const cudaError_t err = cudaLaunchKernelEx(
      &cfg, combine_rmsnorm_kernel, static_cast<const __nv_bfloat16*>(partials), N, H,
      static_cast<const __nv_bfloat16*>(gamma), eps, static_cast<__nv_bfloat16*>(latent),
      static_cast<__nv_bfloat16*>(normed));
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "combine rmsnorm launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

}  // namespace fme
