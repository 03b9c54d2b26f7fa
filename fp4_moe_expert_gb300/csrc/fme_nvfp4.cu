// NVFP4 slot MoE over one local expert range: one persistent sm_103a kernel.
//
// Computes what "nvfp4-megamoe-kernel README.md" describes (slot
// representation; Data Formats; Bugs Found & Fixed 2, 4, 6, 7): a slot is a
// (token, pick) pair whose expert is local; per slot the L1 GEMM on the
// [gate; up] weight, SiLU*Mul, re-quantisation to E2M1 with UE4M3 group-16
// scales, the L2 GEMM; the routing weights are applied once, in the final
// scatter to [M, H]. The design is this library's own:
//
// * One CTA per SM; every CTA derives the same ascending list of touched
//   local experts from topk_ids, so each touched expert streams once.
// * Phase 1 items: 4*rg gate rows plus the matching up rows of one expert
//   (packed E2M1 rows and their UE4M3 scale rows, both contiguous), so
//   SwiGLU finishes in the item. Output h (BF16 value) goes to the workspace.
// * Phase 2 items: 8*rg rows of W2; they wait (bounded) for all phase-1 items
//   of their expert, quantise h per 16 themselves and write the slot outputs
//   o (BF16) to the workspace.
// * Phase 3: every CTA waits (bounded) for all phase-2 items, then sums, for
//   its slice of columns, w[t, r] * o[slot] over the token's local picks in
//   ascending order in FP32 and stores y once as BF16.
// * Weight rows stream through the same cp.async.bulk ring as the FP8
//   kernel; the math is cvt.rn.f16x2.e2m1x2 plus fma.rn.f32.f16 (exact
//   products, exact group sums), times the exact product of the two UE4M3
//   scales of each group.
#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

struct Fp4Args {
  const __nv_bfloat16* x;
  const int32_t* ids;
  const float* tw;  // topk weights
  const uint8_t* w13;
  const uint8_t* s13;
  const uint8_t* w2;
  const uint8_t* s2;
  __nv_bfloat16* y;
  uint32_t* err;
  uint32_t* done;      // [L] phase-1 items completed per local expert
  uint32_t* consumed;  // [L] phase-2 items that passed the wait
  uint32_t* done2;     // phase-2 items completed (all experts)
  uint32_t* passed3;   // CTAs past the phase-3 wait
  float* hbuf;         // [routes, N] SwiGLU output (BF16 values)
  __nv_bfloat16* obuf; // [routes, H] slot outputs
  int M, H, N, L, e0, top_k;
  float limit;
  PhaseGeom g1, g2;  // slices are 16 packed bytes = 32 values
  int gp, r2;
  unsigned long long timeout_ns;
};

constexpr int kFp4Slice = 32;  // values per 16-byte slice

struct Fp4Smem {
  uint8_t ring[kStages][kStageBytes];
  uint64_t full[kStages];
  unsigned long long tokmask[kMaxExperts];
  int16_t ulist[kMaxExperts];
  float red[kComputeWarps][32];
  float ysum[64][kTokChunk];
  int16_t ctx_route[kMaxTokens];
  int16_t ctx_tok[kMaxTokens];
  int ctx_n;
  int U;
  volatile int abort;
};

constexpr size_t kFp4SmemBytes = sizeof(Fp4Smem) + 1024;

__device__ __forceinline__ void fp4_error(const Fp4Args& a, Fp4Smem& S, uint32_t bit) {
  atomicOr(a.err, bit);
  S.abort = 1;
}

__device__ __forceinline__ void fp4_bar() { named_bar_sync(1, kComputeThreads); }

// E4M3 byte (UE4M3 scale) of amax / 6 and the value it stores.
__device__ __forceinline__ float fp4_group_scale(float amax, uint32_t& byte) {
  byte = f32x2_to_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu;
  return e4m3_to_f32(byte);
}

// Quantise 32 values (two groups of 16) to E2M1 nibbles with their group
// scales, as exact f16 pairs: "nvfp4-megamoe-kernel README.md" Bugs Found &
// Fixed 2 (stored scale = block_max / 6, also the divisor; signed E2M1).
__device__ __forceinline__ void fp4_quant32(const float (&v)[32], uint32_t (&out)[16], float (&sc)[2]) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[16 * g + k]));
    uint32_t byte;
    const float d = fp4_group_scale(amax, byte);
    sc[g] = d;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t nib = 0u;
      if (d > 0.0f) nib = f32x2_to_e2m1x2(__fdiv_rn(v[16 * g + 2 * k], d), __fdiv_rn(v[16 * g + 2 * k + 1], d));
      out[8 * g + k] = e2m1x2_to_f16x2(nib);
    }
  }
}

template <int RTC>
__device__ __forceinline__ void fp4_quant_x(const Fp4Args& a, const Fp4Smem& S, int c0, int rt, int gt,
                                            uint32_t (&xa)[kTokChunk][16], float (&xs)[kTokChunk][2]) {
  const PhaseGeom& g = a.g1;
  const int s = gt;
#pragma unroll
  for (int t = 0; t < RTC; ++t) {
    if (s < g.ns && t < rt) {
      const int tok = S.ctx_tok[c0 + t];
      const uint4* p = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * a.H + kFp4Slice * s);
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = __ldg(p + q);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[8 * q + 2 * k] = __uint_as_float(ww[k] << 16);
          v[8 * q + 2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
        }
      }
      fp4_quant32(v, xa[t], xs[t]);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) xa[t][k] = 0u;
      xs[t][0] = xs[t][1] = 0.0f;
    }
  }
}

template <int RTC>
__device__ __forceinline__ void fp4_quant_h(const Fp4Args& a, const Fp4Smem& S, int c0, int rt, int gt,
                                            uint32_t (&xa)[kTokChunk][16], float (&xs)[kTokChunk][2]) {
  const PhaseGeom& g = a.g2;
  const int s = gt;
#pragma unroll
  for (int t = 0; t < RTC; ++t) {
    if (s < g.ns && t < rt) {
      const int route = S.ctx_route[c0 + t];
      const float4* p = reinterpret_cast<const float4*>(a.hbuf + static_cast<size_t>(route) * a.N + kFp4Slice * s);
      float v[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldcg(p + q);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
      }
      fp4_quant32(v, xa[t], xs[t]);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) xa[t][k] = 0u;
      xs[t][0] = xs[t][1] = 0.0f;
    }
  }
}

// acc[q * RTC + t] += dot of row (row0 + q) slice s with token t, per group
// times (weight group scale * activation group scale).
template <int RTC>
__device__ __forceinline__ void fp4_dot_rows(const uint8_t* packed, const uint8_t* scales, int rowbytes,
                                             int scalebytes, int row0, int s, int ns,
                                             const uint32_t (&xa)[kTokChunk][16], const float (&xs)[kTokChunk][2],
                                             float (&acc)[kRowsPerGroup * RTC]) {
  if (s >= ns) return;
#pragma unroll
  for (int q = 0; q < kRowsPerGroup; ++q) {
    const int row = row0 + q;
    const uint4 w = *reinterpret_cast<const uint4*>(packed + static_cast<size_t>(row) * rowbytes + 16 * s);
    const uint32_t sb = *reinterpret_cast<const uint16_t*>(scales + static_cast<size_t>(row) * scalebytes + 2 * s);
    const float sw0 = e4m3_to_f32(sb & 0xFFu), sw1 = e4m3_to_f32(sb >> 8);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint32_t wf[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int b = 0; b < 4; ++b) wf[4 * k + b] = e2m1x2_to_f16x2(ww[k] >> (8 * b));
    }
#pragma unroll
    for (int t = 0; t < RTC; ++t) {
      float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) p0 = fma_f16x2_f32(wf[k], xa[t][k], p0);
#pragma unroll
      for (int k = 8; k < 16; ++k) p1 = fma_f16x2_f32(wf[k], xa[t][k], p1);
      acc[q * RTC + t] = fmaf(p0, __fmul_rn(sw0, xs[t][0]), acc[q * RTC + t]);
      acc[q * RTC + t] = fmaf(p1, __fmul_rn(sw1, xs[t][1]), acc[q * RTC + t]);
    }
  }
}

__device__ void fp4_context(const Fp4Args& a, Fp4Smem& S, int le, int ctid) {
  if (ctid < 32) {
    const int lane = ctid;
    const unsigned long long mask = S.tokmask[le];
    int base = 0;
    for (int t0 = 0; t0 < a.M; t0 += 32) {
      const int t = t0 + lane;
      const bool has = (t < a.M) && ((mask >> t) & 1ull);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
      if (has) {
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        int r = 0;
        for (int k = 0; k < a.top_k; ++k)
          if (__ldg(a.ids + t * a.top_k + k) - a.e0 == le) r = k;
        S.ctx_route[pos] = static_cast<int16_t>(t * a.top_k + r);
        S.ctx_tok[pos] = static_cast<int16_t>(t);
      }
      base += __popc(bal);
    }
    if (lane == 0) S.ctx_n = base;
  }
  fp4_bar();
}

template <int RTC>
__device__ __forceinline__ void fp4_reduce(Fp4Smem& S, float (&acc)[kRowsPerGroup * RTC], int warp, int lane) {
  constexpr int V = kRowsPerGroup * RTC;
  const float s = warp_transpose_sum<V>(acc, lane);
  if ((lane % (32 / V)) == 0) S.red[warp][lane / (32 / V)] = s;
}

template <int RTC>
__device__ void fp4_gemm1_chunk(const Fp4Args& a, Fp4Smem& S, const uint8_t* stage, int h0, int c0, int rt,
                                bool requant, int ctid, int warp, int lane, uint32_t (&xa)[kTokChunk][16],
                                float (&xs)[kTokChunk][2]) {
  const PhaseGeom& g = a.g1;
  const int grp = ctid / g.tpr, gt = ctid % g.tpr;
  if (requant) fp4_quant_x<RTC>(a, S, c0, rt, gt, xa, xs);
  float acc[kRowsPerGroup * RTC];
#pragma unroll
  for (int v = 0; v < kRowsPerGroup * RTC; ++v) acc[v] = 0.0f;
  const int rows = 2 * a.gp;
  const uint8_t* scales = stage + static_cast<size_t>(rows) * (a.H / 2);
  fp4_dot_rows<RTC>(stage, scales, a.H / 2, a.H / 16, grp * kRowsPerGroup, gt, g.ns, xa, xs, acc);
  fp4_reduce<RTC>(S, acc, warp, lane);
  fp4_bar();
  constexpr int V = kRowsPerGroup * RTC;
  const int wpg = g.tpr / 32;
  if (ctid < g.rg * V) {
    const int fg = ctid / V, v = ctid % V;
    float s = 0.0f;
    for (int w = 0; w < wpg; ++w) s += S.red[fg * wpg + w][v];
    S.ysum[fg * kRowsPerGroup + v / RTC][v % RTC] = s;
  }
  fp4_bar();
  if (ctid < a.gp * RTC && ctid % RTC < rt) {
    const int q = ctid / RTC, t = ctid % RTC;
    // L1 rows: [gate; up] (README Bugs Found & Fixed 4); L1 output is BF16.
    const float gate = __bfloat162float(__float2bfloat16_rn(S.ysum[q][t]));
    const float up = __bfloat162float(__float2bfloat16_rn(S.ysum[a.gp + q][t]));
    const float L = a.limit;
    const float gc = fminf(gate, L);
    const float uc = fmaxf(fminf(up, L), -L);
    const float silu = __fdiv_rn(gc, __fadd_rn(1.0f, expf(-gc)));
    const float h = __bfloat162float(__float2bfloat16_rn(__fmul_rn(silu, uc)));
    a.hbuf[static_cast<size_t>(S.ctx_route[c0 + t]) * a.N + h0 + q] = h;
  }
  fp4_bar();
}

template <int RTC>
__device__ void fp4_gemm2_chunk(const Fp4Args& a, Fp4Smem& S, const uint8_t* stage, int m0, int c0, int rt,
                                bool requant, int ctid, int warp, int lane, uint32_t (&xa)[kTokChunk][16],
                                float (&xs)[kTokChunk][2]) {
  const PhaseGeom& g = a.g2;
  const int grp = ctid / g.tpr, gt = ctid % g.tpr;
  if (requant) fp4_quant_h<RTC>(a, S, c0, rt, gt, xa, xs);
  float acc[kRowsPerGroup * RTC];
#pragma unroll
  for (int v = 0; v < kRowsPerGroup * RTC; ++v) acc[v] = 0.0f;
  const uint8_t* scales = stage + static_cast<size_t>(a.r2) * (a.N / 2);
  fp4_dot_rows<RTC>(stage, scales, a.N / 2, a.N / 16, grp * kRowsPerGroup, gt, g.ns, xa, xs, acc);
  fp4_reduce<RTC>(S, acc, warp, lane);
  fp4_bar();
  constexpr int V = kRowsPerGroup * RTC;
  const int wpg = g.tpr / 32;
  if (ctid < g.rg * V && (ctid % V) % RTC < rt) {
    const int fg = ctid / V, v = ctid % V;
    float s = 0.0f;
    for (int w = 0; w < wpg; ++w) s += S.red[fg * wpg + w][v];
    const int m = m0 + fg * kRowsPerGroup + v / RTC;
    a.obuf[static_cast<size_t>(S.ctx_route[c0 + v % RTC]) * a.H + m] = __float2bfloat16_rn(s);
  }
  fp4_bar();
}

struct Fp4Plan {
  long long lo1, hi1, lo2, hi2;
  int per_u1, per_u2;
  __device__ int count() const { return static_cast<int>((hi1 - lo1) + (hi2 - lo2)); }
};

__device__ void fp4_issue(const Fp4Args& a, Fp4Smem& S, const Fp4Plan& P, int it, uint64_t pol) {
  const int s = it % kStages;
  uint8_t* dst = S.ring[s];
  if (it < P.hi1 - P.lo1) {
    const long long i = P.lo1 + it;
    const int u = static_cast<int>(i / P.per_u1);
    const int h0 = static_cast<int>(i % P.per_u1) * a.gp;
    const int le = S.ulist[u];
    const uint32_t pb = static_cast<uint32_t>(a.gp) * (a.H / 2);   // packed bytes per half
    const uint32_t sb = static_cast<uint32_t>(a.gp) * (a.H / 16);  // scale bytes per half
    mbar_arrive_expect_tx(&S.full[s], 2 * (pb + sb));
    const size_t row_g = static_cast<size_t>(le) * 2 * a.N + h0;    // first gate row
    const size_t row_u = row_g + a.N;                               // first up row
    bulk_g2s(dst, a.w13 + row_g * (a.H / 2), pb, &S.full[s], pol);
    bulk_g2s(dst + pb, a.w13 + row_u * (a.H / 2), pb, &S.full[s], pol);
    bulk_g2s(dst + 2 * pb, a.s13 + row_g * (a.H / 16), sb, &S.full[s], pol);
    bulk_g2s(dst + 2 * pb + sb, a.s13 + row_u * (a.H / 16), sb, &S.full[s], pol);
  } else {
    const long long i = P.lo2 + (it - (P.hi1 - P.lo1));
    const int u = static_cast<int>(i / P.per_u2), rb = static_cast<int>(i % P.per_u2);
    const int le = S.ulist[u];
    const uint32_t pb = static_cast<uint32_t>(a.r2) * (a.N / 2);
    const uint32_t sb = static_cast<uint32_t>(a.r2) * (a.N / 16);
    mbar_arrive_expect_tx(&S.full[s], pb + sb);
    const size_t row = static_cast<size_t>(le) * a.H + static_cast<size_t>(rb) * a.r2;
    bulk_g2s(dst, a.w2 + row * (a.N / 2), pb, &S.full[s], pol);
    bulk_g2s(dst + pb, a.s2 + row * (a.N / 16), sb, &S.full[s], pol);
  }
}

__device__ __forceinline__ bool fp4_wait_stage(const Fp4Args& a, Fp4Smem& S, int it) {
  if (!mbar_wait(&S.full[it % kStages], (it / kStages) & 1, a.timeout_ns, &S.abort)) {
    if (!S.abort) fp4_error(a, S, kErrRingWait);
  }
  fp4_bar();
  return !S.abort;
}

__device__ void fp4_drain(const Fp4Args& a, Fp4Smem& S, const Fp4Plan& P, int consumed) {
  if (threadIdx.x != 0) return;
  const int issued = min(P.count(), consumed + kStages);
  for (int k = consumed; k < issued; ++k)
    if (!mbar_wait(&S.full[k % kStages], (k / kStages) & 1, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
}

__device__ bool wait_counter(const Fp4Args& a, Fp4Smem& S, const uint32_t* ctr, uint32_t target) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(ctr) < target) {
      if (globaltimer_ns() - t0 > a.timeout_ns) {
        fp4_error(a, S, kErrCrossWait);
        break;
      }
      __nanosleep(64);
    }
  }
  fp4_bar();
  return !S.abort;
}

__global__ void __launch_bounds__(kThreads, 1) nvfp4_moe_kernel(const __grid_constant__ Fp4Args a) {
  extern __shared__ uint8_t smem_raw[];
  Fp4Smem& S = *reinterpret_cast<Fp4Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    S.abort = 0;
  }
  for (int e = tid; e < a.L; e += kThreads) S.tokmask[e] = 0ull;
  griddep_wait();
  __syncthreads();
  // Local slots: picks whose expert lies in [e0, e0 + L).
  for (int i = tid; i < a.M * a.top_k; i += kThreads) {
    const int le = __ldg(a.ids + i) - a.e0;
    if (le >= 0 && le < a.L) atomicOr(&S.tokmask[le], 1ull << (i / a.top_k));
  }
  __syncthreads();
  if (warp == 0) {
    int U = 0;
    for (int b = 0; b < a.L; b += 32) {
      const int e = b + lane;
      const bool has = (e < a.L) && (S.tokmask[e] != 0ull);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
      if (has) S.ulist[U + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(e);
      U += __popc(bal);
    }
    if (lane == 0) S.U = U;
  }
  __syncthreads();

  const int U = S.U;
  const int G = gridDim.x, c = blockIdx.x;
  Fp4Plan P;
  P.per_u1 = a.N / a.gp;
  P.per_u2 = a.H / a.r2;
  const long long n1 = static_cast<long long>(U) * P.per_u1, n2 = static_cast<long long>(U) * P.per_u2;
  P.lo1 = n1 * c / G;
  P.hi1 = n1 * (c + 1) / G;
  P.lo2 = n2 * c / G;
  P.hi2 = n2 * (c + 1) / G;
  const int n_items = P.count();

  uint64_t pol = 0;
  if (tid == 0 && n_items > 0) {
    pol = l2_evict_first_policy();
    for (int it = 0; it < min(kStages, n_items); ++it) fp4_issue(a, S, P, it, pol);
  }
  const int ctid = tid;
  uint32_t xa[kTokChunk][16];
  float xs[kTokChunk][2];
#pragma unroll
  for (int t = 0; t < kTokChunk; ++t) {
    xs[t][0] = xs[t][1] = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) xa[t][k] = 0u;
  }

  int it = 0, cur_u = -1;
  for (long long i = P.lo1; i < P.hi1; ++i, ++it) {
    const int u = static_cast<int>(i / P.per_u1);
    const int h0 = static_cast<int>(i % P.per_u1) * a.gp;
    const int le = S.ulist[u];
    bool fresh = false;
    if (u != cur_u) {
      fp4_context(a, S, le, ctid);
      cur_u = u;
      fresh = true;
    }
    if (!fp4_wait_stage(a, S, it)) {
      fp4_drain(a, S, P, it);
      return;
    }
    const int nt = S.ctx_n;
    const uint8_t* stage = S.ring[it % kStages];
    for (int c0 = 0; c0 < nt; c0 += kTokChunk) {
      const int rt = min(kTokChunk, nt - c0);
      const bool requant = fresh || nt > kTokChunk;
      switch (rt) {
        case 1: fp4_gemm1_chunk<1>(a, S, stage, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        case 2: fp4_gemm1_chunk<2>(a, S, stage, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        default: fp4_gemm1_chunk<4>(a, S, stage, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
      }
    }
    if (ctid == 0) {
      __threadfence();
      red_release_gpu_add(a.done + le, 1u);
      if (it + kStages < n_items) {
        fence_proxy_async_smem();
        fp4_issue(a, S, P, it + kStages, pol);
      }
    }
  }

  cur_u = -1;
  for (long long i = P.lo2; i < P.hi2; ++i, ++it) {
    const int u = static_cast<int>(i / P.per_u2), rb = static_cast<int>(i % P.per_u2);
    const int le = S.ulist[u];
    const int m0 = rb * a.r2;
    bool fresh = false;
    if (u != cur_u) {
      fp4_context(a, S, le, ctid);
      if (!wait_counter(a, S, a.done + le, static_cast<uint32_t>(P.per_u1))) {
        fp4_drain(a, S, P, it);
        return;
      }
      cur_u = u;
      fresh = true;
    }
    if (!fp4_wait_stage(a, S, it)) {
      fp4_drain(a, S, P, it);
      return;
    }
    const int nt = S.ctx_n;
    const uint8_t* stage = S.ring[it % kStages];
    for (int c0 = 0; c0 < nt; c0 += kTokChunk) {
      const int rt = min(kTokChunk, nt - c0);
      const bool requant = fresh || nt > kTokChunk;
      switch (rt) {
        case 1: fp4_gemm2_chunk<1>(a, S, stage, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        case 2: fp4_gemm2_chunk<2>(a, S, stage, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        default: fp4_gemm2_chunk<4>(a, S, stage, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
      }
    }
    if (ctid == 0) {
      __threadfence();
      red_release_gpu_add(a.done2, 1u);
      const uint32_t old = atomicAdd(a.consumed + le, 1u);
      if (old + 1u == static_cast<uint32_t>(P.per_u2)) {
        atomicExch(a.done + le, 0u);
        atomicExch(a.consumed + le, 0u);
      }
      if (it + kStages < n_items) {
        fence_proxy_async_smem();
        fp4_issue(a, S, P, it + kStages, pol);
      }
    }
  }

  // ---- phase 3: y[t, m] = bf16(sum over t's local picks, ascending, of w * o)
  if (!wait_counter(a, S, a.done2, static_cast<uint32_t>(n2))) return;
  const int chunks = a.H / 8;  // 8 columns (16 bytes of BF16) per thread item
  const int per_cta = (chunks + G - 1) / G;
  const int ch0 = c * per_cta, nch = max(0, min(chunks, ch0 + per_cta) - ch0);
  for (int w = tid; w < a.M * nch; w += kThreads) {
    const int tt = w / nch;
    const int ch = ch0 + w % nch;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    for (int r = 0; r < a.top_k; ++r) {
      const int le = __ldg(a.ids + tt * a.top_k + r) - a.e0;
      if (le < 0 || le >= a.L) continue;
      const float wt = __ldg(a.tw + tt * a.top_k + r);
      const uint4 o = __ldcg(reinterpret_cast<const uint4*>(a.obuf + static_cast<size_t>(tt * a.top_k + r) * a.H + 8 * ch));
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[2 * k] = __fadd_rn(acc[2 * k], __fmul_rn(wt, __uint_as_float(ow[k] << 16)));
        acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], __fmul_rn(wt, __uint_as_float(ow[k] & 0xFFFF0000u)));
      }
    }
    uint4 out;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k + 1]));
      ow[k] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(a.y + static_cast<size_t>(tt) * a.H + 8 * ch) = out;
  }
  __syncthreads();
  if (tid == 0) {
    // The last CTA past the phase-3 wait re-arms the global counters.
    const uint32_t old = atomicAdd(a.passed3, 1u);
    if (old + 1u == static_cast<uint32_t>(G)) {
      atomicExch(a.done2, 0u);
      atomicExch(a.passed3, 0u);
    }
  }
}

// ---------------------------------------------------------------- host side
static PhaseGeom fp4_geom(int K) {
  PhaseGeom g;
  g.ns = K / kFp4Slice;
  int tpr = 32;
  while (tpr < g.ns && tpr < kComputeThreads) tpr *= 2;
  g.tpr = tpr;
  g.rg = kComputeThreads / tpr;
  g.nspt = (g.ns + tpr - 1) / tpr;
  return g;
}

struct Fp4Workspace {
  uint32_t *err, *done, *consumed, *done2, *passed3;
  float* hbuf;
  __nv_bfloat16* obuf;
  size_t bytes;
};

static size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

static Fp4Workspace fp4_layout(void* base, int M, int H, int N, int L, int top_k) {
  Fp4Workspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.err = reinterpret_cast<uint32_t*>(p + off);
  off += 256;
  w.done = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L));
  w.consumed = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L));
  w.done2 = reinterpret_cast<uint32_t*>(p + off);
  w.passed3 = w.done2 + 1;
  off += 256;
  const size_t routes = static_cast<size_t>(M) * top_k;
  w.hbuf = reinterpret_cast<float*>(p + off);
  off += a256(4 * routes * N);
  w.obuf = reinterpret_cast<__nv_bfloat16*>(p + off);
  off += a256(2 * routes * H);
  w.bytes = off;
  return w;
}

size_t nvfp4_workspace_bytes(int M, int H, int N, int L, int top_k) {
  return fp4_layout(nullptr, M, H, N, L, top_k).bytes;
}

int routed_nvfp4(const void* x, const int32_t* ids, const float* weights, const uint8_t* w13, const uint8_t* s13,
                 const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int e0, int top_k, float limit,
                 void* y, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  const Fp4Workspace w = fp4_layout(workspace, M, H, N, L, top_k);
  if (workspace == nullptr || workspace_bytes < w.bytes)
    return set_last_error(FME_EWORKSPACE, "workspace of %zu bytes needed, %zu given", w.bytes, workspace_bytes);
  Fp4Args a = {};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ids = ids;
  a.tw = weights;
  a.w13 = w13;
  a.s13 = s13;
  a.w2 = w2;
  a.s2 = s2;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.err = w.err;
  a.done = w.done;
  a.consumed = w.consumed;
  a.done2 = w.done2;
  a.passed3 = w.passed3;
  a.hbuf = w.hbuf;
  a.obuf = w.obuf;
  a.M = M;
  a.H = H;
  a.N = N;
  a.L = L;
  a.e0 = e0;
  a.top_k = top_k;
  a.limit = limit;
  a.g1 = fp4_geom(H);
  a.g2 = fp4_geom(N);
  a.gp = kRowsPerGroup * a.g1.rg / 2;
  a.r2 = kRowsPerGroup * a.g2.rg;
  a.timeout_ns = wait_timeout_ns();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_last_error(FME_ECUDA, "cudaGetDevice failed");
  const int sms = device_sm_count(dev);
  if (sms <= 0) return set_last_error(FME_ECUDA, "cannot query the SM count");
  if (!ensure_smem_attr(dev, reinterpret_cast<const void*>(nvfp4_moe_kernel), kFp4SmemBytes)) return FME_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kFp4SmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, nvfp4_moe_kernel, a);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "nvfp4 kernel launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

}  // namespace fme
