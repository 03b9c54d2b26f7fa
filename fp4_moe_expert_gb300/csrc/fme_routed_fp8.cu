// Routed FP8 MoE layer and FP8 shared expert: one persistent sm_103a kernel.
//
// Computes what "vllm.models.glm5next.nvidia.specialized_decode.mega_moe"
// (MegaExperts / _MegaKernel) and ".../shared_expert" (SharedExpert,
// _GateUpKernel, _DownKernel, _group_scale) define; the design is this
// library's own:
//
// * One CTA per SM. Every CTA redoes the routing of all M tokens (warp per
//   token) and derives the same ascending list of the unique experts touched,
//   so each touched expert's weights stream from HBM once per call whatever
//   the number of routes that picked it (the page streams per route).
// * Work items: GEMM1 items are 4*rg rows of "first half" W13 rows plus the
//   matching 4*rg rows of the second half (so SwiGLU finishes inside the
//   item); GEMM2 items are 8*rg rows of W2. Every CTA owns an equal slice of
//   the GEMM1 items, then an equal slice of the GEMM2 items.
// * Thread 0 streams each item's rows with cp.async.bulk into a 3-stage
//   shared-memory ring (one mbarrier per stage, L2 evict-first), kStages
//   items ahead of the compute; every item ends on a CTA barrier, after which
//   its stage is refilled, also across the GEMM1 -> GEMM2 boundary.
// * Eight warps hold the quantised activations of up to four tokens
//   in registers (as exact f16 pairs) and stream weight rows from the ring:
//   cvt.rn.f16x2.e4m3x2 then fma.rn.f32.f16 (exact products, f32 sums); each
//   16-element partial is multiplied by its block's (weight scale * activation
//   scale) product, and a warp transpose-reduction plus a fixed-order
//   cross-warp sum give each row's dot product.
// * GEMM1 items write the SwiGLU output (f32) to the workspace and release a
//   per-expert counter; GEMM2 items wait (bounded) for all GEMM1 items of
//   their expert, then quantise the hidden per 128 themselves.
#include <cstdio>

#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

enum : int { kModeRouted = 0, kModeShared = 1 };

struct Fp8Args {
  const __nv_bfloat16* x;
  const void* logits;
  const float* bias;
  const uint8_t* w13;
  const float* s13;
  const uint8_t* w2;
  const float* s2;
  __nv_bfloat16* out;
  int32_t* ids;
  float* weights;
  __nv_bfloat16* gate_up;  // shared mode, optional
  uint32_t* err;
  uint32_t* done;      // [E] GEMM1 items completed per expert
  uint32_t* consumed;  // [E] GEMM2 items that passed the wait
  float* hbuf;         // [routes, I] SwiGLU output
  int M, H, I, E, top_k;
  float limit, scale;
  int ue8m0, logits_f32, mode;
  PhaseGeom g1, g2;
  int gp;  // first-half rows per GEMM1 item (the item has 2 * gp rows)
  int r2;  // rows per GEMM2 item
  unsigned long long timeout_ns;
};

struct Fp8Smem {
  uint8_t ring[kStages][kStageBytes];
  uint64_t full[kStages];
  unsigned long long tokmask[kMaxExperts];
  int16_t rid[kMaxTokens * kMaxTopK];
  int16_t ulist[kMaxExperts];
  float red[kComputeWarps][32];
  float ysum[64][kTokChunk];
  int16_t ctx_route[kMaxTokens];
  int16_t ctx_tok[kMaxTokens];
  int ctx_n;
  int U;
  volatile int abort;
};

constexpr size_t kFp8SmemBytes = sizeof(Fp8Smem) + 1024;

__device__ __forceinline__ void set_error(const Fp8Args& a, Fp8Smem& S, uint32_t bit) {
  atomicOr(a.err, bit);
  S.abort = 1;
}

// ---------------------------------------------------------------- routing
// One warp routes token t ("mega_moe" _MegaKernel.top_k_pick): sigmoid scores
// (accurate expf, IEEE divide), keys score + bias as monotone uint32, top_k
// rounds of warp max key then lowest expert among equals, weights
// score / (float sum in pick order) * scale.
__device__ void route_token(const Fp8Args& a, Fp8Smem& S, int t, float* sc, uint32_t* ky, int lane,
                            bool write_out) {
  const int E = a.E;
  for (int e = lane; e < E; e += 32) {
    float l;
    if (a.logits_f32)
      l = __ldg(static_cast<const float*>(a.logits) + static_cast<size_t>(t) * E + e);
    else
      l = __bfloat162float(static_cast<const __nv_bfloat16*>(a.logits)[static_cast<size_t>(t) * E + e]);
    const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
    sc[e] = s;
    ky[e] = ordered_key(__fadd_rn(s, __ldg(a.bias + e)));
  }
  __syncwarp();
  float total = 0.0f;
  float mine = 0.0f;
  int mine_e = 0;
  for (int r = 0; r < a.top_k; ++r) {
    uint32_t best = 0u;
    for (int e = lane; e < E; e += 32) best = max(best, ky[e]);
    const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
    uint32_t cand = 0xFFFFFFFFu;
    for (int e = lane; e < E; e += 32)
      if (ky[e] == top) {
        cand = static_cast<uint32_t>(e);
        break;
      }
    const int win = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
    const float s = sc[win];
    total = __fadd_rn(total, s);
    if (lane == r) {
      mine = s;
      mine_e = win;
    }
    __syncwarp();
    if (lane == 0) ky[win] = 0u;
    __syncwarp();
  }
  if (lane < a.top_k) {
    const int route = t * a.top_k + lane;
    S.rid[route] = static_cast<int16_t>(mine_e);
    atomicOr(&S.tokmask[mine_e], 1ull << t);
    if (write_out) {
      a.ids[route] = mine_e;
      a.weights[route] = __fmul_rn(__fdiv_rn(mine, total), a.scale);
    }
  }
}

// ---------------------------------------------------------------- activations
// Quantise the x slices this thread owns for tokens ctx_tok[c0 .. c0+RTC):
// per 128-block sx = max(amax, 1e-10) / 448 (UE8M0 round-up when asked),
// q = e4m3(x * (1 / sx)); stored as exact f16 pairs.
template <int RTC>
__device__ __forceinline__ void quant_x(const Fp8Args& a, const Fp8Smem& S, int c0, int rt, int gt,
                                        uint32_t (&xa)[kMaxSlicesPerThread][kTokChunk][8],
                                        float (&sx)[kMaxSlicesPerThread][kTokChunk]) {
  const PhaseGeom& g = a.g1;
#pragma unroll
  for (int i = 0; i < kMaxSlicesPerThread; ++i) {
    const int s = gt + g.tpr * i;
#pragma unroll
    for (int t = 0; t < RTC; ++t) {
      // Token slots t >= rt pad a 3-token chunk to 4: zero activations.
      const bool valid = (i < g.nspt) && (s < g.ns) && (t < rt);
      float v[16];
      float amax = 0.0f;
      if (!valid) {
#pragma unroll
        for (int k = 0; k < 8; ++k) xa[i][t][k] = 0u;
      }
      if (valid) {
        const int tok = S.ctx_tok[c0 + t];
        const uint4* p = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * a.H + 16 * s);
        const uint4 q0 = __ldg(p), q1 = __ldg(p + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[2 * k] = __uint_as_float(w[k] << 16);
          v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
      if (valid) {
        float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        if (a.ue8m0) scale = ue8m0_ceil(scale);
        const float inv = __fdiv_rn(1.0f, scale);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(v[4 * k], inv), __fmul_rn(v[4 * k + 1], inv));
          const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(v[4 * k + 2], inv), __fmul_rn(v[4 * k + 3], inv));
          e4m3x4_to_f16x2x2(lo | (hi << 16), xa[i][t][2 * k], xa[i][t][2 * k + 1]);
        }
        sx[i][t] = scale;
      }
    }
  }
}

// Quantise the hidden slices this thread owns for routes ctx_route[c0 ..):
// sh = max(amax, 1e-10) / 448 (UE8M0 when asked); routed: qh = e4m3(h / sh)
// ("mega_moe" hidden_block divides); shared: qh = e4m3(h * (1 / sh))
// ("shared_expert" _DownKernel multiplies by the _group_scale inverse).
template <int RTC>
__device__ __forceinline__ void quant_h(const Fp8Args& a, const Fp8Smem& S, int c0, int rt, int gt,
                                        uint32_t (&xa)[kMaxSlicesPerThread][kTokChunk][8],
                                        float (&sh)[kMaxSlicesPerThread][kTokChunk]) {
  const PhaseGeom& g = a.g2;
#pragma unroll
  for (int i = 0; i < kMaxSlicesPerThread; ++i) {
    const int s = gt + g.tpr * i;
#pragma unroll
    for (int t = 0; t < RTC; ++t) {
      const bool valid = (i < g.nspt) && (s < g.ns) && (t < rt);
      float v[16];
      float amax = 0.0f;
      if (!valid) {
#pragma unroll
        for (int k = 0; k < 8; ++k) xa[i][t][k] = 0u;
      }
      if (valid) {
        const int route = S.ctx_route[c0 + t];
        const float4* p = reinterpret_cast<const float4*>(a.hbuf + static_cast<size_t>(route) * a.I + 16 * s);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 f = __ldcg(p + k);
          v[4 * k] = f.x;
          v[4 * k + 1] = f.y;
          v[4 * k + 2] = f.z;
          v[4 * k + 3] = f.w;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
      if (valid) {
        float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        if (a.ue8m0) scale = ue8m0_ceil(scale);
        float q[16];
        if (a.mode == kModeRouted) {
#pragma unroll
          for (int k = 0; k < 16; ++k) q[k] = __fdiv_rn(v[k], scale);
        } else {
          const float inv = __fdiv_rn(1.0f, scale);
#pragma unroll
          for (int k = 0; k < 16; ++k) q[k] = __fmul_rn(v[k], inv);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = f32x2_to_e4m3x2(q[4 * k], q[4 * k + 1]);
          const uint32_t hi = f32x2_to_e4m3x2(q[4 * k + 2], q[4 * k + 3]);
          e4m3x4_to_f16x2x2(lo | (hi << 16), xa[i][t][2 * k], xa[i][t][2 * k + 1]);
        }
        sh[i][t] = scale;
      }
    }
  }
}

// ---------------------------------------------------------------- row dot products
// acc[q * RTC + t] += sum over this thread's slices of the 16-element dot of
// row (row0 + q) with token t's activations, times the slice's scale product.
// `split`: rows >= split use comb[.][1], others comb[.][0].
template <int RTC>
__device__ __forceinline__ void dot_rows(const uint8_t* stage, int rowbytes, int row0, int split, int gt,
                                         const PhaseGeom& g,
                                         const uint32_t (&xa)[kMaxSlicesPerThread][kTokChunk][8],
                                         const float (&comb)[kMaxSlicesPerThread][2][kTokChunk],
                                         float (&acc)[kRowsPerGroup * RTC]) {
#pragma unroll
  for (int q = 0; q < kRowsPerGroup; ++q) {
    const int row = row0 + q;
    const bool second = row >= split;
    const uint8_t* rp = stage + static_cast<size_t>(row) * rowbytes;
#pragma unroll
    for (int i = 0; i < kMaxSlicesPerThread; ++i) {
      const int s = gt + g.tpr * i;
      if ((i < g.nspt) && (s < g.ns)) {
        const uint4 w = *reinterpret_cast<const uint4*>(rp + 16 * s);
        uint32_t wf[8];
        e4m3x4_to_f16x2x2(w.x, wf[0], wf[1]);
        e4m3x4_to_f16x2x2(w.y, wf[2], wf[3]);
        e4m3x4_to_f16x2x2(w.z, wf[4], wf[5]);
        e4m3x4_to_f16x2x2(w.w, wf[6], wf[7]);
#pragma unroll
        for (int t = 0; t < RTC; ++t) {
          float p = 0.0f;
#pragma unroll
          for (int k = 0; k < 8; ++k) p = fma_f16x2_f32(wf[k], xa[i][t][k], p);
          const float c = second ? comb[i][1][t] : comb[i][0][t];
          acc[q * RTC + t] = fmaf(p, c, acc[q * RTC + t]);
        }
      }
    }
  }
}

// Reduce acc over the threads of each row group; results land in
// S.red[warp][v] (v = q * RTC + t) for the group's warps. Caller syncs.
template <int RTC>
__device__ __forceinline__ void reduce_to_smem(Fp8Smem& S, float (&acc)[kRowsPerGroup * RTC], int warp,
                                               int lane) {
  constexpr int V = kRowsPerGroup * RTC;
  const float s = warp_transpose_sum<V>(acc, lane);
  if ((lane % (32 / V)) == 0) S.red[warp][lane / (32 / V)] = s;
}

__device__ __forceinline__ void compute_bar() { named_bar_sync(1, kComputeThreads); }

// ---------------------------------------------------------------- context (routes of an expert)
__device__ void build_context(const Fp8Args& a, Fp8Smem& S, int e, int ctid) {
  if (ctid < 32) {
    const int lane = ctid;
    if (a.mode == kModeShared) {
      for (int t = lane; t < a.M; t += 32) {
        S.ctx_route[t] = static_cast<int16_t>(t);
        S.ctx_tok[t] = static_cast<int16_t>(t);
      }
      if (lane == 0) S.ctx_n = a.M;
    } else {
      const unsigned long long mask = S.tokmask[e];
      int base = 0;
      for (int t0 = 0; t0 < a.M; t0 += 32) {
        const int t = t0 + lane;
        const bool has = (t < a.M) && ((mask >> t) & 1ull);
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
        if (has) {
          const int pos = base + __popc(bal & ((1u << lane) - 1u));
          int r = 0;
          for (int k = 0; k < a.top_k; ++k)
            if (S.rid[t * a.top_k + k] == e) r = k;
          S.ctx_route[pos] = static_cast<int16_t>(t * a.top_k + r);
          S.ctx_tok[pos] = static_cast<int16_t>(t);
        }
        base += __popc(bal);
      }
      if (lane == 0) S.ctx_n = base;
    }
  }
  compute_bar();
}

// ---------------------------------------------------------------- GEMM1 item
template <int RTC>
__device__ __forceinline__ void gemm1_chunk(const Fp8Args& a, Fp8Smem& S, const uint8_t* stage, int e, int j,
                                            int h0, int c0, int rt, bool requant, int ctid, int warp, int lane,
                                            uint32_t (&xa)[kMaxSlicesPerThread][kTokChunk][8],
                                            float (&sx)[kMaxSlicesPerThread][kTokChunk]) {
  const PhaseGeom& g = a.g1;
  const int grp = ctid / g.tpr, gt = ctid % g.tpr;
  if (requant) quant_x<RTC>(a, S, c0, rt, gt, xa, sx);
  // Scale products of the two row blocks (first half: block j; second: I/128 + j).
  const int nb = a.H / 128, nrb = 2 * a.I / 128;
  float comb[kMaxSlicesPerThread][2][kTokChunk];
#pragma unroll
  for (int i = 0; i < kMaxSlicesPerThread; ++i) {
    const int s = gt + g.tpr * i;
    const int b = min(s, g.ns - 1) / 8;
    const float w0 = __ldg(a.s13 + (static_cast<size_t>(e) * nrb + j) * nb + b);
    const float w1 = __ldg(a.s13 + (static_cast<size_t>(e) * nrb + a.I / 128 + j) * nb + b);
#pragma unroll
    for (int t = 0; t < RTC; ++t) {
      comb[i][0][t] = __fmul_rn(w0, sx[i][t]);
      comb[i][1][t] = __fmul_rn(w1, sx[i][t]);
    }
  }
  float acc[kRowsPerGroup * RTC];
#pragma unroll
  for (int v = 0; v < kRowsPerGroup * RTC; ++v) acc[v] = 0.0f;
  dot_rows<RTC>(stage, a.H, grp * kRowsPerGroup, a.gp, gt, g, xa, comb, acc);
  reduce_to_smem<RTC>(S, acc, warp, lane);
  compute_bar();
  // Fixed-order sum over the group's warps -> S.ysum[row][t].
  constexpr int V = kRowsPerGroup * RTC;
  const int wpg = g.tpr / 32;
  if (ctid < g.rg * V) {
    const int fg = ctid / V, v = ctid % V;
    float s = 0.0f;
    for (int w = 0; w < wpg; ++w) s += S.red[fg * wpg + w][v];
    S.ysum[fg * kRowsPerGroup + v / RTC][v % RTC] = s;
  }
  compute_bar();
  // SwiGLU of hidden indices h0 .. h0 + gp for the chunk's tokens.
  if (ctid < a.gp * RTC && ctid % RTC < rt) {
    const int q = ctid / RTC, t = ctid % RTC;
    const float first = S.ysum[q][t];
    const float second = S.ysum[a.gp + q][t];
    const int route = S.ctx_route[c0 + t];
    const float L = a.limit;
    float h;
    if (a.mode == kModeRouted) {
      // W31: up rows first, then gate rows ("mega_moe" module docstring).
      const float gate = fminf(second, L);
      const float up = fmaxf(fminf(first, L), -L);
      h = __fmul_rn(__fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate))), up);
    } else {
      // Shared gate_up: gate rows first, BF16 gate_up and BF16 h.
      const __nv_bfloat16 gb = __float2bfloat16_rn(first);
      const __nv_bfloat16 ub = __float2bfloat16_rn(second);
      if (a.gate_up != nullptr) {
        a.gate_up[static_cast<size_t>(route) * 2 * a.I + h0 + q] = gb;
        a.gate_up[static_cast<size_t>(route) * 2 * a.I + a.I + h0 + q] = ub;
      }
      const float gate = fminf(__bfloat162float(gb), L);
      const float up = fmaxf(fminf(__bfloat162float(ub), L), -L);
      const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
      h = __bfloat162float(__float2bfloat16_rn(__fmul_rn(silu, up)));
    }
    a.hbuf[static_cast<size_t>(route) * a.I + h0 + q] = h;
  }
  compute_bar();
}

// ---------------------------------------------------------------- GEMM2 item
template <int RTC>
__device__ __forceinline__ void gemm2_chunk(const Fp8Args& a, Fp8Smem& S, const uint8_t* stage, int e, int m0,
                                            int c0, int rt, bool requant, int ctid, int warp, int lane,
                                            uint32_t (&xa)[kMaxSlicesPerThread][kTokChunk][8],
                                            float (&sh)[kMaxSlicesPerThread][kTokChunk]) {
  const PhaseGeom& g = a.g2;
  const int grp = ctid / g.tpr, gt = ctid % g.tpr;
  if (requant) quant_h<RTC>(a, S, c0, rt, gt, xa, sh);
  const int nb = a.I / 128, nrb = a.H / 128;
  float comb[kMaxSlicesPerThread][2][kTokChunk];
#pragma unroll
  for (int i = 0; i < kMaxSlicesPerThread; ++i) {
    const int s = gt + g.tpr * i;
    const int b = min(s, g.ns - 1) / 8;
    const float w = __ldg(a.s2 + (static_cast<size_t>(e) * nrb + m0 / 128) * nb + b);
#pragma unroll
    for (int t = 0; t < RTC; ++t) {
      comb[i][0][t] = a.mode == kModeRouted ? __fmul_rn(w, sh[i][t]) : __fmul_rn(sh[i][t], w);
      comb[i][1][t] = comb[i][0][t];
    }
  }
  float acc[kRowsPerGroup * RTC];
#pragma unroll
  for (int v = 0; v < kRowsPerGroup * RTC; ++v) acc[v] = 0.0f;
  dot_rows<RTC>(stage, a.I, grp * kRowsPerGroup, 1 << 30, gt, g, xa, comb, acc);
  reduce_to_smem<RTC>(S, acc, warp, lane);
  compute_bar();
  constexpr int V = kRowsPerGroup * RTC;
  const int wpg = g.tpr / 32;
  if (ctid < g.rg * V && (ctid % V) % RTC < rt) {
    const int fg = ctid / V, v = ctid % V;
    float s = 0.0f;
    for (int w = 0; w < wpg; ++w) s += S.red[fg * wpg + w][v];
    const int m = m0 + fg * kRowsPerGroup + v / RTC;
    const int route = S.ctx_route[c0 + v % RTC];
    a.out[static_cast<size_t>(route) * a.H + m] = __float2bfloat16_rn(s);
  }
  compute_bar();
}

// ---------------------------------------------------------------- kernel
__device__ __forceinline__ void item_range(long long n, int c, int G, long long& lo, long long& hi) {
  lo = n * c / G;
  hi = n * (c + 1) / G;
}

struct ItemPlan {
  long long lo1, hi1, lo2, hi2;
  int per_u1, parts, per_u2;
  __device__ int count() const { return static_cast<int>((hi1 - lo1) + (hi2 - lo2)); }
};

// Issue the bulk copies of the CTA's item number `it` into stage it % kStages.
__device__ void issue_item(const Fp8Args& a, Fp8Smem& S, const ItemPlan& P, int it, uint64_t pol) {
  const int s = it % kStages;
  uint8_t* dst = S.ring[s];
  if (it < P.hi1 - P.lo1) {
    const long long i = P.lo1 + it;
    const int u = static_cast<int>(i / P.per_u1), rem = static_cast<int>(i % P.per_u1);
    const int e = S.ulist[u];
    const int h0 = (rem / P.parts) * 128 + (rem % P.parts) * a.gp;
    const uint32_t half_bytes = static_cast<uint32_t>(a.gp) * a.H;
    mbar_arrive_expect_tx(&S.full[s], 2 * half_bytes);
    const uint8_t* base = a.w13 + static_cast<size_t>(e) * 2 * a.I * a.H;
    bulk_g2s(dst, base + static_cast<size_t>(h0) * a.H, half_bytes, &S.full[s], pol);
    bulk_g2s(dst + half_bytes, base + static_cast<size_t>(a.I + h0) * a.H, half_bytes, &S.full[s], pol);
  } else {
    const long long i = P.lo2 + (it - (P.hi1 - P.lo1));
    const int u = static_cast<int>(i / P.per_u2), rb = static_cast<int>(i % P.per_u2);
    const int e = S.ulist[u];
    const uint32_t bytes = static_cast<uint32_t>(a.r2) * a.I;
    mbar_arrive_expect_tx(&S.full[s], bytes);
    bulk_g2s(dst, a.w2 + (static_cast<size_t>(e) * a.H + static_cast<size_t>(rb) * a.r2) * a.I, bytes,
             &S.full[s], pol);
  }
}

// Wait (all threads) for item `it`'s stage; false (uniformly) on abort.
__device__ __forceinline__ bool wait_stage(const Fp8Args& a, Fp8Smem& S, int it) {
  const int s = it % kStages;
  if (!mbar_wait(&S.full[s], (it / kStages) & 1, a.timeout_ns, &S.abort)) {
    if (!S.abort) set_error(a, S, kErrRingWait);
  }
  compute_bar();
  return !S.abort;
}

// After item `it` (ends on a CTA barrier): thread 0 refills its stage with
// item it + kStages.
__device__ __forceinline__ void refill(const Fp8Args& a, Fp8Smem& S, const ItemPlan& P, int it, uint64_t pol) {
  if (threadIdx.x == 0 && it + kStages < P.count()) {
    fence_proxy_async_smem();
    issue_item(a, S, P, it + kStages, pol);
  }
}

// Before exit: thread 0 waits until every copy it issued has landed.
__device__ void drain(const Fp8Args& a, Fp8Smem& S, const ItemPlan& P, int consumed) {
  if (threadIdx.x != 0) return;
  const int issued = min(P.count(), consumed + kStages);
  for (int k = consumed; k < issued; ++k)
    if (!mbar_wait(&S.full[k % kStages], (k / kStages) & 1, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
}

__global__ void __launch_bounds__(kThreads, 1) fp8_moe_kernel(const __grid_constant__ Fp8Args a) {
  extern __shared__ uint8_t smem_raw[];
  Fp8Smem& S = *reinterpret_cast<Fp8Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    S.abort = 0;
  }
  for (int e = tid; e < a.E; e += kThreads) S.tokmask[e] = 0ull;
  griddep_wait();
  __syncthreads();

  // ---- routing and the unique-expert list (scratch overlays the ring)
  if (a.mode == kModeRouted) {
    float* sc = reinterpret_cast<float*>(&S.ring[0][0]) + warp * 2 * kMaxExperts;
    uint32_t* ky = reinterpret_cast<uint32_t*>(sc + kMaxExperts);
    for (int t = warp; t < a.M; t += kThreads / 32) route_token(a, S, t, sc, ky, lane, blockIdx.x == 0);
    __syncthreads();
    if (warp == 0) {
      int U = 0;
      for (int b = 0; b < a.E; b += 32) {
        const int e = b + lane;
        const bool has = (e < a.E) && (S.tokmask[e] != 0ull);
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
        if (has) S.ulist[U + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(e);
        U += __popc(bal);
      }
      if (lane == 0) S.U = U;
    }
  } else if (tid == 0) {
    S.U = 1;
    S.ulist[0] = 0;
  }
  __syncthreads();

  const int U = S.U;
  const int G = gridDim.x, c = blockIdx.x;
  ItemPlan P;
  P.per_u1 = a.I / a.gp;  // GEMM1 items per expert (I/128 blocks x 128/gp parts)
  P.parts = 128 / a.gp;
  P.per_u2 = a.H / a.r2;  // GEMM2 items per expert
  item_range(static_cast<long long>(U) * P.per_u1, c, G, P.lo1, P.hi1);
  item_range(static_cast<long long>(U) * P.per_u2, c, G, P.lo2, P.hi2);
  const int n_items = P.count();
  if (n_items == 0) return;

  uint64_t pol = 0;
  if (tid == 0) {
    pol = l2_evict_first_policy();
    fence_proxy_async_smem();  // the routing scratch overlaid the ring
    for (int it = 0; it < min(kStages, n_items); ++it) issue_item(a, S, P, it, pol);
  }

  const int ctid = tid;
  uint32_t xa[kMaxSlicesPerThread][kTokChunk][8];
  float xs[kMaxSlicesPerThread][kTokChunk];
#pragma unroll
  for (int i = 0; i < kMaxSlicesPerThread; ++i)
#pragma unroll
    for (int t = 0; t < kTokChunk; ++t) {
      xs[i][t] = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) xa[i][t][k] = 0u;
    }

  int it = 0;
  int cur_u = -1;
  for (long long i = P.lo1; i < P.hi1; ++i, ++it) {
    const int u = static_cast<int>(i / P.per_u1), rem = static_cast<int>(i % P.per_u1);
    const int e = S.ulist[u];
    const int j = rem / P.parts;
    const int h0 = j * 128 + (rem % P.parts) * a.gp;
    bool fresh = false;
    if (u != cur_u) {
      build_context(a, S, e, ctid);
      cur_u = u;
      fresh = true;
    }
    if (!wait_stage(a, S, it)) {
      drain(a, S, P, it);
      return;
    }
    const int nt = S.ctx_n;
    const bool single = nt <= kTokChunk;
    const uint8_t* stage = S.ring[it % kStages];
    for (int c0 = 0; c0 < nt; c0 += kTokChunk) {
      const int rt = min(kTokChunk, nt - c0);
      const bool requant = fresh || !single;
      // 8 rows x 1, 2 or 4 token slots per lane keep the warp reduction a power of two.
      switch (rt) {
        case 1: gemm1_chunk<1>(a, S, stage, e, j, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        case 2: gemm1_chunk<2>(a, S, stage, e, j, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        default: gemm1_chunk<4>(a, S, stage, e, j, h0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
      }
    }
    if (ctid == 0) {
      __threadfence();
      red_release_gpu_add(a.done + e, 1u);
    }
    refill(a, S, P, it, pol);
  }

  cur_u = -1;
  for (long long i = P.lo2; i < P.hi2; ++i, ++it) {
    const int u = static_cast<int>(i / P.per_u2), rb = static_cast<int>(i % P.per_u2);
    const int e = S.ulist[u];
    const int m0 = rb * a.r2;
    bool fresh = false;
    if (u != cur_u) {
      build_context(a, S, e, ctid);
      if (ctid == 0) {
        const uint32_t target = static_cast<uint32_t>(P.per_u1);
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(a.done + e) < target) {
          if (globaltimer_ns() - t0 > a.timeout_ns) {
            set_error(a, S, kErrCrossWait);
            break;
          }
          __nanosleep(64);
        }
      }
      compute_bar();
      if (S.abort) {
        drain(a, S, P, it);
        return;
      }
      cur_u = u;
      fresh = true;
    }
    if (!wait_stage(a, S, it)) {
      drain(a, S, P, it);
      return;
    }
    const int nt = S.ctx_n;
    const bool single = nt <= kTokChunk;
    const uint8_t* stage = S.ring[it % kStages];
    for (int c0 = 0; c0 < nt; c0 += kTokChunk) {
      const int rt = min(kTokChunk, nt - c0);
      const bool requant = fresh || !single;
      // 8 rows x 1, 2 or 4 token slots per lane keep the warp reduction a power of two.
      switch (rt) {
        case 1: gemm2_chunk<1>(a, S, stage, e, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        case 2: gemm2_chunk<2>(a, S, stage, e, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
        default: gemm2_chunk<4>(a, S, stage, e, m0, c0, rt, requant, ctid, warp, lane, xa, xs); break;
      }
    }
    if (ctid == 0) {
      // The last GEMM2 item of this expert re-arms its counters for the next call.
      const uint32_t old = atomicAdd(a.consumed + e, 1u);
      if (old + 1u == static_cast<uint32_t>(P.per_u2)) {
        atomicExch(a.done + e, 0u);
        atomicExch(a.consumed + e, 0u);
      }
    }
    refill(a, S, P, it, pol);
  }
}

// ---------------------------------------------------------------- host side
static PhaseGeom make_geom(int K) {
  PhaseGeom g;
  g.ns = K / 16;
  int tpr = 32;
  while (tpr < g.ns && tpr < kComputeThreads) tpr *= 2;
  g.tpr = tpr;
  g.rg = kComputeThreads / tpr;
  g.nspt = (g.ns + tpr - 1) / tpr;
  return g;
}

struct Fp8Workspace {
  uint32_t* err;
  uint32_t* done;
  uint32_t* consumed;
  float* hbuf;
  size_t bytes;
};

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static Fp8Workspace fp8_workspace_layout(void* base, int routes, int I, int E) {
  Fp8Workspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.err = reinterpret_cast<uint32_t*>(p + off);
  off += 256;
  w.done = reinterpret_cast<uint32_t*>(p + off);
  off += align256(sizeof(uint32_t) * E);
  w.consumed = reinterpret_cast<uint32_t*>(p + off);
  off += align256(sizeof(uint32_t) * E);
  w.hbuf = reinterpret_cast<float*>(p + off);
  off += align256(sizeof(float) * static_cast<size_t>(routes) * I);
  w.bytes = off;
  return w;
}

size_t fp8_workspace_bytes(int routes, int I, int E) {
  return fp8_workspace_layout(nullptr, routes, I, E).bytes;
}

static int launch_fp8(Fp8Args& a, void* workspace, size_t workspace_bytes, int routes, cudaStream_t st) {
  const Fp8Workspace w = fp8_workspace_layout(workspace, routes, a.I, a.mode == kModeShared ? 1 : a.E);
  if (workspace == nullptr || workspace_bytes < w.bytes)
    return set_last_error(FME_EWORKSPACE, "workspace of %zu bytes needed, %zu given", w.bytes, workspace_bytes);
  a.err = w.err;
  a.done = w.done;
  a.consumed = w.consumed;
  a.hbuf = w.hbuf;
  a.g1 = make_geom(a.H);
  a.g2 = make_geom(a.I);
  a.gp = kRowsPerGroup * a.g1.rg / 2;
  a.r2 = kRowsPerGroup * a.g2.rg;
  a.timeout_ns = wait_timeout_ns();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_last_error(FME_ECUDA, "cudaGetDevice failed");
  const int sms = device_sm_count(dev);
  if (sms <= 0) return set_last_error(FME_ECUDA, "cannot query the SM count");
  if (!ensure_smem_attr(dev, reinterpret_cast<const void*>(fp8_moe_kernel), kFp8SmemBytes))
    return set_last_error(FME_ECUDA, "cudaFuncSetAttribute(max dynamic smem) failed");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kFp8SmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, fp8_moe_kernel, a);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "fp8 kernel launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

int routed_fp8(const void* x, const void* logits, int logits_dtype, const float* bias, const uint8_t* w13,
               const float* s13, const uint8_t* w2, const float* s2, int M, int H, int I, int E, int top_k,
               float limit, float scale, int ue8m0, void* out, int32_t* ids, float* weights, void* workspace,
               size_t workspace_bytes, cudaStream_t st) {
  Fp8Args a = {};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.logits = logits;
  a.bias = bias;
  a.w13 = w13;
  a.s13 = s13;
  a.w2 = w2;
  a.s2 = s2;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ids = ids;
  a.weights = weights;
  a.gate_up = nullptr;
  a.M = M;
  a.H = H;
  a.I = I;
  a.E = E;
  a.top_k = top_k;
  a.limit = limit;
  a.scale = scale;
  a.ue8m0 = ue8m0 ? 1 : 0;
  a.logits_f32 = logits_dtype == FME_F32 ? 1 : 0;
  a.mode = kModeRouted;
  return launch_fp8(a, workspace, workspace_bytes, M * top_k, st);
}

int shared_fp8(const void* x, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2, int M,
               int H, int I, float limit, int ue8m0, void* gate_up, void* out, void* workspace,
               size_t workspace_bytes, cudaStream_t st) {
  Fp8Args a = {};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w13 = w13;
  a.s13 = s13;
  a.w2 = w2;
  a.s2 = s2;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.gate_up = static_cast<__nv_bfloat16*>(gate_up);
  a.M = M;
  a.H = H;
  a.I = I;
  a.E = 1;
  a.top_k = 1;
  a.limit = limit;
  a.scale = 1.0f;
  a.ue8m0 = ue8m0 ? 1 : 0;
  a.mode = kModeShared;
  return launch_fp8(a, workspace, workspace_bytes, M, st);
}

}  // namespace fme
