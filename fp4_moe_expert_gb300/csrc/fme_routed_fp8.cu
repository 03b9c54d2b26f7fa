// Routed FP8 MoE layer and FP8 shared expert on the sm_103a tensor cores.
//
// Computes what "vllm.models.glm5next.nvidia.specialized_decode.mega_moe"
// (MegaExperts / _MegaKernel) and ".../shared_expert" (SharedExpert,
// _GateUpKernel, _DownKernel, _group_scale) define. The design is this
// library's own:
//
// * One persistent CTA per SM, eight warps: warp 0 streams weight tiles with
//   TMA (128-byte swizzle, 8 x 16 KB ring, L2 evict-first); warp 1 owns TMEM
//   and issues tcgen05.mma kind::f8f6f4 (M = 128 weight rows, N = 16 *
//   ceil(tokens / 16), K = 32); warps 2-5 read the accumulators and run the
//   epilogue; warps 6-7 quantise the activations into the B operand. Every
//   CTA redoes the routing of all tokens, so each derives the same list of
//   the unique experts touched and each expert's weights stream once.
// * The block scales are FP32 and not powers of two, so the MMA cannot apply
//   them: each 128-wide K block accumulates into its own group of TMEM
//   columns, and the epilogue multiplies every block's partial by
//   (weight scale x activation scale) and sums (the page's one-column-per-K-
//   block idea, with the tokens as the columns of one group).
// * Work is split stream-K style: GEMM1 is (expert, tile of 64 first-half
//   rows + the 64 matching second-half rows, K block) slots, GEMM2 is
//   (expert, tile of 128 rows, K block) slots; every CTA owns an equal
//   contiguous slice of each phase. A tile cut by slice boundaries is summed
//   by its first contributor, in CTA order, from partials in the workspace.
// * A finished GEMM1 tile writes its SwiGLU output (f32) to the workspace and
//   releases a per-expert counter; GEMM2 work of that expert waits for all of
//   its GEMM1 tiles (bounded wait), then quantises the hidden per 128 itself.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fme_common.cuh"
#include "fme_internal.h"
#include "fme_plan.cuh"

namespace fme {

constexpr int kTcThreads = 256;  // TMA, MMA, 4 accumulate, 2 fill warps
// Above this many routes on one expert the GEMM1 fills copy from a per-call
// image of x instead of quantising per chunk.
constexpr int kXImageRoutes = 4;
constexpr int kFillThreads = 64;
constexpr int kTcStages = 8;
constexpr int kAStageBytes = 128 * 128;  // one 128-row x 128-byte K block of weights
constexpr int kBBufBytes = 256 * 128;    // K blocks x N token rows x 128 bytes <= 256 rows
constexpr int kTmemCols = 512;
constexpr int kTmemBuf = 256;            // two accumulator buffers
// The MX kernel keeps its scale vectors in tensor memory beside two
// 192-column accumulator buffers. A block-scaled MMA reads its scale factors
// from a 4-column-aligned address (byte sf_id of each 32-bit cell; B tokens
// 32 .. 63 one column further), so every K block takes 4 columns: the
// weights' (all 2^0) in columns 384..387, B buffer b's token scales from
// 388 + 60 b, K block j at + 4 j (at most 15 K blocks). Its fill stages those
// cells in the B buffer from 24 KB on (a chunk's codes take at most 192
// columns x 128 bytes = 24 KB), 512 bytes per K block.
template <bool MX>
__host__ __device__ constexpr int tmem_buf() { return MX ? 192 : kTmemBuf; }
constexpr uint32_t kSfaCol = 384;
constexpr uint32_t kSfbCol = 388;
constexpr uint32_t kSfbBuf = 60;
constexpr int kMxSfStage = 24 * 1024;
constexpr int kMaxKc = 16;
struct TcArgs {
  CUtensorMap map13;   // routed W13 as [E * 2I rows, H bytes], box 64 rows x 128 bytes
  CUtensorMap map2;    // routed W2 as [E * H rows, I bytes]
  CUtensorMap smap13;  // shared-expert gate_up as [2I rows, H bytes]
  CUtensorMap smap2;   // shared-expert down as [H rows, I bytes]
  const __nv_bfloat16* x;
  const uint8_t* xq;   // MXFP8 input (the MX kernel): x as E4M3 [M, H] and E8M0 [M, H/32]
  const uint8_t* xsc;
  const void* logits;
  const float* bias;
  const float* s13;
  const float* s2;
  const float* ss13;   // shared-expert block scales
  const float* ss2;
  __nv_bfloat16* out;   // routed rows [M * top_k, H]
  __nv_bfloat16* sout;  // shared-expert rows [M, H]
  int32_t* ids;
  float* weights;
  __nv_bfloat16* gate_up;
  uint32_t* err;     // device error word
  uint32_t* done;    // [E + 1] GEMM1 tiles finished per expert (id E: the shared expert)
  uint32_t* passed;  // [E + 1] CTAs whose GEMM2 work passed the wait
  uint32_t* cnt1;    // [(E + 1) * I/64] contributors arrived per GEMM1 tile (expert id, tile)
  uint32_t* cnt2;    // [(E + 1) * H/128] per GEMM2 tile
  float* hbuf;       // [M * top_k + M, I] SwiGLU output (routed routes, then shared tokens)
  uint8_t* ximg;     // [M, H] x quantised per 128 (E4M3), built once per call when experts take many tokens
  float* ximg_sc;    // [M, H/128] its scales
  uint32_t* xsync;   // [2]: CTAs whose share of the image is written; CTAs past the wait for it
  int32_t* picks;    // [M, top_k] expert picks, when the CTAs share the routing
  uint32_t* rsync;   // [2]: tokens routed; CTAs past the wait for them
  float* part;       // [2 phases][kFp8MaxCtas][2 slots][tokens][128 rows] split-tile partials
  int M, H, I, E, top_k;  // E routed experts (0: shared expert only)
  int ptok;          // token rows of one partial slot (min(M, 64))
  float limit, scale;
  float slimit;      // shared-expert SwiGLU clamp
  int ue8m0, logits_f32, has_shared;
  // Phases this launch runs (1 = GEMM1 .. SwiGLU, 2 = hidden re-quant ..
  // GEMM2): 1..2 for the one persistent launch; the two-kernel chain runs
  // 1..1, then 2..2 as a programmatic dependent launch that streams its W2
  // tiles before it waits for the first kernel.
  int phase_lo, phase_hi;
  int sue8m0;        // shared-expert activation scales rounded up to powers of two
  unsigned long long timeout_ns;
};

struct TcSmem {
  uint8_t A[kTcStages][kAStageBytes];
  uint8_t B[2][kBBufBytes];
  float xs[2][kMaxTokens][kMaxKc];  // activation block scales per B buffer
  float wsc[2][2][kMaxKc];          // weight block scales per B buffer: [row half][K block]
  float ysm[16][128];               // GEMM1 epilogue exchange (16 tokens x 128 tile rows)
  uint64_t full[kTcStages], empty[kTcStages];
  uint64_t bfull[2], accfull[2], tmemfree[2], mfree[2], final_bar;
  unsigned long long tokmask[kMaxExperts];
  int16_t rid[kMaxTokens * kMaxTopK];
  int16_t ulist[kMaxExperts + 1];  // [0]: the shared expert, when present
  Heavy heavy;  // the heavy units of the cost-weighted split (at most the shared one)
  int16_t hu[1];
  uint16_t he[1];
  uint32_t hce[2];
  int16_t ctx_route[3][kMaxTokens];  // routes of each B buffer's expert, in token order; [2]: the fill's next
  int16_t ctx_tok[kMaxTokens];       // the tokens of ctx_route[2]
  int btag[2];                       // what each B buffer holds: a GEMM2 (unit, K range), or -1
  alignas(1024) uint32_t sfa_one[128];  // 32 rows x 16 bytes of 2^0 scales (MX kernel)
  int ctx_n[3];
  int16_t seg_route[kMaxTokens];     // the accumulate warps' copy for the current segment
  int seg_n;
  uint32_t tmem_base;
  int U, rmax;
  int flag;
  volatile int abort;
};

constexpr size_t kTcSmemBytes = sizeof(TcSmem) + 1024;
static_assert(kTcSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ void tc_error(const TcArgs& a, TcSmem& S, uint32_t bit) {
  atomicOr(a.err, bit);
  S.abort = 1;
}

// What differs per work expert: (when present) the shared expert as unit 0,
// routed to every token, then the routed experts of the unique list.
// The shared expert follows "shared_expert" (gate rows first, BF16 gate_up and
// h, re-quant by multiplying with the inverse); routed experts follow
// "mega_moe" (up rows first, FP32 h, re-quant by dividing).
struct XInfo {
  bool shared;
  int id;     // counter index: routed expert id, or E for the shared expert
  int row_e;  // expert index within its tensor maps
  const CUtensorMap* m13;
  const CUtensorMap* m2;
  const float* s13;
  const float* s2;
  float limit;
  bool ue8m0;
};

__device__ __forceinline__ XInfo xinfo(const TcArgs& a, const TcSmem& S, int u) {
  XInfo x;
  x.shared = a.has_shared && u == 0;
  if (x.shared) {
    x.id = a.E;
    x.row_e = 0;
    x.m13 = &a.smap13;
    x.m2 = &a.smap2;
    x.s13 = a.ss13;
    x.s2 = a.ss2;
    x.limit = a.slimit;
    x.ue8m0 = a.sue8m0 != 0;
  } else {
    x.id = S.ulist[u];
    x.row_e = x.id;
    x.m13 = &a.map13;
    x.m2 = &a.map2;
    x.s13 = a.s13;
    x.s2 = a.s2;
    x.limit = a.limit;
    x.ue8m0 = a.ue8m0 != 0;
  }
  return x;
}

// The four accumulate warps and the two fill warps each sync among themselves.
__device__ __forceinline__ void epi_bar() { named_bar_sync(1, 128); }
__device__ __forceinline__ void fill_bar() { named_bar_sync(2, kFillThreads); }

// ---------------------------------------------------------------- routing
// Routing ("mega_moe" _MegaKernel.top_k_pick): sigmoid scores (accurate
// expf, IEEE divide), keys score + bias as monotone uint32, the top_k keys
// with the lowest expert first among equal keys, weights score / (float sum
// of the picked scores in pick order) * scale. The 8 warps of a CTA split a
// token's experts (wpt = 8, 4 or 2 warps per token, expert blocks of 32 dealt
// round-robin), each warp picks its top_k by that rule into shared memory,
// then one warp per token merges the candidates by the same rule; the merge
// gives the same picks as one pass over all experts.
struct RouteCand {
  uint32_t key;
  int e;
  float score;
};

// Tokens t0 .. t0 + ntok - 1 (ntok <= 8 / wpt), wpt warps each; E <= 128 wpt.
// gpicks == nullptr: the picks go to S.rid / S.tokmask; else to gpicks[t][r]
// in global memory (the routing shared between CTAs).
template <int WPT = 0>  // warps per token when known at compile time (else wpt)
__device__ void route_split(const TcArgs& a, TcSmem& S, int warp, int lane, bool write_out, int t0, int ntok, int wpt,
                            int32_t* gpicks) {
  if constexpr (WPT > 0) wpt = WPT;
  const int tl = warp / wpt, sl = warp % wpt;
  const int t = t0 + tl;
  const int k = a.top_k;
  // candidates [token][slice][k] in the idle B buffer (no fill has started yet)
  RouteCand* cand = reinterpret_cast<RouteCand*>(S.B[0]);
  if (tl < ntok && t < a.M) {
    constexpr int J = 4;  // expert blocks of 32 per slice: E <= 4 x 32 x wpt
    float sc[J], bs[J];
    uint32_t ky[J];
    int ex[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {  // every load issued before any sigmoid
      ex[j] = lane + 32 * (sl + wpt * j);
      sc[j] = 0.0f;
      bs[j] = 0.0f;
      if (ex[j] < a.E) {
        sc[j] = a.logits_f32
                    ? __ldg(static_cast<const float*>(a.logits) + static_cast<size_t>(t) * a.E + ex[j])
                    : __bfloat162float(static_cast<const __nv_bfloat16*>(a.logits)[static_cast<size_t>(t) * a.E + ex[j]]);
        bs[j] = __ldg(a.bias + ex[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float sgm = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-sc[j])));
      sc[j] = sgm;
      ky[j] = ex[j] < a.E ? ordered_key(__fadd_rn(sgm, bs[j])) : 0u;
    }
    RouteCand* mine = cand + (tl * 8 + sl) * k;
    for (int r = 0; r < k; ++r) {
      uint32_t best = 0u;
#pragma unroll
      for (int j = 0; j < J; ++j) best = max(best, ky[j]);
      const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
      uint32_t c = 0xFFFFFFFFu;
#pragma unroll
      for (int j = J - 1; j >= 0; --j)
        if (ky[j] == top && top != 0u) c = static_cast<uint32_t>(ex[j]);
      const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, c);
      float sv = 0.0f;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (static_cast<uint32_t>(ex[j]) == win) {
          sv = sc[j];
          ky[j] = 0u;
        }
      // the winner's lane holds its score; an exhausted slice offers key 0
      const float s = __shfl_sync(0xFFFFFFFFu, sv, win == 0xFFFFFFFFu ? 0 : static_cast<int>(win & 31u));
      if (lane == 0) mine[r] = RouteCand{top, win == 0xFFFFFFFFu ? 0x7FFFFFFF : static_cast<int>(win), s};
    }
  }
  __syncthreads();
  if (warp < ntok && t0 + warp < a.M) {
    const int tt = t0 + warp;
    const RouteCand* cs = cand + warp * 8 * k;
    const int n = wpt * k;  // <= 8 x 8 (E <= 256 caps k at what 8 blocks hold per slice)
    constexpr int JM = 8;
    uint32_t ky[JM];
    int ex[JM];
    float sc[JM];
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int i = lane + 32 * j;  // slice i / k, rank i % k
      ky[j] = 0u;
      ex[j] = 0x7FFFFFFF;
      sc[j] = 0.0f;
      if (i < n) {
        const RouteCand c = cs[i];
        ky[j] = c.key;
        ex[j] = c.e;
        sc[j] = c.score;
      }
    }
    float total = 0.0f, mine_s = 0.0f;
    int mine_e = 0;
    for (int r = 0; r < k; ++r) {
      uint32_t best = 0u;
#pragma unroll
      for (int j = 0; j < JM; ++j) best = max(best, ky[j]);
      const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
      uint32_t c = 0xFFFFFFFFu;
#pragma unroll
      for (int j = 0; j < JM; ++j)
        if (ky[j] == top && static_cast<uint32_t>(ex[j]) < c) c = static_cast<uint32_t>(ex[j]);
      const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, c);
      float sv = 0.0f;
      int holder = 0;
#pragma unroll
      for (int j = 0; j < JM; ++j)
        if (ky[j] == top && static_cast<uint32_t>(ex[j]) == win) {
          sv = sc[j];
          ky[j] = 0u;
          holder = 1;
        }
      const int src = __ffs(__ballot_sync(0xFFFFFFFFu, holder)) - 1;
      const float s = __shfl_sync(0xFFFFFFFFu, sv, src < 0 ? 0 : src);
      total = __fadd_rn(total, s);
      if (lane == r) {
        mine_s = s;
        mine_e = static_cast<int>(win);
      }
    }
    if (lane < k) {
      const float w = __fmul_rn(__fdiv_rn(mine_s, total), a.scale);
      const int route = tt * k + lane;
      if (gpicks != nullptr) {
        gpicks[route] = mine_e;
      } else {
        S.rid[route] = static_cast<int16_t>(mine_e);
        atomicOr(&S.tokmask[mine_e], 1ull << tt);
      }
      if (write_out) {
        a.ids[route] = mine_e;
        a.weights[route] = w;
      }
    }
  }
}

// ---------------------------------------------------------------- B operand fill
// Routes of expert u (token order) into the fill warps' staging slot ctx_route[2].
__device__ void fill_context(const TcArgs& a, TcSmem& S, int u, int fid) {
  constexpr int b = 2;
  if (fid < 32) {
    const int lane = fid;
    if (a.has_shared && u == 0) {
      // The shared expert's rows follow the routed ones in hbuf: M*top_k + t.
      for (int t = lane; t < a.M; t += 32) {
        S.ctx_route[b][t] = static_cast<int16_t>(a.M * a.top_k + t);
        S.ctx_tok[t] = static_cast<int16_t>(t);
      }
      if (lane == 0) S.ctx_n[b] = a.M;
    } else {
      const int e = S.ulist[u];
      const unsigned long long mask = S.tokmask[e];
      int base = 0;
      for (int t0 = 0; t0 < a.M; t0 += 32) {
        const int t = t0 + lane;
        const bool has = (t < a.M) && ((mask >> t) & 1ull);
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
        if (has) {
          int r = 0;
          for (int k = 0; k < a.top_k; ++k)
            if (S.rid[t * a.top_k + k] == e) r = k;
          const int i = base + __popc(bal & ((1u << lane) - 1u));
          S.ctx_route[b][i] = static_cast<int16_t>(t * a.top_k + r);
          S.ctx_tok[i] = static_cast<int16_t>(t);
        }
        base += __popc(bal);
      }
      if (lane == 0) S.ctx_n[b] = base;
    }
  }
  fill_bar();
}

// MXFP8 input, GEMM1 chunk: one B row per route, the token's E4M3 codes as
// they are (cp.async into the swizzled layout); the four E8M0 bytes of each
// (route, K block) -- one per 32-value block -- are staged for the MMA
// thread, which copies them into tensor memory (tcgen05.cp) where the
// block-scaled MMA applies them to each 32-value partial. Cell (K block j,
// route t) is column 4 j + t / 32, lane t % 32 of the buffer's scale columns,
// staged as copy j (512 bytes), row t % 32, word t / 32. The activation scale
// of the accumulate step is then 1. Routed experts only (the MX entry has no
// shared expert).
template <int TOK>
__device__ bool fill_b_mx(const TcArgs& a, TcSmem& S, const Plan& P, const Chunk& ch, int b, int ci, int fid) {
  const int r = TOK == 1 ? 1 : S.ctx_n[2];  // one token: one route per unit
  const int N = P.N;
  uint8_t* B = S.B[b];
  uint32_t* stage = reinterpret_cast<uint32_t*>(B + kMxSfStage);
  const XInfo xi = xinfo(a, S, ch.u);
  float wsv = 0.0f;
  if (fid < 2 * kMaxKc) {
    const int half = fid / kMaxKc, j = fid % kMaxKc;
    if (j < ch.kc) {
      const int rb = (half == 0 ? 0 : a.I / 128) + ch.T / 2;
      wsv = __ldg(xi.s13 + (static_cast<size_t>(xi.row_e) * (2 * a.I / 128) + rb) * (a.H / 128) + ch.kb0 + j);
    }
  }
  if (ci >= 2) {
    if (!mbar_wait(&S.mfree[b], ((ci >> 1) - 1) & 1, a.timeout_ns, &S.abort)) {
      if (!S.abort) tc_error(a, S, kErrRingWait);
    }
    fill_bar();
    if (S.abort) return false;
  }
  for (int t = fid; t < r; t += kFillThreads) S.ctx_route[b][t] = S.ctx_route[2][t];
  if (fid == 0) S.ctx_n[b] = r;
  const int items = ch.kc * r * 8;
  {
    ItemWalk it(fid >> 3, kFillThreads / 8, r);
    const int sub = fid & 7;
    for (int w = fid; w < items; w += kFillThreads, it.next()) {
      const int t = it.t, j = it.j;
      const int tok = S.ctx_tok[t];
      cp_async_16(B + j * N * 128 + t * 128 + ((sub ^ (t & 7)) << 4),
                  a.xq + static_cast<size_t>(tok) * a.H + (ch.kb0 + j) * 128 + sub * 16);
    }
  }
  ItemWalk iw(fid, kFillThreads, r);
  for (int w = fid; w < ch.kc * r; w += kFillThreads, iw.next()) {
    const int t = iw.t, j = iw.j;
    const int tok = S.ctx_tok[t];
    const uint8_t* e = a.xsc + static_cast<size_t>(tok) * (a.H / 32) + (ch.kb0 + j) * 4;
    // The four bytes in one load when the array is 4-byte aligned (rows are
    // H / 32 bytes, a multiple of 4); bytes [e, e + 3] little-endian either way.
    const uint32_t packed = (reinterpret_cast<uintptr_t>(a.xsc) & 3u) == 0u
                                ? __ldg(reinterpret_cast<const uint32_t*>(e))
                                : static_cast<uint32_t>(__ldg(e)) | (static_cast<uint32_t>(__ldg(e + 1)) << 8) |
                                      (static_cast<uint32_t>(__ldg(e + 2)) << 16) |
                                      (static_cast<uint32_t>(__ldg(e + 3)) << 24);
    stage[j * 128 + (t & 31) * 4 + (t >> 5)] = packed;
    S.xs[b][t][j] = 1.0f;
  }
  if (fid < 2 * kMaxKc) S.wsc[b][fid / kMaxKc][fid % kMaxKc] = wsv;
  if (fid == 0) S.btag[b] = -1;
  cp_async_wait_all();
  fence_proxy_async_smem();
  fill_bar();
  if (fid == 0) mbar_arrive(&S.bfull[b]);
  return true;
}

// GEMM1 chunk from the per-call x image: each (route, K block) row is eight
// 16-byte copies into the swizzled B layout (cp.async, no registers), its
// scale one load; the weight scales as in fill_b.
__device__ bool fill_b_copy(const TcArgs& a, TcSmem& S, const Plan& P, const Chunk& ch, int b, int ci, int fid) {
  const int r = S.ctx_n[2];
  const int N = P.N;
  uint8_t* B = S.B[b];
  const XInfo xi = xinfo(a, S, ch.u);
  const int nbx = a.H / 128;
  float wsv = 0.0f;
  if (fid < 2 * kMaxKc) {
    const int half = fid / kMaxKc, j = fid % kMaxKc;
    if (j < ch.kc) {
      const int rb = (half == 0 ? 0 : a.I / 128) + ch.T / 2;
      wsv = __ldg(xi.s13 + (static_cast<size_t>(xi.row_e) * (2 * a.I / 128) + rb) * (a.H / 128) + ch.kb0 + j);
    }
  }
  if (ci >= 2) {
    if (!mbar_wait(&S.mfree[b], ((ci >> 1) - 1) & 1, a.timeout_ns, &S.abort)) {
      if (!S.abort) tc_error(a, S, kErrRingWait);
    }
    fill_bar();
    if (S.abort) return false;
  }
  for (int t = fid; t < r; t += kFillThreads) S.ctx_route[b][t] = S.ctx_route[2][t];
  if (fid == 0) S.ctx_n[b] = r;
  const int items = ch.kc * r * 8;
  {
    ItemWalk it(fid >> 3, kFillThreads / 8, r);
    const int sub = fid & 7;
    for (int w = fid; w < items; w += kFillThreads, it.next()) {
      const int t = it.t, j = it.j;
      const int tok = S.ctx_tok[t];
      cp_async_16(B + j * N * 128 + t * 128 + ((sub ^ (t & 7)) << 4),
                  a.ximg + static_cast<size_t>(tok) * a.H + (ch.kb0 + j) * 128 + sub * 16);
    }
  }
  ItemWalk iw(fid, kFillThreads, r);
  for (int w = fid; w < ch.kc * r; w += kFillThreads, iw.next()) {
    const int t = iw.t, j = iw.j;
    const int tok = S.ctx_tok[t];
    S.xs[b][t][j] = __ldcg(a.ximg_sc + static_cast<size_t>(tok) * nbx + ch.kb0 + j);
  }
  if (fid < 2 * kMaxKc) S.wsc[b][fid / kMaxKc][fid % kMaxKc] = wsv;
  if (fid == 0) S.btag[b] = -1;
  cp_async_wait_all();
  fence_proxy_async_smem();
  fill_bar();
  if (fid == 0) mbar_arrive(&S.bfull[b]);
  return true;
}

// Quantise the activations of chunk `ch` into B buffer b: for each token row
// t < r and K block j of the chunk, 128 values -> E4M3 by the pages' rule.
// Phase 1 reads x (BF16): sx = max(amax, 1e-10) / 448 [UE8M0], q = e4m3(x * (1/sx)).
// Phase 2 reads the SwiGLU output: sh likewise; routed q = e4m3(h / sh)
// ("mega_moe" hidden_block), shared q = e4m3(h * (1/sh)) ("shared_expert" _DownKernel).
// Row t of K block j sits at j*N*128 + t*128, its 16-byte chunk c at c ^ (t % 8)
// (the 128-byte swizzle the MMA descriptor names). Rows r..N-1 are left as
// they are: they only feed accumulator columns nobody reads.
// The scales and the first batch of activations are loaded before waiting
// for buffer b (chunk ci - 2's accumulators read), hiding their latency.
// Returns false when the wait gave up.
template <int TOK, bool MX>
__device__ bool fill_b(const TcArgs& a, TcSmem& S, const Plan& P, const Chunk& ch, int b, int ci, int fid) {
  if constexpr (MX) {
    if (ch.phase == 1) return fill_b_mx<TOK>(a, S, P, ch, b, ci, fid);
  }
  if (ch.phase == 1 && P.ximage) return fill_b_copy(a, S, P, ch, b, ci, fid);
  const int r = TOK == 1 ? 1 : S.ctx_n[2];  // one token: one route per unit
  const int N = P.N;
  uint8_t* B = S.B[b];
  const XInfo xi = xinfo(a, S, ch.u);
  // Weight block scales of the chunk's K blocks ([first/second row half][j]
  // for GEMM1: row blocks T/2 and I/128 + T/2; [0][j] for GEMM2: row block T).
  float wsv = 0.0f;
  if (fid < 2 * kMaxKc) {
    const int half = fid / kMaxKc, j = fid % kMaxKc;
    const int e = xi.row_e;
    if (j < ch.kc) {
      if (ch.phase == 1) {
        const int rb = (half == 0 ? 0 : a.I / 128) + ch.T / 2;
        wsv = __ldg(xi.s13 + (static_cast<size_t>(e) * (2 * a.I / 128) + rb) * (a.H / 128) + ch.kb0 + j);
      } else if (half == 0) {
        wsv = __ldg(xi.s2 + (static_cast<size_t>(e) * (a.H / 128) + ch.T) * (a.I / 128) + ch.kb0 + j);
      }
    }
  }
  // A GEMM2 chunk over the same unit and K range as the one buffer b holds
  // (the next 128 rows of W2, usually) takes the same quantised hidden rows:
  // only its weight scales are new.
  const int tag = ch.phase == 2 ? (ch.u * 64 + ch.kb0) * 32 + ch.kc : -1;
  const bool reuse = tag >= 0 && S.btag[b] == tag;
  const int items = reuse ? 0 : ch.kc * r * 8;
  const int K = ch.phase == 1 ? a.H : a.I;
  // Items per thread per round (all loads first, then quantise). Four were
  // tried: the larger unrolled code made every M slower (M = 8: 388 against
  // 380 us); many routes per expert take the copy fill above instead.
  constexpr int IPT = 2;
  float v[IPT][16], vn[IPT][16];
  int tt[IPT], jj[IPT], ttn[IPT], jjn[IPT];
  // Item w = base + q * kFillThreads + fid: 16-byte piece w & 7 of item
  // (row, K block) w >> 3, walked per q without dividing by r.
  ItemWalk walk[IPT] = {ItemWalk(fid >> 3, kFillThreads * IPT / 8, r),
                        ItemWalk(kFillThreads / 8 + (fid >> 3), kFillThreads * IPT / 8, r)};
  static_assert(IPT == 2, "one walk per item of a round");
  auto load_batch = [&](float (&v)[IPT][16], int (&tt)[IPT], int (&jj)[IPT], int base) {
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
      const int w = base + q * kFillThreads + fid;
      const int sub = w & 7;
      tt[q] = -1;
      jj[q] = 0;
      if (w < items) {
        tt[q] = walk[q].t;
        jj[q] = walk[q].j;
        const int route = S.ctx_route[2][tt[q]];
        const int col = (ch.kb0 + jj[q]) * 128 + sub * 16;
        if (ch.phase == 1) {
          const int tok = S.ctx_tok[tt[q]];
          const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * K + col);
          const uint4 q0 = __ldg(src), q1 = __ldg(src + 1);
          const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[q][2 * k] = __uint_as_float(wd[k] << 16);
            v[q][2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
          }
        } else {
          const float4* src = reinterpret_cast<const float4*>(a.hbuf + static_cast<size_t>(route) * K + col);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 f = __ldcg(src + k);
            v[q][4 * k] = f.x;
            v[q][4 * k + 1] = f.y;
            v[q][4 * k + 2] = f.z;
            v[q][4 * k + 3] = f.w;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[q][k] = 0.0f;
      }
      walk[q].next();
    }
  };
  auto store_batch = [&](int base) {  // quantises v (tt, jj) of the round at `base`
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
      if (base + q * kFillThreads >= items) break;  // uniform over the fill warps
      const int sub = (base + q * kFillThreads + fid) & 7;
      float amax = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[q][k]));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
      if (tt[q] >= 0) {
        const int t = tt[q], j = jj[q];
        float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
        if (xi.ue8m0) scale = ue8m0_ceil(scale);
        float qv[16];
        if (ch.phase == 2 && !xi.shared) {
#pragma unroll
          for (int k = 0; k < 16; ++k) qv[k] = __fdiv_rn(v[q][k], scale);
        } else {
          const float inv = __fdiv_rn(1.0f, scale);
#pragma unroll
          for (int k = 0; k < 16; ++k) qv[k] = __fmul_rn(v[q][k], inv);
        }
        uint32_t wq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          wq[k] = f32x2_to_e4m3x2(qv[4 * k], qv[4 * k + 1]) | (f32x2_to_e4m3x2(qv[4 * k + 2], qv[4 * k + 3]) << 16);
        uint8_t* dst = B + j * N * 128 + t * 128 + ((sub ^ (t & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        if (sub == 0) S.xs[b][t][j] = scale;
      }
    }
  };
  load_batch(v, tt, jj, 0);
  if (ci >= 2) {
    if (!mbar_wait(&S.mfree[b], ((ci >> 1) - 1) & 1, a.timeout_ns, &S.abort)) {
      if (!S.abort) tc_error(a, S, kErrRingWait);
    }
    fill_bar();
    if (S.abort) return false;
  }
  // Buffer b is free: publish the chunk's routes, then quantise.
  if (!reuse) {
    for (int t = fid; t < r; t += kFillThreads) S.ctx_route[b][t] = S.ctx_route[2][t];
    if (fid == 0) S.ctx_n[b] = r;
  }
  if (fid == 0) S.btag[b] = tag;
  // Rounds of IPT items per thread; the next round's loads are in flight
  // while this round is quantised.
  for (int base = 0; base < items; base += kFillThreads * IPT) {
    const bool more = base + kFillThreads * IPT < items;  // uniform over the fill warps
    if (more) load_batch(vn, ttn, jjn, base + kFillThreads * IPT);
    store_batch(base);
    if (more) {
#pragma unroll
      for (int q = 0; q < IPT; ++q) {
        tt[q] = ttn[q];
        jj[q] = jjn[q];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[q][k] = vn[q][k];
      }
    }
  }
  if (fid < 2 * kMaxKc) S.wsc[b][fid / kMaxKc][fid % kMaxKc] = wsv;
  fence_proxy_async_smem();
  fill_bar();
  if (fid == 0) mbar_arrive(&S.bfull[b]);
  return true;
}

// ---------------------------------------------------------------- epilogue pieces
// Finish one GEMM1 tile: y of a first-half row (threads 0..63) or a
// second-half row (64..127) -> SwiGLU of hidden 64T + q -> hbuf, then release
// the expert counter. Tokens go 16 at a time through shared memory, and the
// SwiGLU loop is not unrolled: this code runs once per tile, and keeping it
// small keeps it in the instruction cache.
template <int TOK>
__device__ void finish_gemm1(const TcArgs& a, TcSmem& S, const Chunk& ch, int b, const float (&y)[TOK],
                             int row, int etid) {
  const int r = S.seg_n;
  const XInfo xi = xinfo(a, S, ch.u);
  const bool shared = xi.shared;
  const int q = row & 63;
  const float L = xi.limit;
  constexpr int GS = TOK < 16 ? TOK : 16;  // tokens per pass through shared memory
  for (int g = 0; g * GS < r; ++g) {
#pragma unroll
    for (int gg = 0; gg < TOK / GS; ++gg) {
      if (gg == g) {
#pragma unroll
        for (int t = 0; t < GS; ++t) S.ysm[t][row] = y[gg * GS + t];
      }
    }
    epi_bar();
    if (row < 64) {
      const int n = min(GS, r - g * GS);
#pragma unroll 1
      for (int t = 0; t < n; ++t) {
        const int route = S.seg_route[g * GS + t];
        const float first = S.ysm[t][q], sec = S.ysm[t][q + 64];
        float h;
        if (!shared) {
          // W31: up rows first, then gate rows ("mega_moe" module docstring).
          const float gate = fminf(sec, L);
          const float up = fmaxf(fminf(first, L), -L);
          h = __fmul_rn(__fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate))), up);
        } else {
          // Shared gate_up: gate rows first; BF16 gate_up and BF16 h.
          const __nv_bfloat16 gb = __float2bfloat16_rn(first);
          const __nv_bfloat16 ub = __float2bfloat16_rn(sec);
          if (a.gate_up != nullptr) {
            const size_t tok = static_cast<size_t>(route - a.M * a.top_k);
            a.gate_up[tok * 2 * a.I + 64 * ch.T + q] = gb;
            a.gate_up[tok * 2 * a.I + a.I + 64 * ch.T + q] = ub;
          }
          const float gate = fminf(__bfloat162float(gb), L);
          const float up = fmaxf(fminf(__bfloat162float(ub), L), -L);
          const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
          h = __bfloat162float(__float2bfloat16_rn(__fmul_rn(silu, up)));
        }
        a.hbuf[static_cast<size_t>(route) * a.I + 64 * ch.T + q] = h;
      }
    }
    epi_bar();
  }
  // The barrier above orders every thread's hidden values before this
  // release (the same pattern publishes the partials).
  if (etid == 0) red_release_gpu_add(a.done + xi.id, 1u);
}

template <int TOK>
__device__ void finish_gemm2(const TcArgs& a, TcSmem& S, const Chunk& ch, int b, const float (&y)[TOK],
                             int row) {
  const int r = S.seg_n;
  const int m = 128 * ch.T + row;
  const bool shared = a.has_shared && ch.u == 0;
  // Routed rows go to out[route]; the shared expert's (routes M*top_k + t) to sout[t].
  __nv_bfloat16* dst = shared ? a.sout : a.out;
  const int row0 = shared ? a.M * a.top_k : 0;
  const int rows = shared ? a.M : a.M * a.top_k;
#pragma unroll
  for (int t = 0; t < TOK; ++t) {
    const int o = S.seg_route[t] - row0;
    if (t < r) {
      if (o >= 0 && o < rows)
        dst[static_cast<size_t>(o) * a.H + m] = __float2bfloat16_rn(y[t]);
      else
        atomicOr(a.err, kErrRoute);
    }
  }
}

__device__ __forceinline__ float* part_slot(const TcArgs& a, int w, int phase, int c, int slot) {
  return a.part + (((static_cast<size_t>(w) * 2 + phase - 1) * kFp8MaxCtas + c) * 2 + slot) * a.ptok * 128;
}

// End of a segment: finish the tile directly when this CTA owns all of it.
// A split tile is finished by its first contributor cf, which holds the
// tile's first K blocks at the END of its slice: the others (holding later K
// blocks at the START of theirs, or whole slices inside the tile) publish
// their partials and move on without waiting, and cf, usually the last to get
// there, adds them to its own in CTA order.
template <int TOK>
__device__ void end_segment(const TcArgs& a, TcSmem& S, const Plan& P, const Chunk& ch, int b, float (&y)[TOK],
                            int row, int etid) {
  const PhasePlan& pp = ch.pp;
  const int cf = pp.cta_of(ch.t0), cl = pp.cta_of(ch.t0 + pp.nb - 1);
  const int r = S.seg_n;
  if (cf != cl) {
    const int e = xinfo(a, S, ch.u).id;
    uint32_t* cnt = ch.phase == 1 ? a.cnt1 + static_cast<size_t>(e) * pp.tiles + ch.T
                                  : a.cnt2 + static_cast<size_t>(e) * pp.tiles + ch.T;
    if (P.c != cf) {
      float* mine = part_slot(a, pp.w, ch.phase, P.c, pp.lo >= ch.t0 ? 0 : 1);
#pragma unroll
      for (int t = 0; t < TOK; ++t)
        if (t < r) __stcg(mine + t * 128 + row, y[t]);
      // The barrier orders every thread's partial before one release.
      epi_bar();
      if (etid == 0) red_release_gpu_add(cnt, 1u);
      return;
    }
    if (etid == 0) {
      const uint32_t want = static_cast<uint32_t>(cl - cf);
      const uint64_t t0 = globaltimer_ns();
      bool ok = true;
      while (ld_acquire_gpu(cnt) < want) {
        if (S.abort || globaltimer_ns() - t0 > a.timeout_ns) {
          ok = false;
          break;
        }
        __nanosleep(32);
      }
      if (ok) {
        atomicExch(cnt, 0u);  // every contributor has arrived: re-arm for the next call
      } else if (!S.abort) {
        tc_error(a, S, kErrCrossWait);
      }
    }
    epi_bar();
    if (S.abort) return;
    // Add the other contributors' partials, four at a time (all loads in
    // flight), in CTA order after this CTA's own.
    for (int c0 = cf + 1; c0 <= cl; c0 += 4) {
      const float* src[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cc = min(c0 + q, cl);
        src[q] = part_slot(a, pp.w, ch.phase, cc, pp.lo_of(cc) >= ch.t0 ? 0 : 1) + row;
      }
      const int nq = min(4, cl - c0 + 1);
#pragma unroll
      for (int t = 0; t < TOK; ++t) {
        if (t < r) {
          float v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = __ldcg(src[q] + t * 128);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q < nq) y[t] += v[q];
        }
      }
    }
  }
  if (ch.phase == 1)
    finish_gemm1<TOK>(a, S, ch, b, y, row, etid);
  else
    finish_gemm2<TOK>(a, S, ch, b, y, row);
}

// Wait until every GEMM1 tile of expert u is finished. (pass_hidden counts
// the CTA in afterwards, off the path to the first GEMM2 MMA.)
__device__ bool wait_hidden(const TcArgs& a, TcSmem& S, const Plan& P, const Chunk& ch, int fid) {
  const int u = ch.u;
  if (a.phase_lo == 2) {
    // The chain's second kernel: the first kernel (every GEMM1 tile) has
    // completed and its writes are visible once this returns.
    griddep_wait();
    fill_bar();
    return true;
  }
  if (fid == 0) {
    const int e = xinfo(a, S, u).id;
    const uint32_t target = static_cast<uint32_t>(P.tiles[0]);
    const uint64_t t0 = globaltimer_ns();
    bool ok = true;
    while (ld_acquire_gpu(a.done + e) < target) {
      if (S.abort || globaltimer_ns() - t0 > a.timeout_ns) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
    if (!ok && !S.abort) tc_error(a, S, kErrCrossWait);
  }
  fill_bar();
  return !S.abort;
}

// Count this CTA past expert u's wait; the last CTA with GEMM2 work on it
// re-arms both counters for the next call (every such CTA has read `done`
// by then).
__device__ void pass_hidden(const TcArgs& a, TcSmem& S, const Chunk& ch) {
  const int e = xinfo(a, S, ch.u).id;
  const PhasePlan& p2 = ch.pp;
  const int s0 = (ch.u - p2.u0) * p2.tiles * p2.nb;
  const int s1 = s0 + p2.tiles * p2.nb - 1;
  const uint32_t ctas = static_cast<uint32_t>(p2.cta_of(s1) - p2.cta_of(s0) + 1);
  const uint32_t old = atomicAdd(a.passed + e, 1u);
  if (old + 1u == ctas) {
    atomicExch(a.done + e, 0u);
    atomicExch(a.passed + e, 0u);
  }
}

// Wait until every CTA has written its share of the x image; the last CTA
// past the wait re-arms both counters for the next call.
__device__ bool wait_ximage(const TcArgs& a, TcSmem& S, int fid) {
  if (fid == 0) {
    const uint32_t target = gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    bool ok = true;
    while (ld_acquire_gpu(a.xsync) < target) {
      if (S.abort || globaltimer_ns() - t0 > a.timeout_ns) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
    if (ok) {
      if (atomicAdd(a.xsync + 1, 1u) + 1u == target) {
        atomicExch(a.xsync, 0u);
        atomicExch(a.xsync + 1, 0u);
      }
    } else if (!S.abort) {
      tc_error(a, S, kErrCrossWait);
    }
  }
  fill_bar();
  return !S.abort;
}

// Scaled sum of one chunk's per-K-block partials: y[t] += D[j][t] *
// (w_scale[j] * x_scale[t][j]) for this thread's row. Loads LD columns per
// tcgen05.ld, GROUPS groups of them per K block, KB K blocks per wait.
template <int LD, int GROUPS, int KB, int TOK>
__device__ __forceinline__ void accumulate(uint32_t tbase, int N, int kc, int r, const float (&ws)[kMaxKc],
                                           const float (&xs)[kMaxTokens][kMaxKc], float (&y)[TOK]) {
#pragma unroll
  for (int j0 = 0; j0 < kMaxKc; j0 += KB) {
    if (j0 < kc) {
#pragma unroll
      for (int g = 0; g < GROUPS; ++g) {
        if (g * LD < r) {
          uint32_t v[KB][LD];
#pragma unroll
          for (int jb = 0; jb < KB; ++jb)
            if (j0 + jb < kc) tmem_ld<LD>(tbase + (j0 + jb) * N + g * LD, v[jb]);
          tc_wait_ld();
#pragma unroll
          for (int jb = 0; jb < KB; ++jb) {
            if (j0 + jb < kc) {
#pragma unroll
              for (int t = 0; t < LD; ++t) {
                if (g * LD + t < r) {
                  const float c = __fmul_rn(ws[j0 + jb], xs[g * LD + t][j0 + jb]);
                  y[g * LD + t] = fmaf(__uint_as_float(v[jb][t]), c, y[g * LD + t]);
                }
              }
            }
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
// TOK: token capacity of the accumulators (1, 4, 8, 16, 32 or 64: the
// smallest that holds M): the per-token loops are unrolled to it, so the
// smaller cases keep their code small enough to stay in the instruction
// caches, and code that cannot run at that capacity (the x image, the
// distributed router at one token) is left out.
template <int TOK, bool MX>
__global__ void __launch_bounds__(kTcThreads, 1) fp8_moe_tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& S = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.bfull[b], 1);
      mbar_init(&S.accfull[b], 1);
      mbar_init(&S.tmemfree[b], 4);
      mbar_init(&S.mfree[b], 4);
    }
    mbar_init(&S.final_bar, 1);
    fence_mbar_init();
    S.abort = 0;
    S.btag[0] = S.btag[1] = -1;
    if (a.E > 0) {
      prefetch_tmap(&a.map13);
      prefetch_tmap(&a.map2);
    }
    if (a.has_shared) {
      prefetch_tmap(&a.smap13);
      prefetch_tmap(&a.smap2);
    }
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  for (int e = tid; e < a.E; e += kTcThreads) S.tokmask[e] = 0ull;
  if (MX) {
    if (tid < 128) S.sfa_one[tid] = 0x7F7F7F7Fu;  // E8M0 2^0 in every byte
    fence_proxy_async_smem();
  }
  // The chain's second kernel reads only the inputs the first one read after
  // its own wait (logits, bias, weights) until its fill waits for the hidden
  // rows; every other launch waits for its predecessor here.
  if (a.phase_lo == 1) griddep_wait();
  if (a.phase_hi == 1) griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- routing and the unit list (the shared expert first, when present, then the routed ones)
  if (a.E > 0) {
    const int wpt = a.M == 1 ? 8 : (a.M == 2 ? 4 : 2);
    static_assert(kMaxExperts <= 128 * 8, "one token always takes the split router");
    if constexpr (TOK == 1) {
      route_split<8>(a, S, warp, lane, blockIdx.x == 0 && a.phase_lo == 1, 0, 1, 8, nullptr);
    } else if (a.M <= 4 && a.E <= 128 * wpt) {
      route_split(a, S, warp, lane, blockIdx.x == 0 && a.phase_lo == 1, 0, a.M, wpt, nullptr);
    } else {
      // Many tokens or experts: CTA c routes tokens c, c + G, ... with all its
      // warps, publishes the picks, and every CTA reads all of them back.
      int mine = 0;
      for (int t = blockIdx.x; t < a.M; t += gridDim.x) {
        route_split(a, S, warp, lane, a.phase_lo == 1, t, 1, 8, a.picks);
        __syncthreads();
        ++mine;
      }
      if (tid == 0) {
        if (mine > 0) {
          __threadfence();
          red_release_gpu_add(a.rsync, static_cast<uint32_t>(mine));
        }
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(a.rsync) < static_cast<uint32_t>(a.M)) {
          if (globaltimer_ns() - t0 > a.timeout_ns) {
            tc_error(a, S, kErrCrossWait);
            break;
          }
          __nanosleep(64);
        }
      }
      __syncthreads();
      if (!S.abort) {
        for (int i = tid; i < a.M * a.top_k; i += kTcThreads) {
          const int e = __ldcg(a.picks + i);
          if (e >= 0 && e < a.E) {
            S.rid[i] = static_cast<int16_t>(e);
            atomicOr(&S.tokmask[e], 1ull << (i / a.top_k));
          } else {
            atomicOr(a.err, kErrRoute);
          }
        }
        // the last CTA past the wait re-arms both counters for the next call
        if (tid == 0 && atomicAdd(a.rsync + 1, 1u) + 1u == gridDim.x) {
          atomicExch(a.rsync, 0u);
          atomicExch(a.rsync + 1, 0u);
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // The shared expert, when present, is unit 0 (its weights stream in the
      // first wave, so its GEMM1 -> GEMM2 hand-over overlaps the routed
      // experts' stream); the routed experts follow in ascending order.
      int U = a.has_shared ? 1 : 0, rmax = 0;
      if (lane == 0 && a.has_shared) S.ulist[0] = -1;
      for (int b = 0; b < a.E; b += 32) {
        const int e = b + lane;
        const unsigned long long m = e < a.E ? S.tokmask[e] : 0ull;
        const bool has = m != 0ull;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
        if (has) S.ulist[U + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(e);
        U += __popc(bal);
        rmax = max(rmax, static_cast<int>(__reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(__popcll(m)))));
      }
      if (lane == 0) {
        S.U = U;
        S.rmax = a.has_shared ? max(rmax, a.M) : rmax;
      }
      if constexpr (TOK > kLightRows) {
        // The one-launch layer's shared unit holds every token: above
        // kLightRows tokens its slots carry more fill, accumulate and
        // epilogue work than the routed units' and the split weighs them so
        // (M = 16: 683 -> 664 us). Routed units with many tokens measured no
        // better weighted (Latent shape, M = 16 / 32: 395 / 608 against 405 /
        // 616 us) and stay unweighted.
        if (lane == 0) {
          const int nh = a.has_shared && a.M > kLightRows ? 1 : 0;
          S.hu[0] = 0;
          S.he[0] = static_cast<uint16_t>(min(a.M, 64) - kLightRows);
          S.hce[0] = 0;
          S.hce[1] = S.he[0];
          S.heavy.nh = nh;
          S.heavy.hu = S.hu;
          S.heavy.he = S.he;
          S.heavy.hce = S.hce;
        }
      }
    }
  } else if (tid == 0) {
    S.U = 1;  // shared expert only
    S.rmax = a.M;
    S.heavy.nh = 0;
  }
  __syncthreads();

  // Many tokens on one expert: quantise x once per call into the image (every
  // CTA a share of the (token, K block) groups, one warp per group, the same
  // arithmetic as fill_b), so the GEMM1 fills only copy rows. With few routes
  // per expert the per-chunk quantisation is cheaper than the grid-wide wait.
  const bool ximage =
      !MX && TOK > kXImageRoutes && a.E > 0 && S.rmax > kXImageRoutes && (!a.has_shared || a.sue8m0 == a.ue8m0);
  if (ximage) {
    const int nbx = a.H / 128;
    const int groups = a.M * nbx;
    for (int g = blockIdx.x * (kTcThreads / 32) + warp; g < groups; g += gridDim.x * (kTcThreads / 32)) {
      const int t = g / nbx, kb = g - t * nbx;
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(a.x + static_cast<size_t>(t) * a.H + kb * 128 + lane * 4));
      const float v0 = __uint_as_float(raw.x << 16), v1 = __uint_as_float(raw.x & 0xFFFF0000u);
      const float v2 = __uint_as_float(raw.y << 16), v3 = __uint_as_float(raw.y & 0xFFFF0000u);
      float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      float scale = __fdiv_rn(fmaxf(amax, 1e-10f), 448.0f);
      if (a.ue8m0) scale = ue8m0_ceil(scale);
      const float inv = __fdiv_rn(1.0f, scale);
      const uint32_t q = f32x2_to_e4m3x2(__fmul_rn(v0, inv), __fmul_rn(v1, inv)) |
                         (f32x2_to_e4m3x2(__fmul_rn(v2, inv), __fmul_rn(v3, inv)) << 16);
      *reinterpret_cast<uint32_t*>(a.ximg + static_cast<size_t>(t) * a.H + kb * 128 + lane * 4) = q;
      if (lane == 0) a.ximg_sc[g] = scale;
    }
    __syncthreads();  // every share written before the one release
    if (tid == 0) {
      __threadfence();
      red_release_gpu_add(a.xsync, 1u);
    }
  }

  Plan P;
  P.U = S.U;
  P.ximage = ximage;
  P.N = 16 * ((S.rmax + 15) / 16);
  P.kcmax = min(kMaxKc, tmem_buf<MX>() / P.N);
  // Up to 4 tokens a GEMM2 chunk is at most the ring's depth, so the first
  // one after the GEMM1 -> GEMM2 hand-over finds all its weights already in
  // shared memory (M = 4: 213 -> 210 us; at 8 tokens, where the waves overlap
  // the hand-over, the longer chunks measured faster).
  P.kcmax2 = TOK <= 4 ? min(P.kcmax, kTcStages) : P.kcmax;
  // Up to kLightRows tokens no unit is heavy: those kernels split by slot
  // counts only and hold none of the cost-weighted code.
  P.hv = TOK > kLightRows ? &S.heavy : nullptr;
  P.N1 = P.N;
  P.kcmax1 = P.kcmax;
  P.c = blockIdx.x;
  P.G = gridDim.x;
  // (One token: one wave either way, known here so the schedule folds.)
  P.W = TOK == 1 || a.phase_lo == a.phase_hi ? 1
                                             : min(P.U, a.has_shared ? layer_waves(a.ptok) : max_waves(a.ptok));
  static_assert(max_waves(1) == 1 && layer_waves(1) == 1, "one wave at one token");
  P.phase_lo = a.phase_lo;
  P.phase_hi = a.phase_hi;
  P.tiles[0] = a.I / 64;
  P.nb[0] = a.H / 128;
  P.tiles[1] = a.H / 128;
  P.nb[1] = a.I / 128;
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      // Rows (two 64-row boxes) and tensor map of K block j of a chunk.
      auto coords = [&](const Chunk& c, int& ra, int& rb, const void*& map) {
        const XInfo xi = xinfo(a, S, c.u);
        const int e = xi.row_e;
        if (c.phase == 1) {
          ra = e * 2 * a.I + 64 * c.T;
          rb = ra + a.I;
          map = xi.m13;
        } else {
          ra = e * a.H + 128 * c.T;
          rb = ra + 64;
          map = xi.m2;
        }
      };
      Cursor cur;
      Chunk ch;
      int k = 0;
      bool ok = true;
      while (ok && cur.next<MX>(P, ch)) {
        int ra, rb;
        const void* map;
        coords(ch, ra, rb, map);
        for (int j = 0; j < ch.kc; ++j, ++k) {
          const int s = k % kTcStages;
          if (k >= kTcStages) {
            const uint32_t parity = ((k / kTcStages) - 1) & 1;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&S.empty[s], parity)) {
              if (S.abort || globaltimer_ns() - t0 > a.timeout_ns) {
                ok = false;
                break;
              }
            }
            if (!ok) {
              if (!S.abort) tc_error(a, S, kErrRingWait);
              break;
            }
          }
          mbar_arrive_expect_tx(&S.full[s], kAStageBytes);
          const int xk = (ch.kb0 + j) * 128;
          tma_load_2d(S.A[s], map, xk, ra, &S.full[s], pol);
          tma_load_2d(S.A[s] + kAStageBytes / 2, map, xk, rb, &S.full[s], pol);
        }
      }
      // Every load issued must land before the CTA may exit.
      for (int kk = max(0, k - kTcStages); kk < k; ++kk)
        if (!mbar_wait(&S.full[kk % kTcStages], (kk / kTcStages) & 1, a.timeout_ns, nullptr))
          atomicOr(a.err, kErrDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = f8_idesc(128, P.N);
      if (MX) {
        // The weights' scales: 2^0 for every row (their FP32 block scales are
        // applied by the accumulate warps).
        tc_cp_32x128b_x4(tmem + kSfaCol, rows16_desc(smem_u32(S.sfa_one)));
      }
      Cursor cur;
      Chunk ch;
      int k = 0, ci = 0;
      bool ok = true;
      while (ok && cur.next<MX>(P, ch)) {
        const int b = ci & 1;
        if (!mbar_wait(&S.bfull[b], (ci >> 1) & 1, a.timeout_ns, &S.abort) ||
            (ci >= 2 && !mbar_wait(&S.tmemfree[b], ((ci >> 1) - 1) & 1, a.timeout_ns, &S.abort))) {
          if (!S.abort) tc_error(a, S, kErrRingWait);
          break;
        }
        tc_fence_after();
        const uint32_t bbase = smem_u32(S.B[b]);
        const bool mx1 = MX && ch.phase == 1;
        const uint32_t sfb = tmem + kSfbCol + kSfbBuf * static_cast<uint32_t>(b);
        if (mx1) {
          // this chunk's token scales into tensor memory, ahead of its MMAs
          for (int q = 0; q < ch.kc; ++q)
            tc_cp_32x128b_x4(sfb + 4 * q, rows16_desc(bbase + kMxSfStage + 512 * q));
        }
        for (int j = 0; j < ch.kc; ++j, ++k) {
          const int s = k % kTcStages;
          if (!mbar_wait(&S.full[s], (k / kTcStages) & 1, a.timeout_ns, &S.abort)) {
            if (!S.abort) tc_error(a, S, kErrRingWait);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t abase = smem_u32(S.A[s]);
          const uint32_t d = tmem + b * tmem_buf<MX>() + j * P.N;
          if (mx1) {
            // MX GEMM1: each 32-value partial scaled by its token's E8M0 byte kk
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_mxf8(d, sw128_desc(abase + 32 * kk), sw128_desc(bbase + j * P.N * 128 + 32 * kk),
                          mxf8_idesc(128, P.N, static_cast<uint32_t>(kk)), tmem + kSfaCol, sfb + 4 * j,
                          kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f8(d, sw128_desc(abase + 32 * kk), sw128_desc(bbase + j * P.N * 128 + 32 * kk), idesc,
                        kk > 0 ? 1u : 0u);
          }
          tc_commit(&S.empty[s]);
        }
        if (!ok) break;
        tc_commit(&S.accfull[b]);
        ++ci;
      }
      // Every MMA issued must complete before TMEM is released.
      tc_commit(&S.final_bar);
      if (!mbar_wait(&S.final_bar, 0, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ accumulate
    const int etid = tid - 64;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = tile row
    const int half = row < 64 ? 0 : 1;
    Cursor cur;
    Chunk ch;
    int ci = 0;
    bool seg_first = true;
    float y[TOK];
#pragma unroll
    for (int t = 0; t < TOK; ++t) y[t] = 0.0f;
    while (cur.next<MX>(P, ch)) {
      const int b = ci & 1;
      if (!mbar_wait(&S.accfull[b], (ci >> 1) & 1, a.timeout_ns, &S.abort)) {
        if (!S.abort) tc_error(a, S, kErrRingWait);
      }
      epi_bar();
      if (S.abort) break;
      tc_fence_after();
      const int r = S.ctx_n[b];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16) + b * tmem_buf<MX>();
      {
        float ws[kMaxKc];
#pragma unroll
        for (int j = 0; j < kMaxKc; ++j) ws[j] = S.wsc[b][ch.phase == 1 ? half : 0][j];
        // Load widths by this chunk's route count, none wider than TOK.
        if (TOK == 1 || r == 1) {
          accumulate<1, 1, 16>(tbase, P.N, ch.kc, r, ws, S.xs[b], y);
        } else if (TOK == 4 || r <= 4) {
          if constexpr (TOK >= 4) accumulate<4, 1, 8>(tbase, P.N, ch.kc, r, ws, S.xs[b], y);
        } else if constexpr (TOK == 8) {
          accumulate<8, 1, 4>(tbase, P.N, ch.kc, r, ws, S.xs[b], y);
        } else if (TOK == 16 || r <= 16) {
          if constexpr (TOK >= 16) accumulate<16, 1, 2>(tbase, P.N, ch.kc, r, ws, S.xs[b], y);
        } else {
          if constexpr (TOK > 16) accumulate<16, TOK / 16, 1>(tbase, P.N, ch.kc, r, ws, S.xs[b], y);
        }
      }
      tc_fence_before();
      if (seg_first) {
        // First chunk of a segment: keep its routes for the segment's end.
        for (int t = etid; t < r; t += 128) S.seg_route[t] = S.ctx_route[b][t];
        if (etid == 0) S.seg_n = r;
      }
      epi_bar();
      // TMEM buffer b and B buffer b (tile, scales, routes) may now be reused.
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.tmemfree[b]);
        mbar_arrive(&S.mfree[b]);
      }
      seg_first = ch.last_of_seg;
      if (ch.last_of_seg) {
        end_segment<TOK>(a, S, P, ch, b, y, row, etid);
#pragma unroll
        for (int t = 0; t < TOK; ++t) y[t] = 0.0f;
      }
      ++ci;
    }
  } else {
    // ------------------------------------------------------------ fill
    // Quantise each chunk's activations into the B operand and stage its
    // scales, up to two chunks ahead of the accumulate warps.
    const int fid = tid - 192;
    Cursor cur;
    Chunk ch;
    int ci = 0, ctx_u = -1, ctx_phase = 0;
    bool ok = true;
    if (ximage) ok = wait_ximage(a, S, fid);
    while (ok && cur.next<MX>(P, ch)) {
      const int b = ci & 1;
      if (ch.u != ctx_u) fill_context(a, S, ch.u, fid);
      const bool first2 = ch.phase == 2 && (ch.u != ctx_u || ctx_phase != 2);
      if (first2 && !wait_hidden(a, S, P, ch, fid)) break;
      ctx_u = ch.u;
      ctx_phase = ch.phase;
      if (!fill_b<TOK, MX>(a, S, P, ch, b, ci, fid)) break;
      if (first2 && fid == 0) pass_hidden(a, S, ch);
      ++ci;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte tensor [rows, cols] (row-major), box 64 rows x 128 bytes, 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, unsigned long long rows, unsigned long long cols) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, 64};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcWorkspace {
  uint32_t *err, *done, *passed, *cnt1, *cnt2, *xsync, *rsync;
  int32_t* picks;
  float *hbuf, *part, *xsc;
  uint8_t* ximg;
  int ptok;
  size_t zero_bytes;  // error word and counters: must be zero when a call starts
  size_t bytes;
};

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static TcWorkspace tc_layout(void* base, int M, int routes, int H, int I, int E) {
  TcWorkspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.err = reinterpret_cast<uint32_t*>(p + off);
  w.xsync = reinterpret_cast<uint32_t*>(p + off + 64);  // two words in the error word's 256-byte unit
  w.rsync = reinterpret_cast<uint32_t*>(p + off + 128);  // two more
  off += 256;
  w.done = reinterpret_cast<uint32_t*>(p + off);
  off += align256(4 * static_cast<size_t>(E));
  w.passed = reinterpret_cast<uint32_t*>(p + off);
  off += align256(4 * static_cast<size_t>(E));
  // Counters first, sized by the expert count only: the zeroed prefix is the
  // same for every M, so one workspace serves calls with any M up to its size.
  w.cnt1 = reinterpret_cast<uint32_t*>(p + off);
  off += align256(4 * static_cast<size_t>(E) * (I / 64));
  w.cnt2 = reinterpret_cast<uint32_t*>(p + off);
  off += align256(4 * static_cast<size_t>(E) * (H / 128));
  w.zero_bytes = off;
  w.hbuf = reinterpret_cast<float*>(p + off);
  off += align256(4 * static_cast<size_t>(routes) * I);
  w.ptok = M < kMaxTokens ? M : kMaxTokens;
  w.part = reinterpret_cast<float*>(p + off);
  off += align256(4 * static_cast<size_t>(waves_cap(w.ptok)) * 2 * kFp8MaxCtas * 2 * w.ptok * 128);
  w.ximg = p + off;
  off += align256(static_cast<size_t>(M) * H);
  w.xsc = reinterpret_cast<float*>(p + off);
  off += align256(4 * static_cast<size_t>(M) * (H / 128));
  w.picks = reinterpret_cast<int32_t*>(p + off);
  off += align256(4 * static_cast<size_t>(M) * kMaxTopK);
  w.bytes = off;
  return w;
}

// lay_routes / lay_slots: hidden rows and counter slots of the workspace
// layout (by default this call's own).
static int launch_tc(TcArgs& a, const uint8_t* w13, const uint8_t* w2, const uint8_t* sw13, const uint8_t* sw2,
                     void* workspace, size_t workspace_bytes, cudaStream_t st, int lay_routes = -1,
                     int lay_slots = -1) {
  const int routes = lay_routes >= 0 ? lay_routes : a.M * a.top_k + (a.has_shared ? a.M : 0);
  const TcWorkspace w = tc_layout(workspace, a.M, routes, a.H, a.I, lay_slots >= 0 ? lay_slots : a.E + 1);
  if (workspace == nullptr || workspace_bytes < w.bytes)
    return set_last_error(FME_EWORKSPACE, "workspace of %zu bytes needed, %zu given", w.bytes, workspace_bytes);
  a.err = w.err;
  a.done = w.done;
  a.passed = w.passed;
  a.cnt1 = w.cnt1;
  a.cnt2 = w.cnt2;
  a.hbuf = w.hbuf;
  a.part = w.part;
  a.ximg = w.ximg;
  a.ximg_sc = w.xsc;
  a.picks = w.picks;
  a.rsync = w.rsync;
  a.xsync = w.xsync;
  a.ptok = w.ptok;
  a.timeout_ns = wait_timeout_ns();
  if (a.E > 0 && (!make_map(&a.map13, w13, static_cast<unsigned long long>(a.E) * 2 * a.I, a.H) ||
                  !make_map(&a.map2, w2, static_cast<unsigned long long>(a.E) * a.H, a.I)))
    return set_last_error(FME_ECUDA, "cuTensorMapEncodeTiled failed or unavailable");
  if (a.has_shared && (!make_map(&a.smap13, sw13, static_cast<unsigned long long>(2) * a.I, a.H) ||
                       !make_map(&a.smap2, sw2, static_cast<unsigned long long>(a.H), a.I)))
    return set_last_error(FME_ECUDA, "cuTensorMapEncodeTiled failed or unavailable");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_last_error(FME_ECUDA, "cudaGetDevice failed");
  const int sms = device_sm_count(dev);
  if (sms <= 0) return set_last_error(FME_ECUDA, "cannot query the SM count");
  // The smallest token capacity that holds M (every expert then has <= M rows).
  auto kernel = a.xq != nullptr
                    ? (a.M == 1 ? fp8_moe_tc_kernel<1, true>
                                : a.M <= 4 ? fp8_moe_tc_kernel<4, true>
                                : a.M <= 8 ? fp8_moe_tc_kernel<8, true>
                                : (a.M <= 16 ? fp8_moe_tc_kernel<16, true>
                                             : (a.M <= 32 ? fp8_moe_tc_kernel<32, true>
                                                          : fp8_moe_tc_kernel<kMaxTokens, true>)))
                    : (a.M == 1 ? fp8_moe_tc_kernel<1, false>
                                : a.M <= 4 ? fp8_moe_tc_kernel<4, false>
                                : a.M <= 8 ? fp8_moe_tc_kernel<8, false>
                                : (a.M <= 16 ? fp8_moe_tc_kernel<16, false>
                                             : (a.M <= 32 ? fp8_moe_tc_kernel<32, false>
                                                          : fp8_moe_tc_kernel<kMaxTokens, false>)));
  if (!ensure_smem_attr(dev, reinterpret_cast<const void*>(kernel), kTcSmemBytes)) return FME_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms < kFp8MaxCtas ? sms : kFp8MaxCtas);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, a);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "fp8 kernel launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

// Routed calls as a two-kernel chain instead of one persistent launch
// (FME_FP8_CHAIN=1): kept to compare the two schedules, off by default.
static bool fp8_chain_enabled() {
  const char* env = std::getenv("FME_FP8_CHAIN");
  return env != nullptr && env[0] == '1';
}

static int layer_launch(const RoutedFp8& r, const SharedFp8& sh, int M, int H, int I, void* workspace,
                        size_t workspace_bytes, cudaStream_t st, int lay_routes, int lay_slots);

int layer_fp8(const RoutedFp8& r, const SharedFp8& sh, int M, int H, int I, void* workspace, size_t workspace_bytes,
              cudaStream_t st) {
  // The MXFP8-input kernel reads its tokens from xq only: no shared expert beside it.
  if (r.xq != nullptr && sh.w13 != nullptr)
    return set_last_error(FME_EINVAL, "MXFP8 input with a shared expert is not supported");
  // Above 16 tokens the shared unit, every token on one expert, is far more
  // fill, accumulate and epilogue work per weight byte than the routed units,
  // and the CTAs holding its slices set the launch's time (DeepSeek-V3 shape:
  // M = 32 1394 us in one launch against 1056 + 109 us for the two calls). It
  // then runs alone, followed by the routed experts, on the stream. Both
  // launches use the one-launch call's workspace layout (the shared expert
  // alone takes counter slot 0, zero before and after it), and each leaves
  // the zeroed prefix zero for the next.
  if (r.E > 0 && sh.w13 != nullptr && M > 16) {
    const int lay_routes = M * r.top_k + M, lay_slots = r.E + 1;
    const int err = layer_launch(RoutedFp8{}, sh, M, H, I, workspace, workspace_bytes, st, lay_routes, lay_slots);
    if (err != FME_OK) return err;
    return layer_launch(r, SharedFp8{}, M, H, I, workspace, workspace_bytes, st, lay_routes, lay_slots);
  }
  return layer_launch(r, sh, M, H, I, workspace, workspace_bytes, st, -1, -1);
}

static int layer_launch(const RoutedFp8& r, const SharedFp8& sh, int M, int H, int I, void* workspace,
                        size_t workspace_bytes, cudaStream_t st, int lay_routes, int lay_slots) {
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.phase_lo = 1;
  a.phase_hi = 2;
  a.M = M;
  a.H = H;
  a.I = I;
  a.scale = 1.0f;
  if (r.E > 0) {
    a.x = static_cast<const __nv_bfloat16*>(r.x);
    a.xq = r.xq;
    a.xsc = r.xsc;
    a.logits = r.logits;
    a.bias = r.bias;
    a.s13 = r.s13;
    a.s2 = r.s2;
    a.out = static_cast<__nv_bfloat16*>(r.out);
    a.ids = r.ids;
    a.weights = r.weights;
    a.E = r.E;
    a.top_k = r.top_k;
    a.limit = r.limit;
    a.scale = r.scale;
    a.ue8m0 = r.ue8m0 ? 1 : 0;
    a.logits_f32 = r.logits_dtype == FME_F32 ? 1 : 0;
  }
  if (sh.w13 != nullptr) {
    a.x = static_cast<const __nv_bfloat16*>(sh.x);
    a.has_shared = 1;
    a.ss13 = sh.s13;
    a.ss2 = sh.s2;
    a.sout = static_cast<__nv_bfloat16*>(sh.out);
    a.gate_up = static_cast<__nv_bfloat16*>(sh.gate_up);
    a.slimit = sh.limit;
    a.sue8m0 = sh.ue8m0 ? 1 : 0;
  }
  if (r.E > 0 && sh.w13 == nullptr && r.xq == nullptr && fp8_chain_enabled()) {
    // The two-kernel chain: GEMM1 .. SwiGLU, then the re-quant and GEMM2 as a
    // programmatic dependent launch (the same workspace layout; the second
    // kernel re-arms the hidden counters the first one raised).
    a.phase_hi = 1;
    const int err = launch_tc(a, r.w13, r.w2, sh.w13, sh.w2, workspace, workspace_bytes, st, lay_routes, lay_slots);
    if (err != FME_OK) return err;
    a.phase_lo = a.phase_hi = 2;
  }
  return launch_tc(a, r.w13, r.w2, sh.w13, sh.w2, workspace, workspace_bytes, st, lay_routes, lay_slots);
}

// Counter slots are sized for the routed experts plus the shared expert
// whether or not a call has it, so routed-only and one-launch calls with the
// same sizes lay out their counters alike and can share one workspace.
size_t layer_fp8_workspace_bytes(int M, int H, int I, int E, int top_k, bool shared) {
  return tc_layout(nullptr, M, M * top_k + (shared ? M : 0), H, I, E + 1).bytes;
}

size_t layer_fp8_zero_bytes(int M, int H, int I, int E, int top_k, bool shared) {
  return tc_layout(nullptr, M, M * top_k + (shared ? M : 0), H, I, E + 1).zero_bytes;
}

}  // namespace fme
