// NVFP4 slot MoE over one local expert range: one persistent sm_103a kernel
// on the 5th-generation tensor cores.
//
// Computes what "nvfp4-megamoe-kernel README.md" describes (slot
// representation; Data Formats; Bugs Found & Fixed 2, 4, 6, 7): a slot is a
// (token, pick) pair whose expert is local; per slot the L1 GEMM on the
// [gate; up] weight, SiLU*Mul, re-quantisation to E2M1 with UE4M3 group-16
// scales, the L2 GEMM; the routing weights are applied once, in the final
// scatter to [M, H]. The design is this library's own:
//
// * Both GEMMs run on `tcgen05.mma kind::mxf4nvf4` (block-scaled E2M1 x E2M1
//   with one UE4M3 scale per 16 values on each side, FP32 accumulation):
//   exactly the pages' block-scaled product, with the packed weights read
//   straight from the TMA ring and no dequantisation.
// * Weights: TMA streams the packed E2M1 rows, 128 bytes (256 values) of
//   each of 128 rows per K block, 128-byte swizzle, into a ring; their group
//   scales come ahead through cp.async and four scale warps write them, with
//   the activation scales, into tensor memory for the MMA.
// * Activations: at start every CTA quantises a share of x to E2M1 with
//   UE4M3 group scales into a packed image in the workspace (all tokens, 16
//   or 64 rows); the GEMM1 epilogue quantises each slot's h (groups of 16 lie
//   inside one 64-row tile) into a second packed image whose rows are the
//   slots of each expert, consecutive. A second TMA thread loads image and
//   scales as the B operand; GEMM1 uses every token as a column and reads
//   back the routed ones.
// * Work split, split-tile finishing and bounded waits follow the routed FP8
//   kernel: one CTA per SM, each phase's (expert, tile, K block) list cut
//   into equal slices, a split tile finished by its first contributor.
// * The scatter y[t] = bf16(sum over t's local picks, ascending, of
//   w * o[slot]) in FP32 runs after every GEMM2 tile (bounded wait).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "fme_common.cuh"
#include "fme_internal.h"

namespace fme {

constexpr int kNvThreads = 352;         // A TMA, MMA, B TMA, 4 scale, 4 epilogue warps
constexpr int kNvKB = 256;              // K values per K block
constexpr int kNvRawBytes = 128 * 128;  // one K block: 128 rows x 128 packed bytes

// Weight group scales run kNvScaleAhead K blocks ahead of the scale warps
// (two 8-byte cp.async per row into a small shared ring), so their global
// latency never stalls them.
constexpr int kNvScaleAhead = 4;

// Tensor memory: the accumulators (two buffers of TOK columns) sit in
// columns 0 .. 127, the scale vectors of a K block (16 columns for A, 16 for
// B: four per MMA) in buffers of 32 columns from column 128 on.
constexpr uint32_t kNvTmemCols = 256;
__device__ __forceinline__ uint32_t nv_sfcol(int sf) { return 128u + 32u * static_cast<uint32_t>(sf); }

template <int TOK>
struct NvCfg {
  // Packed-weight ring: 64-80 KB in flight per SM. Deeper rings measured
  // slower (more weight rows open at once in DRAM: 10 stages took M = 8 from
  // 56 to 62 us, 8 stages M = 64 from 177 to 205 us); the activation operand
  // comes from L2 and needs only a short ring of its own: 6 stages from 32
  // tokens up (M = 64: 182.9 -> 180.9 us against 4; 8 took it to 211 us).
  static constexpr int kStages = TOK == 16 ? 4 : 5;
  static constexpr int kBStages = TOK == 16 ? 4 : 6;
  static constexpr int kSfBuf = 4;                // scale-vector buffers in tensor memory
  static constexpr int kBBytes = TOK * 128;       // TOK rows of 128 packed bytes (256 values)
  static constexpr int kBsBytes = TOK * 16;       // their 16 group scales
};

struct NvArgs {
  CUtensorMap map13;  // W13 packed [L * 2N rows, H/2 bytes], box 64 rows x 128 bytes, 128-byte swizzle
  CUtensorMap map2;   // W2 packed [L * H rows, N/2 bytes], same box
  CUtensorMap mapx;   // x image [nb1 * TOK rows, 128 bytes], box TOK rows, 128-byte swizzle
  CUtensorMap mapxs;  // x image scales [nb1 * TOK rows, 16 bytes], box TOK rows
  CUtensorMap maph;   // h image [nb2 * Rp rows, 128 bytes], box TOK rows, 128-byte swizzle
  CUtensorMap maphs;  // h image scales [nb2 * Rp rows, 16 bytes], box TOK rows
  const __nv_bfloat16* x;
  const int32_t* ids;  // [M, top_k] caller's picks (route == 0)
  const float* tw;
  // Fused routing (route != 0): picks from logits [M, E] + bias [E] by the
  // routed FP8 kernel's rule, written to ids_out / tw_out by CTA 0.
  const void* logits;
  const float* bias;
  int32_t* ids_out;
  float* tw_out;
  int route, E, logits_f32;
  float scale;
  const uint8_t* s13;
  const uint8_t* s2;
  __nv_bfloat16* y;
  uint32_t* err;
  uint32_t* sync;     // [6]: x image shares written, CTAs past that wait, GEMM2 tiles done, CTAs past the scatter
                      // wait, CTAs whose tokens are routed, CTAs past that wait
  uint32_t* done;     // [L] GEMM1 tiles finished per local expert
  uint32_t* hpassed;  // [L] CTAs past the expert's hidden wait
  uint32_t* cnt1;     // [L * N/64] contributors per GEMM1 tile
  uint32_t* cnt2;     // [L * H/128]
  uint8_t* ximg;  // [nb1][TOK][128]: packed E2M1 of x, K block kb of token t at row kb * TOK + t
  uint8_t* xsc;   // [nb1][TOK][16]: its UE4M3 group scales
  uint8_t* himg;  // [nb2][Rp][128]: packed E2M1 of h, slot rows of each unit consecutive
  uint8_t* hsc;   // [nb2][Rp][16]
  __nv_bfloat16* obuf;  // [M * top_k, H] slot outputs (route order)
  float* part;          // [2][kFp8MaxCtas][2][TOK][128]
  int M, H, N, L, e0, top_k, Rp;
  float limit;
  unsigned long long timeout_ns;
};

template <int TOK>
struct NvSmem {
  uint8_t B[NvCfg<TOK>::kBStages][NvCfg<TOK>::kBBytes];
  uint8_t R[NvCfg<TOK>::kStages][kNvRawBytes];
  alignas(128) uint8_t Bs[NvCfg<TOK>::kBStages][NvCfg<TOK>::kBsBytes];
  uint64_t fullA[NvCfg<TOK>::kStages], emptyA[NvCfg<TOK>::kStages];
  uint64_t fullB[NvCfg<TOK>::kBStages], emptyB[NvCfg<TOK>::kBStages];
  uint64_t sffull[NvCfg<TOK>::kSfBuf], sffree[NvCfg<TOK>::kSfBuf], accfull[2], tmemfree[2], final_bar;
  float ysm[16][128];
  uint4 sc[kNvScaleAhead][128];  // weight group scales of the next K blocks, by row
  unsigned long long tokmask[kMaxExperts];
  int16_t ulist[kMaxExperts];
  int16_t uidx[kMaxExperts];      // local expert -> unit
  int16_t uoff[kMaxExperts + 1];  // first compact slot row of each unit
  int16_t stok[kMaxTokens * kMaxTopK];
  int16_t sroute[kMaxTokens * kMaxTopK];
  int16_t sid[kMaxTokens * kMaxTopK];  // every route's local expert, -1 when not local
  uint32_t tmem_base;
  int U;
  int direct;  // every token has at most one local slot: y is written by the GEMM2 epilogue
  volatile int abort;
};

// At least 120 KB are requested whatever the rings take, so that a second
// CTA never fits on the SM (see below).
template <int TOK>
constexpr size_t nv_smem_bytes() {
  return sizeof(NvSmem<TOK>) + 1024 > 120 * 1024 ? sizeof(NvSmem<TOK>) + 1024 : 120 * 1024;
}
template <int TOK>
constexpr bool nv_fits() {
  // Shared memory per CTA; tensor memory columns; swizzled TMA destinations
  // (128-byte swizzle) on 1024-byte boundaries; and one CTA per SM: a second
  // CTA would wait in its TMEM allocation while the first may wait on it
  // through the cross-CTA counters, so shared memory keeps it out.
  return nv_smem_bytes<TOK>() <= 232448 && 128 + 32 * NvCfg<TOK>::kSfBuf <= kNvTmemCols &&
         offsetof(NvSmem<TOK>, R) % 1024 == 0 && nv_smem_bytes<TOK>() > 233472 / 2;
}
static_assert(nv_fits<16>() && nv_fits<32>() && nv_fits<64>(), "NVFP4 kernel resources");

__device__ __forceinline__ void nv_epi_bar() { named_bar_sync(1, 128); }

__device__ __forceinline__ void nv_error(const NvArgs& a, volatile int& abort, uint32_t bit) {
  atomicOr(a.err, bit);
  abort = 1;
}

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: A and B E2M1 (type
// code 1 in bits 7-9 and 10-12), both K-major, UE4M3 scales (bit 23 clear),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28, scale-vector ids 0 (four
// scales per row per MMA take the whole 32-bit TMEM cell).
__host__ __device__ constexpr uint32_t nv_idesc(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// D (TMEM) (+)= sum over the 4 groups of 16 of (A x B) * sfa * sfb: A and B
// packed E2M1 in shared memory (64 values, 32 bytes, per row), the scale
// vectors in TMEM.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 2-D tiled TMA load without an L2 cache hint (the activation images are small
// and re-read by every CTA).
__device__ __forceinline__ void tma_load_2d_plain(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 8-byte copy of which the first src_bytes (8 or 0) come from src, the rest zeros.
__device__ __forceinline__ void cp_async8(void* dst, const void* src, uint32_t src_bytes = 8) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// UE4M3 scale byte of a group: e4m3(amax / 6), saturating ("nvfp4-megamoe-kernel
// README.md" Bugs Found & Fixed 2: the stored scale is also the divisor).
__device__ __forceinline__ uint32_t nv_scale_byte(float amax) {
  return f32x2_to_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu;
}
// Two values -> their E2M1 codes (v0 in the low nibble) against the group's
// stored scale d; d == 0 gives zeros (a zero scale quantises its group to
// zeros).
__device__ __forceinline__ uint32_t nv_quant2(float v0, float v1, float d) {
  if (!(d > 0.0f)) return 0u;
  return f32x2_to_e2m1x2(__fdiv_rn(v0, d), __fdiv_rn(v1, d));
}

// ---------------------------------------------------------------- work plan
// Each phase's (unit, tile, K block) slots -- at most 1024 x 128 x 32 = 4.2M --
// split over Ge = min(G, n) CTAs as in the routed FP8 kernel; the products stay
// below 2^32, so unsigned 32-bit arithmetic is exact.
struct NvPhase {
  int n, lo, hi, Ge, tiles, nb;
  __device__ int lo_of(int c) const {
    return c >= Ge ? n : static_cast<int>(static_cast<uint32_t>(n) * static_cast<uint32_t>(c) /
                                          static_cast<uint32_t>(Ge));
  }
  __device__ int cta_of(int x) const {
    return static_cast<int>((static_cast<uint32_t>(x + 1) * static_cast<uint32_t>(Ge) + static_cast<uint32_t>(n) - 1u) /
                            static_cast<uint32_t>(n)) - 1;
  }
};

__device__ NvPhase nv_phase(int n, int tiles, int nb, int G, int c) {
  NvPhase p;
  p.n = n;
  p.tiles = tiles;
  p.nb = nb;
  p.Ge = min(G, n);
  if (c >= p.Ge) {
    p.lo = p.hi = n;
  } else {
    p.lo = p.lo_of(c);
    p.hi = p.lo_of(c + 1);
  }
  return p;
}

// One K block of this CTA's slices, phase 1 then phase 2.
struct NvStep {
  int phase, u, T, kb;
  int t0;            // first slot of the tile
  bool first, last;  // first / last K block of its segment
};

struct NvCursor {
  int pos, phase;
  int u = 0, T = 0, kb = 0;  // of slot pos, once `at` is set (kept by increments, no divisions)
  bool at = false;
  __device__ bool next(const NvPhase (&P)[2], NvStep& st) {
    while (true) {
      const NvPhase& p = P[phase - 1];
      if (pos < p.lo) {
        pos = p.lo;
        at = false;
      }
      if (pos < p.hi) {
        if (!at) {
          const int tile = pos / p.nb;
          kb = pos - tile * p.nb;
          u = tile / p.tiles;
          T = tile - u * p.tiles;
          at = true;
        }
        st.phase = phase;
        st.u = u;
        st.T = T;
        st.kb = kb;
        st.t0 = pos - kb;
        st.first = pos == p.lo || kb == 0;
        st.last = pos + 1 == p.hi || kb == p.nb - 1;
        ++pos;
        if (++kb == p.nb) {
          kb = 0;
          if (++T == p.tiles) {
            T = 0;
            ++u;
          }
        }
        return true;
      }
      if (phase == 2) return false;
      phase = 2;
      pos = P[1].lo;
      at = false;
    }
  }
};

__device__ __forceinline__ float* nv_part(const NvArgs& a, int phase, int c, int slot, int tok) {
  return a.part + ((static_cast<size_t>(phase - 1) * kFp8MaxCtas + c) * 2 + slot) * tok * 128;
}

// ---------------------------------------------------------------- epilogue
// GEMM1 tile T of unit u (rows 0..63 gate 64T + q, 64..127 up): per slot of
// the unit, g = bf16(gate), v = bf16(up), h = bf16(silu(min(g, L)) *
// clamp(v, -L, L)) ("nvfp4-megamoe-kernel README.md" Bugs Found & Fixed 4
// and 6), then h -> E2M1 with a UE4M3 scale per 16 (groups 16j..16j+15 of
// the tile are half-warps), written to the slot's row of the h image: the
// tile's 64 values are bytes 32 (T % 4) .. + 31 of K block T / 4, its four
// scales bytes 4 (T % 4) .. + 3.
template <int TOK>
__device__ void nv_finish1(const NvArgs& a, NvSmem<TOK>& S, int u, int T, const float (&y)[TOK], int row,
                           int etid) {
  const int le = S.ulist[u];
  const int r0 = S.uoff[u], r = S.uoff[u + 1] - r0;
  const int q = row & 63;
  const float L = a.limit;
  for (int g = 0; g * 16 < a.M; ++g) {
#pragma unroll
    for (int gg = 0; gg < TOK / 16; ++gg) {
      if (gg == g) {
#pragma unroll
        for (int t = 0; t < 16; ++t) S.ysm[t][row] = y[gg * 16 + t];
      }
    }
    nv_epi_bar();
    if (row < 64) {
#pragma unroll 1
      for (int i = 0; i < r; ++i) {
        const int t = S.stok[r0 + i];
        if (t < g * 16 || t >= g * 16 + 16) continue;  // uniform over the warp
        const float gate = __bfloat162float(__float2bfloat16_rn(S.ysm[t - g * 16][q]));
        const float up = __bfloat162float(__float2bfloat16_rn(S.ysm[t - g * 16][q + 64]));
        const float gc = fminf(gate, L);
        const float uc = fmaxf(fminf(up, L), -L);
        const float silu = __fdiv_rn(gc, __fadd_rn(1.0f, expf(-gc)));
        const float h = __bfloat162float(__float2bfloat16_rn(__fmul_rn(silu, uc)));
        float amax = fabsf(h);
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 8));
        const uint32_t sb = nv_scale_byte(amax);
        const float d = e4m3_to_f32(sb);
        // Pair with the neighbour lane: one byte (two nibbles) per even lane.
        const float hn = __shfl_xor_sync(0xFFFFFFFFu, h, 1);
        const size_t hrow = static_cast<size_t>(T >> 2) * a.Rp + r0 + i;
        if ((q & 1) == 0) a.himg[hrow * 128 + (T & 3) * 32 + (q >> 1)] = static_cast<uint8_t>(nv_quant2(h, hn, d));
        if ((q & 15) == 0) a.hsc[hrow * 16 + (T & 3) * 4 + (q >> 4)] = static_cast<uint8_t>(sb);
      }
    }
    nv_epi_bar();
  }
  // The barrier orders every thread's image writes before this release.
  if (etid == 0) red_release_gpu_add(a.done + le, 1u);
}

// GEMM2 tile T2 of unit u: o[slot, 128*T2 + row] = bf16(y[i]) for slot i.
template <int TOK>
__device__ void nv_finish2(const NvArgs& a, NvSmem<TOK>& S, int u, int T2, const float (&y)[TOK], int row,
                           int etid) {
  const int r0 = S.uoff[u], r = S.uoff[u + 1] - r0;
  const int m = 128 * T2 + row;
  if (S.direct) {
    // The slot is its token's only local one: y = bf16(w * bf16(o)), exactly
    // the scatter's sum of one term.
#pragma unroll
    for (int i = 0; i < TOK; ++i)
      if (i < r) {
        const int route = S.sroute[r0 + i];
        const float wt = a.route ? __ldcg(a.tw_out + route) : __ldg(a.tw + route);
        const float o = __bfloat162float(__float2bfloat16_rn(y[i]));
        a.y[static_cast<size_t>(S.stok[r0 + i]) * a.H + m] = __float2bfloat16_rn(__fadd_rn(0.0f, __fmul_rn(wt, o)));
      }
    return;
  }
#pragma unroll
  for (int i = 0; i < TOK; ++i)
    if (i < r) a.obuf[static_cast<size_t>(S.sroute[r0 + i]) * a.H + m] = __float2bfloat16_rn(y[i]);
  nv_epi_bar();
  if (etid == 0) red_release_gpu_add(a.sync + 2, 1u);
}

// End of a segment (see the routed FP8 kernel): a split tile is finished by
// its first contributor, which adds the others' partials in CTA order.
template <int TOK>
__device__ void nv_end_segment(const NvArgs& a, NvSmem<TOK>& S, const NvPhase (&P)[2], const NvStep& st,
                               float (&y)[TOK], int row, int etid) {
  const NvPhase& pp = P[st.phase - 1];
  const int cf = pp.cta_of(st.t0), cl = pp.cta_of(st.t0 + pp.nb - 1);
  const int c = blockIdx.x;
  const int ncols = st.phase == 1 ? a.M : S.uoff[st.u + 1] - S.uoff[st.u];
  if (cf != cl) {
    const int le = S.ulist[st.u];
    uint32_t* cnt = st.phase == 1 ? a.cnt1 + static_cast<size_t>(le) * pp.tiles + st.T
                                  : a.cnt2 + static_cast<size_t>(le) * pp.tiles + st.T;
    if (c != cf) {
      float* mine = nv_part(a, st.phase, c, pp.lo >= st.t0 ? 0 : 1, TOK);
#pragma unroll
      for (int t = 0; t < TOK; ++t)
        if (t < ncols) __stcg(mine + t * 128 + row, y[t]);
      nv_epi_bar();
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
      if (ok)
        atomicExch(cnt, 0u);
      else if (!S.abort)
        nv_error(a, S.abort, kErrCrossWait);
    }
    nv_epi_bar();
    if (S.abort) return;
    for (int c0 = cf + 1; c0 <= cl; c0 += 4) {
      const float* src[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int cc = min(c0 + qq, cl);
        src[qq] = nv_part(a, st.phase, cc, pp.lo_of(cc) >= st.t0 ? 0 : 1, TOK) + row;
      }
      const int nq = min(4, cl - c0 + 1);
#pragma unroll
      for (int t = 0; t < TOK; ++t) {
        if (t < ncols) {
          float v[4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) v[qq] = __ldcg(src[qq] + t * 128);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            if (qq < nq) y[t] += v[qq];
        }
      }
    }
  }
  if (st.phase == 1)
    nv_finish1<TOK>(a, S, st.u, st.T, y, row, etid);
  else
    nv_finish2<TOK>(a, S, st.u, st.T, y, row, etid);
}

// Bounded wait of one thread until *ctr >= target.
__device__ bool nv_wait_ge(const NvArgs& a, volatile int& abort, const uint32_t* ctr, uint32_t target) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(ctr) < target) {
    if (abort || globaltimer_ns() - t0 > a.timeout_ns) {
      if (!abort) nv_error(a, abort, kErrCrossWait);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// ---------------------------------------------------------------- kernel
template <int TOK>
__global__ void __launch_bounds__(kNvThreads, 1) nvfp4_tc_kernel(const __grid_constant__ NvArgs a) {
  using C = NvCfg<TOK>;
  constexpr int kS = C::kStages, kSB = C::kBStages;
  extern __shared__ uint8_t smem_raw[];
  NvSmem<TOK>& S = *reinterpret_cast<NvSmem<TOK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(&S.fullA[s], 1);
      mbar_init(&S.emptyA[s], 1);
    }
    for (int s = 0; s < kSB; ++s) {
      mbar_init(&S.fullB[s], 1);
      mbar_init(&S.emptyB[s], 1);
    }
    for (int b = 0; b < C::kSfBuf; ++b) {
      mbar_init(&S.sffull[b], 4);
      mbar_init(&S.sffree[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.accfull[b], 1);
      mbar_init(&S.tmemfree[b], 4);
    }
    mbar_init(&S.final_bar, 1);
    fence_mbar_init();
    S.abort = 0;
    prefetch_tmap(&a.map13);
    prefetch_tmap(&a.map2);
    prefetch_tmap(&a.mapx);
    prefetch_tmap(&a.mapxs);
    prefetch_tmap(&a.maph);
    prefetch_tmap(&a.maphs);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kNvTmemCols);
    tmem_relinquish();
  }
  for (int e = tid; e < a.L; e += kNvThreads) S.tokmask[e] = 0ull;
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- fused routing: token t is routed by warp 0 of CTA t % G (keys in
  // the epilogue's staging buffer, unused until then) into the ids / weights
  // outputs; every CTA reads all of them back after a grid-wide count
  // (below), so the routing overlaps the x image.
  if (a.route) {
    for (int t = c; warp == 0 && t < a.M; t += G) {
      int e;
      float w;
      route_topk_smem(a.logits, a.logits_f32 != 0, a.bias, a.E, a.top_k, a.scale, t, lane,
                      reinterpret_cast<uint32_t*>(&S.ysm[0][0]), e, w);
      if (lane < a.top_k) {
        a.ids_out[t * a.top_k + lane] = e;
        a.tw_out[t * a.top_k + lane] = w;
      }
    }
    __syncthreads();
    if (tid == 0) red_release_gpu_add(a.sync + 4, 1u);  // this CTA's tokens are routed
  }
  // ---- x image: token t, group g of 16 -> 8 packed bytes and a scale byte,
  // all CTAs share the work. Groups past H (an odd number of 128-value
  // halves) get zero data and zero scales, and so do the h image's scales of
  // that kind: the MMA multiplies every group by its scales.
  {
    const int nb1 = (a.H + kNvKB - 1) / kNvKB, nb2 = (a.N + kNvKB - 1) / kNvKB;
    const int gpt = nb1 * (kNvKB / 16);
    for (int i = c * kNvThreads + tid; i < a.M * gpt; i += G * kNvThreads) {
      const int t = i / gpt, g = i % gpt;
      const size_t xrow = static_cast<size_t>(g >> 4) * TOK + t;
      uint32_t lo = 0u, hi = 0u, sb = 0u;
      if (16 * g < a.H) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H + 16 * g);
        const uint4 w0 = __ldg(src), w1 = __ldg(src + 1);
        const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float v[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[2 * k] = __uint_as_float(wd[k] << 16);
          v[2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
        sb = nv_scale_byte(amax);
        const float d = e4m3_to_f32(sb);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo |= nv_quant2(v[2 * k], v[2 * k + 1], d) << (8 * k);
          hi |= nv_quant2(v[8 + 2 * k], v[8 + 2 * k + 1], d) << (8 * k);
        }
      }
      *reinterpret_cast<uint2*>(a.ximg + xrow * 128 + (g & 15) * 8) = make_uint2(lo, hi);
      a.xsc[xrow * 16 + (g & 15)] = static_cast<uint8_t>(sb);
    }
    if (a.N % kNvKB != 0) {
      for (int r = c * kNvThreads + tid; r < a.Rp; r += G * kNvThreads)
        *reinterpret_cast<uint2*>(a.hsc + (static_cast<size_t>(nb2 - 1) * a.Rp + r) * 16 + 8) = make_uint2(0u, 0u);
    }
  }
  // ---- every route's expert and weight into shared memory
  if (a.route) {
    if (tid == 0) {
      nv_wait_ge(a, S.abort, a.sync + 4, static_cast<uint32_t>(G));
      // The last CTA past the routing wait re-arms both counters.
      if (atomicAdd(a.sync + 5, 1u) + 1u == static_cast<uint32_t>(G)) {
        atomicExch(a.sync + 4, 0u);
        atomicExch(a.sync + 5, 0u);
      }
    }
    __syncthreads();
    for (int i = tid; i < a.M * a.top_k; i += kNvThreads) {
      const long long le = static_cast<long long>(__ldcg(a.ids_out + i)) - a.e0;
      S.sid[i] = static_cast<int16_t>(le >= 0 && le < a.L ? le : -1);
    }
  } else {
    for (int i = tid; i < a.M * a.top_k; i += kNvThreads) {
      const long long le = static_cast<long long>(__ldg(a.ids + i)) - a.e0;
      S.sid[i] = static_cast<int16_t>(le >= 0 && le < a.L ? le : -1);
    }
  }
  if (tid == 0) S.direct = 1;
  __syncthreads();
  // ---- local slots and the unit list
  for (int i = tid; i < a.M * a.top_k; i += kNvThreads) {
    const int le = S.sid[i];
    if (le >= 0) atomicOr(&S.tokmask[le], 1ull << (i / a.top_k));
  }
  // Direct mode when no token has two local slots (then y[t] = bf16(w * o) of
  // its one slot, or zero): the GEMM2 epilogue writes y, no scatter pass.
  for (int t = tid; t < a.M; t += kNvThreads) {
    int n = 0;
    for (int r = 0; r < a.top_k; ++r) n += S.sid[t * a.top_k + r] >= 0;
    if (n > 1) S.direct = 0;
  }
  __syncthreads();
  if (tid == 0) red_release_gpu_add(a.sync, 1u);  // this CTA's share of the x image is written
  if (warp == 0) {
    int U = 0, off = 0;
    for (int b0 = 0; b0 < a.L; b0 += 32) {
      const int e = b0 + lane;
      const unsigned long long m = e < a.L ? S.tokmask[e] : 0ull;
      const bool has = m != 0ull;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
      const int cnt = __popcll(m);
      // inclusive prefix of the slot counts over the lanes
      int pre = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, pre, d);
        if (lane >= d) pre += v;
      }
      const int total = __shfl_sync(0xFFFFFFFFu, pre, 31);
      if (has) {
        const int u = U + __popc(bal & ((1u << lane) - 1u));
        S.ulist[u] = static_cast<int16_t>(e);
        S.uidx[e] = static_cast<int16_t>(u);
        S.uoff[u] = static_cast<int16_t>(off + pre - cnt);
      }
      U += __popc(bal);
      off += total;
    }
    if (lane == 0) {
      S.U = U;
      S.uoff[U] = static_cast<int16_t>(off);
    }
  }
  __syncthreads();
  for (int i = tid; i < a.M * a.top_k; i += kNvThreads) {
    const int le = S.sid[i];
    if (le >= 0 && le < a.L) {
      const int t = i / a.top_k;
      const int u = S.uidx[le];
      const int row = S.uoff[u] + __popcll(S.tokmask[le] & ((1ull << t) - 1ull));
      S.stok[row] = static_cast<int16_t>(t);
      S.sroute[row] = static_cast<int16_t>(i);
    }
  }
  __syncthreads();

  const int U = S.U;
  NvPhase P[2];
  // K blocks of 256 values; an odd number of 128-value halves leaves a last
  // block whose second half lies past the row: the weight and activation
  // loads fill it with zeros and its scales are zero.
  const int nb1 = (a.H + kNvKB - 1) / kNvKB, nb2 = (a.N + kNvKB - 1) / kNvKB;
  P[0] = nv_phase(U * (a.N / 64) * nb1, a.N / 64, nb1, G, c);
  P[1] = nv_phase(U * (a.H / 128) * nb2, a.H / 128, nb2, G, c);
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ A producer (packed weights)
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      NvCursor cur{P[0].lo, 1};
      NvStep st;
      int k = 0;
      while (cur.next(P, st)) {
        const int s = k % kS;
        if (k >= kS && !mbar_wait(&S.emptyA[s], ((k / kS) - 1) & 1, a.timeout_ns, &S.abort)) {
          if (!S.abort) nv_error(a, S.abort, kErrRingWait);
          break;
        }
        const int le = S.ulist[st.u];
        int r0, r1;
        const void* map;
        if (st.phase == 1) {
          r0 = le * 2 * a.N + 64 * st.T;  // gate rows
          r1 = r0 + a.N;                  // up rows
          map = &a.map13;
        } else {
          r0 = le * a.H + 128 * st.T;
          r1 = r0 + 64;
          map = &a.map2;
        }
        mbar_arrive_expect_tx(&S.fullA[s], kNvRawBytes);
        tma_load_2d(S.R[s], map, st.kb * (kNvKB / 2), r0, &S.fullA[s], pol);
        tma_load_2d(S.R[s] + kNvRawBytes / 2, map, st.kb * (kNvKB / 2), r1, &S.fullA[s], pol);
        ++k;
      }
      // Let every issued copy land before the CTA can exit.
      for (int kk = max(0, k - kS); kk < k; ++kk)
        if (!mbar_wait(&S.fullA[kk % kS], (kk / kS) & 1, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ B producer (activation images and their scales)
    if (lane == 0) {
      bool ok = nv_wait_ge(a, S.abort, a.sync, static_cast<uint32_t>(G));
      // The last CTA past the x-image wait re-arms both counters.
      if (atomicAdd(a.sync + 1, 1u) + 1u == static_cast<uint32_t>(G)) {
        atomicExch(a.sync, 0u);
        atomicExch(a.sync + 1, 0u);
      }
      NvCursor cur{P[0].lo, 1};
      NvStep st;
      int k = 0, cur_u = -1;
      while (ok && cur.next(P, st)) {
        const int s = k % kSB;
        if (k >= kSB && !mbar_wait(&S.emptyB[s], ((k / kSB) - 1) & 1, a.timeout_ns, &S.abort)) {
          if (!S.abort) nv_error(a, S.abort, kErrRingWait);
          break;
        }
        if (st.phase == 1) {
          mbar_arrive_expect_tx(&S.fullB[s], C::kBBytes + C::kBsBytes);
          tma_load_2d_plain(S.B[s], &a.mapx, 0, st.kb * TOK, &S.fullB[s]);
          tma_load_2d_plain(S.Bs[s], &a.mapxs, 0, st.kb * TOK, &S.fullB[s]);
        } else {
          const int le = S.ulist[st.u];
          if (st.u != cur_u) {
            // Every GEMM1 tile of this expert must be in the h image.
            if (!nv_wait_ge(a, S.abort, a.done + le, static_cast<uint32_t>(a.N / 64))) break;
            cur_u = st.u;
            const int s0 = st.u * P[1].tiles * P[1].nb, s1 = s0 + P[1].tiles * P[1].nb - 1;
            const uint32_t ctas = static_cast<uint32_t>(P[1].cta_of(s1) - P[1].cta_of(s0) + 1);
            if (atomicAdd(a.hpassed + le, 1u) + 1u == ctas) {
              atomicExch(a.done + le, 0u);
              atomicExch(a.hpassed + le, 0u);
            }
          }
          const int y0 = st.kb * a.Rp + S.uoff[st.u];
          mbar_arrive_expect_tx(&S.fullB[s], C::kBBytes + C::kBsBytes);
          tma_load_2d_plain(S.B[s], &a.maph, 0, y0, &S.fullB[s]);
          tma_load_2d_plain(S.Bs[s], &a.maphs, 0, y0, &S.fullB[s]);
        }
        ++k;
      }
      for (int kk = max(0, k - kSB); kk < k; ++kk)
        if (!mbar_wait(&S.fullB[kk % kSB], (kk / kSB) & 1, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = nv_idesc(128, TOK);
      NvCursor cur{P[0].lo, 1};
      NvStep st;
      int k = 0, seg = 0;
      while (cur.next(P, st)) {
        const int s = k % kS, sb = k % kSB, sf = k % C::kSfBuf, tb = seg & 1;
        if (!mbar_wait(&S.fullA[s], (k / kS) & 1, a.timeout_ns, &S.abort) ||
            !mbar_wait(&S.fullB[sb], (k / kSB) & 1, a.timeout_ns, &S.abort) ||
            !mbar_wait(&S.sffull[sf], (k / C::kSfBuf) & 1, a.timeout_ns, &S.abort) ||
            (st.first && seg >= 2 && !mbar_wait(&S.tmemfree[tb], ((seg >> 1) - 1) & 1, a.timeout_ns, &S.abort))) {
          if (!S.abort) nv_error(a, S.abort, kErrRingWait);
          break;
        }
        tc_fence_after();
        // Both operands are 128-byte-swizzled K-major tiles of 128-byte rows
        // (256 values); MMA j takes values 64j .. 64j + 63, 32 bytes further
        // in each row (start address in 16-byte units; shared addresses stay
        // far below 256 KB, so the 14-bit field never carries).
        const uint64_t adesc = sw128_desc(smem_u32(S.R[s]));
        const uint64_t bdesc = sw128_desc(smem_u32(S.B[sb]));
        const uint32_t dtm = tmem + tb * TOK;
        const uint32_t sfa = tmem + nv_sfcol(sf), sfb = sfa + 16;
#pragma unroll
        for (int j = 0; j < kNvKB / 64; ++j)
          tc_mma_nvf4(dtm, adesc + 2 * j, bdesc + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j,
                      (st.first && j == 0) ? 0u : 1u);
        tc_commit(&S.emptyA[s]);
        tc_commit(&S.emptyB[sb]);
        tc_commit(&S.sffree[sf]);
        if (st.last) {
          tc_commit(&S.accfull[tb]);
          ++seg;
        }
        ++k;
      }
      tc_commit(&S.final_bar);
      if (!mbar_wait(&S.final_bar, 0, a.timeout_ns, nullptr)) atomicOr(a.err, kErrDrain);
    }
  } else if (warp < 7) {
    // ------------------------------------------------------------ scale vectors -> TMEM
    // Per K block, MMA j reads four TMEM columns of scale vectors (four
    // UE4M3 bytes per 32-bit cell, groups 4j .. 4j + 3): for A, weight row m
    // from lane m, column m / 32; for B, token column n from lane n % 32,
    // column n / 32, in each lane quadrant. So each warp writes its own
    // quadrant: its 32 weight rows (in every column) and all token columns.
    const int quad = warp & 3;
    const int srow = quad * 32 + lane;  // weight row = TMEM lane
    const uint32_t tq = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    // The 16 scale bytes of weight row `row` of K block q: two 8-byte copies
    // (rows are 8-byte aligned); the second is zeros when the block's second
    // half lies past the row.
    auto fetch_row = [&](uint4* dst, const NvStep& q, int row) {
      const int le = S.ulist[q.u];
      const uint8_t* src;
      int K;
      if (q.phase == 1) {
        const int grow = le * 2 * a.N + (row < 64 ? 64 * q.T + row : a.N + 64 * q.T + row - 64);
        src = a.s13 + static_cast<size_t>(grow) * (a.H / 16) + 16 * q.kb;
        K = a.H;
      } else {
        src = a.s2 + (static_cast<size_t>(le) * a.H + 128 * q.T + row) * (a.N / 16) + 16 * q.kb;
        K = a.N;
      }
      const bool full = (q.kb + 1) * kNvKB <= K;
      cp_async8(dst, src);
      cp_async8(reinterpret_cast<uint8_t*>(dst) + 8, full ? src + 8 : src, full ? 8u : 0u);
    };
    auto fetch = [&](int slot, const NvStep& q) { fetch_row(&S.sc[slot][srow], q, srow); };
    // Slot n % kNvScaleAhead holds K block n; a refill goes to the slot read
    // one iteration earlier (each thread reads only its own copies).
    NvCursor ahead{P[0].lo, 1};
    NvStep qa;
    for (int j = 0; j < kNvScaleAhead - 1; ++j) {
      if (ahead.next(P, qa)) fetch(j, qa);
      cp_async_commit();
    }
    NvCursor cur{P[0].lo, 1};
    NvStep st;
    int k = 0;
    while (cur.next(P, st)) {
      const int sb = k % kSB, sf = k % C::kSfBuf;
      cp_async_wait<kNvScaleAhead - 2>();  // this thread's scales of K block k have landed
      uint32_t ra[16], rb[16];
      {
        const uint4 w = S.sc[k % kNvScaleAhead][srow];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ra[c] = w.x;
          ra[4 + c] = w.y;
          ra[8 + c] = w.z;
          ra[12 + c] = w.w;
        }
      }
      if (ahead.next(P, qa)) fetch((k + kNvScaleAhead - 1) % kNvScaleAhead, qa);
      cp_async_commit();
      if (!mbar_wait(&S.fullB[sb], (k / kSB) & 1, a.timeout_ns, &S.abort) ||
          (k >= C::kSfBuf && !mbar_wait(&S.sffree[sf], ((k / C::kSfBuf) - 1) & 1, a.timeout_ns, &S.abort))) {
        if (!S.abort) nv_error(a, S.abort, kErrRingWait);
        break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = lane + 32 * c;  // token column
        const uint4 w = t < TOK ? *reinterpret_cast<const uint4*>(S.Bs[sb] + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
        rb[c] = w.x;
        rb[4 + c] = w.y;
        rb[8 + c] = w.z;
        rb[12 + c] = w.w;
      }
      tc_fence_after();
      tmem_st16(tq + nv_sfcol(sf), ra);
      tmem_st16(tq + nv_sfcol(sf) + 16, rb);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sffull[sf]);
      ++k;
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------ epilogue (TMEM lane quadrant = warp % 4)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int etid = tid - 224;
    NvCursor cur{P[0].lo, 1};
    NvStep st;
    int seg = 0;
    float y[TOK];
    while (cur.next(P, st)) {
      if (!st.last) continue;
      const int tb = seg & 1;
      if (!mbar_wait(&S.accfull[tb], (seg >> 1) & 1, a.timeout_ns, &S.abort)) {
        if (!S.abort) nv_error(a, S.abort, kErrRingWait);
      }
      nv_epi_bar();
      if (S.abort) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + tb * TOK;
#pragma unroll
      for (int g = 0; g < TOK / 16; ++g) {
        uint32_t v[16];
        tmem_ld<16>(taddr + 16 * g, v);
        tc_wait_ld();
#pragma unroll
        for (int t = 0; t < 16; ++t) y[16 * g + t] = __uint_as_float(v[t]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tmemfree[tb]);
      nv_end_segment<TOK>(a, S, P, st, y, row, etid);
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kNvTmemCols);

  if (S.direct) {
    // Tokens without a local slot get zero rows (a share of the rows per CTA).
    const int chunks = a.H / 8;
    for (int w = c * kNvThreads + tid; w < a.M * chunks; w += G * kNvThreads) {
      const int tt = w / chunks;
      bool any = false;
      for (int r = 0; r < a.top_k; ++r) any |= S.sid[tt * a.top_k + r] >= 0;
      if (!any) *reinterpret_cast<uint4*>(a.y + static_cast<size_t>(tt) * a.H + 8 * (w % chunks)) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  // ---- scatter: y[t, m] = bf16(sum over t's local picks, ascending, of w * o)
  const uint32_t tiles2 = static_cast<uint32_t>(U) * static_cast<uint32_t>(a.H / 128);
  if (tid == 0 && !S.abort) nv_wait_ge(a, S.abort, a.sync + 2, tiles2);
  __syncthreads();
  if (!S.abort) {
    const int chunks = a.H / 8;  // 8 columns (16 bytes of BF16) per thread item
    const int per_cta = (chunks + G - 1) / G;
    const int ch0 = c * per_cta, nch = max(0, min(chunks, ch0 + per_cta) - ch0);
    for (int w = tid; w < a.M * nch; w += kNvThreads) {
      const int tt = w / nch;
      const int chn = ch0 + w % nch;
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
      for (int r = 0; r < a.top_k; ++r) {
        const int le = S.sid[tt * a.top_k + r];
        if (le < 0 || le >= a.L) continue;
        const float wt = a.route ? __ldcg(a.tw_out + tt * a.top_k + r) : __ldg(a.tw + tt * a.top_k + r);
        const uint4 o =
            __ldcg(reinterpret_cast<const uint4*>(a.obuf + static_cast<size_t>(tt * a.top_k + r) * a.H + 8 * chn));
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
      *reinterpret_cast<uint4*>(a.y + static_cast<size_t>(tt) * a.H + 8 * chn) = out;
    }
  }
  __syncthreads();
  if (tid == 0) {
    // The last CTA past the scatter wait re-arms its counters.
    if (atomicAdd(a.sync + 3, 1u) + 1u == static_cast<uint32_t>(G)) {
      atomicExch(a.sync + 2, 0u);
      atomicExch(a.sync + 3, 0u);
    }
  }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 nv_encode_fn() {
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

// 2-D byte tensor [rows, cols] (row-major) with a box of box_rows x box_cols bytes.
static bool nv_map(CUtensorMap* map, const void* base, unsigned long long rows, unsigned long long cols,
                   unsigned box_cols, unsigned box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = nv_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct NvWorkspace {
  uint32_t *err, *sync, *done, *hpassed, *cnt1, *cnt2;
  uint8_t *ximg, *xsc, *himg, *hsc;
  __nv_bfloat16* obuf;
  float* part;
  int tok, Rp;
  size_t bytes;
};

static size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

static NvWorkspace nv_layout(void* base, int M, int H, int N, int L, int top_k) {
  NvWorkspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.tok = M <= 16 ? 16 : (M <= 32 ? 32 : kMaxTokens);  // token capacity of the kernel
  w.Rp = M * top_k > w.tok ? M * top_k : w.tok;  // at least one box of rows
  w.err = reinterpret_cast<uint32_t*>(p + off);
  w.sync = w.err + 1;  // words 1..6 of the first 256 bytes
  off += 256;
  w.done = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L));
  w.hpassed = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L));
  w.cnt1 = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L) * (N / 64));
  w.cnt2 = reinterpret_cast<uint32_t*>(p + off);
  off += a256(4 * static_cast<size_t>(L) * (H / 128));
  const size_t nb1 = static_cast<size_t>((H + kNvKB - 1) / kNvKB), nb2 = static_cast<size_t>((N + kNvKB - 1) / kNvKB);
  w.ximg = p + off;
  off += a256(nb1 * w.tok * 128);
  w.xsc = p + off;
  off += a256(nb1 * w.tok * 16);
  w.himg = p + off;
  off += a256(nb2 * w.Rp * 128);
  w.hsc = p + off;
  off += a256(nb2 * w.Rp * 16);
  w.obuf = reinterpret_cast<__nv_bfloat16*>(p + off);
  off += a256(2 * static_cast<size_t>(M) * top_k * H);
  w.part = reinterpret_cast<float*>(p + off);
  off += a256(4 * static_cast<size_t>(2) * kFp8MaxCtas * 2 * w.tok * 128);
  w.bytes = off;
  return w;
}

size_t nvfp4_workspace_bytes(int M, int H, int N, int L, int top_k) {
  return nv_layout(nullptr, M, H, N, L, top_k).bytes;
}

template <int TOK>
static int nv_launch(NvArgs& a, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_last_error(FME_ECUDA, "cudaGetDevice failed");
  const int sms = device_sm_count(dev);
  if (sms <= 0) return set_last_error(FME_ECUDA, "cannot query the SM count");
  const void* kern = reinterpret_cast<const void*>(nvfp4_tc_kernel<TOK>);
  if (!ensure_smem_attr(dev, kern, nv_smem_bytes<TOK>())) return FME_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms < kFp8MaxCtas ? sms : kFp8MaxCtas);
  cfg.blockDim = dim3(kNvThreads);
  cfg.dynamicSmemBytes = nv_smem_bytes<TOK>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, nvfp4_tc_kernel<TOK>, a);
  if (err != cudaSuccess) return set_last_error(FME_ECUDA, "nvfp4 kernel launch: %s", cudaGetErrorString(err));
  return FME_OK;
}

int routed_nvfp4(const void* x, const int32_t* ids, const float* weights, const uint8_t* w13, const uint8_t* s13,
                 const uint8_t* w2, const uint8_t* s2, int M, int H, int N, int L, int e0, int top_k, float limit,
                 void* y, void* workspace, size_t workspace_bytes, cudaStream_t st, const Nvfp4Routing* route) {
  const NvWorkspace w = nv_layout(workspace, M, H, N, L, top_k);
  if (workspace == nullptr || workspace_bytes < w.bytes)
    return set_last_error(FME_EWORKSPACE, "workspace of %zu bytes needed, %zu given", w.bytes, workspace_bytes);
  NvArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ids = ids;
  a.tw = weights;
  if (route != nullptr) {
    a.route = 1;
    a.logits = route->logits;
    a.logits_f32 = route->logits_dtype == FME_F32 ? 1 : 0;
    a.bias = route->bias;
    a.E = route->E;
    a.scale = route->scale;
    a.ids_out = route->ids;
    a.tw_out = route->weights;
  }
  a.s13 = s13;
  a.s2 = s2;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.err = w.err;
  a.sync = w.sync;
  a.done = w.done;
  a.hpassed = w.hpassed;
  a.cnt1 = w.cnt1;
  a.cnt2 = w.cnt2;
  a.ximg = w.ximg;
  a.xsc = w.xsc;
  a.himg = w.himg;
  a.hsc = w.hsc;
  a.obuf = w.obuf;
  a.part = w.part;
  a.M = M;
  a.H = H;
  a.N = N;
  a.L = L;
  a.e0 = e0;
  a.top_k = top_k;
  a.Rp = w.Rp;
  a.limit = limit;
  a.timeout_ns = wait_timeout_ns();
  const unsigned long long nb1 = static_cast<unsigned long long>((H + kNvKB - 1) / kNvKB);
  const unsigned long long nb2 = static_cast<unsigned long long>((N + kNvKB - 1) / kNvKB);
  if (!nv_map(&a.map13, w13, static_cast<unsigned long long>(L) * 2 * N, H / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !nv_map(&a.map2, w2, static_cast<unsigned long long>(L) * H, N / 2, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !nv_map(&a.mapx, w.ximg, nb1 * w.tok, 128, 128, w.tok, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !nv_map(&a.mapxs, w.xsc, nb1 * w.tok, 16, 16, w.tok, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !nv_map(&a.maph, w.himg, nb2 * w.Rp, 128, 128, w.tok, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !nv_map(&a.maphs, w.hsc, nb2 * w.Rp, 16, 16, w.tok, CU_TENSOR_MAP_SWIZZLE_NONE))
    return set_last_error(FME_ECUDA, "cuTensorMapEncodeTiled failed or unavailable");
  return w.tok == 16 ? nv_launch<16>(a, st) : (w.tok == 32 ? nv_launch<32>(a, st) : nv_launch<kMaxTokens>(a, st));
}

}  // namespace fme
