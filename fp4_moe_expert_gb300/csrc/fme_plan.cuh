// Work decomposition of the routed FP8 kernel (fme_routed_fp8.cu): waves,
// the per-phase stream-K slices and the per-CTA chunk walk. Host and device
// code (the CPU tests walk every CTA's chunks with it).
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define FME_HD __host__ __device__
#else
#define FME_HD
#endif

namespace fme {

FME_HD constexpr int plan_min(int a, int b) { return a < b ? a : b; }

// Waves: the unit list is cut into W consecutive groups; every CTA takes a
// share of every wave and runs GEMM1 of wave w + 1 before GEMM2 of wave w, so
// one wave's GEMM1 -> GEMM2 hand-over (last tiles finishing, hidden rows
// re-quantised) overlaps the next wave's weight stream, and each CTA's work
// mixes experts hit by different token counts. Every wave adds split tiles,
// each with a partial round trip. Measured on the DeepSeek-V3 shape (256
// experts, top 8; L2 flushed, W = 1 / 2 / 3 in microseconds):
//   routed  M = 4: 222 / 224 / 228   M = 6: 293 / 294 / 300   M = 7: 356 / 343 / 332
//           M = 8: 396 / 384 / 367   M = 12: 558 / 532 / 525   M = 24: 918 / 910 / 866
//   + shared M = 3: 205 / 193 / 194  M = 4: 267 / 236 / 232   M = 5: 281 / 267 / 275
//           M = 6: 324 / 304 / 304   M = 8: 406 / 382 / 373   M = 16: 783 / 711 / 683
// (one wave at 1-2 tokens either way). The shared expert is unit 0 of the
// one-launch layer, so it streams in the first wave.
FME_HD constexpr int max_waves(int ptok) { return ptok >= 7 ? 3 : 1; }
FME_HD constexpr int layer_waves(int ptok) {
  return ptok <= 2 ? 1 : (ptok == 3 || ptok == 5 ? 2 : 3);
}
// Waves the partial-sum region is sized for, any call.
FME_HD constexpr int waves_cap(int ptok) {
  return max_waves(ptok) > layer_waves(ptok) ? max_waves(ptok) : layer_waves(ptok);
}

// ---------------------------------------------------------------- work plan
// The units are cut into W waves of consecutive units. The slots of one
// (wave, phase) -- units x tiles x K blocks, at most 1025 x 128 x 64 = 8.4M --
// are split over Ge = min(G, n) CTAs: CTA c < Ge owns [n*c/Ge, n*(c+1)/Ge),
// never empty; CTAs c >= Ge own nothing. The products stay below 8.4M x 161
// < 2^32, so unsigned 32-bit arithmetic is exact.
struct PhasePlan {
  int n, lo, hi;
  int Ge, tiles, nb;
  int w, u0;  // wave and its first unit
  FME_HD int lo_of(int c) const {
    return c >= Ge ? n : static_cast<int>(static_cast<uint32_t>(n) * static_cast<uint32_t>(c) /
                                          static_cast<uint32_t>(Ge));
  }
  // The CTA whose slice holds slot x.
  FME_HD int cta_of(int x) const {
    return static_cast<int>((static_cast<uint32_t>(x + 1) * static_cast<uint32_t>(Ge) + static_cast<uint32_t>(n) - 1u) /
                            static_cast<uint32_t>(n)) - 1;
  }
};

struct Plan {
  int U, N, kcmax, c, G, W;
  bool ximage;  // GEMM1 B rows copied from a per-call quantised image of x
  int kcmax2;  // K blocks per GEMM2 chunk, at most
  int phase_lo, phase_hi;  // phases this launch runs
  int N1, kcmax1;  // the MX kernel's GEMM1 B rows (four per token) and K blocks per chunk
  int tiles[2], nb[2];  // per unit: GEMM1 64-row tiles x H/128 K blocks; GEMM2 128-row tiles x I/128
  FME_HD int wave_lo(int w) const { return U * w / W; }
  // Stage q of 2W: GEMM1 of wave 0, then GEMM1(w + 1) / GEMM2(w) pairs, then
  // the last GEMM2.
  FME_HD void stage(int q, int& w, int& phase) const {
    if (q == 0) {
      w = 0;
      phase = 1;
    } else if (q < 2 * W - 1) {
      w = (q & 1) ? (q + 1) / 2 : q / 2 - 1;
      phase = (q & 1) ? 1 : 2;
    } else {
      w = W - 1;
      phase = 2;
    }
  }
  FME_HD PhasePlan plan(int w, int phase) const {
    PhasePlan pp;
    const int u0 = wave_lo(w), u1 = wave_lo(w + 1);
    const int t = tiles[phase - 1], nbp = nb[phase - 1];
    pp.n = (u1 - u0) * t * nbp;
    pp.tiles = t;
    pp.nb = nbp;
    pp.w = w;
    pp.u0 = u0;
    pp.Ge = plan_min(G, pp.n);
    if (c >= pp.Ge) {
      pp.lo = pp.hi = pp.n;
    } else {
      pp.lo = pp.lo_of(c);
      pp.hi = pp.lo_of(c + 1);
    }
    return pp;
  }
};

struct Chunk {
  int phase, u, T, kb0, kc;
  int t0;  // first slot of the tile within its (wave, phase)
  bool last_of_seg;
  PhasePlan pp;
};

// Walks this CTA's slots stage by stage in chunks of at most kcmax K blocks
// that never cross a tile.
struct Cursor {
  int q = -1, pos = 0, phase = 1;
  PhasePlan pp{};
  template <bool MX>
  FME_HD bool next(const Plan& P, Chunk& ch) {
    while (true) {
      if (q >= 0 && pos < pp.hi) {
        const int tile = pos / pp.nb;
        const int t0 = tile * pp.nb;
        const int seg1 = plan_min(pp.hi, t0 + pp.nb);
        const int uw = tile / pp.tiles;
        ch.phase = phase;
        ch.u = pp.u0 + uw;
        ch.T = tile - uw * pp.tiles;
        ch.t0 = t0;
        ch.kb0 = pos - t0;
        ch.kc = plan_min(phase == 2 ? P.kcmax2 : (MX ? P.kcmax1 : P.kcmax), seg1 - pos);
        ch.last_of_seg = pos + ch.kc == seg1;
        ch.pp = pp;
        pos += ch.kc;
        return true;
      }
      if (++q >= 2 * P.W) return false;
      int w;
      P.stage(q, w, phase);
      if (phase < P.phase_lo || phase > P.phase_hi) {
        pos = pp.hi = 0;  // a stage this launch does not run: nothing to walk
        continue;
      }
      pp = P.plan(w, phase);
      pos = pp.lo;
    }
  }
};

}  // namespace fme
