// Work decomposition of the routed FP8 kernel (fme_routed_fp8.cu): waves,
// the per-phase stream-K slices and the per-CTA chunk walk. Host and device
// code (the CPU tests walk every CTA's chunks with it).
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define FME_HD __host__ __device__
#define FME_HD_COLD __host__ __device__ __noinline__
#else
#define FME_HD
#define FME_HD_COLD
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
// Waves the partial-sum region is sized for: the most any call with up to
// ptok token rows may take, so the workspace never shrinks as M grows and one
// sized for M serves every smaller token count.
FME_HD constexpr int waves_cap(int ptok) {
  int cap = 1;
  for (int p = 1; p <= ptok; ++p) {
    cap = max_waves(p) > cap ? max_waves(p) : cap;
    cap = layer_waves(p) > cap ? layer_waves(p) : cap;
  }
  return cap;
}
constexpr bool waves_cap_holds() {
  for (int p = 1; p <= 64; ++p)
    if (waves_cap(p) < max_waves(p) || waves_cap(p) < layer_waves(p) || (p > 1 && waves_cap(p) < waves_cap(p - 1)))
      return false;
  return true;
}
static_assert(waves_cap_holds(), "the partial-sum region holds every call's waves and grows with M");

// ---------------------------------------------------------------- fill items
// A chunk's items, row (route) t and K block j of its r rows x kc K blocks,
// rows fastest: item p = j * r + t. A thread that steps through them `step`
// at a time keeps (t, j) and advances by (step % r, step / r), so no item costs
// a division by r.
struct ItemWalk {
  int t, j, dt, dj, r;
  FME_HD ItemWalk(int p0, int step, int rows) : r(rows) {
    j = p0 / rows;
    t = p0 - j * rows;
    dj = step / rows;
    dt = step - dj * rows;
  }
  FME_HD void next() {
    t += dt;
    j += dj;
    if (t >= r) {
      t -= r;
      ++j;
    }
  }
};

// ---------------------------------------------------------------- slot costs
// A slot (one K block of one tile of one unit) streams the same weight bytes
// whatever the unit, but its fill, accumulate and epilogue work grows with the
// unit's token rows r. Up to kLightRows rows that work hides under the stream
// and a slot costs kLightRows; a heavy unit's slot costs min(r, 64): the
// split below balances these costs instead of slot counts. The heavy units
// are listed in ascending unit order: unit hu[i] with extra cost he[i] =
// min(r, 64) - kLightRows per slot, hce[i] = he[0] + .. + he[i - 1] (nh + 1
// entries). At most kMaxHeavy of them; a call with more splits by slot counts.
constexpr int kLightRows = 8;
constexpr int kMaxHeavy = 64;
struct Heavy {
  int nh = 0;
  const int16_t* hu = nullptr;
  const uint16_t* he = nullptr;
  const uint32_t* hce = nullptr;
  // Heavy units before unit u.
  FME_HD int before(int u) const {
    int lo = 0, hi = nh;
    while (lo < hi) {
      const int m = (lo + hi) >> 1;
      if (hu[m] < u) lo = m + 1; else hi = m;
    }
    return lo;
  }
};

// ---------------------------------------------------------------- work plan
// The units are cut into W waves of consecutive units. The slots of one
// (wave, phase) -- units x tiles x K blocks, at most 1025 x 128 x 64 = 8.4M --
// are split over Ge = min(G, n) CTAs into contiguous slices, never empty;
// CTAs c >= Ge own nothing.
// - By slot count (no heavy unit in the wave): CTA c < Ge owns
//   [n*c/Ge, n*(c+1)/Ge). The products stay below 8.4M x 161 < 2^32, so
//   unsigned 32-bit arithmetic is exact.
// - By cost: slot x starts at cost position pos(x) (the costs of the slots
//   before it), the wave's total is Wt, and CTA c owns the slots with
//   c*Wt <= pos(x)*Ge < (c+1)*Wt. Every slice holds a slot when no slot costs
//   more than floor(Wt / Ge); a wave where one does splits by slot count.
//   pos(x) <= 8.4M x 64, so 64-bit products are exact.
// The cost-weighted split of one (wave, phase) of n slots, tn per unit, from
// unit u0: see PhasePlan. Out of line and with their arguments by value, so a
// kernel that never splits by cost carries neither their code nor a PhasePlan
// in memory.
struct CostSplit {
  const Heavy* hv;
  uint32_t ce0;  // hv->hce at the wave's first unit
  uint64_t Wt;   // the wave's total cost
  int n, tn, u0, Ge;
  // Cost position of the first slot of unit u (u0 <= u <= u0 + n / tn).
  FME_HD uint64_t ustart(int u) const {
    return static_cast<uint64_t>(tn) * (static_cast<uint64_t>(kLightRows) * static_cast<uint32_t>(u - u0) +
                                        hv->hce[hv->before(u)] - ce0);
  }
  FME_HD uint32_t slot_cost(int u) const {
    const int h = hv->before(u);
    return kLightRows + ((h < hv->nh && hv->hu[h] == u) ? hv->he[h] : 0u);
  }
  FME_HD uint64_t pos(int x) const {
    const int u = u0 + x / tn, o = x - (u - u0) * tn;
    return ustart(u) + static_cast<uint64_t>(o) * slot_cost(u);
  }
};
// The first slot at or past cost ceil(c * Wt / Ge): its unit is the last one
// that starts at or before that cost.
FME_HD_COLD inline int lo_of_by_cost(CostSplit cs, int c) {
  const uint64_t T = (static_cast<uint64_t>(c) * cs.Wt + static_cast<uint64_t>(cs.Ge) - 1) /
                     static_cast<uint64_t>(cs.Ge);
  int lo = 0, hi = cs.n / cs.tn - 1;
  while (lo < hi) {
    const int m = (lo + hi + 1) >> 1;
    if (cs.ustart(cs.u0 + m) <= T) lo = m; else hi = m - 1;
  }
  const int u = cs.u0 + lo;
  const uint64_t cost = cs.slot_cost(u);
  const uint64_t o = (T - cs.ustart(u) + cost - 1) / cost;
  const int x = lo * cs.tn + static_cast<int>(o);
  return x < cs.n ? x : cs.n;
}
FME_HD_COLD inline int cta_of_by_cost(CostSplit cs, int x) {
  return static_cast<int>(cs.pos(x) * static_cast<uint64_t>(cs.Ge) / cs.Wt);
}

struct PhasePlan {
  int n, lo, hi;
  int Ge, tiles, nb;
  int w, u0;  // wave and its first unit
  const Heavy* hv;  // nullptr: split by slot count
  uint32_t ce0;     // hv->hce at the wave's first unit
  uint64_t Wt;      // the wave's total cost
  FME_HD CostSplit cost() const { return CostSplit{hv, ce0, Wt, n, tiles * nb, u0, Ge}; }
  FME_HD int lo_of(int c) const {
    if (c >= Ge) return n;
    if (hv == nullptr)
      return static_cast<int>(static_cast<uint32_t>(n) * static_cast<uint32_t>(c) / static_cast<uint32_t>(Ge));
    return lo_of_by_cost(cost(), c);
  }
  // The CTA whose slice holds slot x.
  FME_HD int cta_of(int x) const {
    if (hv == nullptr)
      return static_cast<int>((static_cast<uint32_t>(x + 1) * static_cast<uint32_t>(Ge) + static_cast<uint32_t>(n) -
                               1u) / static_cast<uint32_t>(n)) - 1;
    return cta_of_by_cost(cost(), x);
  }
  FME_HD uint64_t pos(int x) const { return cost().pos(x); }
};

struct Plan {
  int U, N, kcmax, c, G, W;
  bool ximage;  // GEMM1 B rows copied from a per-call quantised image of x
  int kcmax2;  // K blocks per GEMM2 chunk, at most
  int phase_lo, phase_hi;  // phases this launch runs
  int N1, kcmax1;  // the MX kernel's GEMM1 B rows (four per token) and K blocks per chunk
  int tiles[2], nb[2];  // per unit: GEMM1 64-row tiles x H/128 K blocks; GEMM2 128-row tiles x I/128
  const Heavy* hv = nullptr;  // nullptr or no heavy unit: every split by slot count
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
    pp.hv = nullptr;
    pp.ce0 = 0;
    pp.Wt = 0;
    if (hv != nullptr && hv->nh > 0) {
      // Split this wave by cost when it holds a heavy unit and no slot costs
      // more than a slice's share.
      const int h0 = hv->before(u0), h1 = hv->before(u1);
      uint32_t emax = 0;
      for (int h = h0; h < h1; ++h) emax = hv->he[h] > emax ? hv->he[h] : emax;
      const uint64_t Wt = static_cast<uint64_t>(t * nbp) * (static_cast<uint64_t>(kLightRows) *
                                                                  static_cast<uint32_t>(u1 - u0) +
                                                              hv->hce[h1] - hv->hce[h0]);
      if (h1 > h0 && kLightRows + emax <= Wt / static_cast<uint64_t>(pp.Ge)) {
        pp.hv = hv;
        pp.ce0 = hv->hce[h0];
        pp.Wt = Wt;
      }
    }
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
