// Host check of the routed FP8 kernel's work decomposition (fme_plan.cuh):
// for many (units, tiles, K blocks, CTAs, waves, phase ranges, chunk sizes)
// every CTA walks its chunks with the kernel's own Cursor, and the walk must
// cover every (phase, unit, tile, K block) slot of the launched phases exactly
// once, in chunks of 1..kcmax K blocks inside one tile, each slot on the CTA
// cta_of names, a split tile's first K blocks at the end of its first
// contributor's slice, and no slot of a phase the launch does not run. With
// heavy units (a cost-weighted split) every slice of every stage must also be
// non-empty, and a slice's cost must stay within one slot of its share.
// Prints "OK <cases>" or the first failure; exit status 0 only on success.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "fme_plan.cuh"

using fme::Chunk;
using fme::Cursor;
using fme::Plan;

static int fail(const char* what, int U, int G, int W, int lo, int hi, int c) {
  std::printf("FAIL %s: U=%d G=%d W=%d phases %d..%d cta %d\n", what, U, G, W, lo, hi, c);
  return 1;
}

template <bool MX>
static int check(int U, int tiles1, int nb1, int tiles2, int nb2, int G, int W, int lo, int hi, int kcmax, int kcmax1,
                 int kcmax2, const fme::Heavy& hv) {
  // seen[phase][unit][tile][kb]
  std::vector<int> seen[2];
  seen[0].assign(static_cast<size_t>(U) * tiles1 * nb1, 0);
  seen[1].assign(static_cast<size_t>(U) * tiles2 * nb2, 0);
  for (int c = 0; c < G; ++c) {
    Plan P{};
    P.U = U;
    P.N = 16;
    P.kcmax = kcmax;
    P.N1 = 16;
    P.kcmax1 = kcmax1;
    P.kcmax2 = kcmax2;
    P.hv = &hv;
    P.c = c;
    P.G = G;
    P.W = W;
    P.phase_lo = lo;
    P.phase_hi = hi;
    P.tiles[0] = tiles1;
    P.nb[0] = nb1;
    P.tiles[1] = tiles2;
    P.nb[1] = nb2;
    Cursor cur;
    Chunk ch;
    int guard = 0;
    int last_phase = 0;
    while (cur.next<MX>(P, ch)) {
      if (++guard > 1 << 22) return fail("walk does not end", U, G, W, lo, hi, c);
      if (ch.phase < lo || ch.phase > hi) return fail("phase outside the launch", U, G, W, lo, hi, c);
      const int p = ch.phase - 1;
      const int tl = p == 0 ? tiles1 : tiles2, nb = p == 0 ? nb1 : nb2;
      const int cap = ch.phase == 2 ? kcmax2 : (MX ? kcmax1 : kcmax);
      if (ch.u < 0 || ch.u >= U || ch.T < 0 || ch.T >= tl) return fail("unit or tile out of range", U, G, W, lo, hi, c);
      if (ch.kc < 1 || ch.kc > cap || ch.kb0 < 0 || ch.kb0 + ch.kc > nb)
        return fail("chunk size or K range", U, G, W, lo, hi, c);
      const int tile_in_wave = (ch.u - ch.pp.u0) * tl + ch.T;
      if (ch.t0 != tile_in_wave * nb) return fail("tile start slot", U, G, W, lo, hi, c);
      for (int j = 0; j < ch.kc; ++j) {
        const int slot = ch.t0 + ch.kb0 + j;
        if (ch.pp.cta_of(slot) != c) return fail("cta_of disagrees with the walk", U, G, W, lo, hi, c);
        int& s = seen[p][(static_cast<size_t>(ch.u) * tl + ch.T) * nb + ch.kb0 + j];
        if (s++) return fail("slot walked twice", U, G, W, lo, hi, c);
      }
      // a split tile: its first contributor holds its first K blocks at the end of its slice
      const int cf = ch.pp.cta_of(ch.t0), cl = ch.pp.cta_of(ch.t0 + nb - 1);
      if (cf != cl && c == cf && ch.last_of_seg && ch.t0 + ch.kb0 + ch.kc != ch.pp.hi)
        return fail("first contributor's part not at its slice end", U, G, W, lo, hi, c);
      if (W == 1 && ch.phase < last_phase) return fail("phases out of order", U, G, W, lo, hi, c);
      last_phase = ch.phase;
    }
  }
  // Every stage's slices: contiguous, non-empty, and by cost within one slot
  // of an equal share.
  {
    Plan P{};
    P.U = U;
    P.hv = &hv;
    P.c = 0;
    P.G = G;
    P.W = W;
    P.phase_lo = 1;
    P.phase_hi = 2;
    P.tiles[0] = tiles1;
    P.nb[0] = nb1;
    P.tiles[1] = tiles2;
    P.nb[1] = nb2;
    for (int w = 0; w < W; ++w)
      for (int ph = 1; ph <= 2; ++ph) {
        const fme::PhasePlan pp = P.plan(w, ph);
        if (pp.lo_of(0) != 0 || pp.lo_of(pp.Ge) != pp.n) return fail("slices do not cover the stage", U, G, W, ph, ph, -1);
        for (int c = 0; c < pp.Ge; ++c) {
          const int a = pp.lo_of(c), b = pp.lo_of(c + 1);
          if (b <= a) return fail("empty slice", U, G, W, ph, ph, c);
          if (pp.cta_of(a) != c || pp.cta_of(b - 1) != c) return fail("cta_of at a slice edge", U, G, W, ph, ph, c);
          if (pp.hv != nullptr) {
            const uint64_t cost = (b < pp.n ? pp.pos(b) : pp.Wt) - pp.pos(a);
            const uint64_t share = pp.Wt / static_cast<uint64_t>(pp.Ge);
            if (cost + 64 < share || cost > share + 64 + 1) return fail("slice cost off its share", U, G, W, ph, ph, c);
          }
        }
      }
  }
  for (int p = 0; p < 2; ++p) {
    const bool run = p + 1 >= lo && p + 1 <= hi;
    for (int v : seen[p])
      if (v != (run ? 1 : 0)) return fail(run ? "slot never walked" : "slot of a skipped phase walked", U, G, W, lo, hi, -1);
  }
  return 0;
}

// The fill warps' division-free walk over a chunk's (row, K block) items.
static int check_item_walk() {
  for (int r = 1; r <= 64; ++r)
    for (int step : {1, 3, 8, 16, 64, 128})
      for (int p0 = 0; p0 < step + 9; ++p0) {
        fme::ItemWalk w(p0, step, r);
        for (int k = 0, p = p0; k < 300; ++k, p += step, w.next())
          if (w.t != p % r || w.j != p / r) {
            std::printf("FAIL item walk: r=%d step=%d p0=%d item %d\n", r, step, p0, p);
            return 1;
          }
      }
  return 0;
}

int main() {
  if (check_item_walk()) return 1;
  struct Shape { int tiles1, nb1, tiles2, nb2; };
  const Shape shapes[] = {{32, 56, 56, 16},   // DeepSeek-V3: I 2048, H 7168
                          {32, 28, 28, 16},   // latent: H 3584
                          {4, 4, 4, 2},       // tiny: H 512, I 256
                          {6, 8, 8, 3},       // ragged: H 1024, I 384
                          {2, 1, 1, 1}};      // H = I = 128
  const int units[] = {1, 2, 3, 8, 16, 31, 53, 257};
  const int ctas[] = {1, 3, 148, 152, 160};
  const int ranges[][2] = {{1, 2}, {1, 1}, {2, 2}};
  int cases = 0;
  for (const Shape& s : shapes)
    for (int U : units)
      for (int G : ctas)
        for (int W = 1; W <= 3; ++W)
          for (const auto& r : ranges)
            for (int kc : {16, 8, 4, 1}) {
              if (W > U || (r[0] == r[1] && W != 1)) continue;
              const int kc2 = kc < 8 ? kc : 8;
              // no heavy unit; unit 0 heavy (a one-launch layer's shared
              // expert); every third unit heavy, costs up to 64 rows a slot
              for (int pattern = 0; pattern < 3; ++pattern) {
                std::vector<int16_t> hu;
                std::vector<uint16_t> he;
                for (int u = 0; u < U && static_cast<int>(hu.size()) < fme::kMaxHeavy; ++u) {
                  const bool heavy = pattern == 1 ? u == 0 : (pattern == 2 && u % 3 == 1);
                  if (heavy) {
                    hu.push_back(static_cast<int16_t>(u));
                    he.push_back(static_cast<uint16_t>(pattern == 1 ? 56 : 1 + (u * 7) % 56));
                  }
                }
                std::vector<uint32_t> hce(hu.size() + 1, 0);
                for (size_t i = 0; i < hu.size(); ++i) hce[i + 1] = hce[i] + he[i];
                fme::Heavy hv;
                hv.nh = static_cast<int>(hu.size());
                hv.hu = hu.data();
                hv.he = he.data();
                hv.hce = hce.data();
                if (check<false>(U, s.tiles1, s.nb1, s.tiles2, s.nb2, G, W, r[0], r[1], kc, kc, kc2, hv)) return 1;
                if (check<true>(U, s.tiles1, s.nb1, s.tiles2, s.nb2, G, W, r[0], r[1], kc, kc > 4 ? kc / 4 : 1, kc2,
                                hv))
                  return 1;
                cases += 2;
              }
            }
  std::printf("OK %d\n", cases);
  return 0;
}
