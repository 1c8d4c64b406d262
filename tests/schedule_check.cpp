// Brute-force check of the forward work decomposition (host build).
// For each geometry given on the command line it verifies that
//   * the snake assignment gives every unit to exactly one CTA,
//   * each unit's key walk has exactly n tiles, in CP-step order,
//   * over all units, every (batch, head, query, key) pair the mask allows is
//     computed exactly once and no other pair is.
// Prints "ok" per geometry or the first violation, exit code 1 on failure.
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <vector>

#include "../context_blockwise_causal_gb300/csrc/cp_schedule.cuh"

using namespace cpattn;

static int verify(const CpGeom& g, const std::vector<unsigned char>& count, const char* what);

static int check(int b, int s, int hq, int hkv, int cp, int causal, int grid) {
  CpGeom g;
  g.b = b; g.s = s; g.hq = hq; g.hkv = hkv; g.cp = cp; g.causal = causal;
  g.c = s / (2 * cp);
  g.tpc = (g.c + kTile - 1) / kTile;
  g.npairs = (hq + 1) / 2;
  const int nu = fwd_num_units(g);
  std::vector<int> seen(nu, 0);
  for (int bid = 0; bid < grid; ++bid)
    for (int rd = 0;; ++rd) {
      int idx = snake_unit(rd, bid, grid);
      if (idx >= nu) break;
      seen[idx]++;
    }
  for (int i = 0; i < nu; ++i)
    if (seen[i] != 1) { printf("unit %d assigned %d times\n", i, seen[i]); return 1; }
  // count[(b*hq + h) * s * s + t * s + j]
  std::vector<unsigned char> count(size_t(b) * hq * s * s, 0);
  int prev_n = 1 << 30;
  for (int idx = 0; idx < nu; ++idx) {
    FwdUnit U = fwd_decode_unit(g, idx);
    if (causal && U.n > prev_n) { printf("units not in longest-first order at %d\n", idx); return 1; }
    prev_n = U.n;
    KvWalk w(g, U);
    int chunk, tile, nt = 0;
    bool dg;
    while (w.next(chunk, tile, dg)) {
      ++nt;
      const int rem = g.c - tile * kTile;
      const int nv = rem < kTile ? rem : kTile;
      for (int sub = 0; sub < 2; ++sub) {
        if (sub == 1 && !U.store1) continue;
        const int h = sub ? U.h1 : U.h0;
        if (h / (hq / hkv) != (sub ? U.g1 : U.g0)) { printf("bad kv head\n"); return 1; }
        for (int row = 0; row < U.q_valid; ++row)
          for (int col = 0; col < nv; ++col) {
            if (dg && col > row) continue;
            const int t = U.q_t0 + row, j = chunk * g.c + tile * kTile + col;
            unsigned char& c = count[(size_t(U.bi) * hq + h) * s * s + size_t(t) * s + j];
            if (c) { printf("pair (%d,%d) head %d computed twice\n", t, j, h); return 1; }
            c = 1;
          }
      }
    }
    if (nt != U.n) { printf("unit %d: walk has %d tiles, n = %d\n", idx, nt, U.n); return 1; }
    // the single-step walks, step after step, give the same tiles in order
    KvWalk full(g, U);
    int tot = 0;
    for (int st = 0; st < cp; ++st) {
      KvWalk one(g, U);
      one.only_step(st);
      int c1, t1, c2, t2, ns = 0;
      bool d1, d2;
      while (one.next(c1, t1, d1)) {
        ++ns;
        if (!full.next(c2, t2, d2) || c1 != c2 || t1 != t2 || d1 != d2) {
          printf("unit %d: step %d walk differs from the full walk\n", idx, st);
          return 1;
        }
      }
      if (ns != one.step_tiles(st)) { printf("unit %d: step %d has %d tiles, step_tiles %d\n", idx, st, ns, one.step_tiles(st)); return 1; }
      tot += ns;
    }
    if (tot != U.n) { printf("unit %d: steps sum to %d tiles, n = %d\n", idx, tot, U.n); return 1; }
  }
  if (verify(g, count, "forward")) return 1;
  // backward: key-tile units walking the query tiles that see them
  std::fill(count.begin(), count.end(), 0);
  const int nb = bwd_num_units(g);
  const int G = hq / hkv;
  int prev_items = 1 << 30;
  for (int idx = 0; idx < nb; ++idx) {
    BwdUnit U = bwd_decode_unit(g, idx);
    if (causal && U.items > prev_items) { printf("bwd units not longest-first at %d\n", idx); return 1; }
    prev_items = U.items;
    QWalk w(g, U);
    int chunk, tile, nt = 0;
    bool dg;
    while (w.next(chunk, tile, dg)) {
      ++nt;
      const int rem = g.c - tile * kTile;
      const int qv = rem < kTile ? rem : kTile;
      for (int h = U.g * G; h < (U.g + 1) * G; ++h)
        for (int row = 0; row < qv; ++row)
          for (int col = 0; col < U.k_valid; ++col) {
            if (dg && col > row) continue;
            const int t = chunk * g.c + tile * kTile + row, j = U.k_t0 + col;
            unsigned char& c = count[(size_t(U.bi) * hq + h) * s * s + size_t(t) * s + j];
            if (c) { printf("bwd pair (%d,%d) head %d computed twice\n", t, j, h); return 1; }
            c = 1;
          }
    }
    if (nt != U.nq) { printf("bwd unit %d: walk has %d tiles, nq = %d\n", idx, nt, U.nq); return 1; }
    if (U.items != nt * G) { printf("bwd unit %d: items mismatch\n", idx); return 1; }
  }
  return verify(g, count, "backward");
}

static int verify(const CpGeom& g, const std::vector<unsigned char>& count, const char* what) {
  const int b = g.b, hq = g.hq, s = g.s, causal = g.causal;
  for (int bi = 0; bi < b; ++bi)
    for (int h = 0; h < hq; ++h)
      for (int t = 0; t < s; ++t)
        for (int j = 0; j < s; ++j) {
          const int want = (!causal || j <= t) ? 1 : 0;
          if (count[(size_t(bi) * hq + h) * s * s + size_t(t) * s + j] != want) {
            printf("%s pair (%d,%d) batch %d head %d: count %d want %d\n", what, t, j, bi, h,
                   count[(size_t(bi) * hq + h) * s * s + size_t(t) * s + j], want);
            return 1;
          }
        }
  return 0;
}

int main(int argc, char** argv) {
  // args: groups of 7 ints: b s hq hkv cp causal grid
  int fails = 0;
  for (int i = 1; i + 6 < argc; i += 7) {
    int v[7];
    for (int k = 0; k < 7; ++k) v[k] = atoi(argv[i + k]);
    int rc = check(v[0], v[1], v[2], v[3], v[4], v[5], v[6]);
    printf("%s b=%d s=%d hq=%d hkv=%d cp=%d causal=%d grid=%d\n", rc ? "FAIL" : "ok", v[0], v[1], v[2], v[3], v[4],
           v[5], v[6]);
    fails += rc;
  }
  return fails ? 1 : 0;
}
