// Brute-force check of the kernels' work decomposition (host build).
// For each geometry given on the command line it verifies that
//   * the snake assignment gives every unit to exactly one CTA,
//   * units come longest-first, each key walk has exactly n tiles in CP-step
//     order, and the single-step walks, step after step, give the same tiles,
//   * over all forward units, over all dQ units, and over all backward
//     (key-tile) units, every (head, query, key) pair the mask allows is
//     computed exactly once and no other pair is -- in particular no pair
//     crosses a packed-sample boundary.
// Geometries: "U b s hq hkv cp causal grid" (a uniform batch),
// "P nseq len_1 .. len_nseq hq hkv cp causal grid" (packed samples), or
// "R b s hq hkv cp causal grid" (the rank-local form: every rank's call,
// with its rows mapped back to the sequence, must together cover each pair
// exactly once -- for the all-gather form, for the ring form step by step,
// and for the backward's key-tile units -- and every row a call addresses
// must lie inside its buffer).
// Prints "ok" per geometry or the first violation, exit code 1 on failure.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <vector>

#include "../context_blockwise_causal_gb300/csrc/cp_schedule.cuh"

using namespace cpattn;

struct Rows {
  int total;                 // token rows
  std::vector<int> seq_of;   // sequence of each row
  std::vector<int> pos_of;   // position of each row within its sequence
};

static Rows rows_of(const CpGeom& g) {
  Rows R;
  R.total = g.b * g.s;
  R.seq_of.assign(R.total, 0);
  R.pos_of.assign(R.total, 0);
  for (int i = 0; i < num_seqs(g); ++i) {
    const int t0 = g.nseq > 0 ? g.cu[i] : i * g.s;
    const int len = g.nseq > 0 ? g.cu[i + 1] - g.cu[i] : g.s;
    for (int t = 0; t < len; ++t) {
      R.seq_of[t0 + t] = i;
      R.pos_of[t0 + t] = t;
    }
  }
  return R;
}

static int verify(const CpGeom& g, const Rows& R, const std::vector<unsigned char>& count, const char* what) {
  const size_t T = R.total;
  for (int h = 0; h < g.hq; ++h)
    for (int qa = 0; qa < R.total; ++qa)
      for (int ka = 0; ka < R.total; ++ka) {
        const bool same = R.seq_of[qa] == R.seq_of[ka];
        const int want = same && (!g.causal || R.pos_of[ka] <= R.pos_of[qa]) ? 1 : 0;
        const int got = count[size_t(h) * T * T + size_t(qa) * T + ka];
        if (got != want) {
          printf("%s pair (%d,%d) head %d: count %d want %d\n", what, qa, ka, h, got, want);
          return 1;
        }
      }
  return 0;
}

static int mark(std::vector<unsigned char>& count, const Rows& R, int h, int qa, int ka, const char* what) {
  unsigned char& c = count[size_t(h) * R.total * R.total + size_t(qa) * R.total + ka];
  if (c) {
    printf("%s pair (%d,%d) head %d computed twice\n", what, qa, ka, h);
    return 1;
  }
  c = 1;
  return 0;
}

// Rank-local form: the sequence row (b*s layout) of a row of the rank's
// query shard [b, 2c], and of a row of the key/value buffer -- rank-major
// shards (kv_rank_rows = b*2c), or the one shard of rank `owner` (0).
static int rank_q_row(const CpGeom& g, int row) {
  const int local = 2 * g.c, bi = row / local, u = row % local;
  return bi * g.s + (u < g.c ? g.rank * g.c + u : (2 * g.cp - 1 - g.rank) * g.c + (u - g.c));
}
static int rank_kv_row(const CpGeom& g, int row, int owner) {
  const int local = 2 * g.c;
  int rest = row;
  if (g.kv_rank_rows > 0) {
    owner = row / g.kv_rank_rows;
    rest = row % g.kv_rank_rows;
  }
  const int bi = rest / local, u = rest % local;
  return bi * g.s + (u < g.c ? owner * g.c + u : (2 * g.cp - 1 - owner) * g.c + (u - g.c));
}

// Buffer rows -> sequence rows, and the buffers' row counts.
struct RowMap {
  int q_rows, kv_rows;  // rows of the query-side and key/value buffers
  int owner;            // ring step form: the rank whose shard the K/V buffer holds
  int q(const CpGeom& g, int r) const { return g.rank >= 0 ? rank_q_row(g, r) : r; }
  int kv(const CpGeom& g, int r) const { return g.rank >= 0 ? rank_kv_row(g, r, owner) : r; }
};

static RowMap natural_map(const CpGeom& g) { return RowMap{g.b * g.s, g.b * g.s, -1}; }

// Walk one query-tile unit (forward sub-tile `sub` or a dQ unit) and mark its pairs.
static int walk_query_unit(const CpGeom& g, const Rows& R, const FwdUnit& U, int h, std::vector<unsigned char>& count,
                           const char* what, KvWalk w, const RowMap& M, int sub = 0, int step = -1) {
  int chunk, tile, nt = 0;
  bool walk_dg, dg, dead;
  const int q_t = sub ? U.q_t1 : U.q_t0, q_valid = sub ? U.q_valid1 : U.q_valid;
  const int jd = fwd_dead_pos(g, U, sub, step);
  while (w.next(chunk, tile, walk_dg)) {
    fwd_pos_mask(jd, nt, walk_dg, dg, dead);
    ++nt;
    if (dead) continue;
    const int rem = U.c - tile * kTile;
    const int nv = rem < kTile ? rem : kTile;
    for (int row = 0; row < q_valid; ++row)
      for (int col = 0; col < nv; ++col) {
        if (dg && col > row) continue;
        const int qb = U.tok0 + q_t + row, kb = U.tok0 + kv_chunk_row(g, chunk, U.c) + tile * kTile + col;
        if (qb < 0 || qb >= M.q_rows || kb < 0 || kb >= M.kv_rows) {
          printf("%s: row outside its buffer (query %d of %d, key %d of %d)\n", what, qb, M.q_rows, kb, M.kv_rows);
          return -1;
        }
        if (mark(count, R, h, M.q(g, qb), M.kv(g, kb), what)) return -1;
      }
  }
  return nt;
}
static int walk_query_unit(const CpGeom& g, const Rows& R, const FwdUnit& U, int h, std::vector<unsigned char>& count,
                           const char* what, int sub = 0) {
  return walk_query_unit(g, R, U, h, count, what, KvWalk(g, U), natural_map(g), sub);
}

static int check(const CpGeom& g, int grid) {
  const Rows R = rows_of(g);
  std::vector<unsigned char> count(size_t(g.hq) * R.total * R.total, 0);
  // ---- forward
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
  int prev_n = 1 << 30, prev_seq = -1;
  for (int idx = 0; idx < nu; ++idx) {
    const FwdUnit U = fwd_decode_unit(g, idx);
    if (U.n == 0) continue;  // an empty packed sample, or an empty slot of a unit block
    if (g.nseq > 0 && U.seq != prev_seq) prev_n = 1 << 30;  // packed samples come one after another
    if (g.tp_block > 0 && idx % g.tp_slots == 0) prev_n = 1 << 30;  // unit blocks come one after another
    prev_seq = U.seq;
    if (g.causal && U.n > prev_n) { printf("units not in longest-first order at %d\n", idx); return 1; }
    prev_n = U.n;
    for (int sub = 0; sub < 2; ++sub) {
      if (sub == 1 && !U.store1) continue;
      const int h = sub ? U.h1 : U.h0;
      if (h / (g.hq / g.hkv) != (sub ? U.g1 : U.g0)) { printf("bad kv head\n"); return 1; }
      const int nt = walk_query_unit(g, R, U, h, count, "forward", sub);
      if (nt < 0) return 1;
      if (nt != U.n) { printf("unit %d: walk has %d tiles, n = %d\n", idx, nt, U.n); return 1; }
    }
    // the single-step walks, step after step, give the same tiles in order
    KvWalk full(g, U);
    int tot = 0;
    for (int st = 0; st < g.cp; ++st) {
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
      if (ns != one.step_tiles(st)) {
        printf("unit %d: step %d has %d tiles, step_tiles %d\n", idx, st, ns, one.step_tiles(st));
        return 1;
      }
      tot += ns;
    }
    if (tot != U.n) { printf("unit %d: steps sum to %d tiles, n = %d\n", idx, tot, U.n); return 1; }
  }
  if (verify(g, R, count, "forward")) return 1;
  // ---- dQ units: one query tile of one head
  std::fill(count.begin(), count.end(), 0);
  const int nd = dq_num_units(g);
  for (int idx = 0; idx < nd; ++idx) {
    const FwdUnit U = dq_decode_unit(g, idx);
    if (U.n == 0) continue;
    const int nt = walk_query_unit(g, R, U, U.h0, count, "dq");
    if (nt < 0) return 1;
    if (nt != U.n) { printf("dq unit %d: walk has %d tiles, n = %d\n", idx, nt, U.n); return 1; }
  }
  if (verify(g, R, count, "dq")) return 1;
  // ---- backward: key-tile units walking the query tiles that see them
  std::fill(count.begin(), count.end(), 0);
  const int nb = bwd_num_units(g);
  const int G = g.hq / g.hkv;
  int prev_items = 1 << 30;
  prev_seq = -1;
  for (int idx = 0; idx < nb; ++idx) {
    const BwdUnit U = bwd_decode_unit(g, idx);
    if (U.items == 0) continue;
    if (g.nseq > 0 && U.seq != prev_seq) prev_items = 1 << 30;
    prev_seq = U.seq;
    if (g.causal && U.items > prev_items) { printf("bwd units not longest-first at %d\n", idx); return 1; }
    prev_items = U.items;
    QWalk w(g, U);
    int chunk, tile, nt = 0;
    bool dg;
    while (w.next(chunk, tile, dg)) {
      ++nt;
      const int rem = U.c - tile * kTile;
      const int qv = rem < kTile ? rem : kTile;
      for (int h = U.g * G; h < (U.g + 1) * G; ++h)
        for (int row = 0; row < qv; ++row)
          for (int col = 0; col < U.k_valid; ++col) {
            if (dg && col > row) continue;
            const int qa = U.tok0 + chunk * U.c + tile * kTile + row, ka = U.tok0 + U.k_t0 + col;
            if (mark(count, R, h, qa, ka, "bwd")) return 1;
          }
    }
    if (nt != U.nq) { printf("bwd unit %d: walk has %d tiles, nq = %d\n", idx, nt, U.nq); return 1; }
    if (U.items != nt * G) { printf("bwd unit %d: items mismatch\n", idx); return 1; }
  }
  return verify(g, R, count, "backward");
}

// The rank-local form: each rank's forward (all-gather form and ring steps),
// dQ and key-tile backward units, mapped back to sequence rows.
static int check_rank(const CpGeom& base, int grid, int kv_per_block) {
  const Rows R = rows_of(base);
  const size_t T = R.total;
  std::vector<unsigned char> fwd(size_t(base.hq) * T * T, 0), ring(fwd.size(), 0), dq(fwd.size(), 0),
      bwd(fwd.size(), 0);
  const int G = base.hq / base.hkv;
  for (int r = 0; r < base.cp; ++r) {
    CpGeom g = base;
    g.rank = r;
    g.kv_rank_rows = g.b * 2 * g.c;
    set_tile_pair_blocks(g, grid, kv_per_block);  // as the library sets it, per launch
    const RowMap gathered{g.b * 2 * g.c, g.cp * g.b * 2 * g.c, -1};
    // ---- forward units: snake assignment, longest first, the rank's tiles only
    const int nu = fwd_num_units(g);
    const int blocks = g.tp_block > 0 ? (g.b * g.hq + g.tp_block - 1) / g.tp_block : 0;
    if (nu != (blocks ? blocks * g.tp_slots : g.tile_pairs ? g.hq * g.b * g.tpc : g.npairs * g.b * 2 * g.tpc)) {
      printf("rank %d: %d forward units\n", r, nu);
      return 1;
    }
    std::vector<int> seen(nu, 0);
    for (int bid = 0; bid < grid; ++bid)
      for (int rd = 0;; ++rd) {
        const int idx = snake_unit(rd, bid, grid);
        if (idx >= nu) break;
        seen[idx]++;
      }
    for (int i = 0; i < nu; ++i)
      if (seen[i] != 1) { printf("rank %d: unit %d assigned %d times\n", r, i, seen[i]); return 1; }
    int prev_n = 1 << 30;
    for (int idx = 0; idx < nu; ++idx) {
      if (g.tp_block > 0 && idx % g.tp_slots == 0) prev_n = 1 << 30;
      const FwdUnit U = fwd_decode_unit(g, idx);
      if (U.n == 0) continue;  // an empty slot of a unit block
      if (U.r != r) { printf("rank %d: unit %d belongs to rank %d\n", r, idx, U.r); return 1; }
      if (g.causal && U.n > prev_n) { printf("rank %d: units not longest-first at %d\n", r, idx); return 1; }
      prev_n = U.n;
      for (int sub = 0; sub < 2; ++sub) {
        if (sub == 1 && !U.store1) continue;
        const int h = sub ? U.h1 : U.h0;
        const int nt = walk_query_unit(g, R, U, h, fwd, "rank forward", KvWalk(g, U), gathered, sub);
        if (nt < 0) return 1;
        if (nt != U.n) { printf("rank %d unit %d: walk has %d tiles, n = %d\n", r, idx, nt, U.n); return 1; }
        // ring form: step st reads only the shard of rank (r - st) mod cp
        CpGeom gs = g;
        gs.kv_rank_rows = 0;
        for (int st = 0; st < g.cp; ++st) {
          const RowMap one{g.b * 2 * g.c, g.b * 2 * g.c, ((r - st) % g.cp + g.cp) % g.cp};
          KvWalk w(gs, U);
          w.only_step(st);
          if (walk_query_unit(gs, R, U, h, ring, "rank ring step", w, one, sub, st) < 0) return 1;
        }
      }
    }
    // ---- dQ units
    const int nd = dq_num_units(g);
    for (int idx = 0; idx < nd; ++idx) {
      const FwdUnit U = dq_decode_unit(g, idx);
      if (U.r != r) { printf("rank %d: dq unit %d belongs to rank %d\n", r, idx, U.r); return 1; }
      const int nt = walk_query_unit(g, R, U, U.h0, dq, "rank dq", KvWalk(g, U), gathered);
      if (nt < 0) return 1;
      if (nt != U.n) { printf("rank %d dq unit %d: %d tiles, n = %d\n", r, idx, nt, U.n); return 1; }
    }
    // ---- backward: every key tile of the gathered shards, the rank's query tiles
    const int nb = bwd_num_units(g);
    int prev_items = 1 << 30;
    for (int idx = 0; idx < nb; ++idx) {
      const BwdUnit U = bwd_decode_unit(g, idx);
      if (U.k_valid <= 0) { printf("rank %d: bwd unit %d is not a real key tile\n", r, idx); return 1; }
      if (g.causal && U.items > prev_items) { printf("rank %d: bwd units not longest-first at %d\n", r, idx); return 1; }
      prev_items = U.items;
      QWalk w(g, U);
      int chunk, tile, nt = 0;
      bool dg;
      while (w.next(chunk, tile, dg)) {
        ++nt;
        const int rem = U.c - tile * kTile;
        const int qv = rem < kTile ? rem : kTile;
        for (int h = U.g * G; h < (U.g + 1) * G; ++h)
          for (int row = 0; row < qv; ++row)
            for (int col = 0; col < U.k_valid; ++col) {
              if (dg && col > row) continue;
              const int qb = U.tok0 + q_chunk_row(g, chunk, U.c) + tile * kTile + row, kb = U.tok0 + U.k_t0 + col;
              if (qb >= gathered.q_rows || kb >= gathered.kv_rows) { printf("rank bwd: row outside its buffer\n"); return 1; }
              if (mark(bwd, R, h, gathered.q(g, qb), gathered.kv(g, kb), "rank bwd")) return 1;
            }
      }
      if (nt != U.nq) { printf("rank %d bwd unit %d: walk has %d tiles, nq = %d\n", r, idx, nt, U.nq); return 1; }
      if (U.items != nt * G) { printf("rank %d bwd unit %d: items mismatch\n", r, idx); return 1; }
    }
  }
  return verify(base, R, fwd, "rank forward") || verify(base, R, ring, "rank ring steps") ||
         verify(base, R, dq, "rank dq") || verify(base, R, bwd, "rank backward");
}

// FastDiv against plain division: every divisor up to 5000 with dividends
// around each multiple and at the ends of the range, and pseudo-random
// (divisor, dividend) pairs over the whole range (xorshift, fixed seed).
static int check_fastdiv() {
  auto one = [](int d, int n) {
    const FastDiv f = make_fastdiv(d);
    if (f.div(n) != n / d || f.mod(n) != n % d) {
      printf("fastdiv %d / %d: %d (expected %d)\n", n, d, f.div(n), n / d);
      return 1;
    }
    return 0;
  };
  for (int d = 1; d <= 5000; ++d) {
    for (int k = 0; k <= 64; ++k)
      for (int e = -2; e <= 2; ++e) {
        const int64_t n = int64_t(k) * d + e;
        if (n >= 0 && one(d, int(n))) return 1;
      }
    for (int e = 0; e < 4; ++e)
      if (one(d, 0x7fffffff - e)) return 1;
  }
  uint64_t x = 0x9e3779b97f4a7c15ull;
  for (int i = 0; i < 2000000; ++i) {
    x ^= x << 13;
    x ^= x >> 7;
    x ^= x << 17;
    const int d = int((x >> 33) % 0x7fffffffu) + 1, n = int(x & 0x7fffffffu);
    if (one(d, n) || one(d & 0xffff ? d & 0xffff : 1, n)) return 1;
  }
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 2 && !strcmp(argv[1], "D")) {
    const int rc = check_fastdiv();
    printf("%s fastdiv\n", rc ? "FAIL" : "ok");
    return rc;
  }
  int fails = 0, i = 1;
  int kv_per_block = 0;  // "K n": tile-pair unit blocks of n KV pairs for the geometries that follow
  while (i < argc) {
    if (!strcmp(argv[i], "K") && i + 1 < argc) {
      kv_per_block = atoi(argv[i + 1]);
      i += 2;
      continue;
    }
    CpGeom g;
    char desc[256];
    int grid;
    const bool ranked = !strcmp(argv[i], "R");
    if ((!strcmp(argv[i], "U") || ranked) && i + 7 < argc) {
      g.b = atoi(argv[i + 1]);
      g.s = atoi(argv[i + 2]);
      g.hq = atoi(argv[i + 3]);
      g.hkv = atoi(argv[i + 4]);
      g.cp = atoi(argv[i + 5]);
      g.causal = atoi(argv[i + 6]);
      grid = atoi(argv[i + 7]);
      g.c = g.s / (2 * g.cp);
      g.tpc = (g.c + kTile - 1) / kTile;
      g.nseq = 0;
      snprintf(desc, sizeof desc, "%sb=%d s=%d hq=%d hkv=%d cp=%d causal=%d grid=%d%s", ranked ? "rank-local " : "",
               g.b, g.s, g.hq, g.hkv, g.cp, g.causal, grid,
               (g.hq / g.hkv) % 2 == 1 && (g.s / (2 * g.cp) + kTile - 1) / kTile % 2 == 0 ? " (tile pairs)" : "");
      i += 8;
    } else if (!strcmp(argv[i], "P") && i + 1 < argc) {
      const int n = atoi(argv[i + 1]);
      if (n < 1 || n > kMaxSeqs || i + 2 + n + 4 >= argc) { printf("bad packed spec\n"); return 1; }
      g.nseq = n;
      g.cu[0] = 0;
      for (int k = 0; k < n; ++k) g.cu[k + 1] = g.cu[k] + atoi(argv[i + 2 + k]);
      int j = i + 2 + n;
      g.hq = atoi(argv[j]);
      g.hkv = atoi(argv[j + 1]);
      g.cp = atoi(argv[j + 2]);
      g.causal = atoi(argv[j + 3]);
      grid = atoi(argv[j + 4]);
      finish_packed(g);
      snprintf(desc, sizeof desc, "packed nseq=%d total=%d hq=%d hkv=%d cp=%d causal=%d grid=%d", n, g.s, g.hq,
               g.hkv, g.cp, g.causal, grid);
      i = j + 5;
    } else {
      printf("bad arguments at %s\n", argv[i]);
      return 1;
    }
    g.npairs = (g.hq + 1) / 2;
    g.tile_pairs = use_tile_pairs(g) ? 1 : 0;  // as the library sets it
    set_fast_divs(g);
    {
      CpGeom t = g;
      if (ranked) t.rank = 0;
      set_tile_pair_blocks(t, grid, kv_per_block);
      if (t.tp_block > 0) {
        const size_t n = strlen(desc);
        snprintf(desc + n, sizeof desc - n, " [blocks of %d heads, %d slots]", t.tp_block, t.tp_slots);
      }
      if (!ranked) g = t;
    }
    const int rc = ranked ? check_rank(g, grid, kv_per_block) : check(g, grid);
    printf("%s %s\n", rc ? "FAIL" : "ok", desc);
    fails += rc;
  }
  return fails ? 1 : 0;
}
