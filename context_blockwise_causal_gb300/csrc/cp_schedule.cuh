// Context-parallel work decomposition shared by the kernels.
//
// Zigzag split ("大模型面试宝典 · Megatron-LM 篇", 3.4; "超大规模集群下大语言模型训练
// 实操指南", CP 与其他技术结合): 2*cp chunks of c tokens, virtual rank r owns
// chunks r and 2cp-1-r. Each chunk is cut into tpc = ceil(c/128) tiles that
// start at the chunk's first token (the last one may be ragged).
//
// A forward work unit is one 128-row query tile of one chunk, for a pair of
// query heads (two sub-tiles that walk the same key tiles), for one batch
// element -- or, when the head groups are odd (tile_pairs), two adjacent query
// tiles of one head, so that the two sub-tiles still share their K/V tiles. Its key tiles are visited in the order of the rank's CP steps:
//   step 0      : the rank's own chunks, causal (the one masked "diagonal"
//                 tile is where the query tile meets its own chunk);
//   1 <= i <= r : chunk j = r - i (first half of rank j's pair), unmasked;
//   i > r       : only for queries in chunk 2cp-1-r: chunks j and 2cp-1-j
//                 with j = r - i + cp, unmasked.
// Without the causal mask every step covers both chunks of rank
// j = (r - i) mod cp.
#pragma once
#include <cstdint>

#ifndef __CUDACC__  // host-only builds (the schedule's CPU test)
#define __host__
#define __device__
#endif

namespace cpattn {

constexpr int kTile = 128;
constexpr int kMaxSeqs = 512;  // packed samples per call (their offsets travel as kernel parameters)

// Division by a value fixed for a launch, as a multiply and a shift
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): for 0 <= n < 2^31 and 1 <= d <= 2^31, with
// s = ceil(log2 d) and m = ceil(2^(31+s) / d), which is below 2^32,
// floor(n / d) = floor(n * m / 2^(31+s)): n*m / 2^(31+s) exceeds n/d by
// less than 2^-s <= 1/d. The backward's unit decodes run once per work unit
// in every role of a CTA; a plain integer division there is a long
// dependent chain.
struct FastDiv {
  int d = 1;
  uint32_t m = 0x80000000u;
  int shift = 31;
  __host__ __device__ int div(int n) const { return int((uint64_t(uint32_t(n)) * m) >> shift); }
  __host__ __device__ int mod(int n) const { return n - div(n) * d; }
};
__host__ __device__ inline FastDiv make_fastdiv(int d) {
  FastDiv f;
  f.d = d;
  int s = 0;
  while ((int64_t(1) << s) < d) ++s;
  f.m = uint32_t(((uint64_t(1) << (31 + s)) + uint64_t(d) - 1) / uint64_t(d));
  f.shift = 31 + s;
  return f;
}

// Geometry of a call. Either a uniform batch (nseq == 0: b sequences of s
// tokens, chunk length c, tpc tiles per chunk) or packed samples (nseq > 0:
// b == 1, s == total tokens, sample i is tokens [cu[i], cu[i+1]) with its own
// chunk length; tpc is the largest sample's tile count).
//
// Rank-local form (rank >= 0, uniform batch only): the call is the share of
// one rank of a CP group spread over several GPUs. The query side (q, o,
// lse, dO, dq) then holds only that rank's two chunks, 2c rows per batch
// element: chunk `rank` at local rows [0, c), chunk 2cp-1-rank at [c, 2c).
// The key/value side holds rank-major shards laid out the same way: rank j's
// shard of batch element bi starts at row j * kv_rank_rows + bi * 2c
// (kv_rank_rows = b * 2c after an all-gather of every rank's shard; 0 when
// the buffer holds the one shard a ring step received).
struct CpGeom {
  int b, s, hq, hkv, cp, causal;
  int c;       // chunk length (uniform batch)
  int tpc;     // tiles per chunk (the largest sample's when packed)
  int npairs;  // query-head pairs per batch element: ceil(hq / 2)
  int nseq = 0;
  int rank = -1;         // rank-local form: the rank whose queries the call computes
  int kv_rank_rows = 0;  // rank-local form: rows between consecutive ranks' K/V shards
  int tile_pairs = 0;    // forward units pair two query tiles of one head (see fwd_decode_unit)
  int tp_block = 0;      // tile pairs: (sequence, query head) combinations per unit block (0: one block)
  int tp_slots = 0;      // tile pairs: unit slots per block (its units, then empty slots)
  // divisors of the backward's unit decodes (set_fast_divs; set again
  // whenever b, hq, hkv or tpc change)
  FastDiv fd_hq, fd_hkv, fd_G, fd_tpc, fd_bhq, fd_bhkv;
  int cu[kMaxSeqs + 1];     // packed: sample offsets
  int tile0[kMaxSeqs + 1];  // packed: query tiles (2cp * tpc_i) of the samples before sample i
};

__host__ __device__ inline void set_fast_divs(CpGeom& g) {
  g.fd_hq = make_fastdiv(g.hq);
  g.fd_hkv = make_fastdiv(g.hkv);
  g.fd_G = make_fastdiv(g.hq / g.hkv);
  g.fd_tpc = make_fastdiv(g.tpc > 0 ? g.tpc : 1);
  g.fd_bhq = make_fastdiv(g.b * g.hq);
  g.fd_bhkv = make_fastdiv(g.b * g.hkv);
}

// Rows of one sequence on the query side: the whole sequence, or one rank's
// two chunks in the rank-local form.
__host__ __device__ inline int q_seq_rows(const CpGeom& g) { return g.rank >= 0 ? 2 * g.c : g.s; }

// First row of global chunk `chunk` (chunk length c) relative to its
// sequence's first row, on the query side and on the key/value side.
__host__ __device__ inline int q_chunk_row(const CpGeom& g, int chunk, int c) {
  return g.rank >= 0 ? (chunk < g.cp ? 0 : c) : chunk * c;
}
__host__ __device__ inline int kv_chunk_row(const CpGeom& g, int chunk, int c) {
  if (g.rank < 0) return chunk * c;
  const int owner = chunk < g.cp ? chunk : 2 * g.cp - 1 - chunk;  // the rank holding the chunk
  return owner * g.kv_rank_rows + (chunk < g.cp ? 0 : c);
}

// Tile (chunk, tile) of a sequence in the backward's tile-padded row
// vectors: all 2cp*tpc tiles, or the rank's own 2*tpc in the rank-local form.
__host__ __device__ inline int ld_tile(const CpGeom& g, int chunk, int tile, int tpc) {
  return (g.rank >= 0 ? (chunk < g.cp ? 0 : tpc) : chunk * tpc) + tile;
}

// Packed geometry from the sample offsets (cu[0..nseq] set): the largest
// sample's tiles per chunk and the tile prefix sums.
__host__ __device__ inline void finish_packed(CpGeom& g) {
  g.b = 1;
  g.s = g.cu[g.nseq];
  g.c = 0;
  g.tpc = 0;
  g.tile0[0] = 0;
  for (int i = 0; i < g.nseq; ++i) {
    const int c = (g.cu[i + 1] - g.cu[i]) / (2 * g.cp);
    const int tpc = (c + kTile - 1) / kTile;
    g.tpc = tpc > g.tpc ? tpc : g.tpc;
    g.tile0[i + 1] = g.tile0[i] + 2 * g.cp * tpc;
  }
  set_fast_divs(g);
}

// Packed samples: the sample holding global tile position p (a binary
// search over tile0), and p's offset within that sample's tiles.
__host__ __device__ inline int packed_sample_of(const CpGeom& g, int p, int& local) {
  int lo = 0, hi = g.nseq;  // tile0[lo] <= p < tile0[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (g.tile0[mid] <= p) lo = mid; else hi = mid;
  }
  local = p - g.tile0[lo];
  return lo;
}

// A sequence's placement: its first token in the token rows, its chunk
// length and tiles per chunk (0 tiles for an empty sample).
struct SeqGeom {
  int tok0, c, tpc;
};

__host__ __device__ inline int num_seqs(const CpGeom& g) { return g.nseq > 0 ? g.nseq : g.b; }

__host__ __device__ inline SeqGeom seq_geom(const CpGeom& g, int i) {
  SeqGeom q;
  if (g.nseq == 0) {
    q.tok0 = i * q_seq_rows(g);
    q.c = g.c;
    q.tpc = g.tpc;
  } else {
    q.tok0 = g.cu[i];
    q.c = (g.cu[i + 1] - g.cu[i]) / (2 * g.cp);
    q.tpc = (q.c + kTile - 1) / kTile;
  }
  return q;
}

struct FwdUnit {
  int bi;        // batch element (0 for packed samples)
  int seq;       // batch element or packed sample
  int tok0;      // its first token row
  int lse_t0;    // offset of its positions in an LSE row (the sample's start when packed)
  int c, tpc;    // its chunk length and tiles per chunk
  int h0, h1;    // query heads of the two sub-tiles (h1 == h0 for an odd tail)
  int g0, g1;    // their KV heads
  bool store1;   // sub-tile 1 is a distinct head (its output is stored)
  int k;         // global chunk index of the query tile
  int u;         // tile index within the chunk
  int r, half;   // owning virtual rank and which of its two chunks
  int q_t0;      // first row of the query tile relative to its sequence's first row
                 // (its position in the sequence; its local position in the rank-local form)
  int q_valid;   // rows of the tile inside the chunk
  // sub-tile 1's query tile: the same as sub-tile 0's for a head pair; for a
  // tile pair (tile_pairs) the next tile u of the chunk, sub-tile 0 having
  // tile u0 = u - 1. The key walk is always that of tile u.
  int u0, q_t1, q_valid1;
  int n;         // number of key tiles the unit visits (0: no such tile in a shorter packed sample)
};

// Units per head group of a call: every sequence's key tiles, and its
// query tiles (only the rank's own in the rank-local form).
__host__ __device__ inline int all_tiles(const CpGeom& g) {
  return g.nseq > 0 ? g.tile0[g.nseq] : g.b * 2 * g.cp * g.tpc;
}
__host__ __device__ inline int query_tiles(const CpGeom& g) {
  return g.rank >= 0 ? g.b * 2 * g.tpc : all_tiles(g);
}

// Global tile index of the query tile of local position lt (the unit order
// below walks it from the end): every tile of the sequence, or in the
// rank-local form the rank's tiles, chunk `rank` first.
// kFast: divide with the geometry's FastDiv (the backward's decodes; the
// forward's measured slower with it, its register budget being tighter).
template <bool kFast = false>
__host__ __device__ inline int query_tile_of(const CpGeom& g, int lt) {
  if (g.rank < 0) return lt;
  return (lt < g.tpc ? g.rank : 2 * g.cp - 1 - g.rank) * g.tpc + (kFast ? g.fd_tpc.mod(lt) : lt % g.tpc);
}
__host__ __device__ inline int query_tiles_per_seq(const CpGeom& g) {
  return g.rank >= 0 ? 2 * g.tpc : 2 * g.cp * g.tpc;
}

// Tile pairs replace head pairs in the forward when the query heads of a KV
// group are odd in number (MHA among them): two heads of a pair would then
// belong to different KV heads and need separate K/V tiles. Uniform batches
// with an even number of tiles per chunk only.
__host__ __device__ inline bool use_tile_pairs(const CpGeom& g) {
  return g.nseq == 0 && (g.hq / g.hkv) % 2 == 1 && g.tpc % 2 == 0;
}

__host__ __device__ inline int fwd_num_units(const CpGeom& g) {
  if (g.tile_pairs && g.tp_block > 0) return (g.b * g.hq + g.tp_block - 1) / g.tp_block * g.tp_slots;
  return g.tile_pairs ? g.hq * (query_tiles(g) / 2) : g.npairs * query_tiles(g);
}

// Tile-pair units in blocks. When the heads' K/V is larger than L2 keeps,
// units of all heads in flight at once read it from DRAM again and again;
// the (sequence, query head) combinations are then cut into blocks spanning
// at most about kv_per_block (sequence, KV head) pairs, numbered block after
// block, each block longest first. A block is padded with empty slots to a
// whole number of double rounds of the snake assignment (2 * grid), so each
// block balances the CTAs' work on its own; a block holds at least 1.5 * grid
// units, so the padding stays a small part of it. kv_per_block <= 0, or
// blocks of at least half the pairs, leave one block (no padding).
__host__ __device__ inline void set_tile_pair_blocks(CpGeom& g, int grid, int kv_per_block) {
  g.tp_block = 0;
  g.tp_slots = 0;
  const int pairs = g.b * g.hkv;
  const int units_per_pair = (g.hq / g.hkv) * (query_tiles_per_seq(g) / 2);
  if (!g.tile_pairs || kv_per_block <= 0) return;
  const int kv_min = (3 * grid + 2 * units_per_pair - 1) / (2 * units_per_pair);
  if (kv_per_block < kv_min) kv_per_block = kv_min;
  if (2 * kv_per_block >= pairs) return;
  const int nblk = (pairs + kv_per_block - 1) / kv_per_block;
  const int kv = (pairs + nblk - 1) / nblk;  // KV pairs per block, evened out
  g.tp_block = kv * (g.hq / g.hkv);
  g.tp_slots = (kv * units_per_pair + 2 * grid - 1) / (2 * grid) * (2 * grid);
}

// The query tile with global tile index gt of unit U's sequence (U.seq set).
template <bool kFast = false>
__host__ __device__ inline void fill_query_tile(const CpGeom& g, FwdUnit& U, int gt) {
  const SeqGeom q = seq_geom(g, U.seq);
  U.bi = g.nseq > 0 ? 0 : U.seq;
  U.tok0 = q.tok0;
  U.lse_t0 = g.nseq > 0 ? q.tok0 : 0;
  U.c = q.c;
  U.tpc = q.tpc;
  if (gt >= 2 * g.cp * U.tpc) {  // beyond this packed sample's tiles
    U.k = U.u = U.half = U.r = U.q_t0 = U.q_valid = 0;
    U.u0 = U.q_t1 = U.q_valid1 = 0;
    U.n = 0;
    return;
  }
  if (kFast && g.nseq == 0) {  // uniform batch: every sequence has g.tpc tiles per chunk
    U.k = g.fd_tpc.div(gt);
    U.u = gt - U.k * U.tpc;
  } else {
    U.k = gt / U.tpc;
    U.u = gt % U.tpc;
  }
  U.half = U.k >= g.cp ? 1 : 0;
  U.r = U.half ? 2 * g.cp - 1 - U.k : U.k;
  U.q_t0 = q_chunk_row(g, U.k, U.c) + U.u * kTile;
  const int rem = U.c - U.u * kTile;
  U.q_valid = rem < kTile ? rem : kTile;
  U.u0 = U.u;
  U.q_t1 = U.q_t0;
  U.q_valid1 = U.q_valid;
  if (g.causal)
    U.n = (U.half ? (2 * g.cp - 1 - U.r) * U.tpc : U.r * U.tpc) + U.u + 1;
  else
    U.n = 2 * g.cp * U.tpc;
}

// Units are numbered in longest-first order: the causal cost of the query
// tile with global tile index gt is gt+1 key tiles, so index 0 is the last
// tile of the sequence. Packed samples come one after another (units of one
// sample share their K/V tiles in L2), each longest tile first.
// kTilePairs is the geometry's tile_pairs as a compile-time constant: the
// kernels are instantiated for one or the other, so that neither carries the
// other's decode (the branch alone measured 6 % slower in the forward).
template <bool kTilePairs>
__host__ __device__ inline FwdUnit fwd_decode_unit_t(const CpGeom& g, int idx) {
  FwdUnit U;
  int gt, pr;
  if constexpr (kTilePairs) {
    // tiles (u - 1, u), u odd, of one head; longest first by tile u (within
    // a block of (sequence, head) combinations, see set_tile_pair_blocks)
    const int per = g.b * g.hq;
    const int qp = query_tiles_per_seq(g) / 2;
    int lp, combo;
    if (g.tp_block > 0) {
      const int blk = idx / g.tp_slots;
      const int i = idx - blk * g.tp_slots;
      const int c0 = blk * g.tp_block;
      const int nc = per - c0 < g.tp_block ? per - c0 : g.tp_block;
      if (i >= nc * qp) {  // an empty slot
        U.seq = U.bi = U.tok0 = U.lse_t0 = U.c = U.tpc = U.h0 = U.h1 = U.g0 = U.g1 = 0;
        U.store1 = false;
        U.k = U.u = U.half = U.r = U.q_t0 = U.q_valid = U.u0 = U.q_t1 = U.q_valid1 = 0;
        U.n = 0;
        return U;
      }
      lp = qp - 1 - i / nc;
      combo = c0 + i % nc;
    } else {
      lp = qp - 1 - idx / per;
      combo = idx % per;
    }
    U.seq = combo / g.hq;
    U.h0 = U.h1 = combo % g.hq;
    U.g0 = U.g1 = U.h0 / (g.hq / g.hkv);
    fill_query_tile(g, U, query_tile_of(g, 2 * lp + 1));
    U.store1 = true;
    U.u0 = U.u - 1;
    U.q_t1 = U.q_t0;
    U.q_valid1 = U.q_valid;
    U.q_t0 = U.q_t1 - kTile;
    U.q_valid = kTile;  // only a chunk's last tile can be ragged
    return U;
  }
  if (g.nseq > 0) {
    int local;
    U.seq = packed_sample_of(g, idx / g.npairs, local);
    gt = (g.tile0[U.seq + 1] - g.tile0[U.seq]) - 1 - local;
    pr = idx % g.npairs;
  } else {
    const int per = g.b * g.npairs;
    gt = query_tile_of(g, query_tiles_per_seq(g) - 1 - idx / per);
    const int rest = idx % per;
    U.seq = rest / g.npairs;
    pr = rest % g.npairs;
  }
  const int G = g.hq / g.hkv;
  U.h0 = 2 * pr;
  U.store1 = (2 * pr + 1) < g.hq;
  U.h1 = U.store1 ? 2 * pr + 1 : 2 * pr;
  U.g0 = U.h0 / G;
  U.g1 = U.h1 / G;
  fill_query_tile(g, U, gt);
  return U;
}

__host__ __device__ inline FwdUnit fwd_decode_unit(const CpGeom& g, int idx) {
  return g.tile_pairs ? fwd_decode_unit_t<true>(g, idx) : fwd_decode_unit_t<false>(g, idx);
}

// dQ work units: one 128-row query tile of one head, longest first: the
// forward's decomposition with one head per unit (h0 == h1), so the
// forward's CP-step key walk (KvWalk) applies as is.
__host__ __device__ inline int dq_num_units(const CpGeom& g) { return g.hq * query_tiles(g); }

__host__ __device__ inline FwdUnit dq_decode_unit(const CpGeom& g, int idx) {
  FwdUnit U;
  int gt;
  if (g.nseq > 0) {
    int local;
    U.seq = packed_sample_of(g, idx / g.hq, local);
    gt = (g.tile0[U.seq + 1] - g.tile0[U.seq]) - 1 - local;
    U.h0 = U.h1 = idx % g.hq;
  } else {
    const int q = g.fd_bhq.div(idx);
    gt = query_tile_of<true>(g, query_tiles_per_seq(g) - 1 - q);
    const int rest = idx - q * (g.b * g.hq);
    U.seq = g.fd_hq.div(rest);
    U.h0 = U.h1 = rest - U.seq * g.hq;
  }
  U.g0 = U.g1 = g.fd_G.div(U.h0);
  U.store1 = false;
  fill_query_tile<true>(g, U, gt);
  return U;
}

// Tile pairs: sub-tile 0 (query tile u - 1) follows the key walk of tile u,
// which has one tile more than its own: the diagonal tile of sub-tile 1,
// whose keys all lie beyond sub-tile 0's rows. fwd_dead_pos gives that
// tile's position in the walk (-1 when there is none: head pairs, sub-tile 1,
// no causal mask, or a single-step walk of a later step). With the causal
// mask the walk's diagonal run ends step 0, at position (half ? tpc : 0) + u;
// `step` is the step a single-step walk covers (-1: the whole walk).
__host__ __device__ inline int fwd_dead_pos(const CpGeom& g, const FwdUnit& U, int sub, int step) {
  if (sub != 0 || U.u0 == U.u || !g.causal || step > 0) return -1;
  return (U.half ? U.tpc : 0) + U.u;
}

// The mask of walk position j for a sub-tile with dead position jd: `dead`
// (no key counts), else `diag` (each row sees the keys up to its own
// position): the tile before the dead one is the sub-tile's own diagonal.
__host__ __device__ inline void fwd_pos_mask(int jd, int j, bool walk_diag, bool& diag, bool& dead) {
  dead = j == jd;
  diag = jd >= 0 ? j == jd - 1 : walk_diag;
}

// Static "snake" assignment of units to persistent CTAs: round q gives CTA
// `bid` unit q*grid + bid on even rounds and q*grid + grid-1-bid on odd
// rounds, pairing long units with short ones.
__host__ __device__ inline int snake_unit(int round, int bid, int grid) {
  return (round & 1) ? round * grid + (grid - 1 - bid) : round * grid + bid;
}

// Walks a unit's key tiles in CP-step order (all steps, or one step only).
struct KvWalk {
  int cp, r, half, k, u, tpc, causal;
  int step, seg, v;
  int last;  // last step walked

  __host__ __device__ KvWalk(const CpGeom& g, const FwdUnit& U)
      : cp(g.cp), r(U.r), half(U.half), k(U.k), u(U.u), tpc(U.tpc), causal(g.causal), step(0), seg(0), v(0),
        last(g.cp - 1) {}

  // Restrict the walk to the key tiles of CP step `st`.
  __host__ __device__ void only_step(int st) {
    step = st;
    last = st;
    seg = 0;
    v = 0;
  }

  // Number of key tiles the unit visits at CP step `st`.
  __host__ __device__ int step_tiles(int st) const {
    int n = 0, ch, nt, dg;
    for (int sg = 0; segment(st, sg, ch, nt, dg); ++sg) n += nt;
    return n;
  }

  // Segment `sg` of step `st`: a run of tiles [0, ntiles) of chunk `chunk`;
  // `diag` is the masked tile index in it, or -1.
  __host__ __device__ bool segment(int st, int sg, int& chunk, int& ntiles, int& diag) const {
    diag = -1;
    ntiles = tpc;
    if (!causal) {
      if (sg > 1) return false;
      const int j = ((r - st) % cp + cp) % cp;
      chunk = sg == 0 ? j : 2 * cp - 1 - j;
      return true;
    }
    if (st == 0) {
      if (half == 0) {
        if (sg > 0) return false;
        chunk = r;
        ntiles = u + 1;
        diag = u;
        return true;
      }
      if (sg == 0) {
        chunk = r;
        return true;
      }
      if (sg == 1) {
        chunk = k;
        ntiles = u + 1;
        diag = u;
        return true;
      }
      return false;
    }
    if (st <= r) {
      if (sg > 0) return false;
      chunk = r - st;
      return true;
    }
    if (half == 0) return false;
    const int j = r - st + cp;
    if (sg == 0) {
      chunk = j;
      return true;
    }
    if (sg == 1) {
      chunk = 2 * cp - 1 - j;
      return true;
    }
    return false;
  }

  __host__ __device__ bool next(int& chunk, int& tile, bool& is_diag) {
    while (step <= last) {
      int ch, nt, dg;
      if (segment(step, seg, ch, nt, dg)) {
        if (v < nt) {
          chunk = ch;
          tile = v;
          is_diag = (v == dg);
          ++v;
          return true;
        }
        ++seg;
        v = 0;
        continue;
      }
      ++step;
      seg = 0;
      v = 0;
    }
    return false;
  }
};


// ---------------------------------------------------------------- backward
// A backward work unit is one 128-key tile (chunk kc, tile v) of one KV head
// for one batch element. It visits every (query tile, query head of the
// group) block that sees its keys. By the forward's CP rules those blocks
// are: the rank's own step-0 block (the one diagonal tile, masked), and every
// query tile of a later position (steps 1..cp-1, unmasked) -- i.e. all query
// tiles at or after the key tile in global order. The unit walks them from
// the end of the sequence down to its own diagonal tile: every running unit
// then starts at the same query tiles and moves down at the same pace, so
// the dQ rows being accumulated (and the Q/dO tiles being read) are shared
// by the CTAs in flight and stay in L2. dK/dV of the tile accumulate on chip
// over all its blocks. In the rank-local form the units are still every key
// tile of the sequence, but only the rank's own query tiles are visited: the
// result is the rank's share of every key tile's dK/dV (zero for a tile no
// query of the rank sees).
struct BwdUnit {
  int bi, g;      // batch element (0 for packed samples), KV head
  int seq;        // batch element or packed sample
  int tok0;       // its first token row
  int c, tpc;     // its chunk length and tiles per chunk
  int kc, v;      // key chunk and tile within it
  int gt;         // global tile index of the key tile: kc * tpc + v
  int k_t0;       // first row of the key tile relative to its sequence's first row
  int k_valid;    // keys of the tile inside the chunk (0 for a tile a shorter packed sample does not have)
  int nq;         // number of query tiles that see the tile (the rank's own in the rank-local form)
  int items;      // nq * (hq / hkv); 0 when no query sees the tile
};

// Query tiles of chunk `chunk` at or after global tile gt (tpc per chunk).
__host__ __device__ inline int tiles_from(int chunk, int tpc, int gt) {
  const int n = (chunk + 1) * tpc - gt;
  return n < 0 ? 0 : (n > tpc ? tpc : n);
}

__host__ __device__ inline int bwd_num_units(const CpGeom& g) { return g.hkv * all_tiles(g); }

// Longest-first: the key tile with global tile index gt is seen by ntile-gt
// query tiles (causal), so unit 0 is the first tile of the sequence.
__host__ __device__ inline BwdUnit bwd_decode_unit(const CpGeom& g, int idx) {
  BwdUnit U;
  int gt;
  if (g.nseq > 0) {
    U.seq = packed_sample_of(g, idx / g.hkv, gt);
    U.g = idx % g.hkv;
  } else {
    gt = g.fd_bhkv.div(idx);
    const int rest = idx - gt * (g.b * g.hkv);
    U.seq = g.fd_hkv.div(rest);
    U.g = rest - U.seq * g.hkv;
  }
  U.bi = g.nseq > 0 ? 0 : U.seq;
  const SeqGeom q = seq_geom(g, U.seq);
  U.tok0 = q.tok0;
  U.c = q.c;
  U.tpc = q.tpc;
  U.gt = gt;
  const int ntile = 2 * g.cp * U.tpc;
  if (gt >= ntile) {  // beyond this packed sample's tiles
    U.kc = U.v = U.k_t0 = U.k_valid = U.nq = U.items = 0;
    return U;
  }
  if (g.nseq == 0) {
    U.kc = g.fd_tpc.div(gt);
    U.v = gt - U.kc * U.tpc;
  } else {
    U.kc = gt / U.tpc;
    U.v = gt % U.tpc;
  }
  U.k_t0 = kv_chunk_row(g, U.kc, U.c) + U.v * kTile;
  const int rem = U.c - U.v * kTile;
  U.k_valid = rem < kTile ? rem : kTile;
  if (g.rank >= 0)
    U.nq = g.causal ? tiles_from(g.rank, U.tpc, gt) + tiles_from(2 * g.cp - 1 - g.rank, U.tpc, gt) : 2 * U.tpc;
  else
    U.nq = g.causal ? ntile - gt : ntile;
  U.items = U.nq * (g.hq / g.hkv);
  return U;
}

// Walks the query tiles of a backward unit, last tile first (in the
// rank-local form only the rank's own tiles: chunk 2cp-1-rank, then chunk
// rank, each from its end).
// The position is kept as (chunk, tile) and stepped down one tile at a time
// (no division per tile).
struct QWalk {
  int tpc, lo, gt_k, causal, low_chunk, left;
  int ch, t;  // the next tile: chunk and tile within it

  __host__ __device__ QWalk(const CpGeom& g, const BwdUnit& U)
      : tpc(U.tpc), lo(g.causal ? U.gt : 0), gt_k(U.gt), causal(g.causal),
        low_chunk(g.rank >= 0 ? g.rank : -1), left(g.rank >= 0 ? 2 * U.tpc : 2 * g.cp * U.tpc),
        ch(g.rank >= 0 ? 2 * g.cp - 1 - g.rank : 2 * g.cp - 1), t(U.tpc - 1) {}

  __host__ __device__ bool next(int& chunk, int& tile, bool& is_diag) {
    if (left <= 0) return false;
    const int gt = ch * tpc + t;
    if (gt < lo) return false;  // tiles come in decreasing global order
    chunk = ch;
    tile = t;
    is_diag = causal && gt == gt_k;
    --left;
    if (--t < 0) {  // on to the chunk before: the previous one, or the rank's lower chunk
      t = tpc - 1;
      ch = low_chunk >= 0 ? low_chunk : ch - 1;
    }
    return true;
  }
};

}  // namespace cpattn
