// Context-parallel work decomposition shared by the kernels.
//
// Zigzag split ("大模型面试宝典 · Megatron-LM 篇", 3.4; "超大规模集群下大语言模型训练
// 实操指南", CP 与其他技术结合): 2*cp chunks of c tokens, virtual rank r owns
// chunks r and 2cp-1-r. Each chunk is cut into tpc = ceil(c/128) tiles that
// start at the chunk's first token (the last one may be ragged).
//
// A forward work unit is one 128-row query tile of one chunk, for a pair of
// query heads (two sub-tiles that walk the same key tiles), for one batch
// element. Its key tiles are visited in the order of the rank's CP steps:
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

struct CpGeom {
  int b, s, hq, hkv, cp, causal;
  int c;       // chunk length
  int tpc;     // tiles per chunk
  int npairs;  // query-head pairs per batch element: ceil(hq / 2)
};

struct FwdUnit {
  int bi;        // batch element
  int h0, h1;    // query heads of the two sub-tiles (h1 == h0 for an odd tail)
  int g0, g1;    // their KV heads
  bool store1;   // sub-tile 1 is a distinct head (its output is stored)
  int k;         // global chunk index of the query tile
  int u;         // tile index within the chunk
  int r, half;   // owning virtual rank and which of its two chunks
  int q_t0;      // first token of the query tile (within the sequence)
  int q_valid;   // rows of the tile inside the chunk
  int n;         // number of key tiles the unit visits
};

__host__ __device__ inline int fwd_num_units(const CpGeom& g) { return g.b * g.npairs * 2 * g.cp * g.tpc; }

// Units are numbered in longest-first order: the causal cost of the query
// tile with global tile index gt is gt+1 key tiles, so index 0 is the last
// tile of the sequence.
__host__ __device__ inline FwdUnit fwd_decode_unit(const CpGeom& g, int idx) {
  FwdUnit U;
  const int per = g.b * g.npairs;
  const int ntile = 2 * g.cp * g.tpc;
  const int gt = (ntile - 1) - idx / per;
  const int rest = idx % per;
  U.bi = rest / g.npairs;
  const int pr = rest % g.npairs;
  const int G = g.hq / g.hkv;
  U.h0 = 2 * pr;
  U.store1 = (2 * pr + 1) < g.hq;
  U.h1 = U.store1 ? 2 * pr + 1 : 2 * pr;
  U.g0 = U.h0 / G;
  U.g1 = U.h1 / G;
  U.k = gt / g.tpc;
  U.u = gt % g.tpc;
  U.half = U.k >= g.cp ? 1 : 0;
  U.r = U.half ? 2 * g.cp - 1 - U.k : U.k;
  U.q_t0 = U.k * g.c + U.u * kTile;
  const int rem = g.c - U.u * kTile;
  U.q_valid = rem < kTile ? rem : kTile;
  if (g.causal)
    U.n = (U.half ? (2 * g.cp - 1 - U.r) * g.tpc : U.r * g.tpc) + U.u + 1;
  else
    U.n = 2 * g.cp * g.tpc;
  return U;
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
      : cp(g.cp), r(U.r), half(U.half), k(U.k), u(U.u), tpc(g.tpc), causal(g.causal), step(0), seg(0), v(0),
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
// over all its blocks.
struct BwdUnit {
  int bi, g;      // batch element, KV head
  int kc, v;      // key chunk and tile within it
  int gt;         // global tile index of the key tile: kc * tpc + v
  int k_t0;       // first key token
  int k_valid;    // keys of the tile inside the chunk
  int nq;         // number of query tiles that see the tile
  int items;      // nq * (hq / hkv)
};

__host__ __device__ inline int bwd_num_units(const CpGeom& g) { return g.b * g.hkv * 2 * g.cp * g.tpc; }

// Longest-first: the key tile with global tile index gt is seen by ntile-gt
// query tiles (causal), so unit 0 is the first tile of the sequence.
__host__ __device__ inline BwdUnit bwd_decode_unit(const CpGeom& g, int idx) {
  BwdUnit U;
  const int per = g.b * g.hkv;
  const int ntile = 2 * g.cp * g.tpc;
  const int gt = idx / per;
  const int rest = idx % per;
  U.bi = rest / g.hkv;
  U.g = rest % g.hkv;
  U.gt = gt;
  U.kc = gt / g.tpc;
  U.v = gt % g.tpc;
  U.k_t0 = U.kc * g.c + U.v * kTile;
  const int rem = g.c - U.v * kTile;
  U.k_valid = rem < kTile ? rem : kTile;
  U.nq = g.causal ? ntile - gt : ntile;
  U.items = U.nq * (g.hq / g.hkv);
  return U;
}

// Walks the query tiles of a backward unit, last tile first.
struct QWalk {
  int tpc, lo, gt_k, causal, gt;

  __host__ __device__ QWalk(const CpGeom& g, const BwdUnit& U)
      : tpc(g.tpc), lo(g.causal ? U.gt : 0), gt_k(U.gt), causal(g.causal), gt(2 * g.cp * g.tpc - 1) {}

  __host__ __device__ bool next(int& chunk, int& tile, bool& is_diag) {
    if (gt < lo) return false;
    chunk = gt / tpc;
    tile = gt % tpc;
    is_diag = causal && gt == gt_k;
    --gt;
    return true;
  }
};

}  // namespace cpattn
