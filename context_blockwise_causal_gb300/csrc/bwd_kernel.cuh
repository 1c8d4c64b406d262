// Backward kernels for context-parallel causal attention.
//
//   cpattn_bwd_pre_kernel   per query row: D = rowsum(dO * O) and L*log2(e),
//                           into tile-padded vectors.            (HBM-bound)
//   cpattn_bwd_dkdv_kernel  key-tile-stationary: per 128-key tile of a KV
//                           head, over every (query tile, query head of the
//                           group) block that sees it:
//                             S^T = K Q^T, dP^T = V dO^T            (TMEM)
//                             P^T = 2^(S^T*scale*log2e - L*log2e)
//                             dS^T = P^T (dP^T - D)                (TMEM)
//                             dV += P^T dO, dK += dS^T Q           (TMEM)
//                           dK/dV stay on chip across all blocks and are
//                           written once (dK scaled by the softmax scale).
//   cpattn_bwd_dq_kernel    query-tile-stationary: per 128-query tile of one
//                           head, over the key tiles it sees in the order of
//                           its rank's CP steps (the forward's walk):
//                             S = Q K^T, dP = dO V^T               (TMEM)
//                             dS = P (dP - D)                      (TMEM)
//                             dQ += dS K                           (TMEM)
//                           dq written once (scaled by the softmax scale).
// Splitting dQ from dK/dV costs two extra matmuls per block (S and dP are
// formed twice) but needs no atomics and no fp32 accumulator in device
// memory, and lets each kernel keep its TMEM within 512 columns.
//
// The gradient formulas are those of softmax attention (the derivative of
// the forward defined in include/cpattn.h); the blocks and masks are those of
// the forward's CP steps ("大模型面试宝典 · Megatron-LM 篇", 3.4).
#pragma once
#include <cuda_bf16.h>

#include "cp_schedule.cuh"
#include "ptx.cuh"

namespace cpattn {

constexpr int kBwdThreads = 320;

struct BwdArgs {
  CpGeom g;
  int ntp;  // tile-padded row count per (batch, head): 2*cp*tpc*128
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  int64_t lse_stride;  // row stride of lse per (batch, head): s, or a packed tensor's total
  float* lvec;  // [b, hq, ntp]: lse * log2(e)
  float* dvec;  // [b, hq, ntp]: rowsum(dO * O)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float scale_log2;  // log2(e) * the softmax scale
  float scale;       // the softmax scale (1 / sqrt(d) by default)
  unsigned int* status;
  // time limit of the producers' waits for free buffers: kWaitLimitNs, or a
  // short one in the abort self-test (cpattn_selftest_abort)
  uint64_t producer_limit_ns;
  // extents for the checked build (bounds_ok): rows of the query-side and
  // key/value-side tensors, floats of lse and of each row vector
  int64_t q_rows, kv_rows, lse_len, vec_len;
};

enum BwdStatusBits : unsigned int {
  kStatusBwdProducer = 1u << 8,
  kStatusBwdMma = 1u << 9,
  kStatusBwdSoftmax = 1u << 10,
  kStatusBwdSmemAlign = 1u << 11,
  kStatusBwdDrain = 1u << 12,  // copies or MMAs still in flight after the time limit
};

// Row `row` of tile `tile` of chunk `chunk` of sequence `seq` (tpc tiles per
// chunk) for query head `h` in the tile-padded L/D vectors [sequences, hq,
// ntp] (only the rank's own tiles in the rank-local form).
__device__ __forceinline__ int64_t ld_pos(const CpGeom& g, int ntp, int seq, int h, int chunk, int tile, int tpc,
                                          int row) {
  return int64_t(seq * g.hq + h) * ntp + ld_tile(g, chunk, tile, tpc) * kTile + row;
}

// ---------------------------------------------------------------- preprocess
// A warp takes 32 consecutive rows, one per lane for the index arithmetic and
// the writes. The loads are cooperative: each load instruction reads whole
// rows (D/8 lanes x 16 bytes per row, so 32*16/(2D) rows per instruction),
// the partial dot products are summed by xor shuffles inside each row's lane
// group, and the lane that owns the row keeps its sum.
template <int D>
__global__ void __launch_bounds__(256) cpattn_bwd_pre_kernel(const BwdArgs a) {
  constexpr int kLanesPerRow = D / 8;              // 16 (d = 128) or 8 (d = 64)
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;  // rows one warp-wide load covers
  constexpr int kLoads = 32 / kRowsPerLoad;        // loads for the warp's 32 rows
  constexpr int kBatch = 4;                        // loads in flight per lane
  const CpGeom& g = a.g;
  const int srows = q_seq_rows(g);  // rows of a sequence in o / dout
  const int64_t nrows = int64_t(g.b) * srows * g.hq;
  if (!bounds_ok(nrows <= a.q_rows * g.hq, a.status)) return;  // o and dout hold q_rows rows
  const int lane = threadIdx.x & 31;
  const int li = lane % kLanesPerRow;
  const int lr = lane / kLanesPerRow;  // which of a load's rows this lane reads
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 32; r0 < nrows; r0 += nwarps * 32) {
    float mine = 0.f;
#pragma unroll
    for (int l0 = 0; l0 < kLoads; l0 += kBatch) {
      uint4 x[kBatch], y[kBatch];
#pragma unroll
      for (int l = 0; l < kBatch; ++l) {
        const int64_t row = r0 + (l0 + l) * kRowsPerLoad + lr;
        if (row < nrows) {
          x[l] = reinterpret_cast<const uint4*>(a.o + row * D)[li];
          y[l] = reinterpret_cast<const uint4*>(a.dout + row * D)[li];
        } else {
          x[l] = make_uint4(0u, 0u, 0u, 0u);
          y[l] = x[l];
        }
      }
#pragma unroll
      for (int l = 0; l < kBatch; ++l) {
        const uint32_t xs[4] = {x[l].x, x[l].y, x[l].z, x[l].w}, ys[4] = {y[l].x, y[l].y, y[l].z, y[l].w};
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc);
          acc = fmaf(__uint_as_float(xs[k] & 0xffff0000u), __uint_as_float(ys[k] & 0xffff0000u), acc);
        }
#pragma unroll
        for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        // rows (l0 + l) * kRowsPerLoad + j, j < kRowsPerLoad: lane owning row
        // (l0 + l) * kRowsPerLoad + j takes group j's sum
        const int first = (l0 + l) * kRowsPerLoad;
        const float v = __shfl_sync(0xffffffffu, acc, ((lane - first) & (kRowsPerLoad - 1)) * kLanesPerRow);
        if (lane >= first && lane < first + kRowsPerLoad) mine = v;
      }
    }
    const int64_t idx = r0 + lane;
    if (idx >= nrows) continue;
    const float acc = mine;
    const int h = int(idx % g.hq);
    const int64_t bt = idx / g.hq;
    const int t = int(bt % srows);
    const int bi = int(bt / srows);
    // the row's sequence (batch element, or the packed sample holding t)
    int seq = bi, tl = t;
    if (g.nseq > 0) {
      int lo = 0, hi = g.nseq;  // cu[lo] <= t < cu[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.cu[mid] <= t) lo = mid; else hi = mid;
      }
      seq = lo;
      tl = t - g.cu[lo];
    }
    const SeqGeom q = seq_geom(g, seq);
    int chunk = tl / q.c;  // rank-local form: 0 or 1, the rank's first or second chunk
    const int in = tl - chunk * q.c;
    if (g.rank >= 0) chunk = chunk ? 2 * g.cp - 1 - g.rank : g.rank;
    const int64_t pos = ld_pos(g, a.ntp, seq, h, chunk, in / kTile, q.tpc, in % kTile);
    const int64_t li = (int64_t(bi) * g.hq + h) * a.lse_stride + t;
    if (!bounds_ok(pos >= 0 && pos < a.vec_len && li < a.lse_len && idx < a.q_rows * g.hq, a.status)) continue;
    a.dvec[pos] = acc;
    a.lvec[pos] = a.lse[li] * 1.4426950408889634f;
  }
}

// Column of a packed bf16 operand tile for K-step kk (16 elements): the two
// 64-element halves sit at columns [0,32) and [64,96) of their 128-column
// region, each written by the warp that read the fp32 values there.
__device__ __forceinline__ uint32_t half_split_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

// Bits [lo, hi) of a 32-bit mask (lo, hi clipped to [0, 32]).
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  lo = lo < 0 ? 0 : (lo > 32 ? 32 : lo);
  hi = hi < 0 ? 0 : (hi > 32 ? 32 : hi);
  if (hi <= lo) return 0u;
  const uint32_t upto_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
  const uint32_t below_lo = (1u << lo) - 1u;
  return upto_hi & ~below_lo;
}

// ================================================================ dK / dV
// P for one warp's 32 keys x 32 queries held in 16x256b fragments (see
// tmem_ld16x256b_2x2): element 16u + 4r + 2e + j of rs is key row 16u + 8e +
// t/4 and query 8r + 2(t%4) + j. The thread needs L*log2e for only its 8
// queries (lv[r]: queries 8r + 2(t%4) + {0,1} as .x, .y). Output register
// 8u + 2r + e holds the bf16 pair of queries 8r + 2(t%4) + {0,1} for key row
// 16u + 8e + t/4: the packed column 4r + t%4 of the 16x128b fragment (see
// tmem_st16x128b_2x2). When `masked`, bit c of valid[2u + e] keeps query c
// of that key row; masked entries are selected to zero.
template <bool kMasked>
__device__ __forceinline__ void softmax_p_frag(const uint32_t (&rs)[32], float sl2, const float2 (&lv)[4],
                                               const uint32_t (&valid)[4], int c4, uint32_t (&pp)[16]) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 16 * u + 4 * r + 2 * e;
        const int o = 8 * u + 2 * r + e;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[i]), __uint_as_float(rs[i + 1])), sl2x2,
                         f2_pack(-lv[r].x, -lv[r].y)),
                  x0, x1);
        pp[o] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
        if constexpr (kMasked) {
          const uint32_t bits = valid[2 * u + e] >> (8 * r + 2 * c4);
          pp[o] &= (bits & 1u ? 0x0000ffffu : 0u) | (bits & 2u ? 0xffff0000u : 0u);
        }
      }
}

// dS = P (dP - D) for the same fragment: P as the packed bf16 pairs from
// softmax_p_frag, dP as raw fp32 bits in the 16x256b layout, D per query as
// lv above. Output in the packed 16x128b layout; masked entries are selected
// to zero (their dP - D may be anything).
template <bool kMasked>
__device__ __forceinline__ void ds_frag(const uint32_t (&pp)[16], const uint32_t (&rp)[32], const float2 (&dv)[4],
                                        const uint32_t (&valid)[4], int c4, uint32_t (&pd)[16]) {
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 16 * u + 4 * r + 2 * e;
        const int o = 8 * u + 2 * r + e;
        const float p0 = __uint_as_float(pp[o] << 16), p1 = __uint_as_float(pp[o] & 0xffff0000u);
        float g0, g1;
        f2_unpack(f2_mul(f2_pack(p0, p1),
                         f2_sub(f2_pack(__uint_as_float(rp[i]), __uint_as_float(rp[i + 1])), f2_pack(dv[r].x, dv[r].y))),
                  g0, g1);
        pd[o] = pack_bf16x2(g0, g1);
        if constexpr (kMasked) {
          const uint32_t bits = valid[2 * u + e] >> (8 * r + 2 * c4);
          pd[o] &= (bits & 1u ? 0x0000ffffu : 0u) | (bits & 2u ? 0xffff0000u : 0u);
        }
      }
}

template <int D>
struct DkdvCfg {
  static constexpr int kTileBytes = kTile * D * 2;  // 128 x D bf16
  static constexpr int kQStages = 3;                // Q tiles in flight
  static constexpr int kOStages = 2;                // dO tiles (with L, D) in flight
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffdO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffLD = kOffdO + kOStages * kTileBytes;
  static constexpr int kLDBytes = 2 * kTile * 4;  // L[128], D[128] fp32 per dO stage
  static constexpr int kOffBar = kOffLD + kOStages * kLDBytes;
  // kv_full kv_empty q_full[3] q_empty[3] o_full[2] o_empty[2]
  // s_full s_free dp_full p_full dkv_full dkv_empty drain pt_full
  static constexpr int kNumBars = 2 + 2 * kQStages + 2 * kOStages + 8;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kLayoutBytes = kOffMisc + 16;
  // The d=128 layout leaves no room for re-alignment: the dynamic shared
  // memory base must already be 1024-byte aligned (checked at run time).
  static constexpr bool kNeedAlignedBase = (kLayoutBytes + 1024 > 232448);
  static constexpr int kSmemBytes = kNeedAlignedBase ? kLayoutBytes : kLayoutBytes + 1024;
  static_assert(kLayoutBytes <= 232448, "dK/dV shared memory layout too large");
  // TMEM: S^T [0,128), dP^T [128,256) (later P^T | dS^T), dV, dK
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 256 + D;
};

// Key-tile-stationary dK/dV. One CTA per SM, 10 warps:
//   warps 0-7  element-wise; warp w covers TMEM lanes 32*(w%4).. (key rows)
//              and queries 64*(w/4) .. +63 of each block (D/2 columns of
//              dK/dV at the end)
//   warp 8     TMA producer (K/V per unit; Q in 3 stages; dO, L, D in 2)
//   warp 9     TMEM owner and MMA issuer (whole warp, elect.sync)
// Per (query tile, head) block i, all MMAs have N = 128 (or D):
//   S^T(i) = K Q^T -> [0,128)       dP^T(i) = V dO^T -> [128,256)
//   dK += dS^T(i) Q,  dV += P^T(i) dO   (A operands packed in [128,256))
// The element-wise warps read S^T(i) and release its columns at once
// (s_free), compute P in registers, then read dP^T(i) and write packed bf16
// P^T over it (each warp inside the columns it read: P^T to [128+64h, +32))
// and release it (pt_full), then form dS^T into [128+64h+32, +32) (p_full).
// So the tensor core runs S^T(i+1) while the warps finish block i, dV(i)
// while they form dS(i), and the exponentials of block i overlap dK/dV(i-1)
// and dP^T(i):
//   tensor core:  S^T(i+1) | dV(i) dK(i) | dP^T(i+1) | S^T(i+2) | ...
//   warps:        P(i+1) from S^T(i+1) ..............| dS(i+1)  |
// Units walk their query tiles from the end of the sequence down (QWalk), so
// the CTAs in flight read the same Q/dO tiles from L2.
template <int D, bool kShortWaits = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    cpattn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                           const BwdArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if constexpr (!C::kNeedAlignedBase)
    smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBwdSmemAlign);
    return;
  }
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sdO = smem + C::kOffdO;
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = q_full + C::kQStages;
  uint64_t* o_full = q_empty + C::kQStages;
  uint64_t* o_empty = o_full + C::kOStages;
  uint64_t* s_full = o_empty + C::kOStages;
  uint64_t* s_free = s_full + 1;
  uint64_t* dp_full = s_full + 2;
  uint64_t* p_full = s_full + 3;
  uint64_t* dkv_full = s_full + 4;
  uint64_t* dkv_empty = s_full + 5;
  uint64_t* drain = s_full + 6;
  uint64_t* pt_full = s_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const CpGeom& g = a.g;
  const int G = g.hq / g.hkv;
  const int num_units = bwd_num_units(g);
  const int grid = gridDim.x;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int i = 0; i < C::kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < C::kOStages; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 8);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 8);
    mbar_init(drain, 1);
    mbar_init(pt_full, 8);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmdo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the waits for free stages: a short limit only in the abort self-test
      const uint64_t plimit = kShortWaits ? a.producer_limit_ns : kWaitLimitNs;
      bool ok = true;
      uint32_t item = 0;  // blocks loaded so far (their dO tiles issued)
      uint32_t nq = 0;    // Q tiles issued: item, or item + 1 when a dO wait gave up
      uint32_t nkv = 0;   // K/V tile pairs issued
      int ul = 0;
      auto load_item = [&](const BwdUnit& U, int chunk, int tile, int h) -> bool {
        const int row = U.tok0 + q_chunk_row(g, chunk, U.c) + tile * kTile;
        bounds_ok(row >= 0 && row < a.q_rows && h >= 0 && h < g.hq, a.status);
        const uint32_t qs = item % C::kQStages, os = item % C::kOStages;
        if (item >= C::kQStages &&
            !mbar_wait_lean(&q_empty[qs], ((item / C::kQStages) - 1) & 1, abort_flag, plimit))
          return false;
        mbar_arrive_expect_tx(&q_full[qs], C::kTileBytes);
        for (int x = 0; x < D; x += 64)
          tma_load_3d(sQ + qs * C::kTileBytes + (x / 64) * (kTile * 128), &tmq, &q_full[qs], x, h, row);
        ++nq;
        if (item >= C::kOStages &&
            !mbar_wait_lean(&o_empty[os], ((item / C::kOStages) - 1) & 1, abort_flag, plimit))
          return false;
        mbar_arrive_expect_tx(&o_full[os], C::kTileBytes + C::kLDBytes);
        for (int x = 0; x < D; x += 64)
          tma_load_3d(sdO + os * C::kTileBytes + (x / 64) * (kTile * 128), &tmdo, &o_full[os], x, h, row);
        int64_t pos = ld_pos(g, a.ntp, U.seq, h, chunk, tile, U.tpc, 0);
        if (!bounds_ok(pos >= 0 && pos + kTile <= a.vec_len, a.status)) pos = 0;  // stays inside the vectors
        bulk_load(reinterpret_cast<uint8_t*>(sLD) + os * C::kLDBytes, a.lvec + pos, kTile * 4, &o_full[os]);
        bulk_load(reinterpret_cast<uint8_t*>(sLD) + os * C::kLDBytes + kTile * 4, a.dvec + pos, kTile * 4,
                  &o_full[os]);
        ++item;
        return true;
      };
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const BwdUnit U = bwd_decode_unit(g, idx);
        if (U.items == 0) continue;  // a tile a shorter packed sample does not have
        QWalk w(g, U);
        int chunk, tile;
        bool dg;
        bool first = true;
        while (ok && w.next(chunk, tile, dg)) {
          for (int h = U.g * G; h < (U.g + 1) * G && ok; ++h) {
            ok = load_item(U, chunk, tile, h);
            if (ok && first) {
              // K/V of this unit, once its first block is on its way.
              first = false;
              if (ul > 0 && !(ok = mbar_wait_lean(kv_empty, (ul - 1) & 1, abort_flag, plimit))) break;
              mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
              const int krow = U.tok0 + U.k_t0;
              bounds_ok(krow >= 0 && krow < a.kv_rows && U.g < g.hkv, a.status);
              for (int x = 0; x < D; x += 64) {
                tma_load_3d(sK + (x / 64) * (kTile * 128), &tmk, kv_full, x, U.g, krow);
                tma_load_3d(sV + (x / 64) * (kTile * 128), &tmv, kv_full, x, U.g, krow);
              }
              ++nkv;
            }
          }
        }
        ++ul;
      }
      if (!ok) atomicOr(a.status, kStatusBwdProducer);
      // Let every copy still in flight land before the CTA can exit (older
      // ones landed before their stage was handed back). These waits do not
      // stop on the abort flag: the copies complete regardless.
      bool drained = true;
      for (uint32_t i = nq > C::kQStages ? nq - C::kQStages : 0; i < nq; ++i)
        drained &= mbar_wait_drain(&q_full[i % C::kQStages], (i / C::kQStages) & 1, kWaitLimitNs);
      for (uint32_t i = item > C::kOStages ? item - C::kOStages : 0; i < item; ++i)
        drained &= mbar_wait_drain(&o_full[i % C::kOStages], (i / C::kOStages) & 1, kWaitLimitNs);
      if (nkv > 0) drained &= mbar_wait_drain(kv_full, (nkv - 1) & 1, kWaitLimitNs);
      if (!drained) atomicOr(a.status, kStatusBwdDrain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs this role; elect.sync picks the issuing lane)
    {
      constexpr uint32_t idS = make_idesc_bf16(kTile, kTile, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = make_idesc_bf16(kTile, D, false, true);      // dV, dK
      const uint64_t dK_km = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV_km = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQ_km = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t ddO_km = make_sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t dQ_mn = make_sdesc_sw128(smem_u32(sQ), 16384, 1024);
      const uint64_t ddO_mn = make_sdesc_sw128(smem_u32(sdO), 16384, 1024);
      const uint32_t tS = tbase + C::kColS, tdP = tbase + C::kColdP;
      const uint32_t tdV = tbase + C::kColdV, tdK = tbase + C::kColdK;
      auto issue_s = [&](uint32_t i) {  // S^T(i) = K Q^T
        const uint64_t ro = ((i % C::kQStages) * C::kTileBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
          umma_ss_w(tS, dK_km + off, dQ_km + ro + off, idS, kk > 0);
        }
      };
      auto issue_dp = [&](uint32_t i) {  // dP^T(i) = V dO^T
        const uint64_t ro = ((i % C::kOStages) * C::kTileBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
          umma_ss_w(tdP, dV_km + off, ddO_km + ro + off, idS, kk > 0);
        }
      };
      bool ok = true;
      uint32_t i0 = 0;  // blocks before this unit
      int ul = 0;
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const BwdUnit U = bwd_decode_unit(g, idx);
        if (U.items == 0) continue;  // a tile a shorter packed sample does not have
        const int n = U.items;
        // prologue: S^T and dP^T of the unit's first block. The S^T columns
        // are free once the element-wise warps have read the previous S^T;
        // the dP^T columns once the previous dK/dV MMAs (issued) read them.
        ok = mbar_wait_warp_lean(kv_full, ul & 1, abort_flag, kWaitLimitNs) &&
             mbar_wait_warp_lean(&q_full[i0 % C::kQStages], (i0 / C::kQStages) & 1, abort_flag, kWaitLimitNs) &&
             (i0 == 0 || mbar_wait_warp_lean(s_free, (i0 - 1) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        issue_s(i0);
        umma_commit_w(s_full);
        if (!(ok = mbar_wait_warp_lean(&o_full[i0 % C::kOStages], (i0 / C::kOStages) & 1, abort_flag, kWaitLimitNs)))
          break;
        issue_dp(i0);
        umma_commit_w(dp_full);
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t i = i0 + j;
          if (j + 1 < n) {
            // S^T(i+1) as soon as S^T(i) has been read
            ok = mbar_wait_warp_lean(s_free, i & 1, abort_flag, kWaitLimitNs) &&
                 mbar_wait_warp_lean(&q_full[(i + 1) % C::kQStages], ((i + 1) / C::kQStages) & 1, abort_flag,
                                kWaitLimitNs);
            if (!ok) break;
            issue_s(i + 1);
            umma_commit_w(s_full);
          }
          ok = mbar_wait_warp_lean(pt_full, i & 1, abort_flag, kWaitLimitNs) &&
               (j > 0 || ul == 0 || mbar_wait_warp_lean(dkv_empty, (ul - 1) & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          // dV += P^T dO as soon as P^T is in TMEM, then dK += dS^T Q
          const uint64_t rq = ((i % C::kQStages) * C::kTileBytes) >> 4;
          const uint64_t ro = ((i % C::kOStages) * C::kTileBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ts_w(tdV, tdP + half_split_col(kk), ddO_mn + ro + ((kk * 2048) >> 4), idKV,
                      (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&o_empty[i % C::kOStages]);
          if (!(ok = mbar_wait_warp_lean(p_full, i & 1, abort_flag, kWaitLimitNs))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ts_w(tdK, tdP + 32 + half_split_col(kk), dQ_mn + rq + ((kk * 2048) >> 4), idKV,
                      (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&q_empty[i % C::kQStages]);
          if (j + 1 < n) {
            // dP^T(i+1) over P^T/dS^T(i), which the MMAs just issued read first
            if (!(ok = mbar_wait_warp_lean(&o_full[(i + 1) % C::kOStages], ((i + 1) / C::kOStages) & 1, abort_flag,
                                      kWaitLimitNs)))
              break;
            issue_dp(i + 1);
            umma_commit_w(dp_full);
          } else {
            umma_commit_w(kv_empty);
            umma_commit_w(dkv_full);
          }
        }
        i0 += n;
        ++ul;
      }
      if (!ok && lane == 0) atomicOr(a.status, kStatusBwdMma);
      // no MMA in flight when TMEM and shared memory are released
      umma_commit_w(drain);
      if (!mbar_wait_drain_warp(drain, 0, kWaitLimitNs) && lane == 0) atomicOr(a.status, kStatusBwdDrain);
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int wq = warp & 3;
    const int hf = warp >> 2;                 // queries 64*hf .. +63 of each block
    const int jr = wq * 32 + lane;            // TMEM lane = key row (32x32b accesses)
    const int g4 = lane >> 2, c4 = lane & 3;  // 16-lane fragments: row t/4 (+8), column pair t%4
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    constexpr uint32_t kL16 = 16u << 16;  // lanes +16
    const uint32_t tS = tbase + lane_off + C::kColS + 64 * hf;
    const uint32_t tP = tbase + lane_off + C::kColdP + 64 * hf;
    const float sl2 = a.scale_log2;
    const float scale = a.scale;
    const uint32_t none[4] = {0u, 0u, 0u, 0u};
    bool ok = true;
    uint32_t i = 0;  // blocks processed so far
    int ul = 0;
    for (int rd = 0; ok; ++rd) {
      const int idx = snake_unit(rd, blockIdx.x, grid);
      if (idx >= num_units) break;
      const BwdUnit U = bwd_decode_unit(g, idx);
      const bool key_ok = jr < U.k_valid;
      if (U.items == 0) {
        // No query of this call sees the tile. A tile a shorter packed sample
        // does not have has no rows (k_valid == 0); a real one (rank-local
        // form: no query of the rank reaches it) gets a zero share.
        if (key_ok && bounds_ok(int64_t(U.tok0) + U.k_t0 + jr < a.kv_rows && U.g < g.hkv, a.status)) {
          const int64_t off = ((int64_t(U.tok0) + U.k_t0 + jr) * g.hkv + U.g) * D + hf * (D / 2);
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 8) {
            *reinterpret_cast<uint4*>(a.dv + off + c0) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(a.dk + off + c0) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      QWalk w(g, U);
      int chunk = 0, tile = 0;
      bool dg = false;
      int jh = 0;  // item j's head within the group (j mod G, counted)
      for (int j = 0; j < U.items && ok; ++j, ++i, jh = jh + 1 == G ? 0 : jh + 1) {
        if (jh == 0) w.next(chunk, tile, dg);
        const int rem = U.c - tile * kTile;
        const int q_valid = rem < kTile ? rem : kTile;
        const uint32_t os = i % C::kOStages;
        ok = mbar_wait_lean(&o_full[os], (i / C::kOStages) & 1, abort_flag, kWaitLimitNs) &&
             mbar_wait_lean(s_full, i & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        // S^T: this warp's 32 keys x 64 queries, then release the columns
        uint32_t ra[32], rb[32];
        tmem_ld16x256b_2x2(tS, tS + kL16, tS + 32, tS + kL16 + 32, ra, rb);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        // this thread's 16 queries: 64*hf + 32*cb + 8r + 2*c4 + {0, 1}
        const float* Lq = sLD + os * (2 * kTile) + 64 * hf + 2 * c4;
        float2 lv[2][4], dv[2][4];
#pragma unroll
        for (int cb = 0; cb < 2; ++cb)
#pragma unroll
          for (int r = 0; r < 4; ++r) lv[cb][r] = *reinterpret_cast<const float2*>(Lq + 32 * cb + 8 * r);
        // Blocks away from the diagonal and from ragged chunk ends need no mask.
        const bool full = !dg && q_valid == kTile && U.k_valid == kTile;
        uint32_t valid[2][4];
        uint32_t pp[2][16];
        if (full) {
          softmax_p_frag<false>(ra, sl2, lv[0], none, c4, pp[0]);
          softmax_p_frag<false>(rb, sl2, lv[1], none, c4, pp[1]);
        } else {
          // query q (in the block) is valid for key row kr when the key is in
          // its chunk, the query is in its chunk, and (on the diagonal) q >= kr
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              const int kr = wq * 32 + 8 * f + g4;  // key row of fragment row f (16u + 8e = 8f)
              const int qb = 64 * hf + 32 * cb;
              valid[cb][f] = kr < U.k_valid ? bit_range(dg ? kr - qb : 0, q_valid - qb) : 0u;
            }
          softmax_p_frag<true>(ra, sl2, lv[0], valid[0], c4, pp[0]);
          softmax_p_frag<true>(rb, sl2, lv[1], valid[1], c4, pp[1]);
        }
#pragma unroll
        for (int cb = 0; cb < 2; ++cb)
#pragma unroll
          for (int r = 0; r < 4; ++r) dv[cb][r] = *reinterpret_cast<const float2*>(Lq + kTile + 32 * cb + 8 * r);
        // dP^T of the same keys and queries
        if (!(ok = mbar_wait_lean(dp_full, i & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        tmem_ld16x256b_2x2(tP, tP + kL16, tP + 32, tP + kL16 + 32, ra, rb);
        // P^T -> [64h, 64h+32) of the dP^T columns just read: dV may start
        tmem_st16x128b_2x2(tP, tP + kL16, tP + 16, tP + kL16 + 16, pp[0], pp[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pt_full);
        uint32_t pd[2][16];
        if (full) {
          ds_frag<false>(pp[0], ra, dv[0], none, c4, pd[0]);
          ds_frag<false>(pp[1], rb, dv[1], none, c4, pd[1]);
        } else {
          ds_frag<true>(pp[0], ra, dv[0], valid[0], c4, pd[0]);
          ds_frag<true>(pp[1], rb, dv[1], valid[1], c4, pd[1]);
        }
        // dS^T -> [64h+32, 64h+64)
        tmem_st16x128b_2x2(tP + 32, tP + kL16 + 32, tP + 48, tP + kL16 + 48, pd[0], pd[1]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- dK, dV of the tile: TMEM -> bf16 -> global, 32 columns at a time
      if (!(ok = mbar_wait_lean(dkv_full, ul & 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      const int64_t off = ((int64_t(U.tok0) + U.k_t0 + jr) * g.hkv + U.g) * D + hf * (D / 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t rv[32], rk[32];
        tmem_ld32x2(tbase + lane_off + C::kColdV + hf * (D / 2) + c0, tbase + lane_off + C::kColdK + hf * (D / 2) + c0,
                    rv, rk);
        if (c0 + 32 >= D / 2) {
          // last chunk read: the MMA may start the next unit's dV/dK
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dkv_empty);
        }
        if (key_ok && bounds_ok(int64_t(U.tok0) + U.k_t0 + jr < a.kv_rows && U.g < g.hkv, a.status)) {
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            uint4 pv, pk;
            pv.x = pack_bf16x2(__uint_as_float(rv[q]), __uint_as_float(rv[q + 1]));
            pv.y = pack_bf16x2(__uint_as_float(rv[q + 2]), __uint_as_float(rv[q + 3]));
            pv.z = pack_bf16x2(__uint_as_float(rv[q + 4]), __uint_as_float(rv[q + 5]));
            pv.w = pack_bf16x2(__uint_as_float(rv[q + 6]), __uint_as_float(rv[q + 7]));
            // dK accumulated dS^T Q with dS unscaled: apply the softmax scale here
            pk.x = pack_bf16x2(__uint_as_float(rk[q]) * scale, __uint_as_float(rk[q + 1]) * scale);
            pk.y = pack_bf16x2(__uint_as_float(rk[q + 2]) * scale, __uint_as_float(rk[q + 3]) * scale);
            pk.z = pack_bf16x2(__uint_as_float(rk[q + 4]) * scale, __uint_as_float(rk[q + 5]) * scale);
            pk.w = pack_bf16x2(__uint_as_float(rk[q + 6]) * scale, __uint_as_float(rk[q + 7]) * scale);
            *reinterpret_cast<uint4*>(a.dv + off + c0 + q) = pv;
            *reinterpret_cast<uint4*>(a.dk + off + c0 + q) = pk;
          }
        }
      }
      ++ul;
    }
    if (!ok && lane == 0) atomicOr(a.status, kStatusBwdSoftmax);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================ dQ
// P for one query row's 32 keys (raw fp32 bits of S), packed to bf16 pairs:
// P = 2^(S*sl2 - l2); when `masked`, bit i of `valid` keeps key i (masked
// entries are selected to zero).
template <bool kMasked>
__device__ __forceinline__ void p_row32(const uint32_t (&rs)[32], float sl2, float l2, uint32_t valid,
                                        uint32_t (&pp)[16]) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-l2, -l2);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), sl2x2, nl2), x0, x1);
    pp[i] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
    if constexpr (kMasked)
      pp[i] &= ((valid >> (2 * i)) & 1u ? 0x0000ffffu : 0u) | ((valid >> (2 * i + 1)) & 1u ? 0xffff0000u : 0u);
  }
}

// dS = P (dP - D) for the same 32 keys, P as packed bf16 pairs, D per row;
// masked entries are selected to zero (their dP - D may be anything).
template <bool kMasked>
__device__ __forceinline__ void ds_row32(const uint32_t (&pp)[16], const uint32_t (&rp)[32], float dd,
                                         uint32_t valid, uint32_t (&pd)[16]) {
  const uint64_t ddx2 = f2_pack(dd, dd);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float g0, g1;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(pp[i] << 16), __uint_as_float(pp[i] & 0xffff0000u)),
                     f2_sub(f2_pack(__uint_as_float(rp[2 * i]), __uint_as_float(rp[2 * i + 1])), ddx2)),
              g0, g1);
    pd[i] = pack_bf16x2(g0, g1);
    if constexpr (kMasked)
      pd[i] &= ((valid >> (2 * i)) & 1u ? 0x0000ffffu : 0u) | ((valid >> (2 * i + 1)) & 1u ? 0xffff0000u : 0u);
  }
}

template <int D>
struct DqCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSlots = D == 128 ? 5 : 8;  // K/V ring
  static constexpr int kOffQ = 0;
  static constexpr int kOffdO = kOffQ + kTileBytes;
  static constexpr int kOffKV = kOffdO + kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  // q_full q_empty qa_full qa_empty s_full s_free dp_full p_full dq_full
  // dq_empty drain, kv_full[] kv_empty[], p_half
  static constexpr int kNumBars = 12 + 2 * kSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kLayoutBytes = kOffMisc + 16;
  // The d=128 layout leaves no room for re-alignment: the dynamic shared
  // memory base must already be 1024-byte aligned (checked at run time).
  static constexpr bool kNeedAlignedBase = (kLayoutBytes + 1024 > 232448);
  static constexpr int kSmemBytes = kNeedAlignedBase ? kLayoutBytes : kLayoutBytes + 1024;
  static_assert(kLayoutBytes <= 232448, "dQ shared memory layout too large");
  // TMEM: S [0,128), dP [128,256) (later dS, packed), dQ [256,256+D), then Q
  // and dO as bf16 A operands (D/2 columns each).
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdQ = 256, kColQA = 256 + D, kColdOA = 256 + D + D / 2;
};

// Query-tile-stationary dQ. One CTA per SM, 10 warps:
//   warps 0-7  element-wise; warp w covers TMEM lanes 32*(w%4).. (query rows)
//              and keys 64*(w/4) .. +63 of each key tile (D/2 columns of Q,
//              dO and dQ)
//   warp 8     TMA producer (Q, dO per unit; K/V ring in CP-step order)
//   warp 9     TMEM owner and MMA issuer (whole warp, elect.sync)
// At the start of a unit the element-wise warps copy its Q and dO tiles from
// shared memory into TMEM as packed bf16, so every MMA takes its A operand
// from TMEM and reads only B (a K or V tile) from shared memory:
//   S(j) = Q K_j^T -> [0,128)     dP(j) = dO V_j^T -> [128,256)
//   dQ += dS(j) K_j               (dS packed over dP(j); each warp publishes
//                                  its first 32 keys' dS (p_half) before
//                                  forming the other 32, and the MMAs over
//                                  those keys start at once)
// The element-wise warps load S(j) and at once release its columns (s_free),
// compute P in registers, then load dP(j) and write packed bf16 dS over it,
// each warp inside the columns it read. Tensor-core order per key tile:
//   S(j+1) | dQ(j) | dP(j+1) | S(j+2) | ...
// so the exponentials of tile j overlap dQ(j-1) and dP(j), and only the dS
// step of each warp's first 32 keys lies on the tensor core's critical path.
template <int D, bool kShortWaits = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    cpattn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                         const BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if constexpr (!C::kNeedAlignedBase)
    smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBwdSmemAlign);
    return;
  }
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sdO = smem + C::kOffdO;
  uint8_t* sKV = smem + C::kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* qa_full = bars + 2;
  uint64_t* qa_empty = bars + 3;
  uint64_t* s_full = bars + 4;
  uint64_t* s_free = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* dq_full = bars + 8;
  uint64_t* dq_empty = bars + 9;
  uint64_t* drain = bars + 10;
  uint64_t* kv_full = bars + 11;
  uint64_t* kv_empty = bars + 11 + C::kSlots;
  uint64_t* p_half = bars + 11 + 2 * C::kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const CpGeom& g = a.g;
  const int num_units = dq_num_units(g);
  const int grid = gridDim.x;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_empty, 8);
    mbar_init(qa_full, 8);
    mbar_init(qa_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 8);
    mbar_init(drain, 1);
    mbar_init(p_half, 8);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmdo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t plimit = kShortWaits ? a.producer_limit_ns : kWaitLimitNs;
      bool ok = true;
      uint32_t nload = 0;
      int ul = 0;
      auto load = [&](const CUtensorMap* map, int head, int row) -> bool {
        bounds_ok(row >= 0 && row < a.kv_rows && head >= 0 && head < g.hkv, a.status);
        const uint32_t slot = nload % C::kSlots;
        if (nload >= (uint32_t)C::kSlots &&
            !mbar_wait_lean(&kv_empty[slot], ((nload / C::kSlots) - 1) & 1, abort_flag, plimit))
          return false;
        mbar_arrive_expect_tx(&kv_full[slot], C::kTileBytes);
        uint8_t* dst = sKV + slot * C::kTileBytes;
        for (int x = 0; x < D; x += 64)
          tma_load_3d(dst + (x / 64) * (kTile * 128), map, &kv_full[slot], x, head, row);
        ++nload;
        return true;
      };
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const FwdUnit U = dq_decode_unit(g, idx);
        if (U.n == 0) continue;  // a tile a shorter packed sample does not have
        // the Q/dO stage is free once the element-wise warps copied the
        // previous unit's tiles into TMEM
        if (ul > 0 && !(ok = mbar_wait_lean(q_empty, (ul - 1) & 1, abort_flag, plimit))) break;
        mbar_arrive_expect_tx(q_full, 2 * C::kTileBytes);
        const int qrow = U.tok0 + U.q_t0;
        bounds_ok(qrow >= 0 && qrow < a.q_rows && U.h0 < g.hq, a.status);
        for (int x = 0; x < D; x += 64) {
          tma_load_3d(sQ + (x / 64) * (kTile * 128), &tmq, q_full, x, U.h0, qrow);
          tma_load_3d(sdO + (x / 64) * (kTile * 128), &tmdo, q_full, x, U.h0, qrow);
        }
        KvWalk w(g, U);
        int chunk, tile;
        bool dg;
        while (ok && w.next(chunk, tile, dg)) {
          const int row = U.tok0 + kv_chunk_row(g, chunk, U.c) + tile * kTile;
          // V before K: V is released by the dP MMA, K only after dQ
          ok = load(&tmv, U.g0, row) && load(&tmk, U.g0, row);
        }
        ++ul;
      }
      if (!ok) atomicOr(a.status, kStatusBwdProducer);
      // copies still in flight land before the CTA can exit (see above)
      bool drained = true;
      const uint32_t first = nload > (uint32_t)C::kSlots ? nload - C::kSlots : 0;
      for (uint32_t i = first; i < nload; ++i)
        drained &= mbar_wait_drain(&kv_full[i % C::kSlots], (i / C::kSlots) & 1, kWaitLimitNs);
      if (ul > 0) drained &= mbar_wait_drain(q_full, (ul - 1) & 1, kWaitLimitNs);
      if (!drained) atomicOr(a.status, kStatusBwdDrain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs this role; elect.sync picks the issuing lane)
    {
      constexpr uint32_t idS = make_idesc_bf16(kTile, kTile, false, false);  // S, dP
      constexpr uint32_t idQ = make_idesc_bf16(kTile, D, false, true);       // dQ += dS K
      const uint64_t dKV_km = make_sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dKV_mn = make_sdesc_sw128(smem_u32(sKV), 16384, 1024);
      const uint32_t tS = tbase + C::kColS, tdP = tbase + C::kColdP, tdQ = tbase + C::kColdQ;
      const uint32_t tQA = tbase + C::kColQA, tdOA = tbase + C::kColdOA;
      uint32_t ncons = 0;
      auto take = [&](uint32_t& slot, uint32_t& par) {
        slot = ncons % C::kSlots;
        par = (ncons / C::kSlots) & 1;
        ++ncons;
      };
      // S = Q K^T and dP = dO V^T, A (Q, dO) from TMEM, B from the ring
      auto issue_s = [&](uint32_t ks) {
        const uint64_t kb = dKV_km + ((ks * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
          umma_ts_w(tS, tQA + kk * 8, kb + off, idS, kk > 0);
        }
      };
      auto issue_dp = [&](uint32_t vs) {
        const uint64_t vb = dKV_km + ((vs * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
          umma_ts_w(tdP, tdOA + kk * 8, vb + off, idS, kk > 0);
        }
      };
      bool ok = true;
      uint32_t jt = 0;  // key tiles processed so far
      int ul = 0;
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const FwdUnit U = dq_decode_unit(g, idx);
        if (U.n == 0) continue;  // a tile a shorter packed sample does not have
        const int n = U.n;
        // prologue: S and dP of the unit's first key tile, once Q/dO are in
        // TMEM. The S columns are free once the previous S was read; the dP
        // columns once the previous dQ MMAs (issued) read the dS there.
        uint32_t ks, kp, vs, vp;
        take(vs, vp);
        take(ks, kp);
        ok = mbar_wait_warp_lean(qa_full, ul & 1, abort_flag, kWaitLimitNs) &&
             mbar_wait_warp_lean(&kv_full[ks], kp, abort_flag, kWaitLimitNs) &&
             (jt == 0 || mbar_wait_warp_lean(s_free, (jt - 1) & 1, abort_flag, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        issue_s(ks);
        umma_commit_w(s_full);
        if (!(ok = mbar_wait_warp_lean(&kv_full[vs], vp, abort_flag, kWaitLimitNs))) break;
        issue_dp(vs);
        umma_commit_w(dp_full);
        umma_commit_w(&kv_empty[vs]);
        if (n == 1) umma_commit_w(qa_empty);
        for (int j = 0; j < n && ok; ++j, ++jt) {
          const uint32_t cur_ks = ks;
          uint32_t nvs = 0, nvp = 0;
          if (j + 1 < n) {
            // S(jt+1) as soon as S(jt) has been read
            take(nvs, nvp);
            take(ks, kp);
            ok = mbar_wait_warp_lean(s_free, jt & 1, abort_flag, kWaitLimitNs) &&
                 mbar_wait_warp_lean(&kv_full[ks], kp, abort_flag, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            issue_s(ks);
            umma_commit_w(s_full);
          }
          ok = mbar_wait_warp_lean(p_half, jt & 1, abort_flag, kWaitLimitNs) &&
               (j > 0 || ul == 0 || mbar_wait_warp_lean(dq_empty, (ul - 1) & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          // dQ += dS(jt) K_j   (dS from TMEM, K MN-major): first the K-steps of
          // each warp's first 32 keys (0, 1 and 4, 5), then the rest
          const uint64_t kmn = dKV_mn + ((cur_ks * C::kTileBytes) >> 4);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = (q & 1) + 4 * (q >> 1);
            umma_ts_w(tdQ, tdP + half_split_col(kk), kmn + ((kk * 2048) >> 4), idQ, (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (!(ok = mbar_wait_warp_lean(p_full, jt & 1, abort_flag, kWaitLimitNs))) break;
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 2 + (q & 1) + 4 * (q >> 1);
            umma_ts_w(tdQ, tdP + half_split_col(kk), kmn + ((kk * 2048) >> 4), idQ, 1u);
          }
          umma_commit_w(&kv_empty[cur_ks]);
          if (j == n - 1) umma_commit_w(dq_full);
          if (j + 1 < n) {
            // dP(jt+1) over dS(jt), which the dQ MMAs just issued read first
            if (!(ok = mbar_wait_warp_lean(&kv_full[nvs], nvp, abort_flag, kWaitLimitNs))) break;
            issue_dp(nvs);
            umma_commit_w(dp_full);
            umma_commit_w(&kv_empty[nvs]);
            if (j + 1 == n - 1) umma_commit_w(qa_empty);  // the unit's last reads of Q/dO in TMEM
          }
        }
        ++ul;
      }
      if (!ok && lane == 0) atomicOr(a.status, kStatusBwdMma);
      // no MMA in flight when TMEM and shared memory are released
      umma_commit_w(drain);
      if (!mbar_wait_drain_warp(drain, 0, kWaitLimitNs) && lane == 0) atomicOr(a.status, kStatusBwdDrain);
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int wq = warp & 3;
    const int hf = warp >> 2;
    const int jr = wq * 32 + lane;  // TMEM lane = query row
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::kColS + hf * 64;
    const uint32_t tdP = tbase + lane_off + C::kColdP + hf * 64;
    const float sl2 = a.scale_log2;
    const float scale = a.scale;
    bool ok = true;
    uint32_t jt = 0;
    int ul = 0;
    for (int rd = 0; ok; ++rd) {
      const int idx = snake_unit(rd, blockIdx.x, grid);
      if (idx >= num_units) break;
      const FwdUnit U = dq_decode_unit(g, idx);
      if (U.n == 0) continue;  // a tile a shorter packed sample does not have
      // ---- this row's Q and dO (columns hf*D/2 ..) into TMEM as packed bf16
      ok = mbar_wait_lean(q_full, ul & 1, abort_flag, kWaitLimitNs) &&
           (ul == 0 || mbar_wait_lean(qa_empty, (ul - 1) & 1, abort_flag, kWaitLimitNs));
      if (!ok) break;
      tc_fence_after();  // the previous unit's MMAs have finished reading these columns
      {
        // swizzled rows of the TMA tile: 16-byte chunk c of row jr sits at
        // chunk c ^ (jr & 7) of the row's 128 bytes, d-block x at x * 16 KB
        constexpr int kChunks = D / 16;  // 16-byte chunks of this warp's D/2 elements
        uint32_t rq[D / 4], ro[D / 4];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          const int e0 = hf * (D / 2) + c * 8;  // first element of the chunk
          const int x = e0 / 64, cc = (e0 % 64) / 8;
          const uint32_t off = x * (kTile * 128) + jr * 128 + ((cc ^ (jr & 7)) * 16);
          const uint4 vq = *reinterpret_cast<const uint4*>(sQ + off);
          const uint4 vo = *reinterpret_cast<const uint4*>(sdO + off);
          rq[4 * c] = vq.x; rq[4 * c + 1] = vq.y; rq[4 * c + 2] = vq.z; rq[4 * c + 3] = vq.w;
          ro[4 * c] = vo.x; ro[4 * c + 1] = vo.y; ro[4 * c + 2] = vo.z; ro[4 * c + 3] = vo.w;
        }
        const uint32_t tq = tbase + lane_off + C::kColQA + hf * (D / 4);
        const uint32_t to = tbase + lane_off + C::kColdOA + hf * (D / 4);
        if constexpr (D == 128) {
          tmem_st32(tq, rq);
          tmem_st32(to, ro);
        } else {
          tmem_st16(tq, rq);
          tmem_st16(to, ro);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(qa_full);
        mbar_arrive(q_empty);
      }
      // this row's L*log2e and D (padded rows of a ragged tile read arbitrary
      // values; their dQ is never stored)
      int64_t pos = ld_pos(g, a.ntp, U.seq, U.h0, U.k, U.u, U.tpc, jr);
      if (!bounds_ok(pos >= 0 && pos < a.vec_len, a.status)) pos = 0;  // stays inside the vectors
      const float l2 = a.lvec[pos];
      const float dd = a.dvec[pos];
      KvWalk w(g, U);
      // Without ragged tiles the walk's only masked position is the query
      // tile's diagonal, where step 0 ends: follow the positions without the
      // walk itself (as the forward's softmax warps do).
      const bool walkless = (U.c & (kTile - 1)) == 0;
      const int jdiag = g.causal ? (U.half ? U.tpc : 0) + U.u : -1;
      for (int j = 0; j < U.n && ok; ++j, ++jt) {
        int chunk = 0, tile = 0;
        bool dg = false;
        int n_valid = kTile;
        if (walkless) {
          dg = j == jdiag;
        } else {
          w.next(chunk, tile, dg);
          const int rem = U.c - tile * kTile;
          n_valid = rem < kTile ? rem : kTile;
        }
        if (!(ok = mbar_wait_lean(s_full, jt & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32x2(tS, tS + 32, r0, r1);
        // S(jt) is in registers: the MMA may compute S(jt+1) meanwhile
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        const bool full = !dg && n_valid == kTile;
        // key column c (of this warp's 64) is valid when it is inside its
        // chunk and (on the diagonal) c <= jr
        const int cb = hf * 64;
        int hi = n_valid - cb;
        if (dg && jr + 1 - cb < hi) hi = jr + 1 - cb;
        const uint32_t v0 = full ? 0u : bit_range(0, hi), v1 = full ? 0u : bit_range(0, hi - 32);
        uint32_t pp0[16], pp1[16];
        if (full) {
          p_row32<false>(r0, sl2, l2, 0u, pp0);
          p_row32<false>(r1, sl2, l2, 0u, pp1);
        } else {
          p_row32<true>(r0, sl2, l2, v0, pp0);
          p_row32<true>(r1, sl2, l2, v1, pp1);
        }
        if (!(ok = mbar_wait_lean(dp_full, jt & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        tmem_ld32x2(tdP, tdP + 32, r0, r1);
        uint32_t pd0[16], pd1[16];
        // dS packed into [64h, 64h+32) of the dP columns (read above), its
        // first 32 keys published before the second are formed
        if (full)
          ds_row32<false>(pp0, r0, dd, 0u, pd0);
        else
          ds_row32<true>(pp0, r0, dd, v0, pd0);
        tmem_st16(tdP, pd0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_half);
        if (full)
          ds_row32<false>(pp1, r1, dd, 0u, pd1);
        else
          ds_row32<true>(pp1, r1, dd, v1, pd1);
        tmem_st16(tdP + 16, pd1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- dQ of the tile: TMEM -> scale -> bf16 -> global
      if (!(ok = mbar_wait_lean(dq_full, ul & 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      uint32_t rq[D / 2];
      {
        uint32_t q0[32], q1[32];
        tmem_ld32x2(tbase + lane_off + C::kColdQ + hf * (D / 2),
                    tbase + lane_off + C::kColdQ + hf * (D / 2) + (D == 128 ? 32 : 0), q0, q1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          rq[i] = q0[i];
          if constexpr (D == 128) rq[32 + i] = q1[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_empty);
      if (jr < U.q_valid && bounds_ok(int64_t(U.tok0) + U.q_t0 + jr < a.q_rows && U.h0 < g.hq, a.status)) {
        __nv_bfloat16* dst = a.dq + ((int64_t(U.tok0) + U.q_t0 + jr) * g.hq + U.h0) * D + hf * (D / 2);
#pragma unroll
        for (int i = 0; i < D / 2; i += 8) {
          uint4 pk;
          pk.x = pack_bf16x2(__uint_as_float(rq[i]) * scale, __uint_as_float(rq[i + 1]) * scale);
          pk.y = pack_bf16x2(__uint_as_float(rq[i + 2]) * scale, __uint_as_float(rq[i + 3]) * scale);
          pk.z = pack_bf16x2(__uint_as_float(rq[i + 4]) * scale, __uint_as_float(rq[i + 5]) * scale);
          pk.w = pack_bf16x2(__uint_as_float(rq[i + 6]) * scale, __uint_as_float(rq[i + 7]) * scale);
          *reinterpret_cast<uint4*>(dst + i) = pk;
        }
      }
      ++ul;
    }
    if (!ok && lane == 0) atomicOr(a.status, kStatusBwdSoftmax);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace cpattn
