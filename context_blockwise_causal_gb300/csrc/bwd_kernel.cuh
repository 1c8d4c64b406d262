// Backward kernels for context-parallel causal attention.
//
//   cpattn_bwd_pre_kernel     D[t] = rowsum(dO[t] * O[t]) and L[t]*log2(e) per
//                             query row into tile-padded vectors; zeroes the
//                             fp32 dQ accumulator.                (HBM-bound)
//   cpattn_bwd_kernel         key-tile-stationary main kernel: per 128-key
//                             tile it walks every (query head of the group,
//                             query tile) block that sees it in CP-step order
//                             and computes, on tcgen05 tensor cores,
//                               S^T = K Q^T, dP^T = V dO^T          (TMEM)
//                               P^T = 2^(S^T*scale*log2e - L*log2e)
//                               dS^T = P^T (dP^T - D)
//                               dV += P^T dO, dK += dS^T Q          (TMEM)
//                               dQ^T = K^T dS^T -> fp32 reductions into the
//                               accumulator (d = 64: dQ = dS K)
//                             with 1/sqrt(d) applied once to dK at the end and
//                             to dQ in the conversion,
//                             dK/dV of the tile stay in TMEM across all its
//                             blocks and are written once.
//   cpattn_dq_convert_kernel  fp32 dQ accumulator -> bf16 dq.     (HBM-bound)
//
// The gradient formulas are those of softmax attention (the derivative of
// the forward defined in include/cpattn.h); the blocks and masks are the
// forward's CP steps ("大模型面试宝典 · Megatron-LM 篇", 3.4), seen from the key
// side (see QWalk in cp_schedule.cuh).
//
// Main kernel: one CTA per SM, 10 warps.
//   warps 0-7  element-wise work; warp w covers TMEM lanes 32*(w%4).. and
//              column half w/4 (64 query columns of S^T/dP^T, D/2 columns of
//              dQ/dK/dV)
//   warp 8     TMA producer
//   warp 9     TMEM owner and MMA issuer
// TMEM: A [0,128) S^T, then P^T (bf16 pairs: queries 0-63 in columns 0-31,
// 64-127 in columns 64-95); B [128,256) dP^T, then dQ; dV [256,256+D);
// dK [256+D, 256+2D). Units walk query tiles from the end of the sequence
// down (see QWalk), which keeps the dQ rows being reduced into L2-resident.
// Shared memory: K, V tiles; two stages of (Q, dO, L, D); dS^T (bf16,
// 128 keys x 128 queries, laid out as two 64-query blocks of 128-byte
// swizzled rows: K-major for dK's A operand and MN-major for dQ's A operand).
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
  float* dq_acc;  // [b, s, hq, d] fp32
  float* lvec;    // [b, hq, ntp]: lse * log2(e)
  float* dvec;    // [b, hq, ntp]: rowsum(dO * O)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  unsigned int* status;
};

// ---------------------------------------------------------------- preprocess
template <int D>
__global__ void __launch_bounds__(256) cpattn_bwd_pre_kernel(const BwdArgs a) {
  const CpGeom& g = a.g;
  const int64_t nrows = int64_t(g.b) * g.s * g.hq;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < nrows;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int h = int(idx % g.hq);
    const int64_t bt = idx / g.hq;
    const int t = int(bt % g.s);
    const int bi = int(bt / g.s);
    const uint4* po = reinterpret_cast<const uint4*>(a.o + idx * D);
    const uint4* pd = reinterpret_cast<const uint4*>(a.dout + idx * D);
    float acc = 0.f;
#pragma unroll 4
    for (int i = 0; i < D / 8; ++i) {
      const uint4 x = po[i], y = pd[i];
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc);
        acc = fmaf(__uint_as_float(xs[k] & 0xffff0000u), __uint_as_float(ys[k] & 0xffff0000u), acc);
      }
    }
    const int chunk = t / g.c;
    const int in = t - chunk * g.c;
    const int64_t pos = int64_t(bi * g.hq + h) * a.ntp + (chunk * g.tpc + in / kTile) * kTile + in % kTile;
    a.dvec[pos] = acc;
    a.lvec[pos] = a.lse[(int64_t(bi) * g.hq + h) * g.s + t] * 1.4426950408889634f;
    float4* z = reinterpret_cast<float4*>(a.dq_acc + idx * D);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ---------------------------------------------------------------- dQ convert
// dq = bf16(scale * acc): the main kernel accumulates dS K with dS unscaled.
__global__ void __launch_bounds__(256) cpattn_dq_convert_kernel(const float* __restrict__ acc,
                                                                __nv_bfloat16* __restrict__ dq, int64_t n4,
                                                                float scale) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
    const float4 x = reinterpret_cast<const float4*>(acc)[i];
    uint2 p;
    p.x = pack_bf16x2(x.x * scale, x.y * scale);
    p.y = pack_bf16x2(x.z * scale, x.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = p;
  }
}

// ---------------------------------------------------------------- main
template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;  // 128 x D bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;       // two stages
  static constexpr int kOffdO = kOffQ + 2 * kTileBytes;  // two stages
  static constexpr int kOffdS = kOffdO + 2 * kTileBytes;
  static constexpr int kdSBytes = kTile * kTile * 2;
  static constexpr int kOffLD = kOffdS + kdSBytes;  // two stages of (L[128], D[128]) fp32
  static constexpr int kLDBytes = 2 * kTile * 4;
  static constexpr int kOffBar = kOffLD + 2 * kLDBytes;
  // kv_full kv_empty q_full[2] q_empty[2] s_full p_full ds_empty dq_full dq_empty
  // dkv_full dkv_empty drain
  static constexpr int kNumBars = 14;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kLayoutBytes = kOffMisc + 16;
  // The d=128 layout leaves no room for re-alignment: the dynamic shared
  // memory base must already be 1024-byte aligned (checked at run time).
  static constexpr bool kNeedAlignedBase = (kLayoutBytes + 1024 > 232448);
  static constexpr int kSmemBytes = kNeedAlignedBase ? kLayoutBytes : kLayoutBytes + 1024;
  static constexpr uint32_t kColA = 0, kColB = 128, kColdV = 256, kColdK = 256 + D;
};

enum BwdStatusBits : unsigned int {
  kStatusBwdProducer = 1u << 8,
  kStatusBwdMma = 1u << 9,
  kStatusBwdSoftmax = 1u << 10,
  kStatusBwdSmemAlign = 1u << 11,
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    cpattn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                      const BwdArgs a) {
  using C = BwdCfg<D>;
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
  uint8_t* sdS = smem + C::kOffdS;
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = bars + 4;
  uint64_t* s_full = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* ds_empty = bars + 8;
  uint64_t* dq_full = bars + 9;
  uint64_t* dq_empty = bars + 10;
  uint64_t* dkv_full = bars + 11;
  uint64_t* dkv_empty = bars + 12;
  uint64_t* drain = bars + 13;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);
    mbar_init(ds_empty, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 8);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 8);
    mbar_init(drain, 1);
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
      bool ok = true;
      uint32_t item = 0;  // items loaded so far (stage = item & 1)
      int ul = 0;
      auto load_item = [&](const BwdUnit& U, int chunk, int tile, int h) -> bool {
        const uint32_t st = item & 1;
        if (item >= 2 && !mbar_wait_bounded(&q_empty[st], ((item >> 1) - 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        mbar_arrive_expect_tx(&q_full[st], 2 * C::kTileBytes + C::kLDBytes);
        const int row = U.bi * g.s + chunk * g.c + tile * kTile;
        for (int x = 0; x < D; x += 64) {
          tma_load_3d(sQ + st * C::kTileBytes + (x / 64) * (kTile * 128), &tmq, &q_full[st], x, h, row);
          tma_load_3d(sdO + st * C::kTileBytes + (x / 64) * (kTile * 128), &tmdo, &q_full[st], x, h, row);
        }
        const int64_t pos = int64_t(U.bi * g.hq + h) * a.ntp + (chunk * g.tpc + tile) * kTile;
        bulk_load(reinterpret_cast<uint8_t*>(sLD) + st * C::kLDBytes, a.lvec + pos, kTile * 4, &q_full[st]);
        bulk_load(reinterpret_cast<uint8_t*>(sLD) + st * C::kLDBytes + kTile * 4, a.dvec + pos, kTile * 4,
                  &q_full[st]);
        ++item;
        return true;
      };
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const BwdUnit U = bwd_decode_unit(g, idx);
        QWalk w(g, U);
        int chunk, tile;
        bool dg;
        bool first = true;
        while (ok && w.next(chunk, tile, dg)) {
          for (int h = U.g * G; h < (U.g + 1) * G && ok; ++h) {
            ok = load_item(U, chunk, tile, h);
            if (ok && first) {
              // K/V of this unit, after the first query item is on its way.
              first = false;
              if (ul > 0 && !(ok = mbar_wait_bounded(kv_empty, (ul - 1) & 1, abort_flag, kWaitLimitNs))) break;
              mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
              const int krow = U.bi * g.s + U.k_t0;
              for (int x = 0; x < D; x += 64) {
                tma_load_3d(sK + (x / 64) * (kTile * 128), &tmk, kv_full, x, U.g, krow);
                tma_load_3d(sV + (x / 64) * (kTile * 128), &tmv, kv_full, x, U.g, krow);
              }
            }
          }
        }
        ++ul;
      }
      if (!ok) atomicOr(a.status, kStatusBwdProducer);
      // Let every copy still in flight land before the CTA can exit.
      for (uint32_t i = item > 2 ? item - 2 : 0; i < item; ++i)
        mbar_wait_bounded(&q_full[i & 1], (i >> 1) & 1, abort_flag, kWaitLimitNs);
      if (ul > 0) mbar_wait_bounded(kv_full, (ul - 1) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc_bf16(kTile, kTile, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = make_idesc_bf16(kTile, D, false, true);      // dV, dK
      constexpr uint32_t idQ = make_idesc_bf16(kTile, D == 128 ? kTile : D, true, true);  // dQ^T / dQ
      const uint64_t dK_km = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV_km = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dK_mn = make_sdesc_sw128(smem_u32(sK), 16384, 1024);
      const uint64_t dQ_km = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t ddO_km = make_sdesc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t dQ_mn = make_sdesc_sw128(smem_u32(sQ), 16384, 1024);
      const uint64_t ddO_mn = make_sdesc_sw128(smem_u32(sdO), 16384, 1024);
      const uint64_t ddS_km = make_sdesc_sw128(smem_u32(sdS), 16, 1024);
      const uint64_t ddS_mn = make_sdesc_sw128(smem_u32(sdS), 16384, 1024);
      const uint32_t tA = tbase + C::kColA, tB = tbase + C::kColB;
      const uint32_t tdV = tbase + C::kColdV, tdK = tbase + C::kColdK;
      bool ok = true;
      uint32_t item = 0;
      int ul = 0;
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const BwdUnit U = bwd_decode_unit(g, idx);
        for (int it = 0; it < U.items && ok; ++it, ++item) {
          const uint32_t st = item & 1;
          const uint64_t so = (st * C::kTileBytes) >> 4;
          ok = mbar_wait_bounded(&q_full[st], (item >> 1) & 1, abort_flag, kWaitLimitNs) &&
               (it > 0 || mbar_wait_bounded(kv_full, ul & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          // S^T = K Q^T  (region A is free: the previous dV MMA read P^T first)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
            umma_ss(tA, dK_km + off, dQ_km + so + off, idS, kk > 0);
          }
          // dP^T = V dO^T  (region B must have been drained of the previous dQ)
          if (item > 0 && !(ok = mbar_wait_bounded(dq_empty, (item - 1) & 1, abort_flag, kWaitLimitNs))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
            umma_ss(tB, dV_km + off, ddO_km + so + off, idS, kk > 0);
          }
          umma_commit(s_full);
          ok = mbar_wait_bounded(p_full, item & 1, abort_flag, kWaitLimitNs) &&
               (it > 0 || ul == 0 || mbar_wait_bounded(dkv_empty, (ul - 1) & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          const uint32_t acc = it > 0 ? 1u : 0u;
          // dV += P^T dO  (P^T from TMEM)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t pcol = kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
            umma_ts(tdV, tA + pcol, ddO_mn + so + ((kk * 2048) >> 4), idKV, acc | (kk > 0));
          }
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
            umma_ss(tdK, ddS_km + off, dQ_mn + so + ((kk * 2048) >> 4), idKV, acc | (kk > 0));
          }
          // dQ -> region B. d = 128: dQ^T = K^T dS^T (TMEM lanes = head dim, so
          // each warp's reduction into the accumulator is one 128-byte line);
          // d = 64: dQ = dS K (lanes = queries).
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            if constexpr (D == 128)
              umma_ss(tB, dK_mn + ((kk * 2048) >> 4), ddS_mn + ((kk * 2048) >> 4), idQ, kk > 0);
            else
              umma_ss(tB, ddS_mn + ((kk * 2048) >> 4), dK_mn + ((kk * 2048) >> 4), idQ, kk > 0);
          }
          umma_commit(&q_empty[st]);
          umma_commit(ds_empty);
          umma_commit(dq_full);
          if (it == U.items - 1) {
            umma_commit(kv_empty);
            umma_commit(dkv_full);
          }
        }
        ++ul;
      }
      if (!ok) atomicOr(a.status, kStatusBwdMma);
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, abort_flag, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int wq = warp & 3;
    const int hf = warp >> 2;
    const int jr = wq * 32 + lane;  // TMEM lane: key row (S^T, dK, dV) or query row (dQ)
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tA = tbase + lane_off + C::kColA;
    const uint32_t tB = tbase + lane_off + C::kColB;
    const float sl2 = a.scale_log2;
    const float scale = a.scale;
    bool ok = true;
    uint32_t item = 0;
    int ul = 0;
    for (int rd = 0; ok; ++rd) {
      const int idx = snake_unit(rd, blockIdx.x, grid);
      if (idx >= num_units) break;
      const BwdUnit U = bwd_decode_unit(g, idx);
      QWalk w(g, U);
      int chunk = 0, tile = 0;
      bool dg = false;
      for (int it = 0; it < U.items && ok; ++it, ++item) {
        const int hsub = it % G;
        if (hsub == 0) w.next(chunk, tile, dg);
        const int h = U.g * G + hsub;
        const int rem = g.c - tile * kTile;
        const int q_valid = rem < kTile ? rem : kTile;
        const uint32_t st = item & 1;
        ok = mbar_wait_bounded(&q_full[st], (item >> 1) & 1, abort_flag, kWaitLimitNs) &&
             mbar_wait_bounded(s_full, item & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const float* Lv = sLD + st * (2 * kTile);
        const float* Dv = Lv + kTile;
        // Blocks away from the diagonal and from ragged chunk ends need no mask.
        const bool full = !dg && q_valid == kTile && U.k_valid == kTile;
        const bool key_ok = jr < U.k_valid;
        // the previous dQ/dK MMAs must be done reading dS^T
        if (item > 0 && !(ok = mbar_wait_bounded(ds_empty, (item - 1) & 1, abort_flag, kWaitLimitNs))) break;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int sc = 0; sc < 2; ++sc) {
          const int c0 = hf * 64 + sc * 32;  // first query column of this chunk
          uint32_t rs[32], rp[32];
          tmem_ld32(tA + c0, rs);
          tmem_ld32(tB + c0, rp);
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + 2 * i;
            // P = 2^(S*scale*log2e - L*log2e); dS (unscaled) = P (dP - D)
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), sl2x2,
                                      f2_pack(-Lv[c], -Lv[c + 1]));
            float x0, x1;
            f2_unpack(x, x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const uint64_t t = f2_sub(f2_pack(__uint_as_float(rp[2 * i]), __uint_as_float(rp[2 * i + 1])),
                                      f2_pack(Dv[c], Dv[c + 1]));
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(p0, p1), t), d0, d1);
            if (!full) {
              // padded rows of L/D hold arbitrary values: select, never multiply
              const bool v0 = key_ok && c < q_valid && !(dg && jr > c);
              const bool v1 = key_ok && c + 1 < q_valid && !(dg && jr > c + 1);
              p0 = v0 ? p0 : 0.f;
              d0 = v0 ? d0 : 0.f;
              p1 = v1 ? p1 : 0.f;
              d1 = v1 ? d1 : 0.f;
            }
            pp[i] = pack_bf16x2(p0, p1);
            pd[i] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tA + hf * 64 + sc * 16, pp);
          // dS^T row jr, query block hf, 16-byte chunks 4*sc .. 4*sc+3 (swizzled)
          uint8_t* rowp = sdS + hf * (kTile * 128) + jr * 128;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cc = sc * 4 + q4;
            *reinterpret_cast<uint4*>(rowp + ((cc ^ (jr & 7)) << 4)) =
                make_uint4(pd[4 * q4], pd[4 * q4 + 1], pd[4 * q4 + 2], pd[4 * q4 + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        // ---- drain dQ of this block into the fp32 accumulator (unscaled;
        // the conversion kernel applies 1/sqrt(d))
        if (!(ok = mbar_wait_bounded(dq_full, item & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        uint32_t rq[64];
        {
          uint32_t r0[32], r1[32];
          if constexpr (D == 128) {
            tmem_ld32(tB + hf * 64, r0);
            tmem_ld32(tB + hf * 64 + 32, r1);
          } else {
            tmem_ld32(tB + hf * 32, r0);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            rq[i] = r0[i];
            if constexpr (D == 128) rq[32 + i] = r1[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dq_empty);
        const int t0 = chunk * g.c + tile * kTile;
        if constexpr (D == 128) {
          // lane jr holds dQ^T[d = jr][queries hf*64 ..]: a warp adds one
          // contiguous 128-byte line per query row
          float* base = a.dq_acc + ((int64_t(U.bi) * g.s + t0 + hf * 64) * g.hq + h) * D + jr;
          const int64_t row_stride = int64_t(g.hq) * D;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (hf * 64 + i < q_valid) red_add_f32(base + i * row_stride, __uint_as_float(rq[i]));
        } else if (jr < q_valid) {
          float* dst = a.dq_acc + ((int64_t(U.bi) * g.s + t0 + jr) * g.hq + h) * D + hf * (D / 2);
#pragma unroll
          for (int i = 0; i < D / 2; i += 4)
            red_add_v4(dst + i, __uint_as_float(rq[i]), __uint_as_float(rq[i + 1]), __uint_as_float(rq[i + 2]),
                       __uint_as_float(rq[i + 3]));
        }
      }
      if (!ok) break;
      // ---- dK, dV of the tile: TMEM -> bf16 -> global
      if (!(ok = mbar_wait_bounded(dkv_full, ul & 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      uint32_t rv[D / 2], rk[D / 2];
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tbase + lane_off + C::kColdV + hf * (D / 2) + c0, r0);
        tmem_ld32(tbase + lane_off + C::kColdK + hf * (D / 2) + c0, r1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          rv[c0 + i] = r0[i];
          rk[c0 + i] = r1[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dkv_empty);
      if (jr < U.k_valid) {
        const int64_t off = ((int64_t(U.bi) * g.s + U.k_t0 + jr) * g.hkv + U.g) * D + hf * (D / 2);
#pragma unroll
        for (int i = 0; i < D / 2; i += 8) {
          uint4 pv, pk;
          pv.x = pack_bf16x2(__uint_as_float(rv[i]), __uint_as_float(rv[i + 1]));
          pv.y = pack_bf16x2(__uint_as_float(rv[i + 2]), __uint_as_float(rv[i + 3]));
          pv.z = pack_bf16x2(__uint_as_float(rv[i + 4]), __uint_as_float(rv[i + 5]));
          pv.w = pack_bf16x2(__uint_as_float(rv[i + 6]), __uint_as_float(rv[i + 7]));
          // dK accumulated dS^T Q with dS unscaled: apply 1/sqrt(d) here
          pk.x = pack_bf16x2(__uint_as_float(rk[i]) * scale, __uint_as_float(rk[i + 1]) * scale);
          pk.y = pack_bf16x2(__uint_as_float(rk[i + 2]) * scale, __uint_as_float(rk[i + 3]) * scale);
          pk.z = pack_bf16x2(__uint_as_float(rk[i + 4]) * scale, __uint_as_float(rk[i + 5]) * scale);
          pk.w = pack_bf16x2(__uint_as_float(rk[i + 6]) * scale, __uint_as_float(rk[i + 7]) * scale);
          *reinterpret_cast<uint4*>(a.dv + off + i) = pv;
          *reinterpret_cast<uint4*>(a.dk + off + i) = pk;
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
