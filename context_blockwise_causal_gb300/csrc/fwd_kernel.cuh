// Forward kernel: all virtual CP ranks in one persistent launch.
//
// One CTA per SM, 12 warps:
//   warps 0-3  softmax/correction/epilogue for sub-tile 0 (one row per thread)
//   warps 4-7  the same for sub-tile 1
//   warp 8     TMA producer (Q tiles, and the K/V ring)
//   warp 9     TMEM owner and tcgen05.mma issuer
//   warps 10-11 idle (complete the third warpgroup for the register split)
// A work unit is a 128-row query tile (of a batch element or a packed
// sample) for a pair of query heads; the two
// sub-tiles walk the same key tiles (CP-step order, see cp_schedule.cuh) so
// the MMA warp can alternate between them:
//     S0(j)=Q0 K_j^T  S1(j)=Q1 K_j^T  O0+=P0(j) V_j  S0(j+1)  O1+=P1(j) V_j  S1(j+1) ...
// while the softmax warps of one sub-tile work on S(j) the tensor core runs
// the other sub-tile's MMAs.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 after.
// P (bf16, two per column) overwrites the first 64 columns of its S tile and
// feeds the P.V MMA straight from TMEM.
//
// Online softmax and the CP correction ("大模型面试宝典 · Megatron-LM 篇", 3.2
// steps 4-5; the per-step log-sum-exp merge): per row a running maximum m
// (base-2, pre-scaled) and sum l; when a new key tile raises the maximum the
// O accumulator and l are multiplied by 2^(m_old - m_new) (a warp skips the
// TMEM round trip when none of its rows moved). Merging step after step in
// this running form is the two-stage merge L = log sum e^{L_i},
// O = sum e^{L_i - L} O_i applied incrementally; partial O never leaves TMEM.
#pragma once
#include <cuda_bf16.h>

#include "cp_schedule.cuh"
#include "ptx.cuh"

namespace cpattn {

// 12 warps: two softmax warpgroups, and a third with the producer and MMA
// warps (its last two warps only take part in the register split). The
// block is launched with kFwdLaunchRegs registers per thread; the softmax
// warpgroups then grow to kFwdSoftmaxRegs and the third shrinks to
// kFwdOtherRegs: 2*128*200 + 128*96 = 63488 <= 384*168 = 64512.
constexpr int kFwdThreads = 384;
constexpr int kFwdLaunchRegs = 168;
constexpr int kFwdSoftmaxRegs = 200;
constexpr int kFwdOtherRegs = 96;
static_assert(2 * 128 * kFwdSoftmaxRegs + 128 * kFwdOtherRegs <= kFwdThreads * kFwdLaunchRegs,
              "register split exceeds the launch budget");
// A row's running max is moved (and O, l rescaled) as soon as a key tile
// raises it. The largest P of the row is then exactly 1, which bf16 holds
// exactly; with a lagging max (FA4's thresholded rescale) that dominant P
// exceeds 1 and is rounded, which measured about twice the output error on
// peaky rows (Q, K ~ N(0, 4)) for a 2-4% gain in speed.
constexpr float kRescaleThreshold = 0.0f;  // log2 units

struct FwdArgs {
  CpGeom g;
  __nv_bfloat16* o;  // fused form: normalised output, bf16
  float* lse;        // natural-log LSE [b, hq, lse_stride] (of the step, in step form)
  int64_t lse_stride;  // row stride of lse per (batch, head): s, or a packed tensor's total
  float* o_part;     // step form: the step's normalised partial output, fp32
  int step;          // step form: the CP step computed
  float scale_log2;  // log2(e) * the softmax scale
  unsigned int* status;
  // time limit of the producer's waits for free buffers: kWaitLimitNs, or a
  // short one in the abort self-test (cpattn_selftest_abort)
  uint64_t producer_limit_ns;
  // extents for the checked build (bounds_ok): rows of the query-side and
  // key/value-side tensors, floats of lse
  int64_t q_rows, kv_rows, lse_len;
};

// K/V ring of kRing slots. When the two sub-tiles share K/V a key tile takes
// two slots (K, V); when they do not (odd GQA groups, including MHA) it
// takes four (K0, K1, V0, V1), so at d = 128 four slots would hold a single
// tile with nothing prefetched: those launches use five (the shared-memory
// budget holds five 32 KB slots beside the two Q tiles).
template <int D>
constexpr int fwd_ring(bool odd_group) {
  return D == 128 ? (odd_group ? 5 : 4) : 8;
}

template <int D, int kRing = fwd_ring<D>(false)>
struct FwdCfg {
  static constexpr int kQBytes = kTile * D * 2;  // one 128 x D bf16 tile
  static constexpr int kKVBytes = kTile * D * 2;
  static constexpr int kSlots = kRing;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kQBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kKVBytes;
  // barriers: q_full[2] q_empty[2] s_full[2] p_full[2] o_full[2] o_empty[2]
  //           drain, kv_full[kSlots] kv_empty[kSlots], p_half[2]
  static constexpr int kNumBars = 15 + 2 * kSlots;
  // Epilogue staging: 4 KB per softmax warp (32 rows x 128 bytes) to turn its
  // O stores into whole 128-byte lines; only where the ring leaves room (not
  // with the five-slot ring at d = 128).
  static constexpr int kStageBytes = kRing == fwd_ring<D>(false) ? 8 * 32 * 128 : 0;
  static constexpr int kOffStage = (kOffBar + kNumBars * 8 + 127) & ~127;
  static constexpr int kOffMisc = kOffStage + kStageBytes;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static constexpr uint32_t kColO = 256;
};

enum FwdStatusBits : unsigned int {
  kStatusProducer = 1u << 0,
  kStatusMma = 1u << 1,
  kStatusSoftmax = 1u << 2,
  kStatusDrain = 1u << 3,  // copies or MMAs still in flight after the time limit
};

// kStep = false: the fused forward (all CP steps, merged on chip, bf16 O).
// kStep = true: one CP step `a.step` for every rank, unmerged: each query
// row's softmax over that step's keys only, written as an fp32 partial O and
// its LSE ("大模型面试宝典 · Megatron-LM 篇", 3.2 step 4, before correction);
// rows that take no part in the step get O = 0, L = -inf.
// kTP: units are tile pairs (a.g.tile_pairs), not head pairs.
// kShortWaits: the producer's waits for free buffers use a.producer_limit_ns
// (the abort self-test) instead of the compile-time limit.
template <int D, bool kStep, int kRing, bool kTP, bool kShortWaits = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    cpattn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const FwdArgs a) {
  using C = FwdCfg<D, kRing>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sKV = smem + C::kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 2;
  uint64_t* s_full = bars + 4;
  uint64_t* p_full = bars + 6;
  uint64_t* o_full = bars + 8;
  uint64_t* o_empty = bars + 10;
  uint64_t* drain = bars + 12;
  uint64_t* kv_full = bars + 13;
  uint64_t* kv_empty = bars + 13 + C::kSlots;
  uint64_t* p_half = bars + 13 + 2 * C::kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const CpGeom& g = a.g;
  const int num_units = fwd_num_units(g);
  const int grid = gridDim.x;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_half[i], 4);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 4);
    }
    mbar_init(drain, 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp >= 8) {
  reg_dealloc<kFwdOtherRegs>();  // this warpgroup: producer, MMA, two idle warps
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t plimit = kShortWaits ? a.producer_limit_ns : kWaitLimitNs;
      bool ok = true;
      uint32_t nload = 0;
      int ul = 0;
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const FwdUnit U = fwd_decode_unit_t<kTP>(g, idx);
        if (U.n == 0) continue;  // a tile a shorter packed sample does not have
        KvWalk w(g, U);
        if constexpr (kStep) {
          w.only_step(a.step);
          if (w.step_tiles(a.step) == 0) continue;  // no key tile at this step
        }
        if (ul > 0) {
          ok = mbar_wait_bounded(&q_empty[0], (ul - 1) & 1, abort_flag, plimit) &&
               mbar_wait_bounded(&q_empty[1], (ul - 1) & 1, abort_flag, plimit);
          if (!ok) break;
        }
        for (int sub = 0; sub < 2; ++sub) {
          mbar_arrive_expect_tx(&q_full[sub], C::kQBytes);
          const int h = sub ? U.h1 : U.h0;
          const int qrow = U.tok0 + (sub ? U.q_t1 : U.q_t0);
          bounds_ok(qrow >= 0 && qrow < a.q_rows && h >= 0 && h < g.hq, a.status);
          for (int x = 0; x < D; x += 64)
            tma_load_3d(sQ + sub * C::kQBytes + (x / 64) * (kTile * 128), &tmq, &q_full[sub], x, h, qrow);
        }
        const bool shared_kv = U.g0 == U.g1;
        int chunk, tile;
        bool dg;
        auto load = [&](const CUtensorMap* map, int head, int row) -> bool {
          bounds_ok(row >= 0 && row < a.kv_rows && head >= 0 && head < g.hkv, a.status);
          const uint32_t slot = nload % C::kSlots;
          if (nload >= (uint32_t)C::kSlots) {
            if (!mbar_wait_bounded(&kv_empty[slot], ((nload / C::kSlots) - 1) & 1, abort_flag, plimit))
              return false;
          }
          mbar_arrive_expect_tx(&kv_full[slot], C::kKVBytes);
          uint8_t* dst = sKV + slot * C::kKVBytes;
          for (int x = 0; x < D; x += 64) tma_load_3d(dst + (x / 64) * (kTile * 128), map, &kv_full[slot], x, head, row);
          ++nload;
          return true;
        };
        while (ok && w.next(chunk, tile, dg)) {
          const int row = U.tok0 + kv_chunk_row(g, chunk, U.c) + tile * kTile;
          ok = load(&tmk, U.g0, row) && (shared_kv || load(&tmk, U.g1, row)) && load(&tmv, U.g0, row) &&
               (shared_kv || load(&tmv, U.g1, row));
        }
        ++ul;
      }
      if (!ok) atomicOr(a.status, kStatusProducer);
      // Let every copy still in flight land before the CTA can exit (older
      // ones landed before their slot was handed back). These waits do not
      // stop on the abort flag: the copies complete regardless.
      bool drained = true;
      const uint32_t first = nload > (uint32_t)C::kSlots ? nload - C::kSlots : 0;
      for (uint32_t i = first; i < nload; ++i)
        drained &= mbar_wait_drain(&kv_full[i % C::kSlots], (i / C::kSlots) & 1, kWaitLimitNs);
      if (ul > 0) {
        drained &= mbar_wait_drain(&q_full[0], (ul - 1) & 1, kWaitLimitNs);
        drained &= mbar_wait_drain(&q_full[1], (ul - 1) & 1, kWaitLimitNs);
      }
      if (!drained) atomicOr(a.status, kStatusDrain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs this role; elect.sync picks the issuing lane)
    {
      constexpr uint32_t idS = make_idesc_bf16(kTile, kTile, false, false);
      constexpr uint32_t idO = make_idesc_bf16(kTile, D, false, true);
      const uint64_t dQ[2] = {make_sdesc_sw128(smem_u32(sQ), 16, 1024),
                              make_sdesc_sw128(smem_u32(sQ + C::kQBytes), 16, 1024)};
      const uint64_t dKV0 = make_sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dV0 = make_sdesc_sw128(smem_u32(sKV), 16384, 1024);
      auto issue_S = [&](int sub, uint32_t slot) {
        const uint64_t kb = dKV0 + ((slot * C::kKVBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
          umma_ss_w(tbase + sub * kTile, dQ[sub] + off, kb + off, idS, kk > 0);
        }
      };
      // O += P V over keys [64*half, 64*half + 64) (K-steps 4*half .. +3)
      auto issue_PV = [&](int sub, uint32_t slot, bool acc, int half) {
        const uint64_t vb = dV0 + ((slot * C::kKVBytes) >> 4);
#pragma unroll
        for (int q = 0; q < kTile / 32; ++q) {
          const int kk = half * (kTile / 32) + q;
          umma_ts_w(tbase + C::kColO + sub * D, tbase + sub * kTile + kk * 8, vb + ((kk * 2048) >> 4), idO,
                    (acc || kk > 0) ? 1u : 0u);
        }
      };
      uint32_t ncons = 0;
      auto take = [&](uint32_t& slot, uint32_t& par) {
        slot = ncons % C::kSlots;
        par = (ncons / C::kSlots) & 1;
        ++ncons;
      };
      bool ok = true;
      uint32_t pcnt[2] = {0, 0};
      int ul = 0;
      for (int rd = 0; ok; ++rd) {
        const int idx = snake_unit(rd, blockIdx.x, grid);
        if (idx >= num_units) break;
        const FwdUnit U = fwd_decode_unit_t<kTP>(g, idx);
        if (U.n == 0) continue;
        const bool shared_kv = U.g0 == U.g1;
        const int n = kStep ? KvWalk(g, U).step_tiles(a.step) : U.n;
        if (kStep && n == 0) continue;
        ok = mbar_wait_warp(&q_full[0], ul & 1, abort_flag, kWaitLimitNs) &&
             mbar_wait_warp(&q_full[1], ul & 1, abort_flag, kWaitLimitNs);
        if (!ok) break;
        // prologue: S0(0), S1(0)
        uint32_t k0, k0p, k1, k1p;
        take(k0, k0p);
        if (shared_kv) { k1 = k0; k1p = k0p; } else take(k1, k1p);
        // waits on TMA-filled buffers need no tcgen05 fence: the copies and
        // the MMA operand reads are both async-proxy operations ordered by
        // the transaction barrier
        if (!(ok = mbar_wait_warp(&kv_full[k0], k0p, abort_flag, kWaitLimitNs))) break;
        issue_S(0, k0);
        umma_commit_w(&s_full[0]);
        if (!shared_kv) umma_commit_w(&kv_empty[k0]);
        if (n == 1) umma_commit_w(&q_empty[0]);
        if (!shared_kv && !(ok = mbar_wait_warp(&kv_full[k1], k1p, abort_flag, kWaitLimitNs))) break;
        issue_S(1, k1);
        umma_commit_w(&s_full[1]);
        umma_commit_w(&kv_empty[k1]);
        if (n == 1) umma_commit_w(&q_empty[1]);
        for (int j = 0; j < n && ok; ++j) {
          uint32_t v0, v0p, v1, v1p;
          take(v0, v0p);
          if (shared_kv) { v1 = v0; v1p = v0p; } else take(v1, v1p);
          // ---- sub-tile 0: O0 += P0(j) V_j (first half of the keys as soon
          // as their P is in TMEM), then S0(j+1)
          ok = mbar_wait_warp(&kv_full[v0], v0p, abort_flag, kWaitLimitNs) &&
               mbar_wait_warp(&p_half[0], pcnt[0] & 1, abort_flag, kWaitLimitNs) &&
               (j > 0 || ul == 0 || mbar_wait_warp(&o_empty[0], (ul - 1) & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          issue_PV(0, v0, j > 0, 0);
          if (!(ok = mbar_wait_warp(&p_full[0], pcnt[0] & 1, abort_flag, kWaitLimitNs))) break;
          ++pcnt[0];
          tc_fence_after();
          issue_PV(0, v0, j > 0, 1);
          if (!shared_kv) umma_commit_w(&kv_empty[v0]);
          if (j == n - 1) umma_commit_w(&o_full[0]);
          uint32_t nk0 = 0, nk0p = 0, nk1 = 0, nk1p = 0;
          if (j + 1 < n) {
            take(nk0, nk0p);
            if (shared_kv) { nk1 = nk0; nk1p = nk0p; } else take(nk1, nk1p);
            if (!(ok = mbar_wait_warp(&kv_full[nk0], nk0p, abort_flag, kWaitLimitNs))) break;
            issue_S(0, nk0);
            umma_commit_w(&s_full[0]);
            if (!shared_kv) umma_commit_w(&kv_empty[nk0]);
            if (j + 1 == n - 1) umma_commit_w(&q_empty[0]);
          }
          // ---- sub-tile 1: O1 += P1(j) V_j, then S1(j+1)
          ok = (shared_kv || mbar_wait_warp(&kv_full[v1], v1p, abort_flag, kWaitLimitNs)) &&
               mbar_wait_warp(&p_half[1], pcnt[1] & 1, abort_flag, kWaitLimitNs) &&
               (j > 0 || ul == 0 || mbar_wait_warp(&o_empty[1], (ul - 1) & 1, abort_flag, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          issue_PV(1, v1, j > 0, 0);
          if (!(ok = mbar_wait_warp(&p_full[1], pcnt[1] & 1, abort_flag, kWaitLimitNs))) break;
          ++pcnt[1];
          tc_fence_after();
          issue_PV(1, v1, j > 0, 1);
          umma_commit_w(&kv_empty[v1]);
          if (j == n - 1) umma_commit_w(&o_full[1]);
          if (j + 1 < n) {
            if (!shared_kv && !(ok = mbar_wait_warp(&kv_full[nk1], nk1p, abort_flag, kWaitLimitNs))) break;
            issue_S(1, nk1);
            umma_commit_w(&s_full[1]);
            umma_commit_w(&kv_empty[nk1]);
            if (j + 1 == n - 1) umma_commit_w(&q_empty[1]);
          }
        }
        ++ul;
      }
      if (!ok && lane == 0) atomicOr(a.status, kStatusMma);
      // No MMA may be in flight when TMEM is released (nor when the shared
      // memory they read is), whether or not a role gave up.
      umma_commit_w(drain);
      if (!mbar_wait_drain_warp(drain, 0, kWaitLimitNs) && lane == 0) atomicOr(a.status, kStatusDrain);
    }
  }
  } else {
    reg_alloc<kFwdSoftmaxRegs>();  // the two softmax warpgroups
    // ------------------------------------------------------------ softmax
    const int sub = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + sub * kTile;
    const uint32_t tO = tbase + lane_off + C::kColO + sub * D;
    const float sl2 = a.scale_log2;
    bool ok = true;
    uint32_t scnt = 0;
    int ul = 0;
    for (int rd = 0; ok; ++rd) {
      const int idx = snake_unit(rd, blockIdx.x, grid);
      if (idx >= num_units) break;
      const FwdUnit U = fwd_decode_unit_t<kTP>(g, idx);
      if (U.n == 0) continue;
      // this sub-tile's query rows (a second head, or the next query tile)
      const int q_t = sub ? U.q_t1 : U.q_t0;
      const int q_valid = sub ? U.q_valid1 : U.q_valid;
      // tile pairs: the position of sub-tile 0's fully masked tile (-1: none)
      const int jd = kTP ? fwd_dead_pos(g, U, sub, kStep ? a.step : -1) : -1;
      KvWalk w(g, U);
      int n = U.n;
      if constexpr (kStep) {
        w.only_step(a.step);
        n = w.step_tiles(a.step);
        if (n == 0) {
          // the unit's rows take no part in this step: O = 0, L = -inf
          if (row < q_valid && (sub == 0 || U.store1)) {
            const int h = sub ? U.h1 : U.h0;
            const int t = q_t + row;
            const int64_t li = (int64_t(U.bi) * g.hq + h) * a.lse_stride + U.lse_t0 + t;
            if (bounds_ok(int64_t(U.tok0) + t < a.q_rows && h < g.hq && li < a.lse_len, a.status)) {
              float4* dst = reinterpret_cast<float4*>(a.o_part + ((int64_t(U.tok0) + t) * g.hq + h) * D);
#pragma unroll
              for (int c0 = 0; c0 < D / 4; ++c0) dst[c0] = make_float4(0.f, 0.f, 0.f, 0.f);
              a.lse[li] = -INFINITY;
            }
          }
          continue;
        }
      }
      float m_used = -INFINITY;
      float l = 0.f;
      // Without ragged tiles (and outside the step form) the walk's only
      // masked position is the query tile's diagonal, where step 0 ends: the
      // softmax warps then follow the positions without the walk itself.
      const bool walkless = !kStep && (U.c & (kTile - 1)) == 0;
      const int jdiag = g.causal ? (U.half ? U.tpc : 0) + U.u : -1;
      for (int j = 0; j < n; ++j) {
        int chunk = 0, tile = 0;
        bool walk_dg = false, dg = false, dead = false;
        int n_valid = kTile;
        if (walkless) {
          walk_dg = j == jdiag;
        } else {
          w.next(chunk, tile, walk_dg);
          const int rem = U.c - tile * kTile;
          n_valid = rem < kTile ? rem : kTile;
        }
        if constexpr (kTP)
          fwd_pos_mask(jd, j, walk_dg, dg, dead);
        else
          dg = walk_dg;
        if (!(ok = mbar_wait_bounded(&s_full[sub], scnt & 1, abort_flag, kWaitLimitNs))) break;
        ++scnt;
        tc_fence_after();
        float s[kTile];
        float hw_max;
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          float m4[4];
          tmem_ld32x4_max(tS, tS + 32, tS + 64, tS + 96, r0, r1, r2, r3, m4);
          hw_max = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
            s[64 + i] = __uint_as_float(r2[i]);
            s[96 + i] = __uint_as_float(r3[i]);
          }
        }
        // row max: from the load itself, except on a masked tile (the diagonal
        // or a ragged chunk end), where it is taken over the unmasked scores
        float m_raw = hw_max;
        if (dg || dead || n_valid < kTile) {
          const int lim = dead ? -1 : dg ? (row < n_valid - 1 ? row : n_valid - 1) : n_valid - 1;
#pragma unroll
          for (int i = 0; i < kTile; ++i)
            if (i > lim) s[i] = -INFINITY;
          // row max: eight independent chains of 3-input maxima, chain k over
          // the scores k, k+8, ..., k+120
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float m = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
            for (int i = 24; i + 8 < kTile; i += 16) m = fmax3(m, s[i + k], s[i + 8 + k]);
            mx[k] = fmaxf(m, s[kTile - 8 + k]);
          }
          m_raw = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
        }
        const float m_new = m_raw * sl2;
        const bool upd = m_new > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (upd) {
          alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - m_new);
          m_used = m_new;
        }
        const float neg = (m_used == -INFINITY) ? 0.f : -m_used;
        const bool rescale = j > 0 && __any_sync(0xffffffffu, upd);
        // P = 2^(S*scale*log2e - m), packed to bf16 pairs as it is formed so
        // the fp32 scores die early; the row sum uses the fp32 values. The
        // first 64 keys' P goes to TMEM (and to the MMA warp) before the
        // second half is formed, so P.V starts while the warps still work.
        uint32_t pk[32];
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negx2 = f2_pack(neg, neg);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int q = 0; q < kTile / 4; ++q) {
            const int i = hh * (kTile / 4) + q;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sl2x2, negx2), x0, x1);
            const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
            const uint64_t e = f2_pack(e0, e1);
            if ((i & 3) == 0) acc0 = f2_add(acc0, e);
            else if ((i & 3) == 1) acc1 = f2_add(acc1, e);
            else if ((i & 3) == 2) acc2 = f2_add(acc2, e);
            else acc3 = f2_add(acc3, e);
            pk[q] = pack_bf16x2(e0, e1);
          }
          if (hh == 0 && rescale) {
            // Rescale O before any P.V of this tile (the MMA warp waits for
            // p_half). This row's O accumulator is idle: P.V of step j-1
            // completed before S(j) was signalled. The stores are not waited
            // for one by one: the P store below waits for all of them before
            // the fence and the p_half arrival publish the columns.
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(tO + c0, r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32_nowait(tO + c0, r);
            }
          }
          tmem_st32(tS + hh * 32, pk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(hh == 0 ? &p_half[sub] : &p_full[sub]);
        }
        float a0, a1;
        f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a0, a1);
        l = l * alpha + (a0 + a1);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, L = (m + log2 l) ln 2
      if (!(ok = mbar_wait_bounded(&o_full[sub], ul & 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      uint32_t ov[D];
      if constexpr (D == 128) {
        uint32_t r0[64], r1[64];
        tmem_ld64(tO, r0);
        tmem_ld64(tO + 64, r1);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          ov[i] = r0[i];
          ov[64 + i] = r1[i];
        }
      } else {
        uint32_t r0[64];
        tmem_ld64(tO, r0);
#pragma unroll
        for (int i = 0; i < 64; ++i) ov[i] = r0[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[sub]);
      const bool store = row < q_valid && (sub == 0 || U.store1);
      if (kStep && store) {
        const int h = sub ? U.h1 : U.h0;
        const int t = q_t + row;
        const float inv = 1.f / l;
        const int64_t li = (int64_t(U.bi) * g.hq + h) * a.lse_stride + U.lse_t0 + t;
        if (bounds_ok(int64_t(U.tok0) + t < a.q_rows && h < g.hq && li < a.lse_len, a.status)) {
          float4* dst = reinterpret_cast<float4*>(a.o_part + ((int64_t(U.tok0) + t) * g.hq + h) * D);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 4)
            dst[c0 / 4] = make_float4(__uint_as_float(ov[c0]) * inv, __uint_as_float(ov[c0 + 1]) * inv,
                                      __uint_as_float(ov[c0 + 2]) * inv, __uint_as_float(ov[c0 + 3]) * inv);
          a.lse[li] = (m_used + log2f(l)) * 0.69314718055994530942f;
        }
      } else if (!kStep && C::kStageBytes > 0) {
        // O through the warp's staging buffer, 64 columns at a time: each
        // thread writes its row's 128 bytes (16-byte pieces at slot
        // k ^ (row & 7), so neither pass has bank conflicts), then each store
        // covers 4 rows x 128 contiguous bytes, whole lines. Every lane takes
        // part; rows outside the tile's valid part or of a repeated head are
        // not written.
        const int h = sub ? U.h1 : U.h0;
        const float inv = 1.f / l;
        const bool write_head = sub == 0 || U.store1;
        uint4* stg = reinterpret_cast<uint4*>(smem + C::kOffStage + warp * (32 * 128));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c0 = c * 64 + k * 8;
            uint4 pkv;
            pkv.x = pack_bf16x2(__uint_as_float(ov[c0 + 0]) * inv, __uint_as_float(ov[c0 + 1]) * inv);
            pkv.y = pack_bf16x2(__uint_as_float(ov[c0 + 2]) * inv, __uint_as_float(ov[c0 + 3]) * inv);
            pkv.z = pack_bf16x2(__uint_as_float(ov[c0 + 4]) * inv, __uint_as_float(ov[c0 + 5]) * inv);
            pkv.w = pack_bf16x2(__uint_as_float(ov[c0 + 6]) * inv, __uint_as_float(ov[c0 + 7]) * inv);
            stg[lane * 8 + (k ^ (lane & 7))] = pkv;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);  // the warp's row
            const int part = lane & 7;          // 16-byte piece of the 128
            const uint4 v = stg[r * 8 + (part ^ (r & 7))];
            const int trow = wq * 32 + r;       // row within the tile
            if (write_head && trow < q_valid &&
                bounds_ok(int64_t(U.tok0) + q_t + trow < a.q_rows && h < g.hq, a.status))
              *reinterpret_cast<uint4*>(a.o + ((int64_t(U.tok0) + q_t + trow) * g.hq + h) * D + c * 64 + part * 8) = v;
          }
          __syncwarp();
        }
        const int64_t li = (int64_t(U.bi) * g.hq + h) * a.lse_stride + U.lse_t0 + q_t + row;
        if (store && bounds_ok(li < a.lse_len, a.status)) a.lse[li] = (m_used + log2f(l)) * 0.69314718055994530942f;
      } else if (store && bounds_ok(int64_t(U.tok0) + q_t + row < a.q_rows &&
                                        (int64_t(U.bi) * g.hq + (sub ? U.h1 : U.h0)) * a.lse_stride + U.lse_t0 +
                                                q_t + row < a.lse_len,
                                    a.status)) {
        const int h = sub ? U.h1 : U.h0;
        const int t = q_t + row;
        const float inv = 1.f / l;
        __nv_bfloat16* dst = a.o + ((int64_t(U.tok0) + t) * g.hq + h) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 8) {
          uint4 pkv;
          pkv.x = pack_bf16x2(__uint_as_float(ov[c0 + 0]) * inv, __uint_as_float(ov[c0 + 1]) * inv);
          pkv.y = pack_bf16x2(__uint_as_float(ov[c0 + 2]) * inv, __uint_as_float(ov[c0 + 3]) * inv);
          pkv.z = pack_bf16x2(__uint_as_float(ov[c0 + 4]) * inv, __uint_as_float(ov[c0 + 5]) * inv);
          pkv.w = pack_bf16x2(__uint_as_float(ov[c0 + 6]) * inv, __uint_as_float(ov[c0 + 7]) * inv);
          *reinterpret_cast<uint4*>(dst + c0) = pkv;
        }
        a.lse[(int64_t(U.bi) * g.hq + h) * a.lse_stride + U.lse_t0 + t] = (m_used + log2f(l)) * 0.69314718055994530942f;
      }
      ++ul;
    }
    if (!ok && lane == 0) atomicOr(a.status, kStatusSoftmax);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace cpattn
