// Log-sum-exp merge of two partial attention results over disjoint key sets:
// the correction step of context parallelism in its unfused form
// ("大模型面试宝典 · Megatron-LM 篇", 3.2 steps 4-5: L is corrected after
// every step, each partial O by exp(L_i - L) before the sum):
//     L = log(e^{L_a} + e^{L_b}),   O = e^{L_a - L} O_a + e^{L_b - L} O_b.
// Rows with L_a = L_b = -inf (no key seen yet) stay L = -inf, O = 0.
// Element-wise over rows; HBM-bound: per row it reads 2 (d fp32 + 1 fp32)
// and writes d fp32 (or d bf16) + 1 fp32.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace cpattn {

struct MergeArgs {
  int b, s, hq;
  const float* o_a;    // [b, s, hq, d] fp32
  const float* lse_a;  // [b, hq, s] fp32, natural log
  const float* o_b;    // may be null (no second part)
  const float* lse_b;  // null iff o_b is null
  float* o_out;        // may alias o_a; may be null if o_bf16 is set
  float* lse_out;      // may alias lse_a
  __nv_bfloat16* o_bf16;  // optional bf16 copy of the merged O
};

// A warp takes a contiguous run of rows (one row per D/4 lanes: the whole
// warp at d = 128, a half-warp at d = 64) and decodes its first row once;
// the (batch, token, head) of the following rows are stepped, so the loop
// does no integer division.
template <int D>
__global__ void __launch_bounds__(256) cpattn_lse_merge_kernel(const MergeArgs m) {
  constexpr int kV = D / 4;               // float4 per row
  constexpr int kRowsPerStep = 32 / kV;   // rows a warp handles at once
  const int64_t rows = int64_t(m.b) * m.s * m.hq;
  const int lane = threadIdx.x & 31;
  const int c = lane % kV;
  const int sub = lane / kV;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  // rows per warp, a multiple of kRowsPerStep
  const int64_t per = ((rows + nwarps - 1) / nwarps + kRowsPerStep - 1) / kRowsPerStep * kRowsPerStep;
  const int64_t r_begin = warp * per;
  const int64_t r_end = r_begin + per < rows ? r_begin + per : rows;
  if (r_begin >= r_end) return;
  // this lane's first row, decoded once
  int64_t row = r_begin + sub;
  int h = int(row % m.hq);
  int64_t bt = row / m.hq;
  int t = int(bt % m.s);
  int bi = int(bt / m.s);
  for (; row - sub < r_end; row += kRowsPerStep) {
    if (row < r_end) {
      const int64_t lpos = (int64_t(bi) * m.hq + h) * m.s + t;
      const int64_t idx = row * kV + c;
      const float la = m.lse_a[lpos];
      const float lb = m.lse_b ? m.lse_b[lpos] : -INFINITY;
      const float4 oa = reinterpret_cast<const float4*>(m.o_a)[idx];
      const float4 ob = m.o_b ? reinterpret_cast<const float4*>(m.o_b)[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float mx = fmaxf(la, lb);
      float wa = 0.f, wb = 0.f, L = -INFINITY;
      if (mx > -INFINITY) {
        const float ea = expf(la - mx), eb = expf(lb - mx);
        const float sum = ea + eb;
        L = mx + logf(sum);
        wa = ea / sum;
        wb = eb / sum;
      }
      const float4 r = make_float4(wa * oa.x + wb * ob.x, wa * oa.y + wb * ob.y, wa * oa.z + wb * ob.z,
                                   wa * oa.w + wb * ob.w);
      // every lane of the row has read lse_a / o_a before any lane writes
      // (the outputs may alias the first input)
      __syncwarp(kV == 32 ? 0xffffffffu : (0xffffu << (16 * sub)));
      if (m.o_out) reinterpret_cast<float4*>(m.o_out)[idx] = r;
      if (m.o_bf16) {
        uint2 pk;
        pk.x = pack_bf16x2(r.x, r.y);
        pk.y = pack_bf16x2(r.z, r.w);
        reinterpret_cast<uint2*>(m.o_bf16)[idx] = pk;
      }
      if (c == 0) m.lse_out[lpos] = L;
    }
    // step (bi, t, h) by kRowsPerStep rows ([b, s, hq] order)
#pragma unroll
    for (int k = 0; k < kRowsPerStep; ++k) {
      if (++h == m.hq) {
        h = 0;
        if (++t == m.s) {
          t = 0;
          ++bi;
        }
      }
    }
  }
}

}  // namespace cpattn
