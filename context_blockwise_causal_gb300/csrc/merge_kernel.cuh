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

template <int D>
__global__ void __launch_bounds__(256) cpattn_lse_merge_kernel(const MergeArgs m) {
  constexpr int kV = D / 4;  // float4 per row; a row lies within one warp
  const int64_t rows = int64_t(m.b) * m.s * m.hq;
  const int64_t total = rows * kV;  // a multiple of 32: whole warps per iteration
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = idx / kV;  // [b, s, hq] order, as o
    const int c = int(idx % kV);
    const int h = int(row % m.hq);
    const int64_t bt = row / m.hq;
    const int t = int(bt % m.s);
    const int bi = int(bt / m.s);
    const int64_t lpos = (int64_t(bi) * m.hq + h) * m.s + t;
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
    __syncwarp();
    if (m.o_out) reinterpret_cast<float4*>(m.o_out)[idx] = r;
    if (m.o_bf16) {
      uint2 pk;
      pk.x = pack_bf16x2(r.x, r.y);
      pk.y = pack_bf16x2(r.z, r.w);
      reinterpret_cast<uint2*>(m.o_bf16)[idx] = pk;
    }
    if (c == 0) m.lse_out[lpos] = L;
  }
}

}  // namespace cpattn
