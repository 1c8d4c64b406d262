// Rotary position embedding (RoPE) applied in place to q or k with the
// positions context parallelism needs ("Megatron 面试题（一）：模型抽象与训练
// 数据流", item M016): the phase is that of the token's position in the full
// sequence -- for a rank-local zigzag shard, the zigzag map's global position
// of each local token -- and with packed samples the position restarts at
// each sample boundary. Half-rotation layout: pair (x_i, x_{i+d/2}) turns by
// theta = pos * base^(-2i/d).
//
// Accuracy: theta reaches 10^5 radians at long context, beyond what an fp32
// product and fp32 sin/cos can resolve, so the angle is formed in fp64 as
// turns (pos * inv_freq / 2pi, with inv_freq precomputed in fp64 on the
// host), reduced to [-1/2, 1/2] turn, and only then evaluated with fp32
// sincospi. One thread handles two adjacent pairs of one token for every
// head (the angle depends on the token and the pair only). HBM-bound: reads
// and writes x once.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace cpattn {

constexpr int kRopeMaxHalf = 64;  // d/2 for d <= 128

struct RopeArgs {
  __nv_bfloat16* x;  // [b, n, h, d] bf16, rotated in place
  int b, n, h;
  int s, cp, rank;   // rank < 0: natural order (n == s); else rank-local shard of `rank` (n == s / cp)
  const int* cu_seqlens;  // optional [nseq + 1] sample offsets (b == 1), device
  int nseq;
  int inverse;       // rotate by -theta (the gradient of the rotation)
  double turns_per_pos[kRopeMaxHalf];  // base^(-2i/d) / (2 pi), i < d/2
};

__device__ __forceinline__ int rope_position(const RopeArgs& a, int tok) {
  int gpos = tok;
  if (a.rank >= 0) {
    const int c = a.s / (2 * a.cp);
    gpos = tok < c ? a.rank * c + tok : (2 * a.cp - 1 - a.rank) * c + (tok - c);
  }
  if (a.cu_seqlens) {
    // last sample start <= gpos
    int lo = 0, hi = a.nseq;  // cu[lo] <= gpos < cu[hi] for well-formed offsets
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_seqlens[mid] <= gpos) lo = mid; else hi = mid;
    }
    gpos -= a.cu_seqlens[lo];
  }
  return gpos;
}

template <int D>
__global__ void __launch_bounds__(256) cpattn_rope_kernel(const RopeArgs a) {
  constexpr int kHalf = D / 2;
  constexpr int kPairs = kHalf / 2;  // threads per token: two pairs each
  const int64_t total = int64_t(a.b) * a.n * kPairs;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int j = int(idx % kPairs);
    const int64_t bt = idx / kPairs;  // b * n + tok
    const int tok = int(bt % a.n);
    const int i0 = 2 * j;
    const int pos = rope_position(a, tok);
    float sn[2], cs[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      double turns = double(pos) * a.turns_per_pos[i0 + e];
      turns -= rint(turns);
      sincospif(float(2.0 * turns), &sn[e], &cs[e]);
      if (a.inverse) sn[e] = -sn[e];
    }
    __nv_bfloat16* row = a.x + bt * a.h * D;
    for (int hh = 0; hh < a.h; ++hh) {
      __nv_bfloat162* p1 = reinterpret_cast<__nv_bfloat162*>(row + hh * D + i0);
      __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(row + hh * D + kHalf + i0);
      const float2 x1 = __bfloat1622float2(*p1), x2 = __bfloat1622float2(*p2);
      *p1 = __floats2bfloat162_rn(x1.x * cs[0] - x2.x * sn[0], x1.y * cs[1] - x2.y * sn[1]);
      *p2 = __floats2bfloat162_rn(x1.x * sn[0] + x2.x * cs[0], x1.y * sn[1] + x2.y * cs[1]);
    }
  }
}

}  // namespace cpattn
