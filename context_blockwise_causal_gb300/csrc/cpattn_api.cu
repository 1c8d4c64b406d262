// C-ABI entry points declared in include/cpattn.h: argument checks, TMA
// tensor-map encoding and kernel launches. No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/cpattn.h"
#include "bwd_kernel.cuh"
#include "fwd_kernel.cuh"
#include "merge_kernel.cuh"
#include "rope_kernel.cuh"
#include "tmap.h"

namespace cpattn {

// Sticky status word written by kernels that give up waiting.
__device__ unsigned int g_device_status;

// Backward scratch for cpattn_bwd_noalloc (see include/cpattn.h): a fixed
// device array in this library's module, so that entry point needs no
// allocation. Every device that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  bool sm103 = false;
  int num_sms = 0;
  unsigned int* status = nullptr;
  // kernel attributes already set, per kernel; set once, read by any thread
  std::atomic<bool> fwd_attr[17] = {};  // [d == 128][step form][five-slot ring][tile pairs]; 16: self-test
  std::atomic<bool> bwd_attr[3] = {};   // [d == 128]; 2: self-test
};
DeviceInfo g_devs[kMaxDevices];
std::mutex g_mu;
// Cap on the grid of the persistent attention kernels (0: one CTA per SM).
std::atomic<int> g_max_ctas{0};

// Grid of a persistent kernel over `units` work units: one CTA per SM, at
// most the cap set by cpattn_set_max_ctas, at most one per unit.
int persistent_grid(const DeviceInfo* di, int64_t units) {
  const int cap_set = g_max_ctas.load(std::memory_order_relaxed);
  const int cap = cap_set > 0 && cap_set < di->num_sms ? cap_set : di->num_sms;
  return units < cap ? int(units) : cap;
}

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_devs[dev];
  if (!di.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    di.sm103 = (major == 10 && minor == 3);
    di.num_sms = sms;
    if (di.sm103) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return CPATTN_ERR_CUDA;
      di.status = static_cast<unsigned int*>(p);
    }
    di.init = true;
  }
  *out = &di;
  return di.sm103 ? CPATTN_OK : CPATTN_ERR_UNSUPPORTED_ARCH;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_geometry(int b, int s, int hq, int hkv, int d, int cp) {
  if (b < 1 || s < 1 || hq < 1 || hkv < 1 || cp < 1) return CPATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return CPATTN_ERR_INVALID_ARG;
  if (hq % hkv != 0) return CPATTN_ERR_INVALID_ARG;
  if (s % (2 * cp) != 0) return CPATTN_ERR_INVALID_ARG;
  if (int64_t(b) * s >= (int64_t(1) << 31)) return CPATTN_ERR_INVALID_ARG;
  const int64_t units = int64_t(b) * ((hq + 1) / 2) * 2 * cp * ((s / (2 * cp) + kTile - 1) / kTile);
  if (units >= (int64_t(1) << 31)) return CPATTN_ERR_INVALID_ARG;
  // the tile-padded row count of the backward's L/D vectors is an int
  if (int64_t(2) * cp * ((s / (2 * cp) + kTile - 1) / kTile) * kTile >= (int64_t(1) << 31)) return CPATTN_ERR_INVALID_ARG;
  return CPATTN_OK;
}

CpGeom make_geom(int b, int s, int hq, int hkv, int cp, int causal) {
  CpGeom g;
  g.b = b;
  g.s = s;
  g.hq = hq;
  g.hkv = hkv;
  g.cp = cp;
  g.causal = causal ? 1 : 0;
  g.c = s / (2 * cp);
  g.tpc = (g.c + kTile - 1) / kTile;
  g.npairs = (hq + 1) / 2;
  g.tile_pairs = use_tile_pairs(g) ? 1 : 0;
  set_fast_divs(g);
  return g;
}

// K/V bytes of the heads whose tile-pair units may be in flight together
// (see set_tile_pair_blocks): a quarter of L2.
constexpr int64_t kTilePairKvBudget = 32ll << 20;

template <int D, bool kStep, int kRing, bool kTP, bool kShort = false>
int launch_fwd_ring(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& args_in,
                    DeviceInfo* di, cudaStream_t st) {
  using C = FwdCfg<D, kRing>;
  const int slot =
      kShort ? 16 : (D == 128 ? 8 : 0) + (kStep ? 4 : 0) + (kRing == fwd_ring<D>(false) ? 0 : 2) + (kTP ? 1 : 0);
  if (!di->fwd_attr[slot].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(cpattn_fwd_kernel<D, kStep, kRing, kTP, kShort>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    // The in-kernel register split assumes exactly kFwdLaunchRegs registers
    // per thread at launch; with fewer, the growing warpgroups would wait
    // for registers that never come free.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, cpattn_fwd_kernel<D, kStep, kRing, kTP, kShort>) != cudaSuccess) return CPATTN_ERR_CUDA;
    if (fa.numRegs != kFwdLaunchRegs) return CPATTN_ERR_LAUNCH_FAILED;
    di->fwd_attr[slot].store(true, std::memory_order_release);
  }
  FwdArgs args = args_in;
  if (kTP) {  // K/V of one (sequence, KV head): s tokens of K and of V
    const int64_t per_pair = 4ll * args.g.s * D;
    set_tile_pair_blocks(args.g, persistent_grid(di, int64_t(1) << 31), int(kTilePairKvBudget / per_pair));
  }
  const int units = fwd_num_units(args.g);
  const int grid = persistent_grid(di, units);
  cpattn_fwd_kernel<D, kStep, kRing, kTP, kShort><<<grid, kFwdThreads, C::kSmemBytes, st>>>(tq, tk, tv, args);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_LAUNCH_FAILED;
}

// The K/V ring follows the head grouping (see fwd_ring).
template <int D, bool kStep>
int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& args,
               DeviceInfo* di, cudaStream_t st) {
  // head pairs that straddle KV groups need separate K/V tiles (tile pairs share them)
  if (args.g.tile_pairs) return launch_fwd_ring<D, kStep, fwd_ring<D>(false), true>(tq, tk, tv, args, di, st);
  const bool odd_group = (args.g.hq / args.g.hkv) % 2 != 0;
  if (fwd_ring<D>(odd_group) != fwd_ring<D>(false))
    return launch_fwd_ring<D, kStep, fwd_ring<D>(true), false>(tq, tk, tv, args, di, st);
  return launch_fwd_ring<D, kStep, fwd_ring<D>(false), false>(tq, tk, tv, args, di, st);
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

namespace {
bool valid_scale(float scale) { return scale > 0.f && scale <= 3.0e38f; }
double default_scale(int d) { return 1.0 / std::sqrt(double(d)); }
}  // namespace

namespace {
// The fused forward. `geom` overrides the uniform geometry (packed samples,
// or the rank-local form); the query-side tensors then have q_rows rows and
// the key/value side kv_rows (both b * s by default).
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq, int hkv, int d,
             int cp, int causal, double scale, void* stream, int64_t lse_stride = -1, const CpGeom* geom = nullptr,
             uint64_t q_rows = 0, uint64_t kv_rows = 0, uint64_t producer_limit_ns = kWaitLimitNs) {
  if (!q || !k || !v || !o || !lse) return CPATTN_ERR_NULL_PTR;
  int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return CPATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di))) return rc;
  CUtensorMap tq, tk, tv;
  if (q_rows == 0) q_rows = uint64_t(b) * s;
  if (kv_rows == 0) kv_rows = uint64_t(b) * s;
  if (!encode_bf16_rows_heads_d(&tq, q, q_rows, hq, d, kTile) ||
      !encode_bf16_rows_heads_d(&tk, k, kv_rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&tv, v, kv_rows, hkv, d, kTile))
    return CPATTN_ERR_CUDA;
  FwdArgs args;
  args.g = geom ? *geom : make_geom(b, s, hq, hkv, cp, causal);
  args.o = static_cast<__nv_bfloat16*>(o);
  args.lse = lse;
  args.lse_stride = lse_stride < 0 ? s : lse_stride;
  args.q_rows = int64_t(q_rows);
  args.kv_rows = int64_t(kv_rows);
  args.lse_len = int64_t(b) * hq * args.lse_stride;
  args.o_part = nullptr;
  args.step = -1;
  args.scale_log2 = float(1.4426950408889634 * scale);
  args.status = di->status;
  args.producer_limit_ns = producer_limit_ns;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (producer_limit_ns != kWaitLimitNs)  // the abort self-test: d = 128, head pairs sharing K/V (checked there)
    return launch_fwd_ring<128, false, fwd_ring<128>(false), false, true>(tq, tk, tv, args, di, st);
  return d == 128 ? launch_fwd<128, false>(tq, tk, tv, args, di, st) : launch_fwd<64, false>(tq, tk, tv, args, di, st);
}
}  // namespace

extern "C" int cpattn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq,
                             int hkv, int d, int cp, int causal, float scale, void* stream) {
  if (!valid_scale(scale)) return CPATTN_ERR_INVALID_ARG;
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  return fwd_impl(q, k, v, o, lse, b, s, hq, hkv, d, cp, causal, double(scale), stream);
}

extern "C" int cpattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq,
                          int hkv, int d, int cp, int causal, void* stream) {
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  return fwd_impl(q, k, v, o, lse, b, s, hq, hkv, d, cp, causal, default_scale(d), stream);
}

namespace {
// One CP step, unmerged (the step form of the forward kernel); geometry and
// row counts as for fwd_impl.
int step_impl(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int b, int s, int hq,
              int hkv, int d, int cp, int step, int causal, double scale, void* stream, const CpGeom* geom = nullptr,
              uint64_t q_rows = 0, uint64_t kv_rows = 0, int64_t lse_stride = -1) {
  if (!q || !k || !v || !o_part || !lse_part) return CPATTN_ERR_NULL_PTR;
  int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  if (step < 0 || step >= cp) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) || !aligned16(lse_part))
    return CPATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di))) return rc;
  CUtensorMap tq, tk, tv;
  if (q_rows == 0) q_rows = uint64_t(b) * s;
  if (kv_rows == 0) kv_rows = uint64_t(b) * s;
  if (!encode_bf16_rows_heads_d(&tq, q, q_rows, hq, d, kTile) ||
      !encode_bf16_rows_heads_d(&tk, k, kv_rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&tv, v, kv_rows, hkv, d, kTile))
    return CPATTN_ERR_CUDA;
  FwdArgs args;
  args.g = geom ? *geom : make_geom(b, s, hq, hkv, cp, causal);
  args.o = nullptr;
  args.lse = lse_part;
  args.lse_stride = lse_stride < 0 ? s : lse_stride;
  args.q_rows = int64_t(q_rows);
  args.kv_rows = int64_t(kv_rows);
  args.lse_len = int64_t(b) * hq * args.lse_stride;
  args.o_part = o_part;
  args.step = step;
  args.scale_log2 = float(1.4426950408889634 * scale);
  args.status = di->status;
  args.producer_limit_ns = kWaitLimitNs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? launch_fwd<128, true>(tq, tk, tv, args, di, st) : launch_fwd<64, true>(tq, tk, tv, args, di, st);
}
}  // namespace

extern "C" int cpattn_fwd_step(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int b,
                               int s, int hq, int hkv, int d, int cp, int step, int causal, void* stream) {
  return step_impl(q, k, v, o_part, lse_part, b, s, hq, hkv, d, cp, step, causal, default_scale(d), stream);
}

extern "C" int cpattn_lse_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                                float* o_out, float* lse_out, void* o_bf16, int b, int s, int hq, int d,
                                void* stream) {
  if (!o_a || !lse_a || !lse_out || (!o_out && !o_bf16) || (!o_b) != (!lse_b)) return CPATTN_ERR_NULL_PTR;
  if (b < 1 || s < 1 || hq < 1 || (d != 64 && d != 128)) return CPATTN_ERR_INVALID_ARG;
  if (int64_t(b) * s * hq >= (int64_t(1) << 31)) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(o_a) || (o_b && !aligned16(o_b)) || (o_out && !aligned16(o_out)) || (o_bf16 && !aligned16(o_bf16)) ||
      (reinterpret_cast<uintptr_t>(lse_a) & 3u) || (lse_b && (reinterpret_cast<uintptr_t>(lse_b) & 3u)) ||
      (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return CPATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc) return rc;
  MergeArgs m;
  m.b = b;
  m.s = s;
  m.hq = hq;
  m.o_a = o_a;
  m.lse_a = lse_a;
  m.o_b = o_b;
  m.lse_b = lse_b;
  m.o_out = o_out;
  m.lse_out = lse_out;
  m.o_bf16 = static_cast<__nv_bfloat16*>(o_bf16);
  const int64_t threads = int64_t(b) * s * hq * (d / 4);
  int64_t blocks = (threads + 255) / 256;
  const int64_t cap = int64_t(di->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128)
    cpattn_lse_merge_kernel<128><<<int(blocks), 256, 0, st>>>(m);
  else
    cpattn_lse_merge_kernel<64><<<int(blocks), 256, 0, st>>>(m);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_LAUNCH_FAILED;
}

extern "C" int cpattn_rope(void* x, int b, int n, int h, int d, int s, int cp, int rank, const int* cu_seqlens,
                           int nseq, float base, int inverse, void* stream) {
  if (!x) return CPATTN_ERR_NULL_PTR;
  if (b < 1 || n < 1 || h < 1 || s < 1 || cp < 1 || (d != 64 && d != 128) || !(base > 1.0f))
    return CPATTN_ERR_INVALID_ARG;
  if (rank < 0) {
    if (n != s) return CPATTN_ERR_INVALID_ARG;
  } else {
    if (rank >= cp || s % (2 * cp) != 0 || n != s / cp) return CPATTN_ERR_INVALID_ARG;
  }
  if (cu_seqlens && (b != 1 || nseq < 1)) return CPATTN_ERR_INVALID_ARG;
  if (int64_t(b) * n * h * d >= (int64_t(1) << 40)) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))) return CPATTN_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc) return rc;
  RopeArgs a;
  a.x = static_cast<__nv_bfloat16*>(x);
  a.b = b;
  a.n = n;
  a.h = h;
  a.s = s;
  a.cp = cp;
  a.rank = rank < 0 ? -1 : rank;
  a.cu_seqlens = cu_seqlens;
  a.nseq = cu_seqlens ? nseq : 0;
  a.inverse = inverse ? 1 : 0;
  const double two_pi = 6.283185307179586476925;
  for (int i = 0; i < kRopeMaxHalf; ++i)
    a.turns_per_pos[i] = i < d / 2 ? std::pow(double(base), -2.0 * i / d) / two_pi : 0.0;
  const int64_t threads = int64_t(b) * n * (d / 4);
  int64_t blocks = (threads + 255) / 256;
  const int64_t cap = int64_t(di->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128)
    cpattn_rope_kernel<128><<<int(blocks), 256, 0, st>>>(a);
  else
    cpattn_rope_kernel<64><<<int(blocks), 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_LAUNCH_FAILED;
}

namespace cpattn {
namespace {
struct UnfusedLayout {
  size_t o_acc, lse_acc, o_part, lse_part, total;
};
UnfusedLayout unfused_layout(int b, int s, int hq, int d) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t ob = size_t(b) * s * hq * d * 4, lb = size_t(b) * hq * s * 4;
  UnfusedLayout L;
  L.o_acc = 0;
  L.lse_acc = al(ob);
  L.o_part = L.lse_acc + al(lb);
  L.lse_part = L.o_part + al(ob);
  L.total = L.lse_part + al(lb);
  return L;
}
}  // namespace
}  // namespace cpattn

extern "C" size_t cpattn_fwd_unfused_workspace_bytes(int b, int s, int hq, int d) {
  if (b < 1 || s < 1 || hq < 1 || (d != 64 && d != 128)) return 0;
  return unfused_layout(b, s, hq, d).total;
}

extern "C" int cpattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                                  size_t ws_bytes, int b, int s, int hq, int hkv, int d, int cp, int causal,
                                  void* stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return CPATTN_ERR_NULL_PTR;
  int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  const UnfusedLayout L = unfused_layout(b, s, hq, d);
  if (ws_bytes < L.total) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || !aligned16(o) || !aligned16(lse))
    return CPATTN_ERR_MISALIGNED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* o_acc = reinterpret_cast<float*>(ws + L.o_acc);
  float* lse_acc = reinterpret_cast<float*>(ws + L.lse_acc);
  float* o_part = reinterpret_cast<float*>(ws + L.o_part);
  float* lse_part = reinterpret_cast<float*>(ws + L.lse_part);
  // step 0 into the accumulator, then each later step merged into it; the
  // last merge writes the bf16 output and the final LSE
  if ((rc = cpattn_fwd_step(q, k, v, o_acc, lse_acc, b, s, hq, hkv, d, cp, 0, causal, stream))) return rc;
  if (cp == 1) return cpattn_lse_merge(o_acc, lse_acc, nullptr, nullptr, nullptr, lse, o, b, s, hq, d, stream);
  for (int i = 1; i < cp; ++i) {
    if ((rc = cpattn_fwd_step(q, k, v, o_part, lse_part, b, s, hq, hkv, d, cp, i, causal, stream))) return rc;
    const bool last = i == cp - 1;
    if ((rc = cpattn_lse_merge(o_acc, lse_acc, o_part, lse_part, last ? nullptr : o_acc, last ? lse : lse_acc,
                               last ? o : nullptr, b, s, hq, d, stream)))
      return rc;
  }
  return CPATTN_OK;
}

namespace cpattn {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct BwdLayout {
  size_t lvec, dvec, total;
  int ntp;
};

// nseq sequences of up to tpc tiles per chunk
BwdLayout bwd_layout_tiles(int nseq, int tpc, int hq, int cp) {
  BwdLayout L;
  L.ntp = 2 * cp * tpc * kTile;
  L.lvec = 0;
  L.dvec = align256(size_t(nseq) * hq * L.ntp * 4);
  L.total = L.dvec + align256(size_t(nseq) * hq * L.ntp * 4);
  return L;
}

BwdLayout bwd_layout(int b, int s, int hq, int d, int cp) {
  (void)d;
  const int c = s / (2 * cp);
  return bwd_layout_tiles(b, (c + kTile - 1) / kTile, hq, cp);
}

template <int D, bool kShort = false>
int launch_bwd_stage(int stage, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const BwdArgs& args, DeviceInfo* di, cudaStream_t st) {
  const int slot = kShort ? 2 : D == 128 ? 1 : 0;
  if (!di->bwd_attr[slot].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(cpattn_bwd_dkdv_kernel<D, kShort>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkdvCfg<D>::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(cpattn_bwd_dq_kernel<D, kShort>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqCfg<D>::kSmemBytes) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    di->bwd_attr[slot].store(true, std::memory_order_release);
  }
  if (stage == 0) {
    const int64_t rows = int64_t(args.g.b) * q_seq_rows(args.g) * args.g.hq;
    int pre_grid = int((rows + 255) / 256);
    if (pre_grid > di->num_sms * 16) pre_grid = di->num_sms * 16;
    cpattn_bwd_pre_kernel<D><<<pre_grid, 256, 0, st>>>(args);
  } else if (stage == 1) {
    const int units = bwd_num_units(args.g);
    cpattn_bwd_dkdv_kernel<D, kShort><<<persistent_grid(di, units), kBwdThreads,
                                        DkdvCfg<D>::kSmemBytes, st>>>(tq, tk, tv, tdo, args);
  } else {
    const int units = dq_num_units(args.g);
    cpattn_bwd_dq_kernel<D, kShort><<<persistent_grid(di, units), kBwdThreads, DqCfg<D>::kSmemBytes,
                                      st>>>(tq, tk, tv, tdo, args);
  }
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_LAUNCH_FAILED;
}

template <int D, bool kShort = false>
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
               const BwdArgs& args, DeviceInfo* di, cudaStream_t st) {
  for (int stage = 0; stage < 3; ++stage) {
    const int rc = launch_bwd_stage<D, kShort>(stage, tq, tk, tv, tdo, args, di, st);
    if (rc) return rc;
  }
  return CPATTN_OK;
}

}  // namespace
}  // namespace cpattn

extern "C" size_t cpattn_bwd_workspace_bytes(int b, int s, int hq, int hkv, int d, int cp) {
  if (check_geometry(b, s, hq, hkv, d, cp)) return 0;
  return bwd_layout(b, s, hq, d, cp).total;
}

namespace cpattn {
namespace {

// Argument checks and tensor maps shared by cpattn_bwd and cpattn_bwd_stage.
int prepare_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv,
                int d, int cp, int causal, double scale, CUtensorMap* maps, BwdArgs* args, DeviceInfo** di,
                int64_t lse_stride = -1, const CpGeom* packed = nullptr, const CpGeom* ranked = nullptr,
                uint64_t producer_limit_ns = kWaitLimitNs) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return CPATTN_ERR_NULL_PTR;
  int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  for (const void* p : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv), static_cast<const void*>(workspace)})
    if (!aligned16(p)) return CPATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return CPATTN_ERR_MISALIGNED;
  // rank-local form: the row vectors hold the rank's 2*tpc tiles per (batch, head)
  const BwdLayout L = packed   ? bwd_layout_tiles(packed->nseq, packed->tpc, hq, cp)
                      : ranked ? bwd_layout_tiles(b, ranked->tpc, hq, 1)
                               : bwd_layout(b, s, hq, d, cp);
  if (workspace_bytes < L.total) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = device_info(di))) return rc;
  // rows of the query-side tensors (q, o, dout, dq) and of the key/value side
  // (a rank-local call's gathered K/V shards hold cp * b * 2c = b * s rows too)
  const uint64_t q_rows = ranked ? uint64_t(b) * 2 * ranked->c : uint64_t(b) * s;
  const uint64_t kv_rows = uint64_t(b) * s;
  if (!encode_bf16_rows_heads_d(&maps[0], q, q_rows, hq, d, kTile) ||
      !encode_bf16_rows_heads_d(&maps[1], k, kv_rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&maps[2], v, kv_rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&maps[3], dout, q_rows, hq, d, kTile))
    return CPATTN_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  args->g = packed ? *packed : ranked ? *ranked : make_geom(b, s, hq, hkv, cp, causal);
  args->ntp = L.ntp;
  args->o = static_cast<const __nv_bfloat16*>(o);
  args->dout = static_cast<const __nv_bfloat16*>(dout);
  args->lse = lse;
  args->lse_stride = lse_stride < 0 ? s : lse_stride;
  args->q_rows = int64_t(q_rows);
  args->kv_rows = int64_t(kv_rows);
  args->lse_len = int64_t(b) * hq * args->lse_stride;
  args->vec_len = int64_t(num_seqs(args->g)) * hq * L.ntp;
  args->lvec = reinterpret_cast<float*>(ws + L.lvec);
  args->dvec = reinterpret_cast<float*>(ws + L.dvec);
  args->dq = static_cast<__nv_bfloat16*>(dq);
  args->dk = static_cast<__nv_bfloat16*>(dk);
  args->dv = static_cast<__nv_bfloat16*>(dv);
  args->scale = float(scale);
  args->scale_log2 = float(1.4426950408889634 * scale);
  args->status = (*di)->status;
  args->producer_limit_ns = producer_limit_ns;
  return CPATTN_OK;
}

}  // namespace
}  // namespace cpattn

namespace {
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv, int d, int cp,
             int causal, double scale, void* stream, int64_t lse_stride = -1, const CpGeom* packed = nullptr,
             const CpGeom* ranked = nullptr, uint64_t producer_limit_ns = kWaitLimitNs) {
  CUtensorMap maps[4];
  BwdArgs args;
  DeviceInfo* di = nullptr;
  const int rc = prepare_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp,
                             causal, double(scale), maps, &args, &di, lse_stride, packed, ranked, producer_limit_ns);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (producer_limit_ns != kWaitLimitNs)  // the abort self-test (d = 128, checked there)
    return launch_bwd<128, true>(maps[0], maps[1], maps[2], maps[3], args, di, st);
  return d == 128 ? launch_bwd<128>(maps[0], maps[1], maps[2], maps[3], args, di, st)
                  : launch_bwd<64>(maps[0], maps[1], maps[2], maps[3], args, di, st);
}

}  // namespace

extern "C" int cpattn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int b, int s, int hq, int hkv, int d, int cp, int causal, float scale, void* stream) {
  if (!valid_scale(scale)) return CPATTN_ERR_INVALID_ARG;
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp, causal,
                  double(scale), stream);
}

extern "C" int cpattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          int b, int s, int hq, int hkv, int d, int cp, int causal, void* stream) {
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp, causal,
                  default_scale(d), stream);
}

// ---------------------------------------------------------------- packed samples
namespace {
// Checks the host sample offsets; returns the total token count or a
// negative error code.
// Packed-sample geometry (nseq <= kMaxSeqs): one launch covers every sample.
CpGeom packed_geom(const int* cu, int nseq, int hq, int hkv, int cp, int causal) {
  CpGeom g = make_geom(1, cu[nseq], hq, hkv, cp, causal);
  g.nseq = nseq;
  g.tile_pairs = 0;  // packed samples pair heads
  for (int i = 0; i <= nseq; ++i) g.cu[i] = cu[i];
  finish_packed(g);
  return g;
}

bool packed_units_fit(const CpGeom& g) {
  return int64_t(g.tile0[g.nseq]) * (g.npairs > g.hq ? g.npairs : g.hq) < (int64_t(1) << 31);
}

int64_t check_cu(const int* cu, int nseq, int cp) {
  if (!cu) return CPATTN_ERR_NULL_PTR;
  if (nseq < 1 || cp < 1 || cu[0] != 0) return CPATTN_ERR_INVALID_ARG;
  for (int i = 0; i < nseq; ++i) {
    const int64_t len = int64_t(cu[i + 1]) - cu[i];
    if (len < 0 || len % (2 * cp) != 0) return CPATTN_ERR_INVALID_ARG;
  }
  return cu[nseq];
}
}  // namespace

extern "C" int cpattn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const int* cu_seqlens, int nseq, int hq, int hkv, int d, int cp, int causal,
                                 float scale, void* stream) {
  const int64_t total = check_cu(cu_seqlens, nseq, cp);
  if (total < 0) return int(total);
  if (!q || !k || !v || !o || !lse) return CPATTN_ERR_NULL_PTR;
  if (!(scale == 0.f || valid_scale(scale))) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  if (d != 64 && d != 128) return CPATTN_ERR_INVALID_ARG;
  const double sc = scale == 0.f ? default_scale(d) : double(scale);
  if (total == 0) return CPATTN_OK;
  if (nseq <= kMaxSeqs) {
    if (hq < 1 || hkv < 1) return CPATTN_ERR_INVALID_ARG;
    const CpGeom g = packed_geom(cu_seqlens, nseq, hq, hkv, cp, causal);
    if (!packed_units_fit(g)) return CPATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, lse, 1, int(total), hq, hkv, d, cp, causal, sc, stream, total, &g);
  }
  // More samples than one launch's parameters hold: groups of up to
  // kMaxSeqs consecutive samples, one launch per group. Each group's rows,
  // its LSE columns (row stride still the packed total) and its sample
  // offsets are taken relative to its first token.
  if (hq < 1 || hkv < 1) return CPATTN_ERR_INVALID_ARG;
  for (int first = 0; first < nseq; first += kMaxSeqs) {
    const int n = nseq - first < kMaxSeqs ? nseq - first : kMaxSeqs;
    const int start = cu_seqlens[first], len = cu_seqlens[first + n] - start;
    if (len == 0) continue;
    int cu[kMaxSeqs + 1];
    for (int i = 0; i <= n; ++i) cu[i] = cu_seqlens[first + i] - start;
    const CpGeom g = packed_geom(cu, n, hq, hkv, cp, causal);
    if (!packed_units_fit(g)) return CPATTN_ERR_INVALID_ARG;
    const size_t qo = size_t(start) * hq * d * 2, ko = size_t(start) * hkv * d * 2;
    const int rc = fwd_impl(static_cast<const uint8_t*>(q) + qo, static_cast<const uint8_t*>(k) + ko,
                            static_cast<const uint8_t*>(v) + ko, static_cast<uint8_t*>(o) + qo, lse + start, 1, len,
                            hq, hkv, d, cp, causal, sc, stream, total, &g);
    if (rc) return rc;
  }
  return CPATTN_OK;
}

extern "C" size_t cpattn_bwd_varlen_workspace_bytes(const int* cu_seqlens, int nseq, int hq, int hkv, int d, int cp) {
  if (check_cu(cu_seqlens, nseq, cp) < 0 || hq < 1 || hkv < 1 || hq % hkv || (d != 64 && d != 128)) return 0;
  // one launch per group of up to kMaxSeqs samples; the groups share the
  // workspace, so it is sized for the largest
  size_t need = 16;
  for (int first = 0; first < nseq; first += kMaxSeqs) {
    const int n = nseq - first < kMaxSeqs ? nseq - first : kMaxSeqs;
    int cu[kMaxSeqs + 1];
    for (int i = 0; i <= n; ++i) cu[i] = cu_seqlens[first + i] - cu_seqlens[first];
    const CpGeom g = packed_geom(cu, n, hq, hkv, cp, 1);
    if (g.tpc > 0) {
      const size_t b = bwd_layout_tiles(n, g.tpc, hq, cp).total;
      need = b > need ? b : need;
    }
  }
  return need;
}

extern "C" int cpattn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                 size_t workspace_bytes, const int* cu_seqlens, int nseq, int hq, int hkv, int d,
                                 int cp, int causal, float scale, void* stream) {
  const int64_t total = check_cu(cu_seqlens, nseq, cp);
  if (total < 0) return int(total);
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return CPATTN_ERR_NULL_PTR;
  if (!(scale == 0.f || valid_scale(scale))) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  if (d != 64 && d != 128) return CPATTN_ERR_INVALID_ARG;
  const double sc = scale == 0.f ? default_scale(d) : double(scale);
  if (total == 0) return CPATTN_OK;
  if (nseq <= kMaxSeqs) {
    if (hq < 1 || hkv < 1) return CPATTN_ERR_INVALID_ARG;
    const CpGeom g = packed_geom(cu_seqlens, nseq, hq, hkv, cp, causal);
    if (!packed_units_fit(g)) return CPATTN_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, 1, int(total), hq, hkv, d, cp,
                    causal, sc, stream, total, &g);
  }
  // More samples than one launch's parameters hold: groups of up to
  // kMaxSeqs consecutive samples (as in the forward), one after another on
  // the stream, sharing the workspace.
  if (hq < 1 || hkv < 1) return CPATTN_ERR_INVALID_ARG;
  for (int first = 0; first < nseq; first += kMaxSeqs) {
    const int n = nseq - first < kMaxSeqs ? nseq - first : kMaxSeqs;
    const int start = cu_seqlens[first], len = cu_seqlens[first + n] - start;
    if (len == 0) continue;
    int cu[kMaxSeqs + 1];
    for (int i = 0; i <= n; ++i) cu[i] = cu_seqlens[first + i] - start;
    const CpGeom g = packed_geom(cu, n, hq, hkv, cp, causal);
    if (!packed_units_fit(g)) return CPATTN_ERR_INVALID_ARG;
    const size_t qo = size_t(start) * hq * d * 2, ko = size_t(start) * hkv * d * 2;
    const int rc = bwd_impl(static_cast<const uint8_t*>(q) + qo, static_cast<const uint8_t*>(k) + ko,
                            static_cast<const uint8_t*>(v) + ko, static_cast<const uint8_t*>(o) + qo, lse + start,
                            static_cast<const uint8_t*>(dout) + qo, static_cast<uint8_t*>(dq) + qo,
                            static_cast<uint8_t*>(dk) + ko, static_cast<uint8_t*>(dv) + ko, workspace,
                            workspace_bytes, 1, len, hq, hkv, d, cp, causal, sc, stream, total, &g);
    if (rc) return rc;
  }
  return CPATTN_OK;
}

// ---------------------------------------------------------------- rank-local form
namespace {
// Geometry of one rank's share of a multi-GPU CP group (see CpGeom).
int rank_geom(int b, int s, int hq, int hkv, int d, int cp, int rank, int causal, int kv_rank_rows, CpGeom* g) {
  const int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  if (rank < 0 || rank >= cp) return CPATTN_ERR_INVALID_ARG;
  *g = make_geom(b, s, hq, hkv, cp, causal);
  g->rank = rank;
  g->kv_rank_rows = kv_rank_rows;
  return CPATTN_OK;
}

int rank_scale(float scale, int d, double* out) {
  if (!(scale == 0.f || valid_scale(scale))) return CPATTN_ERR_INVALID_ARG;
  *out = scale == 0.f ? default_scale(d) : double(scale);
  return CPATTN_OK;
}
}  // namespace

extern "C" int cpattn_fwd_rank(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq,
                               int hkv, int d, int cp, int rank, int causal, float scale, void* stream) {
  CpGeom g;
  double sc = 0.0;
  int rc = rank_scale(scale, d, &sc);
  if (rc) return rc;
  if ((rc = rank_geom(b, s, hq, hkv, d, cp, rank, causal, b * (s / cp), &g))) return rc;
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  const int local = s / cp;  // 2c rows per batch element on the query side
  return fwd_impl(q, k, v, o, lse, b, s, hq, hkv, d, cp, causal, sc, stream, local, &g, uint64_t(b) * local,
                  uint64_t(b) * s);
}

extern "C" int cpattn_fwd_rank_step(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                                    int b, int s, int hq, int hkv, int d, int cp, int rank, int step, int causal,
                                    float scale, void* stream) {
  CpGeom g;
  double sc = 0.0;
  int rc = rank_scale(scale, d, &sc);
  if (rc) return rc;
  if ((rc = rank_geom(b, s, hq, hkv, d, cp, rank, causal, 0, &g))) return rc;
  const int local = s / cp;
  return step_impl(q, k, v, o_part, lse_part, b, s, hq, hkv, d, cp, step, causal, sc, stream, &g,
                   uint64_t(b) * local, uint64_t(b) * local, local);
}

extern "C" size_t cpattn_bwd_rank_workspace_bytes(int b, int s, int hq, int hkv, int d, int cp) {
  if (check_geometry(b, s, hq, hkv, d, cp)) return 0;
  const int c = s / (2 * cp);
  return bwd_layout_tiles(b, (c + kTile - 1) / kTile, hq, 1).total;
}

extern "C" int cpattn_bwd_rank(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, void* workspace,
                               size_t workspace_bytes, int b, int s, int hq, int hkv, int d, int cp, int rank,
                               int causal, float scale, void* stream) {
  CpGeom g;
  double sc = 0.0;
  int rc = rank_scale(scale, d, &sc);
  if (rc) return rc;
  if ((rc = rank_geom(b, s, hq, hkv, d, cp, rank, causal, b * (s / cp), &g))) return rc;
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp, causal, sc,
                  stream, s / cp, nullptr, &g);
}

extern "C" int cpattn_bwd_rank_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv, int d,
                                     int cp, int rank, int causal, float scale, void* stream) {
  if (stage < 0 || stage > 2) return CPATTN_ERR_INVALID_ARG;
  CpGeom g;
  double sc = 0.0;
  int rc = rank_scale(scale, d, &sc);
  if (rc) return rc;
  if ((rc = rank_geom(b, s, hq, hkv, d, cp, rank, causal, b * (s / cp), &g))) return rc;
  if (lse && !aligned16(lse)) return CPATTN_ERR_MISALIGNED;
  CUtensorMap maps[4];
  BwdArgs args;
  DeviceInfo* di = nullptr;
  if ((rc = prepare_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp, causal,
                        sc, maps, &args, &di, s / cp, nullptr, &g)))
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? launch_bwd_stage<128>(stage, maps[0], maps[1], maps[2], maps[3], args, di, st)
                  : launch_bwd_stage<64>(stage, maps[0], maps[1], maps[2], maps[3], args, di, st);
}

extern "C" int cpattn_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                size_t workspace_bytes, int b, int s, int hq, int hkv, int d, int cp, int causal,
                                void* stream) {
  if (stage < 0 || stage > 2) return CPATTN_ERR_INVALID_ARG;
  CUtensorMap maps[4];
  BwdArgs args;
  DeviceInfo* di = nullptr;
  const int rc = prepare_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp,
                             causal, default_scale(d), maps, &args, &di);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? launch_bwd_stage<128>(stage, maps[0], maps[1], maps[2], maps[3], args, di, st)
                  : launch_bwd_stage<64>(stage, maps[0], maps[1], maps[2], maps[3], args, di, st);
}

namespace cpattn {
namespace {

void* g_noalloc_addr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device. The array's
// name is only a host-side stand-in, so it is resolved here once per device,
// with that device current.
void* noalloc_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_addr[dev] = p;
  }
  return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace cpattn

// Backward for callers that cannot allocate device memory: the workspace is
// the library's own fixed 64 MiB scratch array instead of a caller buffer.
extern "C" int cpattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dout, void* dq, void* dk, void* dv, int b, int s, int hq, int hkv,
                                  int d, int cp, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return CPATTN_ERR_NULL_PTR;
  int rc = check_geometry(b, s, hq, hkv, d, cp);
  if (rc) return rc;
  for (const void* p : {q, k, v, o, static_cast<const void*>(lse), dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!aligned16(p)) return CPATTN_ERR_MISALIGNED;
  const BwdLayout L = bwd_layout(b, s, hq, d, cp);
  if (L.total > kNoAllocScratchBytes) return CPATTN_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di))) return rc;
  void* scratch = noalloc_scratch_address();  // first call on a device resolves it
  if (!scratch) return CPATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t rows = uint64_t(b) * s;
  if (!encode_bf16_rows_heads_d(&tq, q, rows, hq, d, kTile) || !encode_bf16_rows_heads_d(&tk, k, rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&tv, v, rows, hkv, d, kTile) ||
      !encode_bf16_rows_heads_d(&tdo, dout, rows, hq, d, kTile))
    return CPATTN_ERR_CUDA;
  // The preprocess kernel rewrites the L/D vectors on every call, so stale
  // contents of the shared array from an earlier call do not matter.
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  BwdArgs args;
  args.g = make_geom(b, s, hq, hkv, cp, causal);
  args.ntp = L.ntp;
  args.o = static_cast<const __nv_bfloat16*>(o);
  args.dout = static_cast<const __nv_bfloat16*>(dout);
  args.lse = lse;
  args.lse_stride = s;
  args.q_rows = int64_t(rows);
  args.kv_rows = int64_t(rows);
  args.lse_len = int64_t(b) * hq * s;
  args.vec_len = int64_t(b) * hq * L.ntp;
  args.lvec = reinterpret_cast<float*>(ws + L.lvec);
  args.dvec = reinterpret_cast<float*>(ws + L.dvec);
  args.dq = static_cast<__nv_bfloat16*>(dq);
  args.dk = static_cast<__nv_bfloat16*>(dk);
  args.dv = static_cast<__nv_bfloat16*>(dv);
  args.scale = float(1.0 / std::sqrt(double(d)));
  args.scale_log2 = float(1.4426950408889634 / std::sqrt(double(d)));
  args.status = di->status;
  args.producer_limit_ns = kWaitLimitNs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? launch_bwd<128>(tq, tk, tv, tdo, args, di, st) : launch_bwd<64>(tq, tk, tv, tdo, args, di, st);
}

extern "C" size_t cpattn_bwd_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int cpattn_zigzag_index(int s, int cp, int64_t* global_of_local) {
  if (!global_of_local) return CPATTN_ERR_NULL_PTR;
  if (s < 1 || cp < 1 || s % (2 * cp) != 0) return CPATTN_ERR_INVALID_ARG;
  const int64_t c = s / (2 * cp);
  for (int64_t r = 0; r < cp; ++r) {
    int64_t* row = global_of_local + r * 2 * c;
    for (int64_t u = 0; u < c; ++u) row[u] = r * c + u;
    for (int64_t u = 0; u < c; ++u) row[c + u] = (2 * cp - 1 - r) * c + u;
  }
  return CPATTN_OK;
}

// Self-test of the bounded waits: one thread waits on a barrier phase that
// nothing completes. The wait gives up after limit_ns of %globaltimer, the
// kernel records kSelfTestTimeoutBit in the status word and returns; no
// fault, no hang, and the context stays usable.
constexpr unsigned int kSelfTestTimeoutBit = 1u << 16;
__global__ void cpattn_selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns)) atomicOr(status, kSelfTestTimeoutBit);
}

extern "C" int cpattn_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return CPATTN_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc) return rc;
  cpattn_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(di->status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_LAUNCH_FAILED;
}

// Self-test of the abort path in the attention kernels themselves: the fused
// forward, then the backward's three stages, with the producers' waits for
// free buffers limited to limit_ns. A producer gives up at its first wait that
// does not complete at once, raises the CTA's abort flag and records its bit;
// the other roles leave at their next wait; before the CTA frees anything,
// every role waits (with the normal limit) for the copies and MMAs it issued.
// Nothing faults or hangs; the outputs are left incomplete.
extern "C" int cpattn_selftest_abort(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                     size_t workspace_bytes, int b, int s, int hq, int hkv, int d, int cp,
                                     unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns >= kWaitLimitNs) return CPATTN_ERR_INVALID_ARG;
  // the self-test kernels are built for d = 128 with head pairs sharing K/V
  if (d != 128 || hkv < 1 || hq % hkv != 0 || (hq / hkv) % 2 != 0) return CPATTN_ERR_INVALID_ARG;
  int rc = fwd_impl(q, k, v, o, lse, b, s, hq, hkv, d, cp, 1, default_scale(d), stream, -1, nullptr, 0, 0, limit_ns);
  if (rc) return rc;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, b, s, hq, hkv, d, cp, 1,
                  default_scale(d), stream, -1, nullptr, nullptr, limit_ns);
}

// Self-test of a checked build's bounds tests: the fused forward told that
// the query-side tensors hold one row fewer than they do. The last row's
// stores then fail their test and are skipped, and bit 20 of the status word
// is set; the buffers do hold that row, so nothing outside them is touched
// whether or not a test fires. Builds without the tests return
// CPATTN_ERR_INVALID_ARG before any device work.
extern "C" int cpattn_selftest_bounds(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s,
                                      int hq, int hkv, int d, int cp, void* stream) {
#ifdef CPATTN_CHECKS
  if (b < 1 || s < 2) return CPATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, b, s, hq, hkv, d, cp, 1, default_scale(d), stream, -1, nullptr,
                  uint64_t(b) * s - 1, 0);
#else
  (void)q, (void)k, (void)v, (void)o, (void)lse, (void)b, (void)s, (void)hq, (void)hkv, (void)d, (void)cp,
      (void)stream;
  return CPATTN_ERR_INVALID_ARG;
#endif
}

extern "C" int cpattn_checked_build(void) {
#ifdef CPATTN_CHECKS
  return 1;
#else
  return 0;
#endif
}

extern "C" int cpattn_device_status(void* stream, int* status) {
  if (!status) return CPATTN_ERR_NULL_PTR;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int h = 0, zero = 0;
  if (cudaMemcpyAsync(&h, di->status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  *status = int(h);
  return h ? CPATTN_ERR_TIMEOUT : CPATTN_OK;
}

extern "C" int cpattn_set_max_ctas(int max_ctas) {
  if (max_ctas < 0) return CPATTN_ERR_INVALID_ARG;
  g_max_ctas.store(max_ctas, std::memory_order_relaxed);
  return CPATTN_OK;
}

extern "C" const char* cpattn_strerror(int code) {
  switch (code) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_INVALID_ARG: return "invalid argument (unsupported shape or size)";
    case CPATTN_ERR_NULL_PTR: return "null pointer";
    case CPATTN_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case CPATTN_ERR_UNSUPPORTED_ARCH: return "current device is not sm_103 (GB300)";
    case CPATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CPATTN_ERR_LAUNCH_FAILED: return "kernel launch failed";
    case CPATTN_ERR_TIMEOUT: return "a kernel gave up waiting (device status set)";
    case CPATTN_ERR_CUDA: return "CUDA runtime or driver error";
    default: return "unknown error";
  }
}

extern "C" int cpattn_version(void) { return 100; }
