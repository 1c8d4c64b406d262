// Thin inline-PTX wrappers for the sm_103a primitives the attention kernels use:
// mbarriers, TMA tensor loads, and the tcgen05 family (TMEM allocation, MMA,
// commit, TMEM loads/stores and their fences). Everything here is written
// from the public PTX ISA description of these instructions.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace cpattn {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Checked builds (compiled with -DCPATTN_CHECKS, the library's debug form in
// place of a memory checker): the kernels test the rows, heads and vector
// positions of their global accesses against the extents of the buffers and
// record a failure in bit 20 of the device status word; a store out of range
// is skipped and a plain bulk copy's source clamped, so a checked run touches
// nothing outside its buffers (tensor copies clip by themselves). In other
// builds bounds_ok() is constant true and the tests compile away.
constexpr unsigned int kStatusBounds = 1u << 20;
#ifdef CPATTN_CHECKS
__device__ __forceinline__ bool bounds_ok(bool ok, unsigned int* status) {
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
}
#else
__device__ __forceinline__ bool bounds_ok(bool, unsigned int*) { return true; }
#endif

// Time limit of every wait on a barrier inside the kernels.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded waits on phase `parity` of `bar`. They give up when `*abort`
// becomes non-zero (another role already gave up) or after `limit_ns` of wall
// time; in the latter case they raise `*abort` themselves. They return true
// when the phase completed.
//
// The slow path: poll until the phase completes or the wait gives up.
__device__ __forceinline__ bool mbar_wait_loop(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Per-thread bounded wait on a barrier phase; false on timeout or abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_loop(bar, parity, abort, limit_ns);
}

// Warp-uniform bounded wait for roles run by a whole converged warp (the MMA
// issuers): the lanes agree on the outcome, so a lane that timed out can
// never leave the others at a full-mask elect.sync.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_ns) {
  bool ok = __all_sync(0xffffffffu, mbar_try_wait(bar, parity));
  if (!ok) ok = __all_sync(0xffffffffu, mbar_wait_loop(bar, parity, abort, limit_ns));
  return ok;
}

// The same waits with the slow path out of line, so that the fast path
// (phase already complete) is one test and no loop. For kernels without a
// register split (a call inside a setmaxnreg region does not allocate).
__device__ __noinline__ bool mbar_wait_loop_ool(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                uint64_t limit_ns) {
  return mbar_wait_loop(bar, parity, abort, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_lean(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_loop_ool(bar, parity, abort, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_warp_lean(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                    uint64_t limit_ns) {
  bool ok = __all_sync(0xffffffffu, mbar_try_wait(bar, parity));
  if (!ok) ok = __all_sync(0xffffffffu, mbar_wait_loop_ool(bar, parity, abort, limit_ns));
  return ok;
}

// Waits for work that completes by itself -- TMA copies already issued, MMAs
// already committed to a barrier -- before a CTA releases the shared memory
// or TMEM that work writes. Unlike the waits above it ignores the abort
// flag: that work finishes whether or not another role gave up, and leaving
// before it does would let it write memory the CTA no longer owns. Only the
// time limit ends it (false: the caller records it in the status word).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}
// The same for a whole converged warp (the MMA issuers' final commit).
__device__ __forceinline__ bool mbar_wait_drain_warp(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_drain(bar, parity, limit_ns));
}

// Register reallocation between warpgroups (all four warps of a warpgroup
// execute the same instruction). The counts must be multiples of 8.
template <int N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled tensor load into shared memory; completion is signalled on `bar`
// as transaction bytes.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 out).
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 async operation issued so far by
// this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D type (1 = f32); 7-9 A type (1 = bf16); 10-12 B type (1 = bf16)
//   bit 15 A is MN-major; bit 16 B is MN-major; 17-22 N>>3; 24-28 M>>4.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t(N) >> 3) << 17) | ((uint32_t(M) >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start address >> 4; 16-29 leading byte offset >> 4;
//   32-45 stride byte offset >> 4; 46-47 = 1 (descriptor version);
//   61-63 layout = 2 (128-byte swizzle).
// K-major operand (rows of 128 bytes along K, 8-row groups of 1024 bytes):
//   SBO = 1024 (next 8 rows), LBO unused.
// MN-major operand (rows of 128 bytes along M/N, one row per K index):
//   SBO = 1024 (next 8 K indices), LBO = distance to the next 64-element
//   block along M/N.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// TMEM loads: one row (lane) per thread, 32 consecutive 32-bit columns per
// x32 chunk. The wait is folded into the same asm statement so no use of the
// destination registers can be scheduled before the data has landed.
#define CPATTN_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                     "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_R8(0), CPATTN_R8(8), CPATTN_R8(16), CPATTN_R8(24)
      : "r"(taddr)
      : "memory");
}
// Two x32 loads (64 columns starting at taddr) with one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_R8(0), CPATTN_R8(8), CPATTN_R8(16), CPATTN_R8(24), CPATTN_R8(32), CPATTN_R8(40), CPATTN_R8(48),
        CPATTN_R8(56)
      : "r"(taddr)
      : "memory");
}
#undef CPATTN_R8

#define CPATTN_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                     "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
// TMEM stores of 16 / 32 consecutive 32-bit columns, waited on before return.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      CPATTN_W8(0), CPATTN_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      CPATTN_W8(0), CPATTN_W8(8), CPATTN_W8(16), CPATTN_W8(24)
      : "memory");
}
#undef CPATTN_W8

// TMEM store of 32 columns without waiting for completion: a later
// tcgen05.wait::st (before the fence that publishes the columns) covers it.
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// 1-D bulk copy global -> shared, completion as transaction bytes on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Vector atomic add (no return) of four fp32 values at a 16-byte aligned
// global address.
__device__ __forceinline__ void red_add_v4(float* gaddr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}


// Packed two-lane fp32 arithmetic (sm_100+ f32x2 instructions).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Scalar fp32 atomic add (no return).
__device__ __forceinline__ void red_add_f32(float* gaddr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gaddr), "f"(v) : "memory");
}


// Two TMEM loads of 32 columns (from two addresses) with a single wait.
#define CPATTN_RA8(i) "=r"(ra[i + 0]), "=r"(ra[i + 1]), "=r"(ra[i + 2]), "=r"(ra[i + 3]), \
                      "=r"(ra[i + 4]), "=r"(ra[i + 5]), "=r"(ra[i + 6]), "=r"(ra[i + 7])
#define CPATTN_RB8(i) "=r"(rb[i + 0]), "=r"(rb[i + 1]), "=r"(rb[i + 2]), "=r"(rb[i + 3]), \
                      "=r"(rb[i + 4]), "=r"(rb[i + 5]), "=r"(rb[i + 6]), "=r"(rb[i + 7])
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&ra)[32], uint32_t (&rb)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_RA8(0), CPATTN_RA8(8), CPATTN_RA8(16), CPATTN_RA8(24), CPATTN_RB8(0), CPATTN_RB8(8),
        CPATTN_RB8(16), CPATTN_RB8(24)
      : "r"(ta), "r"(tb)
      : "memory");
}
// 16-lane fragments. A 16x256b.x4 access covers 16 TMEM lanes x 32 columns:
// thread t holds lanes t/4 (registers 4r, 4r+1) and t/4 + 8 (registers
// 4r+2, 4r+3) at columns 8r + 2(t%4) and 8r + 2(t%4) + 1, r = 0..3.
// Four such loads (lanes +0 and +16 of two column ranges) with one wait:
// ra[0..15] from ta0, ra[16..31] from ta1, rb likewise from tb0, tb1.
__device__ __forceinline__ void tmem_ld16x256b_2x2(uint32_t ta0, uint32_t ta1, uint32_t tb0, uint32_t tb1,
                                                   uint32_t (&ra)[32], uint32_t (&rb)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n\t"
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_RA8(0), CPATTN_RA8(8), CPATTN_RA8(16), CPATTN_RA8(24), CPATTN_RB8(0), CPATTN_RB8(8),
        CPATTN_RB8(16), CPATTN_RB8(24)
      : "r"(ta0), "r"(ta1), "r"(tb0), "r"(tb1)
      : "memory");
}
#undef CPATTN_RA8
#undef CPATTN_RB8


// Four TMEM loads of 32 columns (from four addresses) with a single wait.
#define CPATTN_RX8(r, i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                         "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32x4(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t td, uint32_t (&ra)[32],
                                            uint32_t (&rb)[32], uint32_t (&rc)[32], uint32_t (&rd)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_RX8(ra, 0), CPATTN_RX8(ra, 8), CPATTN_RX8(ra, 16), CPATTN_RX8(ra, 24), CPATTN_RX8(rb, 0),
        CPATTN_RX8(rb, 8), CPATTN_RX8(rb, 16), CPATTN_RX8(rb, 24), CPATTN_RX8(rc, 0), CPATTN_RX8(rc, 8),
        CPATTN_RX8(rc, 16), CPATTN_RX8(rc, 24), CPATTN_RX8(rd, 0), CPATTN_RX8(rd, 8), CPATTN_RX8(rd, 16),
        CPATTN_RX8(rd, 24)
      : "r"(ta), "r"(tb), "r"(tc), "r"(td)
      : "memory");
}
#undef CPATTN_RX8



// Four TMEM loads of 32 columns that also return the maximum of each load's
// 32 values (tcgen05.ld.red with .max, new in sm_103a): the loaded row's
// maximum comes with the load instead of from a chain of max instructions.
#define CPATTN_RZ8(r, i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                         "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32x4_max(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t td, uint32_t (&ra)[32],
                                                uint32_t (&rb)[32], uint32_t (&rc)[32], uint32_t (&rd)[32], float (&m)[4]) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %128, [%132];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %129, [%133];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, %130, [%134];\n\t"
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, %131, [%135];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_RZ8(ra, 0), CPATTN_RZ8(ra, 8), CPATTN_RZ8(ra, 16), CPATTN_RZ8(ra, 24), CPATTN_RZ8(rb, 0),
        CPATTN_RZ8(rb, 8), CPATTN_RZ8(rb, 16), CPATTN_RZ8(rb, 24), CPATTN_RZ8(rc, 0), CPATTN_RZ8(rc, 8),
        CPATTN_RZ8(rc, 16), CPATTN_RZ8(rc, 24), CPATTN_RZ8(rd, 0), CPATTN_RZ8(rd, 8), CPATTN_RZ8(rd, 16),
        CPATTN_RZ8(rd, 24), "=f"(m[0]), "=f"(m[1]), "=f"(m[2]), "=f"(m[3])
      : "r"(ta), "r"(tb), "r"(tc), "r"(td)
      : "memory");
}
#undef CPATTN_RZ8

// Four TMEM stores of 16 columns (to four addresses) with a single wait.
#define CPATTN_W4(r) "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
__device__ __forceinline__ void tmem_st16x4(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t td,
                                            const uint32_t (&ra)[16], const uint32_t (&rb)[16],
                                            const uint32_t (&rc)[16], const uint32_t (&rd)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], {%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%2], {%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%3], {%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(ta), "r"(tb), "r"(tc), "r"(td),
      "r"(ra[0]), "r"(ra[1]), "r"(ra[2]), "r"(ra[3]), "r"(ra[4]), "r"(ra[5]), "r"(ra[6]), "r"(ra[7]),
      "r"(ra[8]), "r"(ra[9]), "r"(ra[10]), "r"(ra[11]), "r"(ra[12]), "r"(ra[13]), "r"(ra[14]), "r"(ra[15]),
      "r"(rb[0]), "r"(rb[1]), "r"(rb[2]), "r"(rb[3]), "r"(rb[4]), "r"(rb[5]), "r"(rb[6]), "r"(rb[7]),
      "r"(rb[8]), "r"(rb[9]), "r"(rb[10]), "r"(rb[11]), "r"(rb[12]), "r"(rb[13]), "r"(rb[14]), "r"(rb[15]),
      "r"(rc[0]), "r"(rc[1]), "r"(rc[2]), "r"(rc[3]), "r"(rc[4]), "r"(rc[5]), "r"(rc[6]), "r"(rc[7]),
      "r"(rc[8]), "r"(rc[9]), "r"(rc[10]), "r"(rc[11]), "r"(rc[12]), "r"(rc[13]), "r"(rc[14]), "r"(rc[15]),
      "r"(rd[0]), "r"(rd[1]), "r"(rd[2]), "r"(rd[3]), "r"(rd[4]), "r"(rd[5]), "r"(rd[6]), "r"(rd[7]),
      "r"(rd[8]), "r"(rd[9]), "r"(rd[10]), "r"(rd[11]), "r"(rd[12]), "r"(rd[13]), "r"(rd[14]), "r"(rd[15])
      : "memory");
}
#undef CPATTN_W4


__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Three-input fp32 maximum.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two TMEM stores of 32 columns (to two addresses) with a single wait.
__device__ __forceinline__ void tmem_st32x2(uint32_t ta, uint32_t tb, const uint32_t (&ra)[32],
                                            const uint32_t (&rb)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(ta), "r"(tb), "r"(ra[0]), "r"(ra[1]), "r"(ra[2]), "r"(ra[3]), "r"(ra[4]), "r"(ra[5]), "r"(ra[6]), "r"(ra[7]), "r"(ra[8]), "r"(ra[9]), "r"(ra[10]), "r"(ra[11]), "r"(ra[12]), "r"(ra[13]), "r"(ra[14]), "r"(ra[15]), "r"(ra[16]), "r"(ra[17]), "r"(ra[18]), "r"(ra[19]), "r"(ra[20]), "r"(ra[21]), "r"(ra[22]), "r"(ra[23]), "r"(ra[24]), "r"(ra[25]), "r"(ra[26]), "r"(ra[27]), "r"(ra[28]), "r"(ra[29]), "r"(ra[30]), "r"(ra[31]), "r"(rb[0]), "r"(rb[1]), "r"(rb[2]), "r"(rb[3]), "r"(rb[4]), "r"(rb[5]), "r"(rb[6]), "r"(rb[7]), "r"(rb[8]), "r"(rb[9]), "r"(rb[10]), "r"(rb[11]), "r"(rb[12]), "r"(rb[13]), "r"(rb[14]), "r"(rb[15]), "r"(rb[16]), "r"(rb[17]), "r"(rb[18]), "r"(rb[19]), "r"(rb[20]), "r"(rb[21]), "r"(rb[22]), "r"(rb[23]), "r"(rb[24]), "r"(rb[25]), "r"(rb[26]), "r"(rb[27]), "r"(rb[28]), "r"(rb[29]), "r"(rb[30]), "r"(rb[31])
      : "memory");
}


// Warp-collective forms of the MMA issue and commit: every lane of a
// converged warp executes them and elect.sync picks the one lane that
// issues. A single tcgen05 issuing thread has little slack over the tensor
// pipe (an M=128, N=128, K=16 MMA executes in 64 cycles), and issuing from a
// converged warp is markedly cheaper than from a lone divergent lane.
__device__ __forceinline__ void umma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pe, pa;\n\t.reg .b32 re;\n\t"
      "elect.sync re|pe, 0xffffffff;\n\t"
      "setp.ne.b32 pa, %4, 0;\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pa;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pe, pa;\n\t.reg .b32 re;\n\t"
      "elect.sync re|pe, 0xffffffff;\n\t"
      "setp.ne.b32 pa, %4, 0;\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred pe;\n\t.reg .b32 re;\n\t"
      "elect.sync re|pe, 0xffffffff;\n\t"
      "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}


// Three TMEM loads of 32 columns with a single wait.
#define CPATTN_RY8(r, i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                         "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32x3(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t (&ra)[32],
                                            uint32_t (&rb)[32], uint32_t (&rc)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%96];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%97];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%98];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : CPATTN_RY8(ra, 0), CPATTN_RY8(ra, 8), CPATTN_RY8(ra, 16), CPATTN_RY8(ra, 24), CPATTN_RY8(rb, 0),
        CPATTN_RY8(rb, 8), CPATTN_RY8(rb, 16), CPATTN_RY8(rb, 24), CPATTN_RY8(rc, 0), CPATTN_RY8(rc, 8),
        CPATTN_RY8(rc, 16), CPATTN_RY8(rc, 24)
      : "r"(ta), "r"(tb), "r"(tc)
      : "memory");
}
#undef CPATTN_RY8


// Two TMEM stores of 16 columns (to two addresses) with a single wait.
__device__ __forceinline__ void tmem_st16x2(uint32_t ta, uint32_t tb, const uint32_t (&ra)[16],
                                            const uint32_t (&rb)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], {%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(ta), "r"(tb), "r"(ra[0]), "r"(ra[1]), "r"(ra[2]), "r"(ra[3]), "r"(ra[4]), "r"(ra[5]), "r"(ra[6]), "r"(ra[7]), "r"(ra[8]), "r"(ra[9]), "r"(ra[10]), "r"(ra[11]), "r"(ra[12]), "r"(ra[13]), "r"(ra[14]), "r"(ra[15]), "r"(rb[0]), "r"(rb[1]), "r"(rb[2]), "r"(rb[3]), "r"(rb[4]), "r"(rb[5]), "r"(rb[6]), "r"(rb[7]), "r"(rb[8]), "r"(rb[9]), "r"(rb[10]), "r"(rb[11]), "r"(rb[12]), "r"(rb[13]), "r"(rb[14]), "r"(rb[15])
      : "memory");
}

// Four 16x128b.x4 stores with one wait. A 16x128b.x4 access covers 16 lanes
// x 16 columns: thread t writes lane t/4 (register 2r) and lane t/4 + 8
// (register 2r+1) at column 4r + t%4, r = 0..3. ra[0..7] go to ta0,
// ra[8..15] to ta1, rb likewise to tb0, tb1.
__device__ __forceinline__ void tmem_st16x128b_2x2(uint32_t ta0, uint32_t ta1, uint32_t tb0, uint32_t tb1,
                                                   const uint32_t (&ra)[16], const uint32_t (&rb)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%4,%5,%6,%7,%8,%9,%10,%11};\n\t"
      "tcgen05.st.sync.aligned.16x128b.x4.b32 [%1], {%12,%13,%14,%15,%16,%17,%18,%19};\n\t"
      "tcgen05.st.sync.aligned.16x128b.x4.b32 [%2], {%20,%21,%22,%23,%24,%25,%26,%27};\n\t"
      "tcgen05.st.sync.aligned.16x128b.x4.b32 [%3], {%28,%29,%30,%31,%32,%33,%34,%35};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(ta0), "r"(ta1), "r"(tb0), "r"(tb1), "r"(ra[0]), "r"(ra[1]), "r"(ra[2]), "r"(ra[3]), "r"(ra[4]), "r"(ra[5]), "r"(ra[6]), "r"(ra[7]), "r"(ra[8]), "r"(ra[9]), "r"(ra[10]), "r"(ra[11]), "r"(ra[12]), "r"(ra[13]), "r"(ra[14]), "r"(ra[15]), "r"(rb[0]), "r"(rb[1]), "r"(rb[2]), "r"(rb[3]), "r"(rb[4]), "r"(rb[5]), "r"(rb[6]), "r"(rb[7]), "r"(rb[8]), "r"(rb[9]), "r"(rb[10]), "r"(rb[11]), "r"(rb[12]), "r"(rb[13]), "r"(rb[14]), "r"(rb[15])
      : "memory");
}

}  // namespace cpattn
