/*
 * cpattn — context-parallel (CP) causal self-attention on one GB300 GPU.
 *
 * The method (web page "大模型面试宝典 · Megatron-LM 篇", question 3
 * "Context Parallel 篇", sub-questions 3.2 and 3.4; and "超大规模集群下大语言
 * 模型训练实操指南", section "CP 与其他技术结合"):
 *   - the sequence of s tokens is cut into 2*cp chunks of c = s/(2cp)
 *     tokens; virtual rank r holds chunks r and 2cp-1-r (zigzag balance);
 *   - at step i, rank r works on the KV of rank j = (r - i) mod cp:
 *       step 0     local Q vs local KV, causal;
 *       1 <= i <= r all local Q vs the first half of the incoming KV, no mask;
 *       i > r      the second half of Q vs the full incoming KV, no mask;
 *   - each step's partial output O_i and log-sum-exp L_i are corrected and
 *     merged: L = log(sum_i e^{L_i}), O = sum_i e^{L_i - L} O_i.
 * The result equals plain causal softmax attention over the uncut sequence
 * (3.2: each rank's output equals the matching part of the non-CP output).
 * All cp virtual ranks run inside one kernel launch on one GPU; the library
 * itself moves no data between devices (the rank-local calls further down
 * compute one rank's share of a CP group spread over GPUs, and the caller
 * exchanges K/V). The per-step correction is carried on chip, so partial
 * outputs never reach device memory.
 *
 * Conventions shared by every entry point
 *   - Tensors are in natural token order (the zigzag is applied inside).
 *     q, o, dout, dq: [b, s, hq, d]; k, v, dk, dv: [b, s, hkv, d];
 *     bf16, contiguous, head_dim fastest. lse: [b, hq, s] fp32, natural log.
 *   - Grouped-query attention: query head h uses KV head h / (hq / hkv)
 *     (page "Megatron 面试题（一）：模型抽象与训练数据流", item M014).
 *   - Softmax scale is 1/sqrt(d) (any positive scale through cpattn_fwd_ex /
 *     cpattn_bwd_ex). causal != 0 selects the causal mask
 *     (key position <= query position); causal == 0 is full attention with
 *     the same CP chunking (every step unmasked).
 *   - Supported: d in {64, 128}; s divisible by 2*cp; hq divisible by hkv;
 *     b, s, hq, hkv, cp >= 1; b*s < 2^31. Chunk length c need not be a
 *     multiple of the 128-token tile (ragged tiles are masked).
 *   - Pointers: device pointers unless stated otherwise; the caller owns every
 *     buffer. Device buffers must be 16-byte aligned. No call allocates
 *     device memory and none keeps per-call state (the one fixed scratch
 *     array, used only by cpattn_bwd_noalloc, is part of the loaded module).
 *   - Device: calls launch on the calling thread's current CUDA device; the
 *     device buffers and the stream must belong to it. Library state (kernel
 *     attributes, the status word) is kept per device and may be used from
 *     several host threads at once.
 *   - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work and return; results are ready when the stream
 *     is synchronised.
 *   - Return value: 0 on success, a negative CPATTN_ERR_* code otherwise
 *     (nothing is enqueued on an argument error). No C++ exception crosses
 *     this interface.
 *   - Device-side failures: every wait inside the kernels has a time limit.
 *     A kernel that gives up records it in a sticky device status word and
 *     returns without faulting; read it with cpattn_device_status().
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = -1,     /* shape/size outside the supported set   */
  CPATTN_ERR_NULL_PTR = -2,        /* a required pointer is NULL             */
  CPATTN_ERR_MISALIGNED = -3,      /* a device pointer is not 16-byte aligned */
  CPATTN_ERR_UNSUPPORTED_ARCH = -4,/* current device is not sm_103            */
  CPATTN_ERR_WORKSPACE_TOO_SMALL = -5,
  CPATTN_ERR_LAUNCH_FAILED = -6,   /* kernel launch returned a CUDA error     */
  CPATTN_ERR_TIMEOUT = -7,         /* a kernel gave up waiting (device status) */
  CPATTN_ERR_CUDA = -8             /* other CUDA runtime/driver error         */
};

/*
 * Forward pass. Writes o (bf16) and lse (fp32, natural log) for every query
 * of every head: O[t] = sum_{j<=t} softmax_j(q_t.k_j/sqrt(d)) v_j,
 * lse[t] = log sum_{j<=t} exp(q_t.k_j/sqrt(d)).
 * Computed CP-style (steps 0..cp-1 per virtual rank, merge fused on chip).
 */
int cpattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq, int hkv,
               int d, int cp, int causal, void* stream);

/*
 * cpattn_fwd with a caller-chosen softmax scale (scores = scale * q.k instead
 * of q.k / sqrt(d)); lse is then log sum_j exp(scale * q_t.k_j). scale must be
 * positive and finite, else CPATTN_ERR_INVALID_ARG. cpattn_fwd(...) equals
 * cpattn_fwd_ex(..., 1/sqrt(d), stream).
 */
int cpattn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq, int hkv,
                  int d, int cp, int causal, float scale, void* stream);

/*
 * The same forward in the unfused form the pages describe: one launch per CP
 * step, each writing every rank's partial result to device memory, and a
 * log-sum-exp correction after every step ("大模型面试宝典 · Megatron-LM 篇",
 * 3.2 steps 4-5; the two-stage L / O correction of "Megatron 面试题（一）",
 * item M019). Same inputs, outputs and result as cpattn_fwd (up to rounding
 * order); it exists to run the steps one by one (e.g. to overlap them with a
 * KV exchange) and as the baseline against which the fused form is measured.
 * Calls cpattn_fwd_step cp times and cpattn_lse_merge max(cp-1, 1) times.
 *   workspace: device, 256-byte aligned, at least
 *              cpattn_fwd_unfused_workspace_bytes(b, s, hq, d) bytes (two fp32
 *              copies of O and of the LSE); contents need not be initialised
 *              and are overwritten. Errors as cpattn_fwd, plus
 *              CPATTN_ERR_WORKSPACE_TOO_SMALL; workspace misaligned ->
 *              CPATTN_ERR_MISALIGNED.
 */
size_t cpattn_fwd_unfused_workspace_bytes(int b, int s, int hq, int d);
int cpattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                       size_t ws_bytes, int b, int s, int hq, int hkv, int d, int cp, int causal, void* stream);

/*
 * One CP step for every virtual rank, unmerged ("大模型面试宝典 · Megatron-LM
 * 篇", 3.2 steps 2-4, 3.4): at step `step` (0 <= step < cp) rank r computes
 * its block against the KV of rank (r - step) mod cp with the step's mask,
 * each query row taking the softmax over that block's keys only.
 *   o_part:   [b, s, hq, d] fp32: the block's normalised output for each query
 *             row that takes part in the step, 0 for the other rows.
 *   lse_part: [b, hq, s] fp32, natural log: the block's log-sum-exp, -inf for
 *             rows that take no part.
 * Merging the cp steps' results with cpattn_lse_merge gives cpattn_fwd's
 * result. Errors as cpattn_fwd; step outside [0, cp) -> CPATTN_ERR_INVALID_ARG.
 */
int cpattn_fwd_step(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int b, int s,
                    int hq, int hkv, int d, int cp, int step, int causal, void* stream);

/*
 * Log-sum-exp merge of two partial results over disjoint key sets, row by
 * row (the correction of "大模型面试宝典 · Megatron-LM 篇", 3.2 steps 4-5):
 *   L = log(e^{L_a} + e^{L_b}),  O = e^{L_a - L} O_a + e^{L_b - L} O_b;
 * rows with L_a = L_b = -inf give L = -inf, O = 0.
 *   o_a, o_b:     [b, s, hq, d] fp32; lse_a, lse_b: [b, hq, s] fp32 natural log.
 *                 o_b and lse_b may both be NULL (no second part: O_a, L_a are
 *                 passed through, e.g. to convert to bf16).
 *   o_out:        [b, s, hq, d] fp32 merged O, may alias o_a; may be NULL.
 *   lse_out:      [b, hq, s] fp32 merged L, may alias lse_a.
 *   o_bf16:       optional [b, s, hq, d] bf16 copy of the merged O (NULL = none);
 *                 o_out and o_bf16 may not both be NULL.
 * d in {64, 128}. The fp32/bf16 O pointers must be 16-byte aligned, the LSE
 * pointers 4-byte aligned. Errors: NULL_PTR, INVALID_ARG, MISALIGNED,
 * UNSUPPORTED_ARCH, LAUNCH_FAILED.
 */
int cpattn_lse_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, float* o_out,
                     float* lse_out, void* o_bf16, int b, int s, int hq, int d, void* stream);

/*
 * Packed samples (variable lengths): tensors hold several samples back to
 * back -- q, o, dout, dq: [total, hq, d]; k, v, dk, dv: [total, hkv, d];
 * lse: [hq, total] -- and attention stays within each sample. Each sample is
 * split by the zigzag into 2*cp chunks of its own (its length must be
 * divisible by 2*cp; 0 is allowed and skipped) and computed exactly as
 * cpattn_fwd / cpattn_bwd compute a b = 1 sequence.
 *   cu_seqlens: HOST int32 [nseq + 1] sample offsets, 0 = cu[0] <= ... <=
 *               cu[nseq] = total (read during the call only).
 *   scale:      0 selects 1/sqrt(d); otherwise as cpattn_fwd_ex.
 * Up to 512 samples run in one launch per kernel (the offsets travel as
 * kernel parameters; work units are dealt longest tile first across all
 * samples); more samples run as consecutive groups of up to 512, one launch
 * per group and kernel, one after another on `stream`. cpattn_bwd_varlen
 * needs a workspace of cpattn_bwd_varlen_workspace_bytes(...) bytes (per
 * sample of a group two fp32 vectors padded to the group's longest sample's
 * tiles; the largest group's). Errors as cpattn_fwd / cpattn_bwd; malformed
 * offsets -> CPATTN_ERR_INVALID_ARG.
 */
int cpattn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                      int nseq, int hq, int hkv, int d, int cp, int causal, float scale, void* stream);
size_t cpattn_bwd_varlen_workspace_bytes(const int* cu_seqlens, int nseq, int hq, int hkv, int d, int cp);
int cpattn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, const int* cu_seqlens,
                      int nseq, int hq, int hkv, int d, int cp, int causal, float scale, void* stream);

/*
 * Rotary position embedding, in place, with the positions context
 * parallelism needs ("Megatron 面试题（一）：模型抽象与训练数据流", item M016):
 * each token turns by its position in the full sequence, not by its index in
 * a rank's shard, and packed samples restart the position at their start.
 * Pair (x_i, x_{i+d/2}), i < d/2, turns by theta = pos * base^(-2i/d):
 *   x_i' = x_i cos(theta) - x_{i+d/2} sin(theta),
 *   x_{i+d/2}' = x_i sin(theta) + x_{i+d/2} cos(theta).
 *   x:          [b, n, h, d] bf16, rotated in place (q or k; h heads).
 *   rank < 0:   natural token order, n == s, position of token t = t.
 *   rank >= 0:  x is virtual rank `rank`'s zigzag shard (chunk rank, then
 *               chunk 2cp-1-rank; n == s / cp, s divisible by 2cp): local
 *               token u has the zigzag map's global position.
 *   cu_seqlens: optional device int32 [nseq + 1] sample offsets in the full
 *               sequence (0 = cu[0] < ... < cu[nseq] = s); requires b == 1;
 *               the position becomes the token's offset within its sample.
 *               NULL = one sample.
 *   base:       frequency base (> 1), e.g. 10000.
 *   inverse:    non-zero rotates by -theta (the gradient: dx = R^T dy).
 * The angle is formed in fp64 and reduced to one turn before fp32 sin/cos,
 * so long positions keep full accuracy. d in {64, 128}. Errors: NULL_PTR,
 * INVALID_ARG, MISALIGNED (x not 16-byte aligned), UNSUPPORTED_ARCH,
 * LAUNCH_FAILED.
 */
int cpattn_rope(void* x, int b, int n, int h, int d, int s, int cp, int rank, const int* cu_seqlens, int nseq,
                float base, int inverse, void* stream);

/*
 * Bytes of caller-provided device workspace cpattn_bwd needs for these sizes
 * (two fp32 vectors per query row and head: lse * log2(e) and
 * D = rowsum(dO * O), in 128-row tile order). Returns 0 for unsupported sizes.
 */
size_t cpattn_bwd_workspace_bytes(int b, int s, int hq, int hkv, int d, int cp);

/*
 * Backward pass from the forward's saved o and lse: with P = exp(S - lse),
 *   dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)),
 *   dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d),
 * over the same CP steps and masks as the forward; dK/dV of a KV head sum
 * over its query-head group. Writes dq, dk, dv (bf16). `workspace` must hold
 * cpattn_bwd_workspace_bytes(...) bytes (16-byte aligned); its contents on
 * entry do not matter and on exit are unspecified.
 */
int cpattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
               void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv,
               int d, int cp, int causal, void* stream);

/*
 * cpattn_bwd for a forward run with cpattn_fwd_ex's `scale` (the same value
 * must be passed; lse is that forward's). Errors as cpattn_bwd, plus
 * CPATTN_ERR_INVALID_ARG for a scale that is not positive and finite.
 */
int cpattn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv,
                  int d, int cp, int causal, float scale, void* stream);

/*
 * One stage of cpattn_bwd, for callers that schedule or time the backward's
 * kernels themselves. Stage 0 writes the per-row vectors (L*log2(e) and
 * D = rowsum(dO * O)) into the workspace; stage 1 computes dk and dv
 * (key-tile-stationary); stage 2 computes dq (query-tile-stationary, key
 * tiles in CP-step order). Stages 1 and 2 read only the inputs and what
 * stage 0 wrote, so once stage 0 is complete they may run in either order or
 * on different streams. cpattn_bwd runs stages 0, 1, 2 on one stream.
 * Arguments as cpattn_bwd; stage outside 0..2 -> CPATTN_ERR_INVALID_ARG.
 */
int cpattn_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int b,
                     int s, int hq, int hkv, int d, int cp, int causal, void* stream);

/*
 * cpattn_bwd without a workspace argument. The pages describe nothing like
 * it: it exists for callers that cannot allocate device memory when they
 * call the backward -- code that runs under a device-memory budget fixed at
 * start-up, threads that must not enter an allocator, or bindings with no
 * device allocator of their own -- and so cannot hand cpattn_bwd its
 * workspace. The caller still passes every input and output buffer.
 *
 * The workspace is instead a fixed scratch array of
 * cpattn_bwd_noalloc_max_scratch_bytes() bytes (64 MiB) inside the library,
 * held by every device that loads the library until the process exits.
 * Sizes whose workspace (cpattn_bwd_workspace_bytes) exceeds it are rejected
 * with CPATTN_ERR_WORKSPACE_TOO_SMALL before any device work.
 * This entry point calls no cudaMalloc/cudaFree and no allocating routine.
 *
 * The first call of this entry point on a device looks up the scratch
 * array's device address; make that first call before any stream capture. All calls share the one array and each call
 * re-initialises what it needs, but calls that overlap on the GPU (on
 * different streams, or from different threads without ordering) race on
 * it and give wrong results: order them.
 * Arguments, layouts and errors are otherwise those of cpattn_bwd.
 */
int cpattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int b, int s, int hq, int hkv, int d, int cp,
                       int causal, void* stream);

/* Size in bytes of the scratch array cpattn_bwd_noalloc uses. */
size_t cpattn_bwd_noalloc_max_scratch_bytes(void);

/*
 * ---- Rank-local form: one rank's share of a CP group spread over GPUs ----
 *
 * The pages run each CP rank on its own device: rank r holds its zigzag
 * shard of q, k, v (chunks r and 2cp-1-r, c = s/(2cp) tokens each), and the
 * ranks exchange K/V either around a ring, one neighbour per step, with the
 * step's attention computed while the next K/V is in flight ("大模型面试宝典 ·
 * Megatron-LM 篇", 3.1 point 2 and 3.2 steps 2-5), or by an all-gather of K/V
 * in the forward and an all-gather of K/V plus a reduce-scatter of dK/dV in
 * the backward ("超大规模集群下大语言模型训练实操指南", section "超长文本场景
 * 解决方案"). These calls are the device work of one such rank; the exchange
 * itself (NCCL) is the caller's. Each launches on the local GPU only and
 * reads local buffers: nothing here touches another device's memory.
 *
 * Layouts (b batch elements; 2c = s/cp rows per element in a shard):
 *   q, o, dout, dq:  this rank's shard [b, 2c, hq, d] bf16, local rows
 *                    [0, c) = chunk `rank`, [c, 2c) = chunk 2cp-1-rank;
 *   lse:             [b, hq, 2c] fp32, natural log, same local rows;
 *   k_all, v_all:    every rank's shard, rank-major [cp, b, 2c, hkv, d] bf16
 *                    (what an all-gather of the shards along a new leading
 *                    dimension gives);
 *   k_blk, v_blk:    one rank's shard [b, 2c, hkv, d] bf16 (what a ring step
 *                    receives);
 *   dk_part, dv_part: [cp, b, 2c, hkv, d] bf16 like k_all: this rank's share
 *                    of every shard's dK/dV; summing them over the ranks (a
 *                    reduce-scatter) gives each rank its shard's dK/dV.
 * s is the full sequence length (s divisible by 2cp); 0 <= rank < cp;
 * scale 0 selects 1/sqrt(d), otherwise any positive finite value. Other
 * limits, pointers and errors as cpattn_fwd / cpattn_bwd; rank outside
 * [0, cp) -> CPATTN_ERR_INVALID_ARG.
 */

/* Every CP step of rank `rank` in one launch, merged on chip: o and lse of
 * the rank's shard, equal to those rows of cpattn_fwd's result. */
int cpattn_fwd_rank(const void* q, const void* k_all, const void* v_all, void* o, float* lse, int b, int s, int hq,
                    int hkv, int d, int cp, int rank, int causal, float scale, void* stream);

/* CP step `step` of rank `rank` against the shard of rank (rank - step) mod
 * cp, unmerged (3.2 steps 2 and 4): o_part [b, 2c, hq, d] fp32 and lse_part
 * [b, hq, 2c] as cpattn_fwd_step's, rows outside the step 0 / -inf. Merging a
 * rank's cp step results with cpattn_lse_merge (shapes [b, 2c, hq, d]) gives
 * cpattn_fwd_rank's result. step outside [0, cp) -> CPATTN_ERR_INVALID_ARG. */
int cpattn_fwd_rank_step(const void* q, const void* k_blk, const void* v_blk, float* o_part, float* lse_part, int b,
                         int s, int hq, int hkv, int d, int cp, int rank, int step, int causal, float scale,
                         void* stream);

/* Workspace bytes of cpattn_bwd_rank (0 for an unsupported shape). */
size_t cpattn_bwd_rank_workspace_bytes(int b, int s, int hq, int hkv, int d, int cp);

/* The backward of rank `rank` from its saved o and lse: dq of its shard, and
 * its share dk_part, dv_part of every shard's dK/dV (a key tile no query of
 * the rank sees gets zeros). Deterministic, like cpattn_bwd. */
int cpattn_bwd_rank(const void* q, const void* k_all, const void* v_all, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk_part, void* dv_part, void* workspace, size_t workspace_bytes,
                    int b, int s, int hq, int hkv, int d, int cp, int rank, int causal, float scale, void* stream);

/* One stage of cpattn_bwd_rank (as cpattn_bwd_stage is of cpattn_bwd): 0 the
 * row vectors, 1 the shares dk_part/dv_part, 2 dq. After stage 1 the shares
 * are complete, so their reduce-scatter can run while stage 2 computes dq.
 * Arguments as cpattn_bwd_rank; stage outside 0..2 -> CPATTN_ERR_INVALID_ARG. */
int cpattn_bwd_rank_stage(int stage, const void* q, const void* k_all, const void* v_all, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk_part, void* dv_part,
                          void* workspace, size_t workspace_bytes, int b, int s, int hq, int hkv, int d, int cp,
                          int rank, int causal, float scale, void* stream);

/*
 * Host helper: the zigzag index map. Fills global_of_local (HOST memory,
 * cp * 2c int64 values, row-major [cp][2c]) with the global token position
 * of virtual rank r's local position u: chunk r then chunk 2cp-1-r, each in
 * natural order ("大模型面试宝典 · Megatron-LM 篇", 3.4).
 */
int cpattn_zigzag_index(int s, int cp, int64_t* global_of_local);

/*
 * Reads the sticky device status word of the current device into *status
 * (0 = no kernel gave up waiting) and clears it. Synchronises `stream`.
 * Returns CPATTN_ERR_TIMEOUT when the word was non-zero, else 0 or a CUDA
 * error code. Bits: forward producer / MMA / softmax role gave up (0, 1, 2);
 * forward copies or MMAs still in flight at the end after the time limit (3);
 * the same for the backward kernels (8, 9, 10; 12); a backward kernel's
 * shared memory base not 1024-byte aligned (11); the timeout self-test (16);
 * a bounds test of a checked build failed (20).
 * A role that gives up makes the others leave too, but every role first waits
 * for the copies and MMAs it already issued, so no kernel frees memory that
 * asynchronous work still writes.
 *
 * The per-device state behind this word (and the scratch address of
 * cpattn_bwd_noalloc) is looked up once per device ordinal and kept for the
 * life of the process: the library does not survive cudaDeviceReset() of a
 * device it has used (reload the process instead).
 */
int cpattn_device_status(void* stream, int* status);

/*
 * Caps the grid of the persistent attention kernels (forward in every form,
 * dK/dV, dQ) at max_ctas CTAs, one per SM; 0 (the default) uses every SM.
 * Each CTA takes a whole SM (all its registers and nearly all its shared
 * memory), so a kernel launched on another stream -- say a communication
 * library's send/receive kernel during a ring CP step ("大模型面试宝典 ·
 * Megatron-LM 篇", 3.2: the next shard travels while a step computes) --
 * runs meanwhile only on SMs the cap leaves free. Results do not depend on
 * the grid: every work unit is computed the same way on whichever CTA takes
 * it, so outputs are bit-identical. Process-wide; applies to launches made
 * after the call. Returns CPATTN_ERR_INVALID_ARG for max_ctas < 0.
 */
int cpattn_set_max_ctas(int max_ctas);

/*
 * Self-test of the timeout path: launches one block whose single waiting
 * thread waits on a barrier phase that nothing completes, giving up after
 * limit_ns nanoseconds (1 .. 2e9) exactly as the kernels' waits do. It then
 * sets bit 16 (0x10000) of the device status word and returns, without a
 * fault or a hang; cpattn_device_status() reports it afterwards. Returns
 * CPATTN_ERR_INVALID_ARG for a limit outside the range (before any device
 * work), else as a launch.
 */
int cpattn_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * Self-test of the abort path of the attention kernels: runs the fused
 * forward (writing o, lse) and then the three backward stages, as
 * cpattn_fwd and cpattn_bwd with causal = 1 would, but with the TMA
 * producers' waits for free buffers limited to limit_ns nanoseconds
 * (below the kernels' normal 2 s). A producer then gives up mid-run (status bit 0 for the
 * forward, 8 for the backward); the other roles leave at their next wait
 * (bits 1-2, 9-10). Before a CTA frees its shared memory and TMEM, each role
 * waits, with the normal 2 s limit, for the copies and MMAs it issued itself,
 * so no fault follows; bits 3 and 12 would say that such a wait ran out.
 * The outputs are left incomplete. Arguments otherwise as cpattn_bwd, with
 * d = 128 and an even number of query heads per KV head (the self-test
 * kernels are built for that case only); CPATTN_ERR_INVALID_ARG for other
 * shapes or a limit outside 1 .. 2e9 - 1 (before any device work).
 */
int cpattn_selftest_abort(const void* q, const void* k, const void* v, void* o, float* lse, const void* dout,
                          void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int b, int s,
                          int hq, int hkv, int d, int cp, unsigned long long limit_ns, void* stream);

/*
 * Checked builds (libcpattn_checked.so, compiled with -DCPATTN_CHECKS; the
 * library's debug form in place of a memory checker): every kernel tests the
 * rows, heads and vector positions of its global accesses against the
 * extents of the buffers, records a failure in bit 20 (0x100000) of the
 * device status word, skips a store out of range and keeps a plain bulk copy
 * inside its source; results are otherwise those of the normal build, bit
 * for bit. cpattn_checked_build() returns 1 in a checked build, else 0.
 */
int cpattn_checked_build(void);

/*
 * Self-test of a checked build's bounds tests: runs the fused forward (as
 * cpattn_fwd with causal = 1) told that q and o hold one row fewer than they
 * do, so the stores of the last row fail their test and are skipped and bit
 * 20 is set (no access leaves the buffers either way). The last row of o and
 * of lse is left unwritten. Arguments as cpattn_fwd (s >= 2). Returns
 * CPATTN_ERR_INVALID_ARG in builds without the tests, before any device work.
 */
int cpattn_selftest_bounds(const void* q, const void* k, const void* v, void* o, float* lse, int b, int s, int hq,
                           int hkv, int d, int cp, void* stream);

/* Static description of an error code. */
const char* cpattn_strerror(int code);

/* Library version, major*10000 + minor*100 + patch. */
int cpattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
