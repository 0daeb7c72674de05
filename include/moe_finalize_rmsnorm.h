/*
 * moe_finalize_rmsnorm.h — C ABI of the GB300 (sm_103a) MoE finalize +
 * residual + RMSNorm library (libmfr.so).
 *
 * The operation, for every token t in [0, T) and column h in [0, H):
 *
 *   acc          = +0;  for j = 0..k-1:  acc = fma(w[t,j], E[idx[t,j], h], acc)
 *   x            = residual_in[t,h] + acc                          (FP32)
 *   residual_out[t,h] = x
 *   out[t,h]     = bf16( x / sqrt(mean_h(x^2) + eps) * gamma[h] )
 *
 * Where each step is defined:
 *  - Gather of the k expert rows straight from the GEMM2 result, which sits in
 *    expert-grouped order and is reached through the index map
 *    permuted_row_of: "FlashInfer, Muse-Spark-Open을 위한 융합 정규화 및 TP/EP
 *    MoE 최적화로 성능 극대화" (flashinfer PR 6544 analysis), section 2.1.
 *  - Weighted sum with FP32 fused multiply-adds, in a fixed slot order, BF16
 *    only at the end; the unfused finalize is the deterministic one:
 *    "FlashInfer MoE 성능 최적화: CuTe DSL을 활용한 Deterministic Finalize
 *    개선기" (flashinfer PR 5319 analysis), section 1.
 *  - Residual add on the FP32 residual stream, then RMSNorm, in one pass:
 *    "Blackwell 아키텍처를 위한 MoE All-Reduce Fusion 최적화: FlashInfer의
 *    'Cake' 백엔드 분석" (flashinfer PR 4730 analysis), section 2 (fusion
 *    strategy); FP32 residual stream: PR 6544 analysis, section 1.1.
 *  - Programmatic dependent launch: the kernel loads its independent inputs,
 *    then waits for the producing kernel before touching its output:
 *    PR 5319 analysis, section 2.
 *  - A thread-block cluster that reduces through distributed shared memory
 *    for few tokens: PR 4730 analysis, section 2 (cluster-level exchange).
 *  The all-reduce across GPUs that those pages fuse in is not part of this
 *  single-GPU library.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device (or managed) addresses on the
 *    plan's device; the caller owns all of them.  No entry point allocates on
 *    a run: only the *_plan functions allocate (a 4-byte device status word
 *    each), and moe_finalize_rmsnorm_destroy frees it.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Runs are asynchronous on that stream.
 *  - Every function returns MFR_OK or an MFR_ERR_* code and never aborts the
 *    process.  moe_finalize_rmsnorm_last_error() gives a one-line reason for
 *    the last failure on the calling thread.
 *  - Layouts are dense row-major: expert_out [R, H] bf16, permuted_row_of
 *    [T, k] int32, topk_weights [T, k] fp32, residual_in / residual_out
 *    [T, H] fp32, gamma [H] bf16, out [T, H] bf16.
 */
#ifndef MOE_FINALIZE_RMSNORM_H
#define MOE_FINALIZE_RMSNORM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------- */
#define MFR_OK                    0
#define MFR_ERR_INVALID_ARG       1  /* null pointer, eps < 0 or not finite, bad alias, wrong device */
#define MFR_ERR_UNSUPPORTED_SHAPE 2  /* see moe_finalize_rmsnorm_supports */
#define MFR_ERR_MISALIGNED        3  /* 16-byte rule for E/residual/gamma/out, 4-byte for idx/w */
#define MFR_ERR_BAD_DEVICE        4  /* the current device is not compute capability 10.3 */
#define MFR_ERR_LAUNCH            5  /* the kernel launch failed (CUDA error wrapped) */
#define MFR_ERR_CUDA              6  /* another CUDA runtime call failed */
#define MFR_ERR_BAD_INDEX         7  /* a permuted_row_of entry was outside [0, R) */

/* ---- bits of the device status word ------------------------------------- */
#define MFR_STATUS_BAD_INDEX      1  /* some slot index was outside [0, R); that slot added 0 */
#define MFR_STATUS_TIMEOUT        2  /* a bounded on-chip wait gave up (never expected); the
                                        outputs of that call are not valid */

/* ---- kernel variants ---------------------------------------------------- */
#define MFR_VARIANT_AUTO          0  /* chosen from (T, H, k, device) only  */
#define MFR_VARIANT_CLUSTER       1  /* H split over a cluster of CTAs per token, DSMEM reduction */
#define MFR_VARIANT_ROWS          2  /* one CTA per token, rows gathered into registers */
#define MFR_VARIANT_STREAM        3  /* persistent CTAs, rows staged in shared memory by bulk copies */

/* Options of a plan.  Zero-initialise, or call moe_finalize_rmsnorm_default_options. */
typedef struct mfr_options {
    int enable_pdl;    /* 1: launch with programmatic stream serialization; the kernel
                          reads permuted_row_of, topk_weights and gamma BEFORE waiting
                          on the preceding kernel in the stream, and expert_out and
                          residual_in after.  Those three must therefore not be written
                          by a kernel that may still be running when this one starts.
                          0: ordinary stream order. */
    int force_variant; /* MFR_VARIANT_*; AUTO picks by T, H and the device */
    int cluster_size;  /* MFR_VARIANT_CLUSTER: CTAs per token (2, 4, 8 or 16); 0 = auto */
    int debug_checks;  /* 1: run() waits for the kernel and returns MFR_ERR_BAD_INDEX
                          when a slot index was out of range (slow; for debugging) */
    int sentinel_skip; /* 1: a NEGATIVE permuted_row_of entry marks a slot whose expert
                          is not local (expert parallelism): the slot adds nothing and
                          is not an error.  Entries >= R still raise
                          MFR_STATUS_BAD_INDEX.  0: every entry outside [0, R) is an
                          error.  The skip itself follows the non-local-expert path of
                          the PR 6544 analysis, section 2.4. */
} mfr_options;

/* What a plan decided; for tests, benchmarks and logs. */
typedef struct mfr_plan_info {
    int variant;       /* MFR_VARIANT_CLUSTER / _ROWS / _STREAM */
    int grid_x;        /* CTAs launched (tokens x cluster size, or persistent CTAs) */
    int grid_y;        /* always 1 */
    int block;         /* threads per CTA */
    int cluster;       /* CTAs per cluster (1 = none) */
    int smem_bytes;    /* dynamic shared memory per CTA */
    int chunks_per_thread; /* 16-byte column chunks each thread owns per row */
    int sm_count;      /* SMs of the plan's device */
    int slot_registers; /* CLUSTER / ROWS: 1 = slot rows and weights held in registers
                           across the dependency wait, 0 = read from shared memory
                           after it (chosen when the registers would cost a wave).
                           Per-expert RMSNorm plans: 1 = the one-pass form (rows
                           held in registers), 0 = the two-pass form */
} mfr_plan_info;

typedef struct mfr_plan_s* mfr_plan_t;

/* 1 when (H, k) is supported, else 0.  Pure: touches no device.
 * Supported: H % 8 == 0 and 8 <= H <= 16384; 1 <= k <= 16.
 * Fastest at H in {4096, 8192} and k == 8. */
int moe_finalize_rmsnorm_supports(int64_t H, int k);

/* Fills *opt with the defaults: enable_pdl = 1, everything else 0. */
void moe_finalize_rmsnorm_default_options(mfr_options* opt);

/* Creates a plan for T tokens (T >= 0), hidden size H, top-k k and an
 * expert_out of R rows (R >= 0) on the CURRENT device.  opt may be NULL
 * (defaults).  Validates the shape, checks the device is compute capability
 * 10.3, fixes the variant and launch geometry, and allocates the plan's
 * 4-byte device status word (cleared).  On failure *plan is set to NULL.
 * A plan is immutable after creation and may be run concurrently on several
 * streams; they share its status word. */
int moe_finalize_rmsnorm_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                              const mfr_options* opt);

/* Enqueues one call of the fused path on `stream`.
 *  expert_out       device, bf16 [R, H], 16-byte aligned (may be NULL when R == 0)
 *  permuted_row_of  device, int32 [T, k], 4-byte aligned: row of expert_out for (t, j)
 *  topk_weights     device, fp32 [T, k], 4-byte aligned: router weights, used as given
 *  residual_in      device, fp32 [T, H], 16-byte aligned
 *  residual_out     device, fp32 [T, H], 16-byte aligned; may equal residual_in
 *                   (in place) but must not otherwise overlap it
 *  gamma            device, bf16 [H], 16-byte aligned
 *  eps              finite, >= 0 (eps == 0 with an all-zero row gives NaN, as IEEE says)
 *  out              device, bf16 [T, H], 16-byte aligned; overlaps no input
 *  stream           cudaStream_t as void*
 * A slot whose index lies outside [0, R) adds nothing and sets
 * MFR_STATUS_BAD_INDEX in the plan's status word (the kernel never reads out
 * of bounds and never traps).  T == 0 is a no-op returning MFR_OK.
 * The current device must be the plan's device. */
int moe_finalize_rmsnorm_run(mfr_plan_t plan,
                             const void* expert_out, const int32_t* permuted_row_of,
                             const float* topk_weights, const float* residual_in,
                             float* residual_out, const void* gamma, float eps,
                             void* out, void* stream);

/* ---- residual + RMSNorm with an NVFP4 output ----------------------------
 * The same fused call, but the normalised FP32 values are written as NVFP4
 * for the next GEMM instead of bf16: "FlashInfer, Muse-Spark-Open을 위한
 * 융합 정규화 및 TP/EP MoE 최적화로 성능 극대화" (flashinfer PR 6544 analysis),
 * section 2.3, fuses RMSNorm with NVFP4 quantisation; the format follows the
 * public NVFP4 description.  For each block of 16 consecutive columns of a
 * token, with y the FP32 value (x * rsqrt(mean(x^2) + eps)) * gamma:
 *   amax = max |y|;  sf = E4M3((amax / 6) * s_enc)   nearest-even, saturating
 *   dec = value(sf) / s_enc;  enc = sf == 0 ? 0 : 1 / dec
 *   q   = E2M1(y * enc)                              nearest-even, saturating
 * so that y ~ value(q) * value(sf) / s_enc.  Each step is one FP32 operation.
 *  s_enc   the FP32 tensor scale (> 0, finite); the usual choice is
 *          448 * 6 / amax over the tensor, measured offline
 *  out_q   device, uint8 [T, H/2], 4-byte aligned: two codes per byte,
 *          column 2j in the low nibble of byte j
 *  out_sf  device, uint8: E4M3 block scales, [T, H/16] row-major, or for
 *          plans made with MFR_SF_TILED_128x4 the tiled layout below
 * residual_out is written as in moe_finalize_rmsnorm_run.  Needs H % 16 == 0.
 * Plans come from moe_finalize_rmsnorm_nvfp4_plan (same arguments and
 * options as moe_finalize_rmsnorm_plan) and run only with
 * moe_finalize_rmsnorm_nvfp4_run. */
int moe_finalize_rmsnorm_nvfp4_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                    const mfr_options* opt);

/* The same plan with a choice of block-scale layout for out_sf:
 *  MFR_SF_ROW_MAJOR    uint8 [T, H/16], row-major (moe_finalize_rmsnorm_nvfp4_plan)
 *  MFR_SF_TILED_128x4  the layout block-scaled FP4 GEMMs read for their
 *                      operand scales (the public 1-D block-scaling-factor
 *                      layout): the [T, H/16] scale matrix, padded to a
 *                      multiple of 128 rows and of 4 columns, is cut into
 *                      tiles of 128 rows x 4 columns stored as 512 consecutive
 *                      bytes each, tiles in row-major order of (row / 128,
 *                      column / 4); scale (r, c) sits at byte
 *                      (r mod 32) * 16 + ((r / 32) mod 4) * 4 + (c mod 4) of its
 *                      tile.  out_sf then holds ceil(T/128)*128 x
 *                      ceil(H/64)*4 bytes; the padding bytes are not written
 *                      (a GEMM that reads padded rows or columns needs them,
 *                      and the matching rows / columns of out_q, set by the
 *                      caller).  out_q is [T, H/2] as before.
 * Any other sf_layout is MFR_ERR_INVALID_ARG.  moe_finalize_rmsnorm_nvfp4_run
 * runs both kinds. */
#define MFR_SF_ROW_MAJOR   0
#define MFR_SF_TILED_128x4 1
int moe_finalize_rmsnorm_nvfp4_plan_ex(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                       const mfr_options* opt, int sf_layout);

/* Bytes of out_sf for an NVFP4 plan in its layout (T * H/16 row-major); -1
 * for a NULL or non-NVFP4 plan. */
int64_t moe_finalize_rmsnorm_nvfp4_sf_bytes(mfr_plan_t plan);
int moe_finalize_rmsnorm_nvfp4_run(mfr_plan_t plan, const void* expert_out,
                                   const int32_t* permuted_row_of, const float* topk_weights,
                                   const float* residual_in, float* residual_out, const void* gamma,
                                   float eps, float s_enc, void* out_q, void* out_sf, void* stream);

/* ---- plain finalize (no residual, no norm) ------------------------------
 * out[t, h] = bf16( sum_j fma(w[t,j], E[idx[t,j], h], .) ), the FP32 weighted
 * sum in slot order rounded once to bf16: the finalize kernel of
 * "FlashInfer MoE 성능 최적화: CuTe DSL을 활용한 Deterministic Finalize
 * 개선기" (flashinfer PR 5319 analysis), section 1.
 * moe_finalize_plan takes the same arguments and options as
 * moe_finalize_rmsnorm_plan (cluster_size then splits the columns of a token
 * over that many CTAs, without a cluster; nothing is reduced).
 * moe_finalize_run: expert_out bf16 [R, H] and out bf16 [T, H] 16-byte
 * aligned, permuted_row_of / topk_weights [T, k] 4-byte aligned, out overlaps
 * no input; bad indices behave as in moe_finalize_rmsnorm_run.  Each plan
 * kind works only with its own run function (MFR_ERR_INVALID_ARG otherwise);
 * _get_status, _plan_info, _launch_floor and _destroy take either kind. */
int moe_finalize_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                      const mfr_options* opt);
int moe_finalize_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                     const float* topk_weights, void* out, void* stream);

/* ---- end to end from host buffers ----------------------------------------
 * The same call with every tensor in HOST memory.  On `stream`, in order:
 * one cudaMemcpyAsync per input (expert_out, permuted_row_of, topk_weights,
 * residual_in, gamma) into the caller's device workspace, the kernel, and one
 * cudaMemcpyAsync per output (residual_out, out) back to host memory.
 * Asynchronous: the host outputs are complete when `stream` reaches that
 * point.  Host buffers should be page-locked (pinned) for the copies to be
 * asynchronous.  The workspace (device, 256-byte aligned, at least
 * moe_finalize_rmsnorm_host_workspace_bytes(plan) bytes, owned by the caller)
 * holds every tensor of one call; calls whose workspaces differ may overlap
 * on different streams (one call's output copies then run under the next
 * call's input copies).  Only plans made by moe_finalize_rmsnorm_plan.
 * host_workspace_bytes returns -1 for a NULL or plain-finalize plan. */
int64_t moe_finalize_rmsnorm_host_workspace_bytes(mfr_plan_t plan);
int moe_finalize_rmsnorm_run_host(mfr_plan_t plan, const void* h_expert_out,
                                  const int32_t* h_permuted_row_of, const float* h_topk_weights,
                                  const float* h_residual_in, float* h_residual_out,
                                  const void* h_gamma, float eps, void* h_out,
                                  void* d_workspace, int64_t workspace_bytes, void* stream);

/* Waits for `stream`, reads the plan's status word into *device_status
 * (MFR_STATUS_* bits) and clears it.  Returns MFR_OK or a CUDA error code. */
int moe_finalize_rmsnorm_get_status(mfr_plan_t plan, void* stream, int* device_status);

/* Enqueues an EMPTY kernel with exactly the plan's launch geometry (grid,
 * block, cluster, dynamic shared memory, PDL attribute) that only performs the
 * dependent-launch wait and trigger.  Benchmarks time it to get the launch
 * floor of a call.  Touches no memory.  T == 0 is a no-op. */
int moe_finalize_rmsnorm_launch_floor(mfr_plan_t plan, void* stream);

/* The launch-plus-one-pass floor of a call: the same empty kernel with the
 * plan's exact launch geometry and dependent-launch protocol (including the
 * slot-index reads, the cluster barrier and the L2 prefetch that precede the
 * wait), plus, after the wait, the parts of the call's data movement that
 * `work` selects, with no arithmetic:
 *   MFR_FLOOR_LOAD      each thread loads its 16-byte chunks of the k slot
 *                       rows of expert_out and of residual_in (the call's reads)
 *   MFR_FLOOR_EXCHANGE  one barrier over the token's cluster of CTAs (a CTA
 *                       barrier for one-CTA plans): the least a cross-CTA
 *                       reduction costs
 *   MFR_FLOOR_STORE     each thread stores its chunks of residual_out and out
 *                       (the call's writes; their contents are unspecified)
 * work = 0 is moe_finalize_rmsnorm_launch_floor plus the prologue's reads.
 * Benchmarks time it beside a call to split a small call's time into launch,
 * data movement, exchange and the kernel's own work.  Only plans made by
 * moe_finalize_rmsnorm_plan whose variant is MFR_VARIANT_CLUSTER or
 * MFR_VARIANT_ROWS (MFR_ERR_UNSUPPORTED_SHAPE otherwise).  Pointers, sizes,
 * alignment and overlap rules are those of moe_finalize_rmsnorm_run;
 * permuted_row_of is always read, the others only when `work` needs them
 * (NULL allowed otherwise).  work outside [0, 7] is MFR_ERR_INVALID_ARG.  An
 * index outside [0, R) is skipped (no status bit).  T == 0 is a no-op. */
#define MFR_FLOOR_LOAD     1
#define MFR_FLOOR_EXCHANGE 2
#define MFR_FLOOR_STORE    4
int moe_finalize_rmsnorm_launch_floor_work(mfr_plan_t plan, int work, const void* expert_out,
                                           const int32_t* permuted_row_of, const float* residual_in,
                                           float* residual_out, void* out, void* stream);

/* Failure-path self test.  Enqueues one thread that waits on an on-chip
 * barrier with the same bounded-wait routine every kernel of the library uses
 * (each of their waits gives up after about 2 s and sets MFR_STATUS_TIMEOUT),
 * but with a limit of `limit_cycles` SM clock cycles; the barrier receives its
 * arrival only if `arrive` is nonzero.  When the wait runs out the kernel sets
 * MFR_STATUS_TIMEOUT in the plan's status word and returns, so the context
 * stays usable; read it with _get_status.  limit_cycles must be in
 * [1, 2^32], else MFR_ERR_INVALID_ARG. */
int moe_finalize_rmsnorm_wait_selftest(mfr_plan_t plan, int64_t limit_cycles, int arrive, void* stream);

/* Copies what the plan decided into *info. */
int moe_finalize_rmsnorm_plan_info(mfr_plan_t plan, mfr_plan_info* info);

/* Frees the plan and its status word.  NULL is a no-op.  The caller makes
 * sure no run of this plan is still in flight. */
void moe_finalize_rmsnorm_destroy(mfr_plan_t plan);

/* ---- finalize with an RMSNorm per expert row (a reading) ----------------
 * The PR 6544 analysis ("FlashInfer, Muse-Spark-Open을 위한 융합 정규화 및
 * TP/EP MoE 최적화로 성능 극대화", section 2.1) names a tensor-parallel MoE
 * finalize that fuses the TP reduction, an RMSNorm per expert and the
 * weighted accumulation, and gives no formula.  On one GPU the TP reduction
 * is the identity; this entry point computes the plainest reading:
 *     inv_j     = rsqrt(mean_h(E[r_j, :]^2) + eps)          (FP32, per row)
 *     out[t, h] = bf16( sum_j w[t,j] * ((E[r_j, h] * inv_j) * gamma[h]) )
 * with r_j = permuted_row_of[t, j], FP32 fused multiply-adds in slot order
 * j = 0..k-1, the shared gamma, and no residual.  Variants: a cluster of
 * CTAs per token that split H (MFR_VARIANT_CLUSTER, k <= 8; chosen for
 * T*H <= 2^19), one CTA per token (MFR_VARIANT_ROWS), and above one wave
 * of those (T*H > 8192 x the SM count) with k <= 8 and H <= 8192 the
 * persistent ring kernel (MFR_VARIANT_STREAM).  Forcing CLUSTER with k > 8, or STREAM outside its
 * limits, is MFR_ERR_UNSUPPORTED_SHAPE.
 *
 * moe_finalize_expert_rmsnorm_plan: as moe_finalize_rmsnorm_plan (same
 * shape rules and options).
 * moe_finalize_expert_rmsnorm_run: expert_out bf16 [R, H], permuted_row_of
 * int32 [T, k], topk_weights fp32 [T, k], gamma bf16 [H], out bf16 [T, H];
 * device pointers, 16-byte aligned (4 for the index map and weights); out
 * must not overlap an input; eps finite and >= 0.  Slot index rules, the
 * status word, debug_checks and sentinel_skip as for moe_finalize_rmsnorm_run.
 * Asynchronous; returns MFR_OK or an MFR_ERR_* code.  _get_status,
 * _plan_info, _launch_floor and _destroy take this plan too. */
int moe_finalize_expert_rmsnorm_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                     const mfr_options* opt);
int moe_finalize_expert_rmsnorm_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                                    const float* topk_weights, const void* gamma, float eps, void* out,
                                    void* stream);

/* ---- benchmarking stand-in for the producer of expert_out ---------------
 * Enqueues a kernel that follows the protocol the PR 5319 analysis (section
 * 2) gives the FC2 grouped GEMM: wait for the previous kernel, immediately
 * signal dependents, stay busy for `busy_cycles` SM cycles (0 to 4e9; the
 * GEMM's main loop), then copy `rows` x H bf16 values from `src` to
 * `expert_out` (both device, 16-byte aligned, H % 8 == 0).  enable_pdl = 1
 * launches it with programmatic stream serialization.  Used to measure how
 * much of the finalize's prologue hides behind its producer, and to test that
 * the finalize never reads expert_out before the producer is done.  Not part
 * of the finalize itself; returns MFR_OK or an MFR_ERR_* code. */
int moe_finalize_rmsnorm_bench_producer(const void* src, void* expert_out, int64_t rows, int64_t H,
                                        long long busy_cycles, int enable_pdl, void* stream);

/* ---- allocation-free entry point ---------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: engines that own all device memory
 * through their own pool and forbid allocations outside it, and hosts where
 * cudaMalloc's implicit synchronisation is not allowed on the request path.
 * moe_finalize_rmsnorm_plan allocates a device status word with cudaMalloc;
 * this call needs no plan and allocates nothing (no cudaMalloc, no cudaFree,
 * no allocating library routine).
 *
 * Scratch: the kernel's status word lives in a file-scope __device__ array
 * of MFR_NOALLOC_SLOTS ints (256 bytes), which every GPU that loads the
 * library keeps until the process exits.  `slot` picks the word this call
 * uses; a slot outside [0, MFR_NOALLOC_SLOTS) is rejected with
 * MFR_ERR_INVALID_ARG ("beyond the scratch").  The array keeps its contents
 * from call to call: the set-up clears every word once, and after that a
 * word is cleared only right after a call reads it back (host_status not
 * NULL).  A call made with host_status NULL therefore leaves its bits in the
 * word, and the next call on that slot that reads back reports them together
 * with its own (the same sticky rule as a plan's status word and
 * moe_finalize_rmsnorm_get_status).  No memset is queued ahead of the kernel,
 * so nothing stands between the producing kernel and this one on the stream.
 * Calls that use the same slot and overlap on the GPU (different streams, or
 * graph branches) race on that word: give concurrent streams different slots.
 *
 * Set-up: the first call on a device (made with that device current) looks up
 * the array's device address with cudaGetSymbolAddress, clears the array
 * (synchronously), queries the device and sets the kernel's shared-memory
 * attribute; make that first call before any stream capture.  Later calls on
 * the device reuse it.
 *
 * Arguments and layouts are those of moe_finalize_rmsnorm_run, with T, H, k
 * and R passed directly; the library cannot check that the buffers are as
 * large as (T, H, k, R) say.  It always launches the persistent bulk-copy
 * kernel (MFR_VARIANT_STREAM geometry) with programmatic dependent launch on:
 * the kernel reads permuted_row_of, topk_weights and gamma BEFORE waiting on
 * the preceding kernel in the stream, and expert_out and residual_in after,
 * so those three must not be written by a kernel that may still be running
 * when this one starts (the rule of mfr_options.enable_pdl = 1).  If
 * host_status is not NULL the call waits for `stream`, stores the slot's
 * MFR_STATUS_* bits there and clears the word; if it is NULL the call is
 * fully asynchronous and the bits stay in the word. */
#define MFR_NOALLOC_SLOTS 64
int moe_finalize_rmsnorm_run_noalloc(int64_t T, int64_t H, int k, int64_t R,
                                     const void* expert_out, const int32_t* permuted_row_of,
                                     const float* topk_weights, const float* residual_in,
                                     float* residual_out, const void* gamma, float eps, void* out,
                                     int slot, int* host_status, void* stream);

/* Static text for a return code. */
const char* moe_finalize_rmsnorm_strerror(int code);

/* One-line reason for the last failing call on this thread ("" if none). */
const char* moe_finalize_rmsnorm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FINALIZE_RMSNORM_H */
