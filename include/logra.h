/*
 * logra.h — C ABI of the GB300 (sm_103a) LoGRA low-rank gradient-sketching
 * hot path.
 *
 * Source of the method: "LoGRA: Scaling LLM Reinforcement Learning with
 * Low-Rank Gradient Sketches" (summary page on wispaper.ai):
 *   - section "草图如何取代完整梯度缓冲": the d×r sketch S = G Aᵀ replaces the
 *     d×k gradient G; A is r×k, independent of the batch, fixed while
 *     accumulating, not learned, with independent random-sign entries scaled
 *     by 1/√r; each micro-batch's contribution is added into S in fp32 by
 *     projecting the layer inputs before they meet the backward derivatives;
 *     the update W ← W − αηUA (U = S for plain SGD) is merged into W;
 *   - section "同一份草图也压缩策略同步开销": A is regenerated from a seed;
 *   - section "预测 KL 控制防止过大更新破坏学习": q(D) is the mean KL between
 *     the current and proposed next-token distributions at one temperature,
 *     and α = min{α_max, √(δ/q(D))}.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Matrices are row-major with unit inner stride; `ld*` is the row stride
 *    in elements.  W is d×k (out×in), X is T×k, dY is T×d, A is r×k, S is d×r.
 *  - The caller owns every buffer (device memory unless stated otherwise).
 *    No call allocates or frees device memory; scratch is passed in as
 *    `workspace`, whose size the matching *_workspace_bytes() call gives.
 *  - Device calls are asynchronous on `stream` (0 = legacy default stream).
 *    Validation happens on the host before any launch: a failed check
 *    returns a status and launches nothing.  A failed launch returns
 *    LOGRA_ERR_CUDA.  logra_last_error() then describes the failure.
 *  - Device pointers to bf16 / fp32 data must be 16-byte aligned and every
 *    `ld` of a bf16 matrix a multiple of 8 elements (fp32: 4 elements), so
 *    that rows can be moved with 16-byte accesses and the tensor memory
 *    accelerator.  Matrices the tensor memory accelerator moves (X, dY, W)
 *    must also have a row length that is a multiple of 8 elements: the
 *    accelerator does not clip a row end that falls inside a 16-byte unit
 *    exactly, and a partial unit would touch the caller's row padding.
 *    Violations return LOGRA_ERR_ALIGNMENT.  T, the number of rows, and r
 *    are free.
 *  - The projection rank r is 1 ≤ r ≤ 256 (LOGRA_ERR_UNSUPPORTED above).
 *  - Results are bitwise reproducible run to run for a fixed shape.
 *  - Kernels never wait without a limit: a broken pipeline makes the kernel
 *    record a code in the library's device error word and return;
 *    logra_device_error() reads it.
 *
 * The projection A (shared by every call that takes seed / stream_id):
 *   key = (seed mod 2³², seed >> 32), counter = (j >> 7, i, stream_id, 0),
 *   w = Philox4x32-10(counter, key); bit b = (w[(j & 127) >> 5] >> (j & 31)) & 1;
 *   A[i][j] = (b ? −1 : +1) / √r.
 * Philox4x32-10 is the generator of Salmon et al., "Parallel random numbers:
 * as easy as 1, 2, 3" (SC'11).
 */
#ifndef LOGRA_H_
#define LOGRA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* logra_stream_t;

typedef enum logra_status {
  LOGRA_OK = 0,
  LOGRA_ERR_INVALID_ARG = 1, /* null pointer, non-finite or out-of-range scalar */
  LOGRA_ERR_SHAPE = 2,       /* negative size, ld smaller than the row length  */
  LOGRA_ERR_ALIGNMENT = 3,   /* pointer or ld not 16-byte compatible            */
  LOGRA_ERR_WORKSPACE = 4,   /* workspace missing or too small                   */
  LOGRA_ERR_UNSUPPORTED = 5, /* r > 256, dtype unknown, device is not sm_103      */
  LOGRA_ERR_CUDA = 6,        /* a CUDA runtime / driver call failed              */
  LOGRA_ERR_DEVICE = 7       /* a kernel recorded an error (see logra_device_error) */
} logra_status;

/* Element types accepted by logra_predicted_kl. */
#define LOGRA_DTYPE_BF16 0
#define LOGRA_DTYPE_FP32 1

/* Output element types of logra_regen_projection. */
#define LOGRA_PROJ_INT8_PM1 0  /* int8 ±1 (the signs, A·√r)  */
#define LOGRA_PROJ_BF16 1      /* bf16 ±1/√r (A itself)      */
#define LOGRA_PROJ_FP32 2      /* fp32 ±1/√r (A itself)      */
#define LOGRA_PROJ_GAUSS_BF16 3 /* bf16 Ã = bf16_rn(z): the Gaussian operand (A = Ã/√r) */
#define LOGRA_PROJ_GAUSS_FP32 4 /* fp32 Ã/√r (the Gaussian A itself)                      */
#define LOGRA_PROJ_SIGN_BF16 5  /* bf16 ±1: the sign operand Ã = A·√r of the _proj calls     */

/* Message describing the last failure of a call made by this host thread
 * (empty string after success).  The pointer stays valid until the next call
 * from the same thread. */
const char* logra_last_error(void);

/* Static name of a status code. */
const char* logra_status_string(logra_status status);

/* Library version, major·10000 + minor·100 + patch. */
int logra_version(void);

/* ------------------------------------------------------------------------
 * Sketch accumulation  S += dYᵀ (X Aᵀ)
 *
 * Section "草图如何取代完整梯度缓冲": one micro-batch's contribution to the
 * sketch S = G Aᵀ of a d×k weight, with G = dYᵀX the layer's weight gradient,
 * computed by projecting the inputs first (P = X Aᵀ, T×r) so that no d×k
 * gradient is ever formed, and added into S in fp32.
 *
 *  X       bf16 T×k, row stride ldx (layer inputs of the micro-batch)
 *  dY      bf16 T×d, row stride lddy (gradients w.r.t. the layer outputs)
 *  S       fp32 d×r, row stride lds, read and written (S += ...)
 *  seed, stream_id, r   select the projection A (see above)
 *  workspace           device scratch of at least
 *                      logra_sketch_workspace_bytes(T, d, k, r) bytes,
 *                      256-byte aligned; its contents on entry do not matter.
 *
 * d and k must be multiples of 8 (T need not be).  T, d or k equal to 0 is a
 * no-op (S unchanged).  S must not overlap X, dY or
 * the workspace.  Calls that share one workspace must be ordered on the GPU.
 *
 * Arithmetic: P = X·(A√r)ᵀ is formed on the tensor cores in fp32 (the ±1
 * signs are exact in bf16) and S += (1/√r)·dYᵀP is accumulated in fp32 over
 * split ranges of T whose partial sums are then added in ascending split
 * order.  P enters the second product in one of two forms:
 *  - r ≤ 64: split into P_hi = bf16(P) and P_lo = bf16(P − P_hi) (≈16
 *    significant bits), two bf16 MMAs per step;
 *  - r > 64: as fp16(P_t·2^−e_t) per token t, with 2^e_t the power of two that
 *    puts the largest |P| of the token's group of 16 consecutive tokens in
 *    [2^14, 2^15) (11 significant bits; entries down to 2^−28 of that largest
 *    one stay normal fp16); dY is converted to fp16 on the way into tensor
 *    memory with the token's 2^e_t
 *    and a power-of-two scale per row of S that follows the row's magnitude,
 *    divided out at the end, so one fp16 MMA per step.  The bf16 values of dY
 *    are exact in fp16 unless they fall more than 2^24 below their row's
 *    scale.
 * Either way S stays within ~1e-4 relative Frobenius error of the exact sketch
 * on inputs like the workloads' (bf16 rounding of P alone would give ~2e-3).
 *
 * Workspace layout (for inspection; r16 = r rounded up to 16,
 * Tp = T rounded up to 128, dp = d rounded up to 128 (to 256 when r > 64),
 * each region starting on a 256-byte boundary):
 *   r ≤ 64:  P_hi  bf16 [r16][Tp]   P_hi[n][t] = bf16(P[t][n]); rows n ≥ r are zero
 *            P_lo  bf16 [r16][Tp]
 *   r > 64:  Tp/64 blocks of 64 tokens, each two halves of 256 + 64·r16
 *            bytes (one half per CTA of the contraction's CTA pairs): the 64
 *            token scales g[t] = 2^e_t (fp32, equal within each group of 16
 *            tokens), then r16/2 rows of 64 fp16 values
 *            fp16(P[t][n]·2^−e_t) for rows n = h·r16/2 + nl, stored in the
 *            128-byte swizzled K-major image the contraction copies into shared
 *            memory (16-byte chunk (t%64)/8 of local row nl at chunk
 *            ((t%64)/8) ^ (nl%8), element t%8)
 *   then     part  fp32 [splits][dp][r16]   (splits = logra_sketch_splits(...);
 *                                            absent when splits = 1)
 * ---------------------------------------------------------------------- */
size_t logra_sketch_workspace_bytes(int64_t T, int64_t d, int64_t k, int r);

/* Number of split ranges of T used by logra_sketch_accumulate for a shape;
 * it depends on the shape only, never on the device.  The split count is
 * sized for several matrices in flight at once (for instance the projections
 * of a layer, one call each on a few streams): a single call on an otherwise
 * idle GPU does not occupy every SM. */
int logra_sketch_splits(int64_t T, int64_t d, int64_t k, int r);

logra_status logra_sketch_accumulate(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T,
                                     int64_t d, int64_t k, int r, uint64_t seed, uint32_t stream_id, float* S,
                                     int64_t lds, void* workspace, size_t workspace_bytes, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Sketch accumulation with a given projection
 *
 * Section "这些节省能说明什么、不能说明什么" (design-choice experiments): the
 * paper also runs refreshed Rademacher and refreshed Gaussian projections.  A
 * refreshed Rademacher basis needs no new call (pass a new seed, for instance
 * logra_refreshed_seed(base, step)).  For any other basis the caller passes
 * the projection operand Ã, bf16 r×k (row stride lda, a multiple of 8;
 * 16-byte aligned), and the sketch uses A = Ã/√r:
 *
 *     S += (1/√r)·dYᵀ(X·Ãᵀ)
 *
 * with everything else (arguments, workspace, arithmetic, errors) as in
 * logra_sketch_accumulate.  The Gaussian operand comes from
 * logra_regen_projection(..., LOGRA_PROJ_GAUSS_BF16, ...); it is r·k·2 bytes
 * (4.6 MiB at r = 256, k = 18944), read by the kernels from L2.
 * ---------------------------------------------------------------------- */
logra_status logra_sketch_accumulate_proj(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T,
                                          int64_t d, int64_t k, int r, const void* A, int64_t lda, float* S,
                                          int64_t lds, void* workspace, size_t workspace_bytes,
                                          logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Sketch accumulation for projections that share one input X
 *
 * Section "草图如何取代完整梯度缓冲" (the same operation as
 * logra_sketch_accumulate) for up to LOGRA_MAX_SHARED_X_TARGETS weights that
 * are fed the same layer input X — in a decoder layer the q, k and v
 * projections, or gate and up — so X is read from memory once: the sign
 * tiles of all targets are stacked into one tensor-core operand and one pass
 * over X forms every P_j = X·A_jᵀ.  Each target has its own dY, S, seed and
 * stream id; r is common.  n · (r rounded up to 16) must not exceed 512
 * (LOGRA_ERR_UNSUPPORTED).  Every target's d, and k, are multiples of 8.
 *
 * Workspace: logra_sketch_shared_x_workspace_bytes(T, k, n, d[], r) bytes,
 * 256-byte aligned; target j's region (laid out as for
 * logra_sketch_accumulate) starts after the regions of targets 0..j-1, each
 * rounded up to 256 bytes.  The results equal n separate
 * logra_sketch_accumulate calls bit for bit.
 * ---------------------------------------------------------------------- */
#define LOGRA_MAX_SHARED_X_TARGETS 4

typedef struct logra_sketch_target {
  const void* dY;     /* bf16 T×d, row stride lddy                      */
  int64_t lddy;
  int64_t d;
  uint64_t seed;      /* projection of this target                      */
  uint32_t stream_id;
  float* S;           /* fp32 d×r, row stride lds, read and written     */
  int64_t lds;
} logra_sketch_target;

size_t logra_sketch_shared_x_workspace_bytes(int64_t T, int64_t k, int n, const int64_t* d, int r);

logra_status logra_sketch_accumulate_shared_x(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                              const logra_sketch_target* targets, int r, void* workspace,
                                              size_t workspace_bytes, logra_stream_t stream);

/* The same with a given bf16 projection operand per target (A[j], r×k with
 * row stride lda[j], a multiple of 8; 16-byte aligned), as in
 * logra_sketch_accumulate_proj: S_j += (1/√r)·dY_jᵀ(X·Ã_jᵀ).  The seed and
 * stream_id fields of the targets are not read.  For a Gaussian or cached
 * basis on weights that share their input. */
logra_status logra_sketch_accumulate_shared_x_proj(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                                   const logra_sketch_target* targets, const void* const* A,
                                                   const int64_t* lda, int r, void* workspace,
                                                   size_t workspace_bytes, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Sketch accumulation for a set of matrices, one launch per phase
 *
 * Section "草图如何取代完整梯度缓冲": during the backward pass every sketched
 * weight of the model adds its micro-batch contribution into its own S.  A
 * single matrix's call does not occupy a whole GPU (its projection has T/128
 * CTAs, its contraction about a hundred), so called one after another on one
 * stream the matrices of a model would leave most SMs idle.  These calls
 * sketch n matrices together: one projection launch over the token tiles of
 * all of them, one contraction launch over all their row tiles and splits,
 * one launch of the split reduces, each launch ordering its CTAs by
 * decreasing length (the same kernels as the per-matrix call, which find
 * their matrix in the plan).  Each target's S ends bit-identical to
 * logra_sketch_accumulate (A NULL) or logra_sketch_accumulate_proj (A given)
 * on that target.
 *
 * Two steps, as for the merge of a set of weights:
 *  1. logra_sketch_group_plan() validates the targets, lays out the
 *     workspace (logra_sketch_group_workspace_bytes(n, targets, r) bytes,
 *     256-byte aligned, device memory) and writes a plan of
 *     logra_sketch_group_plan_bytes(n) bytes into HOST memory (128-byte
 *     aligned).  It launches nothing.
 *  2. The caller copies the plan unchanged into DEVICE memory (128-byte
 *     aligned, stream-ordered before the launch) and calls
 *     logra_sketch_accumulate_group() with both copies.
 * The plan holds the addresses of X, dY, S, A and of the workspace; it stays
 * valid while they, the shapes, seeds and stream ids are unchanged, so the
 * micro-batches of a step that reuse their buffers plan once.  The workspace
 * belongs to the plan: two launches that may run at the same time need two
 * workspaces (and plans).
 *
 * Targets: each as for logra_sketch_accumulate (X bf16 T×k, dY bf16 T×d,
 * S fp32 d×r read and written, d and k multiples of 8) with its own T, d, k,
 * seed and stream id; A optional as in logra_sketch_accumulate_proj (then
 * seed and stream_id are not read).  r is common.  Targets with T, d or k
 * equal to 0 are skipped.  The S regions of the targets must not overlap
 * (the launches update them without order between matrices): a matrix
 * sketched from two micro-batches takes two launches.
 * Errors: as in logra_sketch_accumulate, per target; S regions that overlap
 * (LOGRA_ERR_INVALID_ARG); a workspace or plan that is too small or
 * misaligned (LOGRA_ERR_WORKSPACE / LOGRA_ERR_ALIGNMENT); a buffer that is
 * not a plan (LOGRA_ERR_INVALID_ARG).
 * ---------------------------------------------------------------------- */
typedef struct logra_sketch_group_target {
  const void* X;      /* bf16 T×k, row stride ldx                       */
  int64_t ldx;
  const void* dY;     /* bf16 T×d, row stride lddy                      */
  int64_t lddy;
  int64_t T;
  int64_t d;
  int64_t k;
  uint64_t seed;      /* projection (when A is NULL)                    */
  uint32_t stream_id;
  const void* A;      /* optional bf16 r×k projection operand, or NULL  */
  int64_t lda;
  float* S;           /* fp32 d×r, row stride lds, read and written     */
  int64_t lds;
} logra_sketch_group_target;

size_t logra_sketch_group_plan_bytes(int n);

/* 0 for invalid arguments (n < 0, r outside [1, 256], negative sizes). */
size_t logra_sketch_group_workspace_bytes(int n, const logra_sketch_group_target* targets, int r);

logra_status logra_sketch_group_plan(int n, const logra_sketch_group_target* targets, int r, void* workspace,
                                     size_t workspace_bytes, void* plan, size_t plan_bytes);

logra_status logra_sketch_accumulate_group(const void* plan, const void* plan_dev, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Merge  W ← bf16(W − αη·S·A)
 *
 * Section "草图如何取代完整梯度缓冲": the update W ← W − αηUA with U = S (the
 * plain SGD variant), merged straight into the bf16 weights with no adapter
 * branch.  Section "同一份草图也压缩策略同步开销": the same call applies a
 * received factor (αη, S, seed) on the rollout side.
 *
 *  W         bf16 d×k, row stride ldw, updated in place; k a multiple of 8,
 *            bytes of a row past column k are never touched
 *  S         fp32 d×r, row stride lds
 *  alpha_eta the product αη (finite), used when alpha_eta_dev is NULL
 *  alpha_eta_dev  optional device fp32 scalar that replaces alpha_eta (so that
 *            a step size computed on the GPU needs no host round trip)
 *
 * Arithmetic: U = S·(A√r) on tensor cores with fp32 accumulation and S split
 * as bf16 hi + lo (ranks below 16 padded with zeros), then
 * W' = bf16_rn(W − (αη/√r)·U).
 * ---------------------------------------------------------------------- */
logra_status logra_merge_update(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                                uint64_t seed, uint32_t stream_id, float alpha_eta, const float* alpha_eta_dev,
                                logra_stream_t stream);

/* Merge with a given projection operand Ã (bf16 r×k, row stride lda, a
 * multiple of 8; 16-byte aligned): W ← bf16_rn(W − (αη/√r)·S·Ã), everything
 * else as in logra_merge_update. */
logra_status logra_merge_update_proj(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                                     const void* A, int64_t lda, float alpha_eta, const float* alpha_eta_dev,
                                     logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Merge of a set of weights in one launch
 *
 * Section "草图如何取代完整梯度缓冲": at the end of a step every sketched
 * weight of the model takes the merge W ← bf16(W − αη·S·A).  These calls do
 * the same for n weights (one common r and αη) in one launch over all their
 * tiles, so that small weights do not each leave the GPU partly idle at the
 * start and end of their own launch.  Each weight's result equals
 * logra_merge_update (A NULL) or logra_merge_update_proj (A given) on that
 * weight bit for bit.
 *
 * Two steps:
 *  1. logra_merge_group_plan() validates the targets and writes a plan of
 *     logra_merge_group_plan_bytes(n) bytes into HOST memory (128-byte
 *     aligned): a header, the tensor maps and the descriptors of every
 *     weight.  It launches nothing and needs no stream.
 *  2. The caller copies the plan unchanged into DEVICE memory (128-byte
 *     aligned; an ordinary stream-ordered copy before the launch), then
 *     calls logra_merge_update_group() with both copies: the host copy gives
 *     the launch shape, the kernels read the device copy.
 * A plan stays valid while the targets' buffers, shapes, seeds and operands
 * are unchanged, so a trainer plans once and merges every step with a new
 * αη.  The device copy must not be rewritten while a launch that reads it
 * may still run (stream order takes care of that).
 *
 * Targets: each as for logra_merge_update / _proj (W bf16 d×k in place, k
 * and ldw multiples of 8; S fp32 d×r; seed and stream_id, or a bf16 operand
 * A (r×k, row stride lda, a multiple of 8, 16-byte aligned)).  Either every
 * target has an operand A or none has (LOGRA_ERR_INVALID_ARG).  Weights with
 * d = 0 or k = 0 are skipped.  The W regions of the targets must not
 * overlap: the plan builder checks this (a weight named twice, or tied
 * weights, must be merged in separate launches).
 * Errors: as in logra_merge_update, per target; W regions that overlap
 * (LOGRA_ERR_INVALID_ARG); plan buffers that are too small or misaligned
 * (LOGRA_ERR_WORKSPACE / LOGRA_ERR_ALIGNMENT); a buffer that is not a plan
 * (LOGRA_ERR_INVALID_ARG).
 * ---------------------------------------------------------------------- */
typedef struct logra_merge_target {
  void* W;            /* bf16 d×k, row stride ldw, updated in place     */
  int64_t ldw;
  int64_t d;
  int64_t k;
  const float* S;     /* fp32 d×r, row stride lds                       */
  int64_t lds;
  uint64_t seed;      /* projection (when A is NULL)                    */
  uint32_t stream_id;
  const void* A;      /* optional bf16 r×k projection operand, or NULL  */
  int64_t lda;
} logra_merge_target;

size_t logra_merge_group_plan_bytes(int n);

logra_status logra_merge_group_plan(int n, const logra_merge_target* targets, int r, void* plan,
                                    size_t plan_bytes);

logra_status logra_merge_update_group(const void* plan, const void* plan_dev, float alpha_eta,
                                      const float* alpha_eta_dev, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Squared Frobenius norm (for the gradient-reconstruction diagnostic)
 *
 * Section "这些节省能说明什么、不能说明什么" reports the cosine between the
 * dense gradient and its reconstruction from the sketch.  This call gives the
 * norms that cosine needs: out_dev (device fp64 scalar) receives
 * ‖x‖_F² = Σ x_ij² of a rows×cols matrix (dtype LOGRA_DTYPE_FP32 or _BF16,
 * row stride ld elements), summed in fp64 in an order fixed by the shape
 * alone; with accumulate != 0 the sum is added to *out_dev instead.
 * workspace: at least logra_sum_squares_workspace_bytes() bytes, 8-byte
 * aligned.  rows or cols equal to 0 writes 0 (or leaves the sum unchanged).
 * ---------------------------------------------------------------------- */
size_t logra_sum_squares_workspace_bytes(void);
logra_status logra_sum_squares(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld, double* out_dev,
                               int accumulate, void* workspace, size_t workspace_bytes, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Per-step seed of a refreshed projection basis
 *
 * Section "这些节省能说明什么、不能说明什么" compares a fixed basis with one
 * redrawn every step but does not say how the redraw is keyed.  Reading taken
 * here: step t uses seed_t = w0 | (w1 << 32), where (w0, w1, ·, ·) are the
 * words of Philox4x32-10 at counter (t mod 2³², t >> 32, 0, 2) under the key
 * (base mod 2³², base >> 32); the fourth counter word 2 keeps these calls apart
 * from the sign (0) and Gaussian (1) draws.  Host function, no GPU needed.
 * ---------------------------------------------------------------------- */
uint64_t logra_refreshed_seed(uint64_t base_seed, uint64_t step);

/* ------------------------------------------------------------------------
 * Momentum on the sketch (a reading; the pages give no rule)
 *
 * Section "草图如何取代完整梯度缓冲" uses U = S and names stateful sketch
 * optimisers only as adding storage of their own.  This call keeps
 * heavy-ball momentum on the sketch:  M ← β·M + S  (one fused multiply-add
 * per element, rounded once to fp32), and, when clear_s != 0, S ← 0 in the
 * same pass so that S is ready for the next step.  The merge is then called
 * with U = M.  It is only meaningful with a fixed projection (the same seed
 * and stream id every step), so that every S lives in one basis.
 *
 *  M        fp32 d×r, row stride ldm, updated in place (caller-owned state,
 *           zero before the first step)
 *  S        fp32 d×r, row stride lds; must not overlap M
 *  beta     finite
 *
 * Errors: LOGRA_ERR_INVALID_ARG for r < 1, null pointers (with d > 0), M == S or a
 * non-finite beta; LOGRA_ERR_UNSUPPORTED for r > 256; LOGRA_ERR_SHAPE for
 * negative d, ldm < r or lds < r;
 * LOGRA_ERR_ALIGNMENT for pointers not 4-byte aligned.  d = 0 is a no-op.
 * ---------------------------------------------------------------------- */
logra_status logra_sketch_momentum(float* M, int64_t ldm, float* S, int64_t lds, int64_t d, int r, float beta,
                                   int clear_s, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Regenerate the projection A from its seed
 *
 * Section "同一份草图也压缩策略同步开销": the rollout engine rebuilds A from a
 * seed instead of receiving it.  Writes the r×k matrix (row stride lda
 * elements) as int8 ±1, bf16 ±1/√r or fp32 ±1/√r (out_kind).  The sketch and
 * merge kernels never call this for the signs: they rebuild tiles of A on
 * chip.
 *
 * The Gaussian kinds write the Gaussian projection of the design-choice
 * experiments (section "这些节省能说明什么、不能说明什么"), which the pages
 * leave unspecified.  Reading taken here: normals z by the Box–Muller
 * transform from Philox4x32-10 at counter (j >> 2, i, stream_id, 1) — for the
 * words (w0, w1, w2, w3), u = (w0 + ½)·2⁻³² and φ = (w1 + ½)·2⁻³² give
 * columns 4q and 4q+1 as √(−2 ln u)·cos 2πφ and √(−2 ln u)·sin 2πφ, and
 * (w2, w3) give 4q+2 and 4q+3 — rounded to bf16: Ã = bf16_rn(z), A = Ã/√r.
 * LOGRA_PROJ_GAUSS_BF16 writes Ã (the operand of the _proj entry points),
 * LOGRA_PROJ_GAUSS_FP32 writes A.  LOGRA_PROJ_SIGN_BF16 writes the signs as
 * the bf16 operand Ã = ±1 of the _proj calls (a cached copy of the Rademacher
 * projection, which those calls then read by TMA instead of regenerating it).  z is evaluated in fp32; where it lies
 * within a few fp32 ulps of a bf16 rounding midpoint the rounded value may be
 * either neighbour.
 * ---------------------------------------------------------------------- */
logra_status logra_regen_projection(uint64_t seed, uint32_t stream_id, int r, int64_t k, int out_kind, void* A_out,
                                    int64_t lda, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Predicted KL q(D)
 *
 * Section "预测 KL 控制防止过大更新破坏学习": for sampled token rows compare the
 * current model's vocabulary distribution p = softmax(a/τ) with the proposed
 * model's p' = softmax(b/τ) at the same temperature τ;
 * KL_t = Σ_v p_v (log p_v − log p'_v) and q(D) = mean of KL_t over the rows
 * whose mask byte is non-zero (all rows when row_mask is NULL; 0 when no row
 * is selected).
 *
 *  cur, prop   rows×V logits (dtype LOGRA_DTYPE_BF16 or _FP32), row stride ld
 *  temperature τ > 0
 *  row_mask    optional device uint8 [rows]
 *  q_dev       device fp64 scalar receiving q(D)
 *  row_kl_dev  optional device fp32 [rows] receiving KL_t
 *  workspace   at least logra_kl_workspace_bytes(rows) bytes, 256-byte aligned
 *
 * Arithmetic: one pass over each row with an online max; with
 * d_v = (b_v − a_v)/τ, KL_t = E_p[e^d − 1 − d] + (log1p(u) − u) where
 * u = E_p[e^d − 1], a form without the cancellation of log Z' − log Z.  Row
 * sums are fp32, the per-row combination and the mean are fp64 in a fixed
 * order.  A −inf current logit contributes nothing; a finite current logit
 * with a −inf proposed logit gives +inf; NaN propagates.
 * ---------------------------------------------------------------------- */
size_t logra_kl_workspace_bytes(int64_t rows);

logra_status logra_predicted_kl(const void* cur, const void* prop, int dtype, int64_t rows, int64_t V, int64_t ld,
                                float temperature, const uint8_t* row_mask, double* q_dev, float* row_kl_dev,
                                void* workspace, size_t workspace_bytes, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Predicted KL without a workspace (the paper has no counterpart of this
 * call; it is an interface convenience)
 *
 * Computes exactly what logra_predicted_kl computes, with the same arguments
 * minus the workspace, and allocates nothing: the per-row scratch is a fixed
 * array inside the library.  It serves callers that cannot obtain device
 * memory where they need q(D): an inference or rollout engine that has handed
 * all device memory to its own pool at start-up, so that a cudaMalloc there
 * would fail or fragment the pool; or a plain C controller that holds only
 * the logits pointers it was given and has no device allocator of its own.
 *
 *  - rows ≤ LOGRA_KL_NOALLOC_MAX_ROWS (65536); a larger call returns
 *    LOGRA_ERR_UNSUPPORTED and launches nothing.
 *  - The fixed array occupies 512 KiB on every GPU that loads the library,
 *    for as long as the process lives.
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *  - Every call uses the same array and it keeps the last call's contents.
 *    Calls whose kernels can overlap on the GPU (different streams, or host
 *    threads without ordering between them) race and can return wrong
 *    values; order them on one stream.  Nothing in the array has to start at
 *    zero: each row's entry is written before it is read.
 * ---------------------------------------------------------------------- */
#define LOGRA_KL_NOALLOC_MAX_ROWS 65536

logra_status logra_predicted_kl_noalloc(const void* cur, const void* prop, int dtype, int64_t rows, int64_t V,
                                        int64_t ld, float temperature, const uint8_t* row_mask, double* q_dev,
                                        float* row_kl_dev, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Step size  α = min(α_max, √(δ/q))
 *
 * Section "预测 KL 控制防止过大更新破坏学习".  Host-only and synchronous.
 * q ≤ 0 gives α_max, q = +inf gives 0, NaN q gives NaN.  δ > 0 and α_max > 0
 * (LOGRA_ERR_INVALID_ARG otherwise).
 * ---------------------------------------------------------------------- */
logra_status logra_step_size(double q, double delta, double alpha_max, double* alpha_out);

/* Device variant: reads q from device memory and writes the fp32 product
 * α·η to *alpha_eta_dev (and α itself to *alpha_dev when not NULL), on
 * `stream`, so that logra_merge_update can take the step without a host
 * synchronisation. */
logra_status logra_step_size_device(const double* q_dev, double delta, double alpha_max, double eta,
                                    float* alpha_eta_dev, double* alpha_dev, logra_stream_t stream);

/* ------------------------------------------------------------------------
 * Device error word
 *
 * Synchronises `stream`, returns in *code the first error code a kernel of
 * this library recorded on the current device since the last call (0 = none),
 * and clears it.  Returns LOGRA_ERR_DEVICE when the code is non-zero.
 * ---------------------------------------------------------------------- */
logra_status logra_device_error(logra_stream_t stream, unsigned int* code);

/* Self-test of the failure reporting above (the paper has no counterpart):
 * enqueues on `stream` a one-thread kernel that waits on a shared-memory
 * barrier nothing ever arrives at.  After the kernels' one-second wait limit
 * it records code 7 in the device error word and returns; no fault, trap or
 * unbounded wait is involved, and the context stays usable.  A following
 * logra_device_error(stream, &code) returns LOGRA_ERR_DEVICE with code 7 and
 * clears the word. */
logra_status logra_self_test_wait_timeout(logra_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOGRA_H_ */
