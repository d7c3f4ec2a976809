// Host-side glue shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/logra.h"

namespace logra {

// Records a failure for logra_last_error() and returns `st`.
logra_status fail(logra_status st, const std::string& msg);
// Clears the thread's last-error message and returns LOGRA_OK.
logra_status ok();
// Maps a CUDA runtime error to LOGRA_ERR_CUDA with context.
logra_status cuda_fail(cudaError_t e, const char* what);

// Device word that kernels write error codes into (current device).
// Returns nullptr and records an error when it cannot be resolved.
unsigned int* device_error_word();

// Checks that the current device is an sm_103 part and returns its SM count.
logra_status require_sm103(int* sm_count);

// 2-D bf16 tensor map with 128-byte swizzle, zero fill out of bounds.
// inner/outer are the tensor extents in elements/rows, row_bytes the row
// stride; box_inner × box_outer is the tile moved by one copy.
// swizzle_bytes: 128 (rows of the box are 128 bytes) or 64 (rows of 64 bytes).
logra_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                               uint32_t swizzle_bytes = 128);
// fp32 2-D tensor map with the 128-byte swizzle (box_inner·4 ≤ 128 bytes).
logra_status make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer);

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- sketch
struct SketchPlan {
  int64_t T, d, k;
  int r, np;          // np = r rounded up to 16 (MMA N)
  int p16;            // 1: P is carried as fp16 with a power-of-two scale per token (np > 64),
                      // 0: as a bf16 hi + lo pair
  int mt;             // 128-row sub-tiles of S per contraction CTA
  int64_t ldp;        // row stride of the P buffers, T rounded up to 128
  int64_t dp;         // d rounded up to 128·mt
  int d_tiles;        // dp / (128·mt)
  int tk;             // tokens per contraction stage (64 or 32)
  int num_kb_t;       // token blocks of tk
  int splits;         // split ranges of T
  int kb_per_split;
  // Workspace regions: Pᵀ_hi (bf16) or Pᵀ (fp16) at off_phi; Pᵀ_lo (bf16) or
  // the per-token scales (fp32, ldp of them) at off_plo; split partials.
  size_t off_phi, off_plo, off_part, bytes;
};
SketchPlan plan_sketch(int64_t T, int64_t d, int64_t k, int r);

logra_status launch_sketch(const SketchPlan& p, const void* X, int64_t ldx, const void* dY, int64_t lddy,
                           uint64_t seed, uint32_t stream_id, float* S, int64_t lds, void* ws, cudaStream_t st);
size_t shared_x_workspace_bytes(int64_t T, int64_t k, int n, const int64_t* d, int r);
// The same with a given bf16 projection operand Ã (r×k, row stride lda); the
// sketch is S += (1/√r)·dYᵀ(X·Ãᵀ).
logra_status launch_sketch_explicit(const SketchPlan& p, const void* X, int64_t ldx, const void* dY, int64_t lddy,
                                    const void* A, int64_t lda, float* S, int64_t lds, void* ws, cudaStream_t st);
// A / lda: per-target bf16 projection operands, or nullptr for signs built on chip.
logra_status launch_sketch_shared_x(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                    const logra_sketch_target* tg, int r, const void* const* A, const int64_t* lda,
                                    void* ws, cudaStream_t st);
// Sketch of a set of matrices with one launch per phase: plan size, the
// workspace the plan lays out, plan construction (host memory; targets
// validated by the caller, ws of at least sketch_group_workspace_bytes),
// plan header check, launch.
size_t sketch_group_plan_bytes(int n);
size_t sketch_group_workspace_bytes(int n, const logra_sketch_group_target* tg, int r);
logra_status build_sketch_group_plan(int n, const logra_sketch_group_target* tg, int r, void* ws, void* plan);
logra_status check_sketch_group_plan(const void* plan, int* n);
logra_status launch_sketch_group(const void* plan, const void* plan_dev, cudaStream_t st);

// ---------------------------------------------------------------- merge
// A (optional): a given bf16 projection operand Ã (r×k, row stride lda) used
// in place of the regenerated signs; the update is then W − (αη/√r)·S·Ã.
logra_status launch_merge(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                          uint64_t seed, uint32_t stream_id, float alpha_eta, const float* alpha_eta_dev,
                          const void* A, int64_t lda, cudaStream_t st);
// Merge of a set of weights in one launch: plan size, plan construction (host
// memory, targets validated by the caller), plan header check, launch.
size_t merge_group_plan_bytes(int n);
logra_status build_merge_group_plan(int n, const logra_merge_target* tg, int r, void* plan, size_t plan_bytes);
logra_status check_merge_group_plan(const void* plan, int* n, int* r);
logra_status launch_merge_group(const void* plan, const void* plan_dev, float alpha_eta, const float* alpha_eta_dev,
                                cudaStream_t st);

// ---------------------------------------------------------------- KL
logra_status launch_kl(const void* cur, const void* prop, int dtype, int64_t rows, int64_t V, int64_t ld,
                       float temperature, const uint8_t* mask, double* q_dev, float* row_kl, void* ws,
                       cudaStream_t st);
logra_status launch_step_size_device(const double* q_dev, double delta, double alpha_max, double eta,
                                     float* alpha_eta_dev, double* alpha_dev, cudaStream_t st);

// ---------------------------------------------------------------- momentum
logra_status launch_momentum(float* M, int64_t ldm, float* S, int64_t lds, int64_t d, int r, float beta, int clear_s,
                             cudaStream_t st);

// ---------------------------------------------------------------- norms
constexpr int kNormBlocks = 1024;  // partial sums per call (fixed: the sum order never depends on the device)
logra_status launch_sum_squares(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld, double* out,
                                int accumulate, void* ws, cudaStream_t st);

// ---------------------------------------------------------------- self-test
logra_status launch_self_test_wait_timeout(cudaStream_t st);

// ---------------------------------------------------------------- regen
logra_status launch_regen(uint64_t seed, uint32_t stream_id, int r, int64_t k, int out_kind, void* A, int64_t lda,
                          cudaStream_t st);

}  // namespace logra
