// Regenerate the projection A from its seed (LoGRA summary page, section
// "同一份草图也压缩策略同步开销": the rollout side rebuilds A from a seed instead
// of receiving it).  Signs: one warp writes one 128-column group of one row,
// each lane taking four consecutive columns, so stores of a warp are
// contiguous.  Gaussian (the refreshed-Gaussian variant of the design-choice
// experiments in section "这些节省能说明什么、不能说明什么"): one thread per four
// consecutive columns of a row (one generator call), written as the bf16
// operand Ã = bf16_rn(z) or as A = Ã/√r in fp32.

#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

__global__ void __launch_bounds__(256)
    regen_kernel(uint64_t seed, uint32_t stream_id, int r, int64_t k, int kind, void* out, int64_t lda,
                 float scale) {
  const int64_t groups = (k + 127) / 128;
  const int64_t item = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (item >= (int64_t)r * groups) return;
  const int row = (int)(item / groups);
  const int64_t g = item % groups;
  const int lane = threadIdx.x & 31;
  const uint4 w = sign_words(seed, stream_id, (uint32_t)row, (uint32_t)g);
  const uint32_t word = word_of(w, lane >> 3);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = lane * 4 + e;
    const int64_t col = g * 128 + j;
    if (col >= k) break;
    const bool neg = (word >> (j & 31)) & 1u;
    const int64_t off = (int64_t)row * lda + col;
    if (kind == LOGRA_PROJ_INT8_PM1)
      static_cast<int8_t*>(out)[off] = neg ? (int8_t)-1 : (int8_t)1;
    else if (kind == LOGRA_PROJ_BF16)
      static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(neg ? -scale : scale);
    else if (kind == LOGRA_PROJ_SIGN_BF16)
      static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(neg ? -1.0f : 1.0f);
    else
      static_cast<float*>(out)[off] = neg ? -scale : scale;
  }
}

__global__ void __launch_bounds__(256)
    regen_gauss_kernel(uint64_t seed, uint32_t stream_id, int r, int64_t k, int kind, void* out, int64_t lda,
                       float scale) {
  const int64_t quads = (k + 3) / 4;
  const int64_t item = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (item >= (int64_t)r * quads) return;
  const int row = (int)(item / quads);
  const int64_t q = item % quads;
  const float4 z = gauss_quad(seed, stream_id, (uint32_t)row, (uint32_t)q);
  const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int64_t col = q * 4 + e;
    if (col >= k) break;
    const __nv_bfloat16 op = __float2bfloat16_rn(zz[e]);
    const int64_t off = (int64_t)row * lda + col;
    if (kind == LOGRA_PROJ_GAUSS_BF16)
      static_cast<__nv_bfloat16*>(out)[off] = op;
    else
      static_cast<float*>(out)[off] = __bfloat162float(op) * scale;
  }
}

}  // namespace

logra_status launch_regen(uint64_t seed, uint32_t stream_id, int r, int64_t k, int out_kind, void* A, int64_t lda,
                          cudaStream_t st) {
  const float scale = (float)(1.0 / std::sqrt((double)r));
  if (out_kind == LOGRA_PROJ_GAUSS_BF16 || out_kind == LOGRA_PROJ_GAUSS_FP32) {
    const int64_t items = (int64_t)r * ((k + 3) / 4);
    regen_gauss_kernel<<<(unsigned)((items + 255) / 256), 256, 0, st>>>(seed, stream_id, r, k, out_kind, A, lda,
                                                                       scale);
  } else {
    const int64_t items = (int64_t)r * ((k + 127) / 128);
    regen_kernel<<<(unsigned)((items + 7) / 8), 256, 0, st>>>(seed, stream_id, r, k, out_kind, A, lda, scale);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch regen_kernel");
  return LOGRA_OK;
}

}  // namespace logra
