// Regenerate the projection A from its seed (LoGRA summary page, section
// "同一份草图也压缩策略同步开销": the rollout side rebuilds A from a seed instead
// of receiving it).  One warp writes one 128-column group of one row: each lane
// takes four consecutive columns, so stores of a warp are contiguous.

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
    else
      static_cast<float*>(out)[off] = neg ? -scale : scale;
  }
}

}  // namespace

logra_status launch_regen(uint64_t seed, uint32_t stream_id, int r, int64_t k, int out_kind, void* A, int64_t lda,
                          cudaStream_t st) {
  const int64_t items = (int64_t)r * ((k + 127) / 128);
  const float scale = (float)(1.0 / std::sqrt((double)r));
  regen_kernel<<<(unsigned)((items + 7) / 8), 256, 0, st>>>(seed, stream_id, r, k, out_kind, A, lda, scale);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch regen_kernel");
  return LOGRA_OK;
}

}  // namespace logra
