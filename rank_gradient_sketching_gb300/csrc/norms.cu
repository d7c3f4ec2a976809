// Squared Frobenius norm ‖x‖² of a matrix (fp32 or bf16) into a device fp64
// scalar, for the gradient-reconstruction diagnostic of the LoGRA summary
// page (section "这些节省能说明什么、不能说明什么": the cosine between the
// dense gradient and its reconstruction from the sketch).
//
// Deterministic: a fixed grid of kNormBlocks CTAs (independent of the device)
// each sums a fixed set of rows in fp64 in a fixed order, and a single CTA
// then adds the per-CTA partials in index order.

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

constexpr int kNormThreads = 256;

template <typename T>
__device__ __forceinline__ double sq(const T* p) {
  const double v = (double)static_cast<float>(*p);
  return v * v;
}
template <>
__device__ __forceinline__ double sq<__nv_bfloat16>(const __nv_bfloat16* p) {
  const double v = (double)__bfloat162float(*p);
  return v * v;
}

__device__ double block_sum(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kNormThreads / 32; ++w) t += red[w];
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    sum_squares_partial_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
                               double* __restrict__ partial) {
  __shared__ double red[kNormThreads / 32];
  double acc = 0.0;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const T* xr = x + row * ld;
    for (int64_t c = threadIdx.x; c < cols; c += kNormThreads) acc += sq(xr + c);
  }
  const double t = block_sum(acc, red);
  if (threadIdx.x == 0) partial[blockIdx.x] = t;
}

__global__ void __launch_bounds__(kNormThreads)
    sum_squares_final_kernel(const double* __restrict__ partial, int n, double* out, int accumulate) {
  __shared__ double red[kNormThreads / 32];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += kNormThreads) acc += partial[i];
  const double t = block_sum(acc, red);
  if (threadIdx.x == 0) *out = accumulate ? *out + t : t;
}

}  // namespace

logra_status launch_sum_squares(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld, double* out,
                                int accumulate, void* ws, cudaStream_t st) {
  double* partial = static_cast<double*>(ws);
  const unsigned blocks = (unsigned)kNormBlocks;
  if (dtype == LOGRA_DTYPE_BF16)
    sum_squares_partial_kernel<__nv_bfloat16><<<blocks, kNormThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), rows, cols, ld, partial);
  else
    sum_squares_partial_kernel<float><<<blocks, kNormThreads, 0, st>>>(static_cast<const float*>(x), rows, cols, ld,
                                                                       partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch sum_squares_partial_kernel");
  sum_squares_final_kernel<<<1, kNormThreads, 0, st>>>(partial, kNormBlocks, out, accumulate);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch sum_squares_final_kernel");
  return LOGRA_OK;
}

}  // namespace logra
