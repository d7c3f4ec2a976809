// Squared Frobenius norm ‖x‖² of a matrix (fp32 or bf16) into a device fp64
// scalar, for the gradient-reconstruction diagnostic of the LoGRA summary
// page (section "这些节省能说明什么、不能说明什么": the cosine between the
// dense gradient and its reconstruction from the sketch).
//
// Deterministic: a fixed grid of kNormBlocks CTAs (independent of the device)
// each sums a fixed set of elements in fp64 in a fixed order (16-byte vectors
// of a contiguous matrix, else rows), and a single CTA then adds the per-CTA
// partials in index order.

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

// Contiguous input as n16 16-byte vectors: each thread walks a fixed
// grid-stride sequence with four independent loads in flight.  The squares of
// one vector are summed in fp32 (a bf16 square is exact in fp32) and the
// vector's sum is added in fp64, so the fp64 pipe, far slower than HBM on this
// part, sees one add per 16 bytes.
template <typename T>
__device__ __forceinline__ double sq_vec(const uint4& v) {
  float a = 0.f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (sizeof(T) == 2) {
      const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
      a = fmaf(lo, lo, a);
      a = fmaf(hi, hi, a);
    } else {
      const float f = __uint_as_float(w[i]);
      a = fmaf(f, f, a);
    }
  }
  return (double)a;
}

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    sum_squares_flat_kernel(const uint4* __restrict__ x, int64_t n16, double* __restrict__ partial) {
  __shared__ double red[kNormThreads / 32];
  const int64_t stride = (int64_t)gridDim.x * kNormThreads;
  int64_t i = (int64_t)blockIdx.x * kNormThreads + threadIdx.x;
  double acc = 0.0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(x + i), b = __ldcs(x + i + stride), c = __ldcs(x + i + 2 * stride),
                d = __ldcs(x + i + 3 * stride);
    acc += sq_vec<T>(a) + sq_vec<T>(b) + sq_vec<T>(c) + sq_vec<T>(d);
  }
  for (; i < n16; i += stride) acc += sq_vec<T>(__ldcs(x + i));
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
  const int64_t esz = dtype == LOGRA_DTYPE_BF16 ? 2 : 4;
  const bool flat = ld == cols && (rows * cols * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  if (flat) {
    const int64_t n16 = rows * cols * esz / 16;
    if (dtype == LOGRA_DTYPE_BF16)
      sum_squares_flat_kernel<__nv_bfloat16><<<blocks, kNormThreads, 0, st>>>(static_cast<const uint4*>(x), n16,
                                                                              partial);
    else
      sum_squares_flat_kernel<float><<<blocks, kNormThreads, 0, st>>>(static_cast<const uint4*>(x), n16, partial);
  } else if (dtype == LOGRA_DTYPE_BF16)
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
