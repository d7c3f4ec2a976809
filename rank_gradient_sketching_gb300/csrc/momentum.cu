// Momentum on the sketch: M ← β·M + S over a d×r fp32 matrix, optionally
// clearing S in the same pass so that it is ready for the next step's
// accumulation.
//
// LoGRA summary page, section "草图如何取代完整梯度缓冲": the plain update
// uses U = S and the page mentions stateful sketch optimisers only as adding
// storage of their own, with no rule.  The reading implemented here is
// heavy-ball momentum kept on the sketch (U = M), which needs a fixed
// projection: every S then lives in the same r-dimensional basis.
//
// The pass is a pure HBM stream: 12 bytes per element (read M and S, write M)
// plus 4 more when S is cleared.  The arithmetic is one fused multiply-add
// per element, rounded once to fp32.

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

constexpr int kMomThreads = 256;

// Both matrices contiguous (row length r), viewed as n4 float4 elements.
__global__ void __launch_bounds__(kMomThreads)
    momentum_flat_kernel(float4* __restrict__ M, float4* __restrict__ S, int64_t n4, float beta, int clear_s) {
  const int64_t stride = (int64_t)gridDim.x * kMomThreads;
  for (int64_t f = (int64_t)blockIdx.x * kMomThreads + threadIdx.x; f < n4; f += stride) {
    const float4 s = __ldcs(S + f);
    float4 m = __ldcs(M + f);
    m.x = fmaf(beta, m.x, s.x);
    m.y = fmaf(beta, m.y, s.y);
    m.z = fmaf(beta, m.z, s.z);
    m.w = fmaf(beta, m.w, s.w);
    __stcs(M + f, m);
    if (clear_s) __stcs(S + f, make_float4(0.f, 0.f, 0.f, 0.f));
  }
}

// Any strides: a CTA walks rows, its threads the columns of a row.
__global__ void __launch_bounds__(kMomThreads)
    momentum_rows_kernel(float* __restrict__ M, int64_t ldm, float* __restrict__ S, int64_t lds, int64_t d, int r,
                         float beta, int clear_s) {
  for (int64_t row = blockIdx.x; row < d; row += gridDim.x) {
    float* mrow = M + row * ldm;
    float* srow = S + row * lds;
    for (int c = threadIdx.x; c < r; c += kMomThreads) {
      const float s = srow[c];
      mrow[c] = fmaf(beta, mrow[c], s);
      if (clear_s) srow[c] = 0.f;
    }
  }
}

}  // namespace

logra_status launch_momentum(float* M, int64_t ldm, float* S, int64_t lds, int64_t d, int r, float beta, int clear_s,
                             cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "query the multiprocessor count");
  const int64_t n = d * (int64_t)r;
  const bool flat = ldm == r && lds == r && n % 4 == 0 && (reinterpret_cast<uintptr_t>(M) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(S) & 15) == 0;
  if (flat) {
    // enough CTAs in flight to cover the memory latency: 8 per SM, each
    // thread then walks a grid-stride loop
    const int64_t n4 = n / 4;
    const int64_t want = (n4 + kMomThreads - 1) / kMomThreads;
    const unsigned blocks = (unsigned)std::min<int64_t>(want, (int64_t)sms * 8);
    momentum_flat_kernel<<<blocks, kMomThreads, 0, st>>>(reinterpret_cast<float4*>(M), reinterpret_cast<float4*>(S),
                                                          n4, beta, clear_s);
  } else {
    const unsigned blocks = (unsigned)std::min<int64_t>(d, (int64_t)sms * 16);
    momentum_rows_kernel<<<blocks, kMomThreads, 0, st>>>(M, ldm, S, lds, d, r, beta, clear_s);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch momentum kernel");
  return LOGRA_OK;
}

}  // namespace logra
