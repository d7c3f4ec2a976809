// Predicted KL q(D) and the step-size controller.
//
// LoGRA summary page, section "预测 KL 控制防止过大更新破坏学习": the current and
// the proposed model's next-token distributions are compared on sampled rows
// at one temperature; q(D) is the mean KL, and α = min{α_max, √(δ/q(D))}.
//
// One CTA per row, one pass over the V logits of both models.  With
// x_v = a_v/τ, d_v = (b_v − a_v)/τ and weights w_v = e^(x_v − m):
//     KL = E_p[φ(d)] + ψ(u),   φ(d) = e^d − 1 − d,   u = E_p[e^d − 1],
//     ψ(u) = log1p(u) − u,
// which is the plain definition Σ p (log p − log p′) rewritten so that no two
// large log-partition functions are subtracted.  Each thread keeps the running
// (m, Σw, Σw(e^d − 1), Σwφ(d)) with an online max; threads merge by warp
// shuffles and one shared-memory step; the row's combination is done in fp64.
// For |d| ≤ 1/2, φ(d) = d²·Σ_{n≥0} dⁿ/(n+2)! (Taylor series of the exponential,
// degree 6), which keeps full fp32 relative accuracy where e^d − 1 − d would
// cancel; larger |d| and non-finite inputs take a per-element path through
// expm1f.  The mean over rows is a second, single-CTA kernel that sums the
// fp64 per-row values in a fixed order.

#include <cmath>
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

constexpr int kKlThreads = 256;
constexpr int kMeanThreads = 1024;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// |d| up to which φ(d) = e^d − 1 − d comes from its Taylor series: φ(d)/d²
// = Σ_{n≥0} dⁿ/(n+2)!, kept to d⁵ (coefficients 1/2!, …, 1/7!).  The first
// omitted term, d⁶/8!, is below 2e-7 of φ(d) ≈ d²/2 for |d| ≤ 3/8.
constexpr float kSeriesMax = 0.375f;
constexpr float kC2 = 1.0f / 2.0f, kC3 = 1.0f / 6.0f, kC4 = 1.0f / 24.0f, kC5 = 1.0f / 120.0f,
                kC6 = 1.0f / 720.0f, kC7 = 1.0f / 5040.0f;

__device__ __forceinline__ float phi_over_d2(float d) {
  float p = kC7;
  p = fmaf(p, d, kC6);
  p = fmaf(p, d, kC5);
  p = fmaf(p, d, kC4);
  p = fmaf(p, d, kC3);
  p = fmaf(p, d, kC2);
  return p;
}

// Pairs of fp32 values in one 64-bit register pair, processed by the packed
// (f32x2) FMA / add / mul instructions: two lanes of arithmetic per issue.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max that returns NaN when either input is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

struct RowAcc {
  float m;    // running max of a·log2(e)/τ
  float s;    // Σ w
  float su;   // Σ w·(e^d − 1)
  float sp;   // Σ w·φ(d)
  uint64_t s2, su2, sp2;  // the same three sums, two lanes, for the packed path
  float mx;   // running max of b·log2(e)/τ over tokens with a = −inf
  float sx;   // Σ e^(b/τ) over those tokens, relative to mx
  bool nan;   // a NaN met where p = 0
};

__device__ __forceinline__ void rescale(RowAcc& r, float new_m) {
  const float f = (r.m == -INFINITY) ? 0.f : ex2_approx(r.m - new_m);
  r.s *= f;
  r.su *= f;
  r.sp *= f;
  const uint64_t f2 = pk2(f, f);
  r.s2 = mul2(r.s2, f2);
  r.su2 = mul2(r.su2, f2);
  r.sp2 = mul2(r.sp2, f2);
  r.m = new_m;
}

// Folds the packed lanes into the scalar sums (once per thread).
__device__ __forceinline__ void fold_pairs(RowAcc& r) {
  float lo, hi;
  upk2(r.s2, lo, hi);
  r.s += lo + hi;
  upk2(r.su2, lo, hi);
  r.su += lo + hi;
  upk2(r.sp2, lo, hi);
  r.sp += lo + hi;
  r.s2 = r.su2 = r.sp2 = 0ull;
}

// Careful per-element path: non-finite inputs and |d| > 1/2.
__device__ __forceinline__ void slow_element(RowAcc& r, float a, float b, float sc, float inv_tau) {
  if (a == -INFINITY) {
    // p_v = 0, so the token adds nothing to E_p[·] — but the proposed
    // normaliser still holds e^(b_v/τ), which enters u (and E_p[φ]) as
    // p'_v·Z'/Z.  That mass is kept apart with its own running max.
    if (b != b) {
      r.nan = true;
    } else if (b != -INFINITY) {
      const float y = b * sc;
      if (y > r.mx) {
        r.sx = (r.mx == -INFINITY) ? 0.f : r.sx * ex2_approx(r.mx - y);
        r.mx = y;
      }
      r.sx += ex2_approx(y - r.mx);
    }
    return;
  }
  const float x = a * sc;
  if (x > r.m) rescale(r, x);
  const float w = ex2_approx(x - r.m);
  const float d = (b - a) * inv_tau;
  float em1, phi;
  if (fabsf(d) <= kSeriesMax) {
    phi = d * d * phi_over_d2(d);
    em1 = d + phi;
  } else {
    em1 = expm1f(d);
    phi = em1 - d;
  }
  r.s += w;
  r.su = fmaf(w, em1, r.su);
  r.sp = fmaf(w, phi, r.sp);
}

// Eight consecutive logits of each model.  a_w / b_w hold them as raw 32-bit
// words of two bf16 each (fp32 inputs are passed as float pairs).
__device__ __forceinline__ void chunk8(RowAcc& r, const float (&a)[8], const float (&b)[8], float sc, float inv_tau) {
  float amax = a[0], dmax = 0.f;
  uint64_t A[4], D[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    A[e] = pk2(a[2 * e], a[2 * e + 1]);
    D[e] = mul2(sub2(pk2(b[2 * e], b[2 * e + 1]), A[e]), pk2(inv_tau, inv_tau));
  }
#pragma unroll
  for (int e = 1; e < 8; ++e) amax = fmaxf(amax, a[e]);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float d0, d1;
    upk2(D[e], d0, d1);
    dmax = fmax_nan(dmax, fmax_nan(fabsf(d0), fabsf(d1)));
  }
  if (dmax <= kSeriesMax) {  // all inputs finite and |d| small: the packed path
    const float xm = amax * sc;
    if (xm > r.m) rescale(r, xm);
    const uint64_t sc2 = pk2(sc, sc), negm2 = pk2(-r.m, -r.m);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x0, x1;
      upk2(fma2(A[e], sc2, negm2), x0, x1);
      const uint64_t W = pk2(ex2_approx(x0), ex2_approx(x1));
      const uint64_t D2 = mul2(D[e], D[e]);
      uint64_t P = fma2(pk2(kC7, kC7), D[e], pk2(kC6, kC6));
      P = fma2(P, D[e], pk2(kC5, kC5));
      P = fma2(P, D[e], pk2(kC4, kC4));
      P = fma2(P, D[e], pk2(kC3, kC3));
      P = fma2(P, D[e], pk2(kC2, kC2));
      const uint64_t PHI = mul2(D2, P);
      r.s2 = add2(r.s2, W);
      r.su2 = fma2(W, add2(D[e], PHI), r.su2);
      r.sp2 = fma2(W, PHI, r.sp2);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) slow_element(r, a[e], b[e], sc, inv_tau);
  }
}

__device__ __forceinline__ void merge_acc(RowAcc& r, float m, float s, float su, float sp, float mx, float sx,
                                          bool nan) {
  const float M = fmaxf(r.m, m);
  const float f1 = (r.m == -INFINITY) ? 0.f : ex2_approx(r.m - M);
  const float f2 = (m == -INFINITY) ? 0.f : ex2_approx(m - M);
  r.s = r.s * f1 + s * f2;
  r.su = r.su * f1 + su * f2;
  r.sp = r.sp * f1 + sp * f2;
  r.m = M;
  const float MX = fmaxf(r.mx, mx);
  const float g1 = (r.mx == -INFINITY) ? 0.f : ex2_approx(r.mx - MX);
  const float g2 = (mx == -INFINITY) ? 0.f : ex2_approx(mx - MX);
  r.sx = r.sx * g1 + sx * g2;
  r.mx = MX;
  r.nan = r.nan || nan;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 u0 = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 u1 = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
  v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
}

__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

template <typename T>
__global__ void __launch_bounds__(kKlThreads, 4)
    kl_rows_kernel(const T* __restrict__ cur, const T* __restrict__ prop, int64_t V, int64_t ld, float inv_tau,
                   double* __restrict__ row_kl64, float* __restrict__ row_kl32) {
  const int64_t row = blockIdx.x;
  const T* a_row = cur + row * ld;
  const T* b_row = prop + row * ld;
  const float sc = inv_tau * kLog2e;
  RowAcc r{-INFINITY, 0.f, 0.f, 0.f, 0ull, 0ull, 0ull, -INFINITY, 0.f, false};

  const int64_t nch = V / 8;
  int64_t ch = threadIdx.x;
  for (; ch + kKlThreads < nch; ch += 2 * kKlThreads) {
    float a0[8], b0[8], a1[8], b1[8];
    load8(a_row + ch * 8, a0);
    load8(b_row + ch * 8, b0);
    load8(a_row + (ch + kKlThreads) * 8, a1);
    load8(b_row + (ch + kKlThreads) * 8, b1);
    chunk8(r, a0, b0, sc, inv_tau);
    chunk8(r, a1, b1, sc, inv_tau);
  }
  if (ch < nch) {
    float a0[8], b0[8];
    load8(a_row + ch * 8, a0);
    load8(b_row + ch * 8, b0);
    chunk8(r, a0, b0, sc, inv_tau);
  }
  for (int64_t v = nch * 8 + threadIdx.x; v < V; v += kKlThreads)
    slow_element(r, load1(a_row + v), load1(b_row + v), sc, inv_tau);
  fold_pairs(r);

  // warp merge
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m = __shfl_xor_sync(0xffffffffu, r.m, off);
    const float s = __shfl_xor_sync(0xffffffffu, r.s, off);
    const float su = __shfl_xor_sync(0xffffffffu, r.su, off);
    const float sp = __shfl_xor_sync(0xffffffffu, r.sp, off);
    const float mx = __shfl_xor_sync(0xffffffffu, r.mx, off);
    const float sx = __shfl_xor_sync(0xffffffffu, r.sx, off);
    const int nan = __shfl_xor_sync(0xffffffffu, (int)r.nan, off);
    merge_acc(r, m, s, su, sp, mx, sx, nan != 0);
  }
  __shared__ float sh[6][kKlThreads / 32];
  __shared__ int shn[kKlThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sh[0][warp] = r.m;
    sh[1][warp] = r.s;
    sh[2][warp] = r.su;
    sh[3][warp] = r.sp;
    sh[4][warp] = r.mx;
    sh[5][warp] = r.sx;
    shn[warp] = r.nan;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    RowAcc t{sh[0][0], sh[1][0], sh[2][0], sh[3][0], 0ull, 0ull, 0ull, sh[4][0], sh[5][0], shn[0] != 0};
    for (int w = 1; w < kKlThreads / 32; ++w)
      merge_acc(t, sh[0][w], sh[1][w], sh[2][w], sh[3][w], sh[4][w], sh[5][w], shn[w] != 0);
    double kl;
    if (t.nan) {
      kl = __longlong_as_double(0x7ff8000000000000LL);
    } else {
      // mass of tokens with p = 0, in the units of s (relative to 2^m)
      const double extra = t.sx > 0.f ? (double)t.sx * exp2((double)t.mx - (double)t.m) : 0.0;
      const double s = t.s, u = ((double)t.su + extra) / s, ephi = ((double)t.sp + extra) / s;
      kl = ephi + (log1p(u) - u);
    }
    row_kl64[row] = kl;
    if (row_kl32) row_kl32[row] = (float)kl;
  }
}

__global__ void __launch_bounds__(kMeanThreads)
    kl_mean_kernel(const double* __restrict__ row_kl, const uint8_t* __restrict__ mask, int64_t rows,
                   double* __restrict__ q) {
  __shared__ double sacc[kMeanThreads];
  __shared__ long long scnt[kMeanThreads];
  double acc = 0.0;
  long long cnt = 0;
  for (int64_t i = threadIdx.x; i < rows; i += kMeanThreads) {
    if (!mask || mask[i]) {
      acc += row_kl[i];
      ++cnt;
    }
  }
  sacc[threadIdx.x] = acc;
  scnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int h = kMeanThreads / 2; h > 0; h >>= 1) {
    if (threadIdx.x < h) {
      sacc[threadIdx.x] += sacc[threadIdx.x + h];
      scnt[threadIdx.x] += scnt[threadIdx.x + h];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *q = scnt[0] ? sacc[0] / (double)scnt[0] : 0.0;
}

__global__ void step_size_kernel(const double* q_dev, double delta, double alpha_max, double eta, float* ae,
                                 double* alpha_out) {
  const double q = *q_dev;
  double alpha;
  if (q != q) alpha = q;
  else if (q <= 0.0) alpha = alpha_max;
  else alpha = fmin(alpha_max, sqrt(delta / q));
  *ae = (float)(alpha * eta);
  if (alpha_out) *alpha_out = alpha;
}

}  // namespace

logra_status launch_kl(const void* cur, const void* prop, int dtype, int64_t rows, int64_t V, int64_t ld,
                       float temperature, const uint8_t* mask, double* q_dev, float* row_kl, void* ws,
                       cudaStream_t st) {
  double* row64 = static_cast<double*>(ws);
  const float inv_tau = (float)(1.0 / (double)temperature);
  cudaError_t e;
  if (rows > 0) {
    if (dtype == LOGRA_DTYPE_BF16)
      kl_rows_kernel<__nv_bfloat16><<<(unsigned)rows, kKlThreads, 0, st>>>(
          static_cast<const __nv_bfloat16*>(cur), static_cast<const __nv_bfloat16*>(prop), V, ld, inv_tau, row64,
          row_kl);
    else
      kl_rows_kernel<float><<<(unsigned)rows, kKlThreads, 0, st>>>(static_cast<const float*>(cur),
                                                                 static_cast<const float*>(prop), V, ld, inv_tau,
                                                                 row64, row_kl);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch kl_rows_kernel");
  }
  kl_mean_kernel<<<1, kMeanThreads, 0, st>>>(row64, mask, rows, q_dev);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch kl_mean_kernel");
  return LOGRA_OK;
}

logra_status launch_step_size_device(const double* q_dev, double delta, double alpha_max, double eta,
                                     float* alpha_eta_dev, double* alpha_dev, cudaStream_t st) {
  step_size_kernel<<<1, 1, 0, st>>>(q_dev, delta, alpha_max, eta, alpha_eta_dev, alpha_dev);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch step_size_kernel");
  return LOGRA_OK;
}

}  // namespace logra

// ---------------------------------------------------------------------------
// logra_predicted_kl_noalloc: the same two kernels as logra_predicted_kl, with
// the per-row scratch in a fixed device array of this file instead of a
// caller-provided workspace, so the call allocates nothing.
// ---------------------------------------------------------------------------
namespace logra {
namespace {

constexpr int64_t kNoAllocMaxRows = LOGRA_KL_NOALLOC_MAX_ROWS;
constexpr int kNoAllocMaxDevices = 64;

// One fp64 per row: 512 KiB, held on every GPU that loads the library until
// the process exits.  Shared by every call of logra_predicted_kl_noalloc.
static __device__ __align__(256) double g_noalloc_row_kl[kNoAllocMaxRows];

// Device address of g_noalloc_row_kl for the current device.  The array's
// name in host code is only a host-side handle, so the address is looked up
// once per device with that device current, and the result is checked.
logra_status noalloc_scratch(double** out) {
  static std::mutex mu;
  static double* addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(LOGRA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_row_kl);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(allocation-free KL scratch)");
    addr[dev] = static_cast<double*>(p);
  }
  *out = addr[dev];
  return LOGRA_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace logra

extern "C" logra_status logra_predicted_kl_noalloc(const void* cur, const void* prop, int dtype, int64_t rows,
                                                   int64_t V, int64_t ld, float temperature,
                                                   const uint8_t* row_mask, double* q_dev, float* row_kl_dev,
                                                   logra_stream_t stream) {
  using namespace logra;
  if (dtype != LOGRA_DTYPE_BF16 && dtype != LOGRA_DTYPE_FP32)
    return fail(LOGRA_ERR_UNSUPPORTED, "unknown dtype " + std::to_string(dtype));
  if (rows < 0 || V < 1)
    return fail(LOGRA_ERR_SHAPE, "need rows >= 0 and V >= 1 (rows=" + std::to_string(rows) +
                                     " V=" + std::to_string(V) + ")");
  if (rows > kNoAllocMaxRows)
    return fail(LOGRA_ERR_UNSUPPORTED, "rows (" + std::to_string(rows) + ") exceeds the " +
                                           std::to_string(kNoAllocMaxRows) +
                                           " rows the allocation-free KL holds; use logra_predicted_kl "
                                           "with a workspace");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(LOGRA_ERR_INVALID_ARG, "temperature must be finite and > 0");
  if (!q_dev) return fail(LOGRA_ERR_INVALID_ARG, "q_dev must be non-null");
  if (rows > 0 && (!cur || !prop)) return fail(LOGRA_ERR_INVALID_ARG, "cur and prop must be non-null");
  if (rows > 0 && ld < V) return fail(LOGRA_ERR_SHAPE, "ld < V");
  const int64_t ld_mult = dtype == LOGRA_DTYPE_BF16 ? 8 : 4;
  if (rows > 0 && (!aligned_to(cur, 16) || !aligned_to(prop, 16) || ld % ld_mult))
    return fail(LOGRA_ERR_ALIGNMENT, "cur and prop must be 16-byte aligned, ld a multiple of 16 bytes");
  if (!aligned_to(q_dev, 8) || (row_kl_dev && !aligned_to(row_kl_dev, 4)))
    return fail(LOGRA_ERR_ALIGNMENT, "q_dev must be 8-byte and row_kl_dev 4-byte aligned");
  logra_status s = require_sm103(nullptr);
  if (s != LOGRA_OK) return s;
  double* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != LOGRA_OK) return s;
  s = launch_kl(cur, prop, dtype, rows, V, ld, temperature, row_mask, q_dev, row_kl_dev, scratch,
                reinterpret_cast<cudaStream_t>(stream));
  if (s == LOGRA_OK) ok();
  return s;
}
