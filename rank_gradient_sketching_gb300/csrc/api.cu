// The extern "C" entry points of include/logra.h: argument validation, error
// reporting, device checks and tensor-map encoding.  Every entry point
// validates on the host and returns before launching anything when a check
// fails; launches are asynchronous on the caller's stream.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace logra {

namespace {
thread_local std::string t_last_error;
constexpr int kMaxDevices = 64;

__device__ unsigned int g_device_error;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

std::string fmt(const char* f, long long a = 0, long long b = 0, long long c = 0) {
  char buf[512];
  std::snprintf(buf, sizeof(buf), f, a, b, c);
  return std::string(buf);
}
}  // namespace

logra_status fail(logra_status st, const std::string& msg) {
  t_last_error = msg;
  return st;
}

logra_status ok() {
  t_last_error.clear();
  return LOGRA_OK;
}

logra_status cuda_fail(cudaError_t e, const char* what) {
  return fail(LOGRA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

unsigned int* device_error_word() {
  static std::mutex mu;
  static unsigned int* cache[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fail(LOGRA_ERR_UNSUPPORTED, "device ordinal out of range");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaGetSymbolAddress(device error word)");
      return nullptr;
    }
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

logra_status require_sm103(int* sm_count) {
  static std::mutex mu;
  static int known[kMaxDevices] = {};  // 0 unknown, 1 ok, 2 wrong arch
  static int sms[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(LOGRA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    int major = 0, minor = 0, count = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    known[dev] = (major == 10 && minor == 3) ? 1 : 2;
    sms[dev] = count;
    if (known[dev] == 2)
      return fail(LOGRA_ERR_UNSUPPORTED,
                  fmt("device is sm_%lld%lld; this library holds sm_103a code only", major, minor));
  }
  if (known[dev] != 1) return fail(LOGRA_ERR_UNSUPPORTED, "device is not sm_103; this library holds sm_103a code only");
  if (sm_count) *sm_count = sms[dev];
  return LOGRA_OK;
}

static logra_status make_tmap_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
                                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                                 uint32_t swizzle_bytes) {
  // The driver entry point is resolved through the runtime so that the library
  // has no link-time dependency on libcuda.
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static cudaError_t resolve_err = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    resolve_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (resolve_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) {
    if (resolve_err != cudaSuccess) return cuda_fail(resolve_err, "resolving cuTensorMapEncodeTiled");
    return fail(LOGRA_ERR_CUDA, "the driver does not provide cuTensorMapEncodeTiled");
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LOGRA_ERR_CUDA, fmt("cuTensorMapEncodeTiled failed with CUresult %lld", (long long)r));
  return LOGRA_OK;
}

logra_status make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, uint32_t swizzle_bytes) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_bytes, box_inner, box_outer,
                      swizzle_bytes);
}

logra_status make_tmap_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, outer, row_bytes, box_inner, box_outer, 128);
}

}  // namespace logra

using namespace logra;

extern "C" {

const char* logra_last_error(void) { return t_last_error.c_str(); }

const char* logra_status_string(logra_status s) {
  switch (s) {
    case LOGRA_OK: return "LOGRA_OK";
    case LOGRA_ERR_INVALID_ARG: return "LOGRA_ERR_INVALID_ARG";
    case LOGRA_ERR_SHAPE: return "LOGRA_ERR_SHAPE";
    case LOGRA_ERR_ALIGNMENT: return "LOGRA_ERR_ALIGNMENT";
    case LOGRA_ERR_WORKSPACE: return "LOGRA_ERR_WORKSPACE";
    case LOGRA_ERR_UNSUPPORTED: return "LOGRA_ERR_UNSUPPORTED";
    case LOGRA_ERR_CUDA: return "LOGRA_ERR_CUDA";
    case LOGRA_ERR_DEVICE: return "LOGRA_ERR_DEVICE";
  }
  return "LOGRA_ERR_UNKNOWN";
}

int logra_version(void) { return 100; }

static logra_status check_rank(int r) {
  if (r < 1) return fail(LOGRA_ERR_INVALID_ARG, fmt("rank r must be >= 1 (got %lld)", r));
  if (r > 256) return fail(LOGRA_ERR_UNSUPPORTED, fmt("rank r must be <= 256 (got %lld)", r));
  return LOGRA_OK;
}

static const int64_t kMaxExtent = (int64_t(1) << 31) - 1;  // TMA coordinates are signed 32-bit

size_t logra_sketch_workspace_bytes(int64_t T, int64_t d, int64_t k, int r) {
  if (T < 0 || d < 0 || k < 0 || r < 1 || r > 256) return 0;
  return plan_sketch(T, d, k, r).bytes;
}

int logra_sketch_splits(int64_t T, int64_t d, int64_t k, int r) {
  if (T < 0 || d < 0 || k < 0 || r < 1 || r > 256) return 0;
  return plan_sketch(T, d, k, r).splits;
}

// Argument checks of one sketched matrix, workspace aside (T, d or k equal
// to 0 returns LOGRA_OK with *empty = true).
static logra_status check_sketch_target(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T,
                                        int64_t d, int64_t k, int r, float* S, int64_t lds, bool* empty) {
  *empty = false;
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (T < 0 || d < 0 || k < 0) return fail(LOGRA_ERR_SHAPE, fmt("sizes must be >= 0 (T=%lld d=%lld k=%lld)", T, d, k));
  if (T > kMaxExtent || d > kMaxExtent || k > kMaxExtent)
    return fail(LOGRA_ERR_SHAPE, "T, d and k must be below 2^31");
  if (T == 0 || d == 0 || k == 0) {
    *empty = true;
    return LOGRA_OK;
  }
  if (!X || !dY || !S) return fail(LOGRA_ERR_INVALID_ARG, "X, dY and S must be non-null");
  if (ldx < k) return fail(LOGRA_ERR_SHAPE, fmt("ldx (%lld) < k (%lld)", ldx, k));
  if (lddy < d) return fail(LOGRA_ERR_SHAPE, fmt("lddy (%lld) < d (%lld)", lddy, d));
  if (lds < r) return fail(LOGRA_ERR_SHAPE, fmt("lds (%lld) < r (%lld)", lds, r));
  if (!aligned(X, 16) || !aligned(dY, 16) || ldx % 8 || lddy % 8)
    return fail(LOGRA_ERR_ALIGNMENT, "X and dY must be 16-byte aligned with ldx, lddy multiples of 8");
  if (d % 8 || k % 8)
    return fail(LOGRA_ERR_ALIGNMENT, fmt("d (%lld) and k (%lld) must be multiples of 8 (rows of 16 bytes)", d, k));
  if (!aligned(S, 4)) return fail(LOGRA_ERR_ALIGNMENT, "S must be 4-byte aligned");
  return LOGRA_OK;
}

// Argument checks shared by the two sketch entry points; on success *plan
// holds the launch plan (T, d or k equal to 0 returns LOGRA_OK with
// *empty = true).
static logra_status check_sketch(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T, int64_t d,
                                 int64_t k, int r, float* S, int64_t lds, void* workspace, size_t workspace_bytes,
                                 SketchPlan* plan, bool* empty) {
  logra_status s = check_sketch_target(X, ldx, dY, lddy, T, d, k, r, S, lds, empty);
  if (s != LOGRA_OK || *empty) return s;
  if (!workspace) return fail(LOGRA_ERR_INVALID_ARG, "workspace must be non-null");
  if (!aligned(workspace, 256)) return fail(LOGRA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  *plan = plan_sketch(T, d, k, r);
  if (workspace_bytes < plan->bytes)
    return fail(LOGRA_ERR_WORKSPACE, fmt("workspace needs %lld bytes, got %lld", (long long)plan->bytes,
                                         (long long)workspace_bytes));
  return LOGRA_OK;
}

// A given projection operand: bf16 r×k, 16-byte aligned rows (TMA).
static logra_status check_operand(const void* A, int64_t lda, int64_t k) {
  if (!A) return fail(LOGRA_ERR_INVALID_ARG, "the projection operand A must be non-null");
  if (lda < k) return fail(LOGRA_ERR_SHAPE, fmt("lda (%lld) < k (%lld)", lda, k));
  if (!aligned(A, 16) || lda % 8)
    return fail(LOGRA_ERR_ALIGNMENT, "A must be 16-byte aligned with lda a multiple of 8");
  return LOGRA_OK;
}

logra_status logra_sketch_accumulate(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T, int64_t d,
                                     int64_t k, int r, uint64_t seed, uint32_t stream_id, float* S, int64_t lds,
                                     void* workspace, size_t workspace_bytes, logra_stream_t stream) {
  SketchPlan p;
  bool empty;
  logra_status s = check_sketch(X, ldx, dY, lddy, T, d, k, r, S, lds, workspace, workspace_bytes, &p, &empty);
  if (s != LOGRA_OK || empty) return s == LOGRA_OK ? ok() : s;
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_sketch(p, X, ldx, dY, lddy, seed, stream_id, S, lds, workspace, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_sketch_accumulate_proj(const void* X, int64_t ldx, const void* dY, int64_t lddy, int64_t T,
                                          int64_t d, int64_t k, int r, const void* A, int64_t lda, float* S,
                                          int64_t lds, void* workspace, size_t workspace_bytes,
                                          logra_stream_t stream) {
  SketchPlan p;
  bool empty;
  logra_status s = check_sketch(X, ldx, dY, lddy, T, d, k, r, S, lds, workspace, workspace_bytes, &p, &empty);
  if (s != LOGRA_OK || empty) return s == LOGRA_OK ? ok() : s;
  if ((s = check_operand(A, lda, k)) != LOGRA_OK) return s;
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_sketch_explicit(p, X, ldx, dY, lddy, A, lda, S, lds, workspace, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

size_t logra_sketch_shared_x_workspace_bytes(int64_t T, int64_t k, int n, const int64_t* d, int r) {
  if (T < 0 || k < 0 || r < 1 || r > 256 || n < 1 || n > LOGRA_MAX_SHARED_X_TARGETS || !d) return 0;
  for (int j = 0; j < n; ++j)
    if (d[j] < 0) return 0;
  return shared_x_workspace_bytes(T, k, n, d, r);
}

// Shared checks and launch of the two shared-input entry points; A / lda are
// the per-target operands of the _proj form, or nullptr.
static logra_status sketch_shared_x(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                    const logra_sketch_target* tg, int r, const void* const* A, const int64_t* lda,
                                    void* workspace, size_t workspace_bytes, logra_stream_t stream) {
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (n < 1 || n > LOGRA_MAX_SHARED_X_TARGETS)
    return fail(LOGRA_ERR_UNSUPPORTED, fmt("n must be in [1, %lld] (got %lld)", LOGRA_MAX_SHARED_X_TARGETS, n));
  if (!tg) return fail(LOGRA_ERR_INVALID_ARG, "targets must be non-null");
  if ((int64_t)n * round_up(r, 16) > 512)
    return fail(LOGRA_ERR_UNSUPPORTED,
                fmt("n (%lld) times r rounded up to 16 (%lld) exceeds 512", n, round_up(r, 16)));
  if (T < 0 || k < 0) return fail(LOGRA_ERR_SHAPE, fmt("sizes must be >= 0 (T=%lld k=%lld)", T, k));
  if (T > kMaxExtent || k > kMaxExtent) return fail(LOGRA_ERR_SHAPE, "T and k must be below 2^31");
  int64_t dv[LOGRA_MAX_SHARED_X_TARGETS];
  for (int j = 0; j < n; ++j) {
    const logra_sketch_target& t = tg[j];
    if (t.d < 1 || t.d > kMaxExtent) return fail(LOGRA_ERR_SHAPE, fmt("target %lld: d must be in [1, 2^31)", j));
    dv[j] = t.d;
  }
  if (T == 0 || k == 0) return ok();
  if (!X || !workspace) return fail(LOGRA_ERR_INVALID_ARG, "X and workspace must be non-null");
  if (ldx < k) return fail(LOGRA_ERR_SHAPE, fmt("ldx (%lld) < k (%lld)", ldx, k));
  if (!aligned(X, 16) || ldx % 8 || k % 8)
    return fail(LOGRA_ERR_ALIGNMENT, "X must be 16-byte aligned with ldx and k multiples of 8");
  for (int j = 0; j < n; ++j) {
    const logra_sketch_target& t = tg[j];
    if (!t.dY || !t.S) return fail(LOGRA_ERR_INVALID_ARG, fmt("target %lld: dY and S must be non-null", j));
    if (t.lddy < t.d || t.lds < r) return fail(LOGRA_ERR_SHAPE, fmt("target %lld: lddy < d or lds < r", j));
    if (!aligned(t.dY, 16) || t.lddy % 8 || t.d % 8)
      return fail(LOGRA_ERR_ALIGNMENT, fmt("target %lld: dY must be 16-byte aligned, lddy and d multiples of 8", j));
    if (!aligned(t.S, 4)) return fail(LOGRA_ERR_ALIGNMENT, fmt("target %lld: S must be 4-byte aligned", j));
  }
  if (!aligned(workspace, 256)) return fail(LOGRA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const size_t need = shared_x_workspace_bytes(T, k, n, dv, r);
  if (workspace_bytes < need)
    return fail(LOGRA_ERR_WORKSPACE, fmt("workspace needs %lld bytes, got %lld", (long long)need,
                                         (long long)workspace_bytes));
  if (A) {
    if (!lda) return fail(LOGRA_ERR_INVALID_ARG, "lda must be non-null");
    for (int j = 0; j < n; ++j)
      if ((s = check_operand(A[j], lda[j], k)) != LOGRA_OK) return s;
  }
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_sketch_shared_x(X, ldx, T, k, n, tg, r, A, lda, workspace, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_sketch_accumulate_shared_x(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                              const logra_sketch_target* tg, int r, void* workspace,
                                              size_t workspace_bytes, logra_stream_t stream) {
  return sketch_shared_x(X, ldx, T, k, n, tg, r, nullptr, nullptr, workspace, workspace_bytes, stream);
}

logra_status logra_sketch_accumulate_shared_x_proj(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                                   const logra_sketch_target* tg, const void* const* A,
                                                   const int64_t* lda, int r, void* workspace,
                                                   size_t workspace_bytes, logra_stream_t stream) {
  if (!A) return fail(LOGRA_ERR_INVALID_ARG, "A must be non-null");
  return sketch_shared_x(X, ldx, T, k, n, tg, r, A, lda, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------ sketch group
size_t logra_sketch_group_plan_bytes(int n) { return n < 0 ? 0 : sketch_group_plan_bytes(n); }

size_t logra_sketch_group_workspace_bytes(int n, const logra_sketch_group_target* targets, int r) {
  if (n < 0 || r < 1 || r > 256 || (n > 0 && !targets)) return 0;
  for (int j = 0; j < n; ++j)
    if (targets[j].T < 0 || targets[j].d < 0 || targets[j].k < 0) return 0;
  return sketch_group_workspace_bytes(n, targets, r);
}

logra_status logra_sketch_group_plan(int n, const logra_sketch_group_target* targets, int r, void* workspace,
                                     size_t workspace_bytes, void* plan, size_t plan_bytes) {
  if (n < 0 || n > (1 << 20)) return fail(LOGRA_ERR_INVALID_ARG, fmt("n (%lld) must be in [0, 2^20]", n));
  if (n > 0 && !targets) return fail(LOGRA_ERR_INVALID_ARG, "targets must be non-null");
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (!plan) return fail(LOGRA_ERR_INVALID_ARG, "plan must be non-null");
  if (!aligned(plan, 128)) return fail(LOGRA_ERR_ALIGNMENT, "plan must be 128-byte aligned");
  if (plan_bytes < sketch_group_plan_bytes(n))
    return fail(LOGRA_ERR_WORKSPACE, fmt("plan needs %lld bytes, got %lld", (long long)sketch_group_plan_bytes(n),
                                         (long long)plan_bytes));
  bool any = false;
  for (int j = 0; j < n; ++j) {
    const logra_sketch_group_target& t = targets[j];
    bool empty;
    s = check_sketch_target(t.X, t.ldx, t.dY, t.lddy, t.T, t.d, t.k, r, t.S, t.lds, &empty);
    if (s != LOGRA_OK) return fail(s, fmt("target %lld: ", j) + logra_last_error());
    if (!empty && t.A && (s = check_operand(t.A, t.lda, t.k)) != LOGRA_OK)
      return fail(s, fmt("target %lld: ", j) + logra_last_error());
    any = any || !empty;
  }
  const size_t need = sketch_group_workspace_bytes(n, targets, r);
  if (any) {
    if (!workspace) return fail(LOGRA_ERR_INVALID_ARG, "workspace must be non-null");
    if (!aligned(workspace, 256)) return fail(LOGRA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (workspace_bytes < need)
      return fail(LOGRA_ERR_WORKSPACE, fmt("workspace needs %lld bytes, got %lld", (long long)need,
                                           (long long)workspace_bytes));
  }
  // The CTAs of one launch update their matrices' S without any order between
  // matrices, so two targets whose S regions share a byte would race.
  {
    std::vector<std::pair<uintptr_t, uintptr_t>> rg;
    rg.reserve((size_t)n);
    for (int j = 0; j < n; ++j) {
      const logra_sketch_group_target& t = targets[j];
      if (t.T == 0 || t.d == 0 || t.k == 0) continue;
      const uintptr_t b = reinterpret_cast<uintptr_t>(t.S);
      rg.emplace_back(b, b + (uintptr_t)(((t.d - 1) * t.lds + r) * 4));
    }
    std::sort(rg.begin(), rg.end());
    for (size_t j = 1; j < rg.size(); ++j)
      if (rg[j].first < rg[j - 1].second)
        return fail(LOGRA_ERR_INVALID_ARG, "the S regions of two targets overlap (sketch them in separate launches)");
  }
  s = build_sketch_group_plan(n, targets, r, workspace, plan);
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_sketch_accumulate_group(const void* plan, const void* plan_dev, logra_stream_t stream) {
  if (!plan || !plan_dev) return fail(LOGRA_ERR_INVALID_ARG, "plan and plan_dev must be non-null");
  if (!aligned(plan, 128) || !aligned(plan_dev, 128))
    return fail(LOGRA_ERR_ALIGNMENT, "plan and plan_dev must be 128-byte aligned");
  int n;
  logra_status s = check_sketch_group_plan(plan, &n);
  if (s != LOGRA_OK) return s;
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_sketch_group(plan, plan_dev, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

static logra_status check_merge(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                                float alpha_eta, const float* alpha_eta_dev, bool* empty) {
  *empty = false;
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (d < 0 || k < 0) return fail(LOGRA_ERR_SHAPE, fmt("sizes must be >= 0 (d=%lld k=%lld)", d, k));
  if (d > kMaxExtent || k > kMaxExtent) return fail(LOGRA_ERR_SHAPE, "d and k must be below 2^31");
  if (!alpha_eta_dev && !std::isfinite(alpha_eta)) return fail(LOGRA_ERR_INVALID_ARG, "alpha_eta must be finite");
  if (d == 0 || k == 0) {
    *empty = true;
    return LOGRA_OK;
  }
  if (!W || !S) return fail(LOGRA_ERR_INVALID_ARG, "W and S must be non-null");
  if (ldw < k) return fail(LOGRA_ERR_SHAPE, fmt("ldw (%lld) < k (%lld)", ldw, k));
  if (lds < r) return fail(LOGRA_ERR_SHAPE, fmt("lds (%lld) < r (%lld)", lds, r));
  if (!aligned(W, 16) || ldw % 8) return fail(LOGRA_ERR_ALIGNMENT, "W must be 16-byte aligned with ldw a multiple of 8");
  if (k % 8) return fail(LOGRA_ERR_ALIGNMENT, fmt("k (%lld) must be a multiple of 8 (rows of 16 bytes)", k));
  if (!aligned(S, 4)) return fail(LOGRA_ERR_ALIGNMENT, "S must be 4-byte aligned");
  if (alpha_eta_dev && !aligned(alpha_eta_dev, 4)) return fail(LOGRA_ERR_ALIGNMENT, "alpha_eta_dev must be 4-byte aligned");
  return LOGRA_OK;
}

logra_status logra_merge_update(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                                uint64_t seed, uint32_t stream_id, float alpha_eta, const float* alpha_eta_dev,
                                logra_stream_t stream) {
  bool empty;
  logra_status s = check_merge(W, ldw, d, k, S, lds, r, alpha_eta, alpha_eta_dev, &empty);
  if (s != LOGRA_OK || empty) return s == LOGRA_OK ? ok() : s;
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_merge(W, ldw, d, k, S, lds, r, seed, stream_id, alpha_eta, alpha_eta_dev, nullptr, 0,
                   reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_merge_update_proj(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                                     const void* A, int64_t lda, float alpha_eta, const float* alpha_eta_dev,
                                     logra_stream_t stream) {
  bool empty;
  logra_status s = check_merge(W, ldw, d, k, S, lds, r, alpha_eta, alpha_eta_dev, &empty);
  if (s != LOGRA_OK || empty) return s == LOGRA_OK ? ok() : s;
  if ((s = check_operand(A, lda, k)) != LOGRA_OK) return s;
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_merge(W, ldw, d, k, S, lds, r, 0, 0, alpha_eta, alpha_eta_dev, A, lda,
                   reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

size_t logra_merge_group_plan_bytes(int n) { return n < 0 ? 0 : merge_group_plan_bytes(n); }

logra_status logra_merge_group_plan(int n, const logra_merge_target* targets, int r, void* plan,
                                    size_t plan_bytes) {
  if (n < 0 || n > (1 << 20)) return fail(LOGRA_ERR_INVALID_ARG, fmt("n (%lld) must be in [0, 2^20]", n));
  if (n > 0 && !targets) return fail(LOGRA_ERR_INVALID_ARG, "targets must be non-null");
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (!plan) return fail(LOGRA_ERR_INVALID_ARG, "plan must be non-null");
  if (!aligned(plan, 128)) return fail(LOGRA_ERR_ALIGNMENT, "plan must be 128-byte aligned");
  if (plan_bytes < merge_group_plan_bytes(n))
    return fail(LOGRA_ERR_WORKSPACE, fmt("plan needs %lld bytes, got %lld", (long long)merge_group_plan_bytes(n), (long long)plan_bytes));
  const bool has_a = n > 0 && targets[0].A != nullptr;
  for (int j = 0; j < n; ++j) {
    const logra_merge_target& t = targets[j];
    if ((t.A != nullptr) != has_a)
      return fail(LOGRA_ERR_INVALID_ARG, fmt("target %lld: either every target has an operand A or none has", j));
    bool empty;
    s = check_merge(t.W, t.ldw, t.d, t.k, t.S, t.lds, r, 0.f, nullptr, &empty);
    if (s != LOGRA_OK) return fail(s, fmt("target %lld: ", j) + logra_last_error());
    if (!empty && has_a && (s = check_operand(t.A, t.lda, t.k)) != LOGRA_OK)
      return fail(s, fmt("target %lld: ", j) + logra_last_error());
  }
  // The CTAs of one launch read and write their weights' tiles without any
  // order between weights, so two targets whose W regions share a byte would
  // race.  Sort the non-empty regions by start and compare neighbours.
  {
    std::vector<std::pair<uintptr_t, uintptr_t>> rg;
    rg.reserve((size_t)n);
    for (int j = 0; j < n; ++j) {
      const logra_merge_target& t = targets[j];
      if (t.d == 0 || t.k == 0) continue;
      const uintptr_t b = reinterpret_cast<uintptr_t>(t.W);
      rg.emplace_back(b, b + (uintptr_t)(((t.d - 1) * t.ldw + t.k) * 2));
    }
    std::sort(rg.begin(), rg.end());
    for (size_t j = 1; j < rg.size(); ++j)
      if (rg[j].first < rg[j - 1].second)
        return fail(LOGRA_ERR_INVALID_ARG, "the W regions of two targets overlap (merge them in separate launches)");
  }
  s = build_merge_group_plan(n, targets, r, plan, plan_bytes);
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_merge_update_group(const void* plan, const void* plan_dev, float alpha_eta,
                                      const float* alpha_eta_dev, logra_stream_t stream) {
  if (!plan || !plan_dev) return fail(LOGRA_ERR_INVALID_ARG, "plan and plan_dev must be non-null");
  if (!aligned(plan, 128) || !aligned(plan_dev, 128))
    return fail(LOGRA_ERR_ALIGNMENT, "plan and plan_dev must be 128-byte aligned");
  int n, r;
  logra_status s = check_merge_group_plan(plan, &n, &r);
  if (s != LOGRA_OK) return s;
  if (!alpha_eta_dev && !std::isfinite(alpha_eta)) return fail(LOGRA_ERR_INVALID_ARG, "alpha_eta must be finite");
  if (alpha_eta_dev && !aligned(alpha_eta_dev, 4)) return fail(LOGRA_ERR_ALIGNMENT, "alpha_eta_dev must be 4-byte aligned");
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_merge_group(plan, plan_dev, alpha_eta, alpha_eta_dev, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_sketch_momentum(float* M, int64_t ldm, float* S, int64_t lds, int64_t d, int r, float beta,
                                   int clear_s, logra_stream_t stream) {
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (d < 0) return fail(LOGRA_ERR_SHAPE, fmt("d must be >= 0 (got %lld)", d));
  if (!std::isfinite(beta)) return fail(LOGRA_ERR_INVALID_ARG, "beta must be finite");
  if (d == 0) return ok();
  if (!M || !S) return fail(LOGRA_ERR_INVALID_ARG, "M and S must be non-null");
  if (M == S) return fail(LOGRA_ERR_INVALID_ARG, "M and S must not overlap");
  if (ldm < r) return fail(LOGRA_ERR_SHAPE, fmt("ldm (%lld) < r (%lld)", ldm, r));
  if (lds < r) return fail(LOGRA_ERR_SHAPE, fmt("lds (%lld) < r (%lld)", lds, r));
  if (!aligned(M, 4) || !aligned(S, 4)) return fail(LOGRA_ERR_ALIGNMENT, "M and S must be 4-byte aligned");
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_momentum(M, ldm, S, lds, d, r, beta, clear_s, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_regen_projection(uint64_t seed, uint32_t stream_id, int r, int64_t k, int out_kind, void* A_out,
                                    int64_t lda, logra_stream_t stream) {
  logra_status s = check_rank(r);
  if (s != LOGRA_OK) return s;
  if (k < 0) return fail(LOGRA_ERR_SHAPE, "k must be >= 0");
  if (k > kMaxExtent) return fail(LOGRA_ERR_SHAPE, "k must be below 2^31");
  if (out_kind != LOGRA_PROJ_INT8_PM1 && out_kind != LOGRA_PROJ_BF16 && out_kind != LOGRA_PROJ_FP32 &&
      out_kind != LOGRA_PROJ_GAUSS_BF16 && out_kind != LOGRA_PROJ_GAUSS_FP32 && out_kind != LOGRA_PROJ_SIGN_BF16)
    return fail(LOGRA_ERR_UNSUPPORTED, fmt("unknown out_kind %lld", out_kind));
  if (k == 0) return ok();
  if (!A_out) return fail(LOGRA_ERR_INVALID_ARG, "A_out must be non-null");
  if (lda < k) return fail(LOGRA_ERR_SHAPE, fmt("lda (%lld) < k (%lld)", lda, k));
  const uintptr_t esz = out_kind == LOGRA_PROJ_INT8_PM1                                  ? 1
                        : out_kind == LOGRA_PROJ_BF16 || out_kind == LOGRA_PROJ_GAUSS_BF16 ||
                                  out_kind == LOGRA_PROJ_SIGN_BF16
                              ? 2
                                                                                           : 4;
  if (!aligned(A_out, esz)) return fail(LOGRA_ERR_ALIGNMENT, "A_out is not aligned to its element size");
  if ((s = require_sm103(nullptr)) != LOGRA_OK) return s;
  s = launch_regen(seed, stream_id, r, k, out_kind, A_out, lda, reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

size_t logra_kl_workspace_bytes(int64_t rows) {
  if (rows < 0) return 0;
  return align256((size_t)(rows > 0 ? rows : 1) * sizeof(double));
}

logra_status logra_predicted_kl(const void* cur, const void* prop, int dtype, int64_t rows, int64_t V, int64_t ld,
                                float temperature, const uint8_t* row_mask, double* q_dev, float* row_kl_dev,
                                void* workspace, size_t workspace_bytes, logra_stream_t stream) {
  if (dtype != LOGRA_DTYPE_BF16 && dtype != LOGRA_DTYPE_FP32)
    return fail(LOGRA_ERR_UNSUPPORTED, fmt("unknown dtype %lld", dtype));
  if (rows < 0 || V < 1) return fail(LOGRA_ERR_SHAPE, fmt("need rows >= 0 and V >= 1 (rows=%lld V=%lld)", rows, V));
  if (rows > kMaxExtent) return fail(LOGRA_ERR_SHAPE, "rows must be below 2^31");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(LOGRA_ERR_INVALID_ARG, "temperature must be finite and > 0");
  if (!q_dev || !workspace) return fail(LOGRA_ERR_INVALID_ARG, "q_dev and workspace must be non-null");
  if (rows > 0 && (!cur || !prop)) return fail(LOGRA_ERR_INVALID_ARG, "cur and prop must be non-null");
  if (rows > 0 && ld < V) return fail(LOGRA_ERR_SHAPE, fmt("ld (%lld) < V (%lld)", ld, V));
  const int64_t ld_mult = dtype == LOGRA_DTYPE_BF16 ? 8 : 4;
  if (rows > 0 && (!aligned(cur, 16) || !aligned(prop, 16) || ld % ld_mult))
    return fail(LOGRA_ERR_ALIGNMENT, "cur and prop must be 16-byte aligned, ld a multiple of 16 bytes");
  if (!aligned(q_dev, 8) || (row_kl_dev && !aligned(row_kl_dev, 4)))
    return fail(LOGRA_ERR_ALIGNMENT, "q_dev must be 8-byte and row_kl_dev 4-byte aligned");
  if (!aligned(workspace, 256)) return fail(LOGRA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (workspace_bytes < logra_kl_workspace_bytes(rows))
    return fail(LOGRA_ERR_WORKSPACE, fmt("workspace needs %lld bytes, got %lld",
                                         (long long)logra_kl_workspace_bytes(rows), (long long)workspace_bytes));
  logra_status s = require_sm103(nullptr);
  if (s != LOGRA_OK) return s;
  s = launch_kl(cur, prop, dtype, rows, V, ld, temperature, row_mask, q_dev, row_kl_dev, workspace,
                reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

size_t logra_sum_squares_workspace_bytes(void) { return (size_t)kNormBlocks * sizeof(double); }

logra_status logra_sum_squares(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld, double* out_dev,
                               int accumulate, void* workspace, size_t workspace_bytes, logra_stream_t stream) {
  if (dtype != LOGRA_DTYPE_BF16 && dtype != LOGRA_DTYPE_FP32)
    return fail(LOGRA_ERR_UNSUPPORTED, fmt("unknown dtype %lld", dtype));
  if (rows < 0 || cols < 0) return fail(LOGRA_ERR_SHAPE, fmt("sizes must be >= 0 (rows=%lld cols=%lld)", rows, cols));
  if (!out_dev) return fail(LOGRA_ERR_INVALID_ARG, "out_dev must be non-null");
  if (!aligned(out_dev, 8)) return fail(LOGRA_ERR_ALIGNMENT, "out_dev must be 8-byte aligned");
  const int64_t n_rows = rows > 0 && cols > 0 ? rows : 0;
  if (n_rows > 0) {
    if (!x) return fail(LOGRA_ERR_INVALID_ARG, "x must be non-null");
    if (ld < cols) return fail(LOGRA_ERR_SHAPE, fmt("ld (%lld) < cols (%lld)", ld, cols));
    if (!aligned(x, dtype == LOGRA_DTYPE_BF16 ? 2 : 4)) return fail(LOGRA_ERR_ALIGNMENT, "x is not aligned to its element size");
  }
  if (!workspace || !aligned(workspace, 8)) return fail(LOGRA_ERR_WORKSPACE, "workspace must be non-null and 8-byte aligned");
  if (workspace_bytes < logra_sum_squares_workspace_bytes())
    return fail(LOGRA_ERR_WORKSPACE, fmt("workspace needs %lld bytes, got %lld",
                                         (long long)logra_sum_squares_workspace_bytes(), (long long)workspace_bytes));
  logra_status s = require_sm103(nullptr);
  if (s != LOGRA_OK) return s;
  s = launch_sum_squares(x, dtype, n_rows, cols, ld, out_dev, accumulate, workspace,
                         reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

// Host Philox4x32-10 (Salmon et al., SC'11, section 3.2), for the per-step
// seeds; the kernels carry their own device copy of the same function.
static void philox_host(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int round = 0; round < 10; ++round) {
    if (round) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)c[0] * 0xD2511F53u, p1 = (uint64_t)c[2] * 0xCD9E8D57u;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0, n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = (uint32_t)p1;
    c[2] = n2;
    c[3] = (uint32_t)p0;
  }
}

uint64_t logra_refreshed_seed(uint64_t base_seed, uint64_t step) {
  uint32_t c[4] = {(uint32_t)step, (uint32_t)(step >> 32), 0u, 2u};
  philox_host(c, (uint32_t)base_seed, (uint32_t)(base_seed >> 32));
  return (uint64_t)c[0] | ((uint64_t)c[1] << 32);
}

logra_status logra_step_size(double q, double delta, double alpha_max, double* alpha_out) {
  if (!alpha_out) return fail(LOGRA_ERR_INVALID_ARG, "alpha_out must be non-null");
  if (!(delta > 0) || !std::isfinite(delta)) return fail(LOGRA_ERR_INVALID_ARG, "delta must be finite and > 0");
  if (!(alpha_max > 0) || !std::isfinite(alpha_max))
    return fail(LOGRA_ERR_INVALID_ARG, "alpha_max must be finite and > 0");
  if (std::isnan(q)) *alpha_out = q;
  else if (q <= 0) *alpha_out = alpha_max;
  else *alpha_out = std::fmin(alpha_max, std::sqrt(delta / q));
  return ok();
}

logra_status logra_step_size_device(const double* q_dev, double delta, double alpha_max, double eta,
                                    float* alpha_eta_dev, double* alpha_dev, logra_stream_t stream) {
  if (!q_dev || !alpha_eta_dev) return fail(LOGRA_ERR_INVALID_ARG, "q_dev and alpha_eta_dev must be non-null");
  if (!(delta > 0) || !std::isfinite(delta)) return fail(LOGRA_ERR_INVALID_ARG, "delta must be finite and > 0");
  if (!(alpha_max > 0) || !std::isfinite(alpha_max))
    return fail(LOGRA_ERR_INVALID_ARG, "alpha_max must be finite and > 0");
  if (!std::isfinite(eta)) return fail(LOGRA_ERR_INVALID_ARG, "eta must be finite");
  if (!aligned(q_dev, 8) || !aligned(alpha_eta_dev, 4) || (alpha_dev && !aligned(alpha_dev, 8)))
    return fail(LOGRA_ERR_ALIGNMENT, "q_dev / alpha_dev must be 8-byte and alpha_eta_dev 4-byte aligned");
  logra_status s = require_sm103(nullptr);
  if (s != LOGRA_OK) return s;
  s = launch_step_size_device(q_dev, delta, alpha_max, eta, alpha_eta_dev, alpha_dev,
                              reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_self_test_wait_timeout(logra_stream_t stream) {
  logra_status s = require_sm103(nullptr);
  if (s != LOGRA_OK) return s;
  s = launch_self_test_wait_timeout(reinterpret_cast<cudaStream_t>(stream));
  return s == LOGRA_OK ? ok() : s;
}

logra_status logra_device_error(logra_stream_t stream, unsigned int* code) {
  if (!code) return fail(LOGRA_ERR_INVALID_ARG, "code must be non-null");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(device error word)");
  *code = v;
  if (v) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(device error word)");
    return fail(LOGRA_ERR_DEVICE, fmt("a kernel recorded device error code %lld", v));
  }
  return ok();
}

}  // extern "C"
