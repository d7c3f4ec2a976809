// Device-side building blocks shared by the sm_103a kernels of the LoGRA
// sketching library: the counter-based sign generator, mbarrier waits with a
// time limit, TMA copies and the tcgen05 (5th-generation tensor core) wrappers.
//
// Everything here is written for sm_103a only; there is no fallback path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/logra.h"

namespace logra {

// ----------------------------------------------------------------------------
// Error words written by kernels (first error wins).  The host passes the
// address of one device word to every launch and reads it back on request.
// ----------------------------------------------------------------------------
enum DeviceError : unsigned int {
  kDevOk = 0,
  kDevTimeoutTmaFull = 1,     // a TMA stage never arrived
  kDevTimeoutStageFree = 2,   // a pipeline stage was never released by the MMA
  kDevTimeoutOperand = 3,     // a generated operand tile never became ready
  kDevTimeoutAccum = 4,       // the accumulator never completed
  kDevTimeoutAccumFree = 5,   // the epilogue never released an accumulator
  kDevTimeoutTeardown = 6,    // outstanding copies did not drain at exit
  kDevTimeoutSelfTest = 7,    // the self-test wait (nothing ever arrives) ran out, as it should
};

// Wall-clock limit for any single wait inside a kernel (nanoseconds).  A
// healthy wait lasts microseconds; one second means the pipeline is broken.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(unsigned int* err, unsigned int code) {
  if (err) atomicCAS(err, 0u, code);
}

// ----------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11, section 3.2): ten rounds of two 32×32→64 multiplies with
// a Weyl-sequence key schedule.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 key) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round) {
      key.x += 0x9E3779B9u;
      key.y += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(c.x, 0xD2511F53u), lo0 = c.x * 0xD2511F53u;
    const uint32_t hi1 = __umulhi(c.z, 0xCD9E8D57u), lo1 = c.z * 0xCD9E8D57u;
    c = make_uint4(hi1 ^ c.y ^ key.x, lo1, hi0 ^ c.w ^ key.y, lo0);
  }
  return c;
}

// The 128 sign bits of row `row` of the projection A, columns
// [128·group, 128·group + 128): bit (j & 31) of word (j & 127) >> 5 belongs to
// column j, and a set bit means −1.  Counter (group, row, stream, 0), key =
// the two halves of the 64-bit seed.
__device__ __forceinline__ uint4 sign_words(uint64_t seed, uint32_t stream_id, uint32_t row, uint32_t group) {
  return philox4x32_10(make_uint4(group, row, stream_id, 0u),
                       make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

// Normals for row `row`, columns [4·quad, 4·quad + 4) of the Gaussian
// projection: the four words of Philox4x32-10 at counter
// (quad, row, stream, 1) — the fourth counter word keeps these calls apart
// from the sign calls — turned into four normals by the Box–Muller transform
// (Box and Muller, Ann. Math. Stat. 29, 1958): with u = (a + ½)·2⁻³² and
// φ = (b + ½)·2⁻³² from a pair of words (a, b), the outputs are
// √(−2 ln u)·cos 2πφ and √(−2 ln u)·sin 2πφ.  For u ≥ ½, ln u is taken as
// log1p(−(1 − u)) with 1 − u = (~a + ½)·2⁻³² formed from the integer, so the
// radius keeps its relative accuracy for u close to 1.  The angle needs more
// than the 24 bits an fp32 conversion of b keeps (near a zero of the cosine an
// error of 2⁻²⁴ rad in the angle is a large relative error in z): with b read
// as a signed integer the angle is π·x, x = (b + ½)·2⁻³¹ ∈ (−1, 1) (the same
// point on the circle), split exactly as x = x_hi + x_lo with x_hi from the
// top 24 bits; sincospi gives the point at π·x_hi and the rotation by the
// small angle π·x_lo (< 2⁻²² rad) is applied to first order, whose neglected
// second-order term is below 2⁻⁴⁵.
__device__ __forceinline__ float2 box_muller(uint32_t a, uint32_t b) {
  const float ln_u = a >= 0x80000000u ? log1pf(-((float)(~a) + 0.5f) * 0x1.0p-32f)
                                      : logf(((float)a + 0.5f) * 0x1.0p-32f);
  const float rho = sqrtf(-2.0f * ln_u);
  const int32_t bs = (int32_t)b;
  const float x_hi = (float)(bs & ~0xFF) * 0x1.0p-31f;             // exact: 24 significant bits
  const float t_lo = ((float)(bs & 0xFF) + 0.5f) * 0x1.0p-31f * 3.14159265358979f;  // π·x_lo
  float sn, cs;
  sincospif(x_hi, &sn, &cs);
  const float s2 = fmaf(cs, t_lo, sn), c2 = fmaf(-sn, t_lo, cs);
  return make_float2(rho * c2, rho * s2);
}

__device__ __forceinline__ float4 gauss_quad(uint64_t seed, uint32_t stream_id, uint32_t row, uint32_t quad) {
  const uint4 w = philox4x32_10(make_uint4(quad, row, stream_id, 1u),
                                make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  const float2 z01 = box_muller(w.x, w.y), z23 = box_muller(w.z, w.w);
  return make_float4(z01.x, z01.y, z23.x, z23.y);
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// Two sign bits → two bf16 values ±1 packed little-endian (bit 0 → low half).
// With x ∈ {0..3}, x·0x40008000 = (x << 15) + (x << 30) places bit 0 of x at
// bit 15 and bit 1 at bit 31 (the two shifted copies do not overlap), which
// are exactly the sign bits of the two halves of 0x3F803F80 (1.0, 1.0).
__device__ __forceinline__ uint32_t pm1_pair(uint32_t bits) {
  return (((bits & 3u) * 0x40008000u) & 0x80008000u) | 0x3F803F80u;
}

// Two floats → a bf16 pair, each rounded to nearest even, x0 in the low half
// (one packed conversion).
__device__ __forceinline__ uint32_t bf16x2_rn(float x0, float x1) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
  return r;
}

// A float pair split into bf16 hi + lo pairs: hi = bf16_rn(x), lo =
// bf16_rn(x − hi) per element (x − hi is exact in fp32).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = bf16x2_rn(x0, x1);
  lo = bf16x2_rn(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

// Eight sign bits (bit i → element i) → eight bf16 ±1 values (16 bytes).
__device__ __forceinline__ uint4 pm1_octet(uint32_t byte) {
  return make_uint4(pm1_pair(byte), pm1_pair(byte >> 2), pm1_pair(byte >> 4), pm1_pair(byte >> 6));
}

// ----------------------------------------------------------------------------
// Shared memory, mbarriers and proxies
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, letting the hardware suspend the thread for up to `ns`
// nanoseconds while the phase is incomplete (it resumes as soon as the phase
// completes); a waiting warp then issues no instructions instead of polling.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Position in a ring of pipeline stages: the stage index and the parity of
// its current phase, advanced without a division by the (run-time) stage
// count.
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
  // k ≤ n stages at once
  __device__ __forceinline__ void advance_by(int k, int n) {
    s += k;
    if (s >= n) {
      s -= n;
      ph ^= 1u;
    }
  }
};

// mbar_wait with suspended polling (20 µs per test at most): for kernels
// whose waiting warps share the schedulers with warps that have work.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* err,
                                                unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, code);
      *abort = 1;
      return false;
    }
  }
}

// Waits until the barrier phase with the given parity has completed.  Gives
// up after kWaitLimitNs, or as soon as another thread of the CTA has given up
// (*abort != 0); on its own timeout it records `code` in *err and raises
// *abort.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* err,
                                          unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, code);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns, to every participating thread, whether
// any of them passed pred = true (so a group can leave a loop together).
__device__ __forceinline__ bool named_barrier_any(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// ----------------------------------------------------------------------------
// Group plans: a launch over the tiles of many matrices finds the matrix of
// its CTA from the first CTA of every matrix, cta_begin[0..n] (ascending).
// ----------------------------------------------------------------------------
// The position m of this CTA: the matrix with cta_begin[m] ≤ blockIdx.x <
// cta_begin[m + 1] (matrices without CTAs, whose two bounds are equal, are
// never chosen).  Every thread of the CTA takes part.  Up to blockDim.x
// matrices it counts, with one barrier, the matrices whose last CTA lies
// before blockIdx.x (one coalesced load per thread); beyond, each thread
// runs a binary search over the ascending array (log₂ n loads).
__device__ __forceinline__ int plan_find(const int32_t* __restrict__ cta_begin, int n) {
  const int bid = (int)blockIdx.x;
  if (n <= (int)blockDim.x) {
    const int j = (int)threadIdx.x;
    return __syncthreads_count(j < n && __ldg(cta_begin + j + 1) <= bid);
  }
  int lo = 0, hi = n;  // cta_begin[lo] ≤ bid < cta_begin[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cta_begin + mid) <= bid)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// Copies a plan record from global to shared memory, one 32-bit word per
// thread (the caller synchronises before reading it).
template <class T>
__device__ __forceinline__ void copy_record_to_shared(T* dst, const T* src) {
  static_assert(sizeof(T) % 4 == 0, "record of whole words");
  for (int i = (int)threadIdx.x; i < (int)(sizeof(T) / 4); i += (int)blockDim.x)
    reinterpret_cast<uint32_t*>(dst)[i] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor).  Coordinates are in elements, innermost first.
// ----------------------------------------------------------------------------
// A tensor map in global memory is read by the tensor-map proxy; this orders
// the earlier generic-proxy writes of its 128 bytes before that use.  The
// maps of a group plan are written by a copy from the host, so the fence has
// system scope (a device buffer that held an earlier plan must not serve the
// earlier descriptors).
__device__ __forceinline__ void tmap_acquire(const CUtensorMap* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.sys [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Waits until at most one committed bulk store group is still reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- CTA pairs (cta_group::2): two CTAs of a cluster share each MMA.  The
// tensor memory of both is allocated collectively (one warp of each CTA
// issues the same allocation and both receive the same address); an MMA
// issued by the even CTA of the pair computes M = 256 rows, rows 0..127 from
// the A operand and into the accumulator of the even CTA, rows 128..255 from
// and into the odd one, with the B operand split by N across the two CTAs'
// shared memory at the same offset (the even CTA holds columns 0..N/2).
// (Checked on GB300 with a probe MMA against a host reference.)
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by a shared::cluster address (this CTA's or the
// peer's), with the default release at CTA scope: what the arrival publishes
// here is the completion of the caller's tensor-memory stores (waited for
// before the arrival), which needs no cluster-wide memory fence; a
// cluster-scope release measured as a fence stall on every arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Warp-collective pair MMA (issued by the even CTA): D[256 × N] (+)= A·B with
// A in tensor memory, B from shared memory.
__device__ __forceinline__ void warp_mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Commit of the pair MMAs issued so far: one arrival on the mbarrier at the
// same offset in both CTAs of the pair.
__device__ __forceinline__ void warp_mma_commit_pair(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// tcgen05.mma kind::f16 (bf16 inputs, fp32 accumulation into D in tensor
// memory), A from shared memory (_ss) or from tensor memory (_ts: row m of the
// tile in lane m, K packed two bf16 per 32-bit column, lower K index in the
// low half), and the commit that arrives once on an mbarrier when all MMAs
// issued before it have completed (their shared-memory operands may then be
// overwritten).
//
// All three are warp-collective: every lane of the issuing warp makes the
// call with the same arguments and one lane, chosen by elect.sync, issues.
// The issuing loop then runs in warp-uniform control flow and its
// descriptors stay warp-uniform; measured on GB300 with an unrolled loop, an
// M = 128, N = 64, K = 16 MMA with A in tensor memory issues every 32 cycles
// this way (the tensor core's own rate) against 44 from a loop run by a
// single thread.  elect.sync picks the same lane every time in a converged
// warp, so the commit tracks the MMAs of that lane.
__device__ __forceinline__ void warp_mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void warp_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void warp_mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 lanes × 16 consecutive 32-bit columns; thread i of the warp gets lane
// (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes × 16 consecutive 32-bit columns written; thread i of the warp
// writes lane (base lane + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// 32 lanes × 8 consecutive 32-bit columns written.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 lanes × 8 consecutive 32-bit columns written by one warp, in the
// register layout of the 16×16 (16-bit) fragments of ldmatrix: thread t puts
// v[0] at (lane t/4, column t%4), v[1] at (lane t/4 + 8, column t%4), v[2] at
// (lane t/4, column 4 + t%4) and v[3] at (lane t/4 + 8, column 4 + t%4),
// relative to the lane and column of taddr.  (This mapping was checked on
// GB300 by writing tagged values and reading them back with the 32x32b shape.)
__device__ __forceinline__ void tmem_st_16x128b_x2(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                                   uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x2.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}

// Two tcgen05.st.16x128b.x2 column blocks (8 columns each, a then b) in one
// instruction: 16 lanes × 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_16x128b_x4(uint32_t taddr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                   uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(b2), "r"(b3)
               : "memory");
}

// 16 lanes × 8 consecutive 32-bit columns, the register layout of a 16×8
// fp32 MMA accumulator fragment: thread t holds v[0], v[1] at (lane t/4,
// columns 2(t%4), 2(t%4) + 1) and v[2], v[3] at (lane t/4 + 8, the same
// columns), relative to taddr (checked on GB300 like the shape above).
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}

// Four 8×8 matrices of 16-bit elements from registers to shared memory,
// transposed: register i of thread t holds elements (t/4, 2(t%4)) and
// (t/4, 2(t%4) + 1) of matrix i, which land in row 2(t%4) (+1), column t/4
// of the 16-byte rows whose addresses lanes 8i .. 8i + 7 give.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Two fp32 values as the packed operand of the f32x2 instructions.
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

// fp16 pair (lo in the low half) of two fp32 bit patterns times (s.x, s.y):
// one packed multiply, one packed round-to-nearest conversion.
__device__ __forceinline__ uint32_t half2_scaled(uint32_t lo, uint32_t hi, uint64_t s) {
  uint64_t v, p;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(lo), "r"(hi));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(v), "l"(s));
  uint32_t h;
  asm("{\n\t.reg .f32 a, b;\n\tmov.b64 {a, b}, %1;\n\tcvt.rn.f16x2.f32 %0, b, a;\n\t}" : "=r"(h) : "l"(p));
  return h;
}

// Bulk copy shared → global (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tmem_st_16x256b(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

// Four 8×8 16-bit matrices from shared memory, transposed: lane t supplies the
// address of row t % 8 of matrix t / 8 (16 contiguous bytes); register i then
// holds, of matrix i, the elements (row 2(t%4), column t/4) in its low half and
// (row 2(t%4) + 1, column t/4) in its high half.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// One-dimensional bulk copy global → shared (both 16-byte aligned, bytes a
// multiple of 16), completing on an mbarrier with its byte count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B, fp32 D,
// M = 128.  a_mn / b_mn select the MN-major (transposed) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16_m128(uint32_t n, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4)              // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | (a_mn << 15)         // A major-ness (0 = K-major)
         | (b_mn << 16)         // B major-ness
         | ((n >> 3) << 17)     // N / 8
         | ((128u >> 4) << 24); // M / 16
}

// fp16 A and B (kind::f16 takes both operands in one type), M = 256 (a CTA pair).
__host__ __device__ constexpr uint32_t idesc_f16_m256(uint32_t n) {
  return (1u << 4)              // D format: f32
         | (0u << 7)            // A format: f16
         | (0u << 10)           // B format: f16
         | ((n >> 3) << 17) | ((256u >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// base is 1024-byte aligned (the swizzle pattern repeats every 8 rows of 128
// bytes).  lbo / sbo are byte offsets:
//   K-major : sbo = distance between 8-row groups along M/N (1024 when dense);
//             lbo is not used for swizzled K-major operands.
//   MN-major: lbo = distance between 64-element chunks along M/N,
//             sbo = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46)  // descriptor version for tcgen05
         | (2ull << 61);                                           // swizzle mode: 128 B
}

// The same for a K-major operand with the 64-byte swizzle: rows of 64 bytes
// (32 bf16 along K), 8-row groups of 512 bytes (sbo), base 512-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46)     // descriptor version for tcgen05
         | (4ull << 61);  // swizzle mode: 64 B
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile laid
// out as 128-byte rows with the 128-byte swizzle (what TMA SWIZZLE_128B
// writes, and what the descriptors above describe).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

}  // namespace logra
