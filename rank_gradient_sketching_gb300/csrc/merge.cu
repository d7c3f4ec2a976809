// Merge W ← bf16(W − αη·S·A) into bf16 weights, in place.
//
// LoGRA summary page, section "草图如何取代完整梯度缓冲": the update
// W ← W − αηUA (U = S in the plain SGD variant) is merged straight into the
// weights, with no resident adapter branch; section "同一份草图也压缩策略同步开
// 销": the receiving side regenerates A from the seed and applies αηU.
//
// The kernel streams W once (read + write) and rebuilds A on chip:
// U(128×64) = S(128×r)·A±1(r×64) per 64-column chunk on tcgen05, with S split
// as bf16 hi + lo (fp32-like accuracy, two MMAs per step) and held in tensor
// memory as the A operand, the ±1 tile built in shared memory in the MN-major
// layout (8 consecutive columns of one rank = one byte of generator output =
// one 16-byte chunk), W tiles moved in and out by TMA.  Ranks below 16 are
// padded to 16 with zero rows of S and of the ±1 tile.  The merge is bound by
// HBM at every rank; even at r ≤ 8, where the MMAs do next to nothing, this
// pipeline (a deep TMA ring of W tiles, warp-specialised roles) measured well
// ahead of a CUDA-core kernel with 16-byte loads (7B set at r = 4: 91.6 %
// against 65.5 % of HBM).
// With a given projection operand Ã (the Gaussian basis, or cached signs) the
// ±1 tiles are replaced by tiles of Ã copied by TMA.
// W' = bf16_rn(float(W) − c·U) with c = αη/√r in fp32.

#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

// ------------------------------------------------------------ merge plan
// A plan merges a set of weights in one launch (logra_merge_update_group):
// a header, the first CTA of every weight (cta_begin[0..n]), then one entry
// per weight with its tensor maps and descriptors.  A CTA finds its weight by
// counting the weights whose CTAs all come before it.
constexpr uint32_t kPlanMagic = 0x4C474D50u;  // "LGMP"
constexpr size_t kPlanHeaderBytes = 128;

struct MergePlanHeader {
  uint32_t magic;
  int32_t n, r, np;
  int32_t path;  // 1: two CTAs per SM (np ≤ 128); 2: one CTA per SM
  int32_t total_ctas;
  int32_t w_stages, b_stages;
  uint32_t tmem_cols, smem_bytes;
  int32_t s_tma, explicit_a;
};
static_assert(sizeof(MergePlanHeader) <= kPlanHeaderBytes, "plan header");

struct alignas(128) MergeEntry {
  CUtensorMap tw;  // W (tensor-core path)
  CUtensorMap ta;  // the given projection operand (explicit_a)
  CUtensorMap ts;  // S staging (s_tma)
  __nv_bfloat16* W;
  int64_t ldw, d, k;
  const float* S;
  int64_t lds;
  const __nv_bfloat16* A;
  int64_t lda;
  uint64_t seed;
  uint32_t stream_id;
  int32_t s_vec4;
  int32_t num_chunks;      // 64-column chunks
  int32_t chunks_per_cta;  // chunks of one CTA
  int32_t groups;          // CTAs across the columns of one 128-row tile
  int32_t ctas;
};
static_assert(sizeof(MergeEntry) == 512, "plan entry");

__host__ __device__ inline size_t plan_begin_bytes(int n) { return ((size_t)(n + 1) * 4 + 127) / 128 * 128; }
__host__ __device__ inline size_t plan_entries_offset(int n) { return kPlanHeaderBytes + plan_begin_bytes(n); }

// The weight of a CTA: plan_find over cta_begin.

// ---------------------------------------------------------- tensor-core path
// warp 0: TMA loads of W tiles; warp 1: TMEM allocation and the MMAs (whole
// warp); EPI epilogue threads: S into tensor memory first (warps 2-5, or all
// epilogue warps when S is staged by TMA), then the accumulators into W' (a
// warp reaches one quarter of the tensor-memory lanes); then the threads
// that build the ±1 tiles (tc_gen: two rank rows each up to np = 128, one
// row each above).  EPI = 128 keeps two CTAs
// per SM up to np = 128.  Above, one CTA per SM runs eight epilogue warps
// in two groups of four that take alternate chunks, so that two per-chunk
// epilogue chains (W from shared memory, tensor-memory loads, the update,
// the store into the output tile, two barriers) overlap, as the chains of
// two CTAs per SM do below.  There a second issuing warp follows the ±1
// warps: the two issuers take alternate chunks (each its own ±1 stage and
// accumulator, so their MMAs are independent), and one warp's batch of MMAs
// keeps the tensor pipe busy through the other's gap between batches (a
// single issuer left the pipe idle for ~25 % of each chunk at np = 256).
// With two issuers the ±1 builders set the pace of a chunk; eight builder
// warps instead of four (608 threads, 96 registers a thread) made the
// np = 256 merge 4 % faster.
constexpr int kGen = 128;
constexpr int kTcMaxWStages = 8;  // W tiles in flight
constexpr int kTcMaxBStages = 3;  // ±1 tiles
constexpr uint32_t kSmemBudget = 230400;    // one CTA per SM
constexpr uint32_t kSmemTwoPerSm = 113664;  // two CTAs per SM
constexpr uint32_t kWTileBytes = 128 * 128;  // 128 rows × 64 bf16

// Threads of the tensor-core kernel and the warp of its second MMA issuer
// (none below np = 128).
constexpr int tc_gen(int epi) { return epi == 256 ? 256 : kGen; }
constexpr int tc_threads(int epi) { return 64 + epi + tc_gen(epi) + (epi == 256 ? 32 : 0); }
constexpr int tc_issuer2(int epi) { return epi == 256 ? (64 + epi + tc_gen(epi)) / 32 : -1; }

struct MergeTcArgs {
  int64_t d, k;
  int r, np;
  int chunks_per_cta, num_chunks;
  int w_stages, b_stages;
  uint32_t tmem_cols;
  float c;
  const float* alpha_eta_dev;
  float inv_sqrt_r;
  const float* S;
  int64_t lds;
  int s_vec4;  // rows of S can be read with 16-byte loads
  __nv_bfloat16* W;
  int64_t ldw;
  uint64_t seed;
  uint32_t stream_id;
  int explicit_a;  // 1: the ±1 tiles are replaced by tiles of a given projection, loaded by TMA
  int s_tma;       // 1: the S tile is staged in the W ring by TMA before the W stream starts
  unsigned int* err;
};

// One 64-column chunk: U = S_hi·A±1 + S_lo·A±1 over NK steps of 16 ranks,
// both halves of S read from tensor memory (16 ranks = 8 columns).  NK is a
// template parameter so the issuing loop is fully unrolled.
template <int NK>
__device__ __forceinline__ void merge_mma_chunk_t(uint32_t d_tmem, uint32_t t_shi, uint32_t t_slo, uint64_t bo,
                                                  uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < NK; ++ks) {
    const uint64_t bd = bo + (uint64_t)(ks * 128);  // 16 ranks = 2048 bytes further
    warp_mma_bf16_ts(d_tmem, t_shi + (uint32_t)(ks * 8), bd, idesc, ks != 0);
    warp_mma_bf16_ts(d_tmem, t_slo + (uint32_t)(ks * 8), bd, idesc, 1);
  }
}

__device__ __forceinline__ void merge_mma_chunk(int nk, uint32_t d_tmem, uint32_t t_shi, uint32_t t_slo, uint64_t bo,
                                                uint32_t idesc) {
  switch (nk) {
#define LOGRA_MERGE_NK(K) \
  case K:                 \
    merge_mma_chunk_t<K>(d_tmem, t_shi, t_slo, bo, idesc); \
    break;
    LOGRA_MERGE_NK(1)
    LOGRA_MERGE_NK(2)
    LOGRA_MERGE_NK(3)
    LOGRA_MERGE_NK(4)
    LOGRA_MERGE_NK(5)
    LOGRA_MERGE_NK(6)
    LOGRA_MERGE_NK(7)
    LOGRA_MERGE_NK(8)
    LOGRA_MERGE_NK(9)
    LOGRA_MERGE_NK(10)
    LOGRA_MERGE_NK(11)
    LOGRA_MERGE_NK(12)
    LOGRA_MERGE_NK(13)
    LOGRA_MERGE_NK(14)
    LOGRA_MERGE_NK(15)
    LOGRA_MERGE_NK(16)
#undef LOGRA_MERGE_NK
    default:
      break;
  }
}

// U(128 × 64) = S(128 × r)·A±1(r × 64) per 64-column chunk of a 128-row tile
// of W.  S is split into bf16 hi + lo and kept in tensor memory as the A
// operand of both MMAs (the K = r dimension packed two per column), so the
// MMAs read only the small ±1 tile from shared memory.  W tiles come in by
// TMA (each slot is released as soon as its rows are in registers); the
// updated tile goes out through one of two output tiles by TMA store.
// The S-staging copy exists only in the eight-warp kernel (np > 128): in the
// four-warp kernel its tensor map and branches, although never taken, cost
// about 3 % of merge throughput in a step (measured), so they are compiled
// out there.
template <int EPI>
struct StageMap {
  CUtensorMap s;
};
template <>
struct StageMap<128> {};

// GROUP: the kernel merges the weights of a plan (a 1-D grid, the CTA's
// weight, maps and chunk range read from the plan in device memory); the
// per-weight fields of the arguments and the map parameters are then unused.
template <bool GROUP>
struct GroupRef {
  const uint8_t* plan;
  int n;
};
template <>
struct GroupRef<false> {};

// What one CTA merges: the tensor maps (parameter or plan memory), S, the
// seed, its 128-row tile and its range of 64-column chunks.
struct TcJob {
  const CUtensorMap* tw;
  const CUtensorMap* ta;
  const CUtensorMap* ts;
  const float* S;
  int64_t d, lds;
  uint64_t seed;
  uint32_t stream_id;
  int s_vec4;
  int64_t d0;
  int c_begin, nch;
};

template <int EPI, bool GROUP>
__global__ void __launch_bounds__(tc_threads(EPI), EPI == 128 ? 2 : 1)
    merge_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ StageMap<EPI> stage, const MergeTcArgs a, const GroupRef<GROUP> grp) {
  constexpr bool kStage = EPI != 128;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_w_full[kTcMaxWStages];
  __shared__ __align__(8) uint64_t bar_w_empty[kTcMaxWStages];
  __shared__ __align__(8) uint64_t bar_b_full[kTcMaxBStages];
  __shared__ __align__(8) uint64_t bar_b_empty[kTcMaxBStages];
  __shared__ __align__(8) uint64_t bar_acc_full[2];
  __shared__ __align__(8) uint64_t bar_acc_empty[2];
  __shared__ __align__(8) uint64_t bar_s_ready;
  __shared__ __align__(8) uint64_t bar_s_full;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t b_bytes = (uint32_t)a.np * 128;      // np ranks × 64 columns
  const uint32_t b_base = smem_addr(smem);
  const uint32_t w_base = b_base + a.b_stages * b_bytes;
  const uint32_t o_base = w_base + a.w_stages * kWTileBytes;  // two output tiles for TMA stores

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A plan's job is kept in shared memory (one thread writes it before the
  // barrier below) and each role reads the fields it uses, instead of every
  // thread holding all of them in registers; a single weight's job is formed
  // from the parameters in registers.
  __shared__ TcJob job_s;
  TcJob job_r;
  if constexpr (GROUP) {
    const int32_t* cta_begin = reinterpret_cast<const int32_t*>(grp.plan + kPlanHeaderBytes);
    const int m = plan_find(cta_begin, grp.n);
    if (threadIdx.x == 0) {
      const MergeEntry* e = reinterpret_cast<const MergeEntry*>(grp.plan + plan_entries_offset(grp.n)) + m;
      const int li = (int)blockIdx.x - __ldg(cta_begin + m);
      const int groups = e->groups, cpc = e->chunks_per_cta;
      job_s.tw = &e->tw;
      job_s.ta = &e->ta;
      job_s.ts = &e->ts;
      job_s.S = e->S;
      job_s.d = e->d;
      job_s.lds = e->lds;
      job_s.seed = e->seed;
      job_s.stream_id = e->stream_id;
      job_s.s_vec4 = e->s_vec4;
      job_s.d0 = (int64_t)(li / groups) * 128;
      job_s.c_begin = (li % groups) * cpc;
      job_s.nch = min(e->num_chunks, job_s.c_begin + cpc) - job_s.c_begin;
    }
  } else {
    job_r.tw = &tmap_w;
    job_r.ta = &tmap_a;
    if constexpr (kStage)
      job_r.ts = &stage.s;
    else
      job_r.ts = nullptr;
    job_r.S = a.S;
    job_r.d = a.d;
    job_r.lds = a.lds;
    job_r.seed = a.seed;
    job_r.stream_id = a.stream_id;
    job_r.s_vec4 = a.s_vec4;
    job_r.d0 = (int64_t)blockIdx.x * 128;
    job_r.c_begin = blockIdx.y * a.chunks_per_cta;
    job_r.nch = min(a.num_chunks, job_r.c_begin + a.chunks_per_cta) - job_r.c_begin;
  }
  if constexpr (GROUP) __syncthreads();
  const TcJob& job = [&]() -> const TcJob& {
    if constexpr (GROUP)
      return job_s;
    else
      return job_r;
  }();
  const int64_t d0 = job.d0;
  const int c_begin = job.c_begin;
  const int nch = job.nch;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.w_stages; ++s) {
      mbar_init(smem_addr(&bar_w_full[s]), 1);
      mbar_init(smem_addr(&bar_w_empty[s]), 128);  // one epilogue group takes each chunk
    }
    for (int s = 0; s < a.b_stages; ++s) {
      mbar_init(smem_addr(&bar_b_full[s]), a.explicit_a ? 1 : tc_gen(EPI));
      mbar_init(smem_addr(&bar_b_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&bar_acc_full[i]), 1);
      mbar_init(smem_addr(&bar_acc_empty[i]), 128);
    }
    // S is converted by every epilogue warp when it is staged by TMA (the
    // boxes are split between the warps of a lane quarter), else by warps 2-5
    mbar_init(smem_addr(&bar_s_ready), kStage && a.s_tma ? EPI : 128);
    mbar_init(smem_addr(&bar_s_full), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&tmem_slot), a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // tensor memory: [0, 128) two 64-column accumulators, then S_hi and S_lo,
  // each written 32 ranks (16 columns) at a time, so each region spans
  // round_up(np, 32) / 2 columns.  (A deeper accumulator ring, up to four fit
  // next to S at np = 256, measured no faster.)
  const uint32_t s_cols = (uint32_t)((a.np + 31) / 32 * 16);
  const uint32_t t_shi = tmem + 128, t_slo = t_shi + s_cols;

  // S staged by TMA: one 128-row × 32-rank box (16 KB, 128-byte swizzle) per
  // 32 ranks, all in flight at once, in the W ring (which starts right after
  // the ±1 ring and runs into the output tiles, so it holds the whole tile)
  const int s_boxes = (a.np + 31) / 32;
  if (warp == 0) {
    if (lane == 0) {
      if constexpr (GROUP) tmap_acquire(job.tw);
      tma_prefetch_desc(job.tw);
      bool go = true;
      if constexpr (kStage) {
        if (a.s_tma) {
          if constexpr (GROUP) tmap_acquire(job.ts);
          tma_prefetch_desc(job.ts);
          mbar_arrive_expect_tx(smem_addr(&bar_s_full), (uint32_t)s_boxes * 16384u);
          for (int j = 0; j < s_boxes; ++j)
            tma_load_2d(w_base + (uint32_t)j * 16384u, job.ts, smem_addr(&bar_s_full), 32 * j, (int32_t)d0);
          // the W stream may overwrite the staging area once S is in tensor memory
          go = mbar_wait(smem_addr(&bar_s_ready), 0, abort_p, a.err, kDevTimeoutOperand);
        }
      }
      int issued = 0;
      for (int i = 0; i < (go ? nch : 0); ++i) {
        const int s = i % a.w_stages;
        const uint32_t ph = (i / a.w_stages) & 1;
        if (!mbar_wait(smem_addr(&bar_w_empty[s]), ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
        mbar_arrive_expect_tx(smem_addr(&bar_w_full[s]), kWTileBytes);
        tma_load_2d(w_base + s * kWTileBytes, job.tw, smem_addr(&bar_w_full[s]), (c_begin + i) * 64, (int32_t)d0);
        issued = i + 1;
      }
      for (int i = (issued > a.w_stages ? issued - a.w_stages : 0); i < issued; ++i) {
        volatile int no_abort = 0;
        mbar_wait(smem_addr(&bar_w_full[i % a.w_stages]), (i / a.w_stages) & 1, &no_abort, a.err,
                  kDevTimeoutTeardown);
      }
      if (kStage && a.s_tma) {  // the staging copies must have landed before the CTA exits
        volatile int no_abort = 0;
        mbar_wait(smem_addr(&bar_s_full), 0, &no_abort, a.err, kDevTimeoutTeardown);
      }
    } else if (lane == 1 && a.explicit_a) {
      // tiles A[0:np, 64·chunk : 64·chunk + 64] of the given projection into
      // the B ring (rows past r and columns past k arrive as zeros); the 128-
      // byte swizzle of the copy is the layout the MMA descriptor reads
      if constexpr (GROUP) tmap_acquire(job.ta);
      tma_prefetch_desc(job.ta);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int s = i % a.b_stages;
        const uint32_t ph = (i / a.b_stages) & 1;
        if (!mbar_wait(smem_addr(&bar_b_empty[s]), ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
        mbar_arrive_expect_tx(smem_addr(&bar_b_full[s]), b_bytes);
        tma_load_2d(b_base + s * b_bytes, job.ta, smem_addr(&bar_b_full[s]), (c_begin + i) * 64, 0);
        issued = i + 1;
      }
      for (int i = (issued > a.b_stages ? issued - a.b_stages : 0); i < issued; ++i) {
        volatile int no_abort = 0;
        mbar_wait(smem_addr(&bar_b_full[i % a.b_stages]), (i / a.b_stages) & 1, &no_abort, a.err,
                  kDevTimeoutTeardown);
      }
    }
  } else if (warp == 1 || warp == tc_issuer2(EPI)) {
    // The whole warp runs the issue loop with warp-uniform waits; one elected
    // lane issues each MMA (the per-chunk loop is unrolled for the rank).
    // With two issuers, warp 1 takes the even chunks and the other the odd.
    // A = S (tensor memory, K-major), B = ±1 tile (N = 64 columns, K = ranks, MN-major)
    const uint32_t idesc = idesc_bf16_m128(64, 0, 1);
    const uint64_t b0 = sdesc_sw128(b_base, b_bytes, 1024);  // stage 0; stage s adds its offset >> 4
    const int nk = a.np / 16;
    constexpr int kStep = tc_issuer2(EPI) < 0 ? 1 : 2;
    int done = 0;  // one past the last chunk this warp issued
    if (__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_s_ready), 0, abort_p, a.err, kDevTimeoutOperand))) {
      tc_fence_after_sync();
      for (int i = warp == 1 ? 0 : 1; i < nch; i += kStep) {
        const int s = i % a.b_stages;
        const int acc = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_b_full[s]), (i / a.b_stages) & 1, abort_p, a.err,
                                               kDevTimeoutOperand)))
          break;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_acc_empty[acc]), ((i >> 1) & 1) ^ 1, abort_p, a.err,
                                               kDevTimeoutAccumFree)))
          break;
        tc_fence_after_sync();
        const uint64_t bo = b0 + (uint64_t)((uint32_t)s * (b_bytes >> 4));
        merge_mma_chunk(nk, tmem + (uint32_t)(acc * 64), t_shi, t_slo, bo, idesc);
        warp_mma_commit(smem_addr(&bar_b_empty[s]));
        warp_mma_commit(smem_addr(&bar_acc_full[acc]));
        done = i + 1;
      }
    }
    // Before the CTA may free tensor memory, the last MMAs must have ended.
    if (done > 0 && lane == 0) {
      volatile int no_abort = 0;
      const int i = done - 1;
      mbar_wait(smem_addr(&bar_acc_full[i & 1]), (i >> 1) & 1, &no_abort, a.err, kDevTimeoutTeardown);
    }
  } else if (warp >= 2 + EPI / 32) {
    // ---------------- ±1 tiles: row n (rank) holds 64 consecutive columns
    const int g = threadIdx.x - 64 - EPI;  // 0 .. tc_gen(EPI) - 1
    uint4 words[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    for (int i = 0; i < (a.explicit_a ? 0 : nch); ++i) {
      const int s = i % a.b_stages;
      const int chunk = c_begin + i;
      if (!mbar_wait(smem_addr(&bar_b_empty[s]), ((i / a.b_stages) & 1) ^ 1, abort_p, a.err, kDevTimeoutStageFree))
        break;
      const uint32_t bt = b_base + s * b_bytes;
#pragma unroll
      for (int h = 0; h < 256 / tc_gen(EPI); ++h) {
        const int n = g + tc_gen(EPI) * h;
        if (n < a.np) {
          if (n < a.r) {
            if ((chunk & 1) == 0 || i == 0)
              words[h] = sign_words(job.seed, job.stream_id, (uint32_t)n, (uint32_t)(chunk >> 1));
            const uint32_t w0 = (chunk & 1) ? words[h].z : words[h].x;
            const uint32_t w1 = (chunk & 1) ? words[h].w : words[h].y;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              const uint32_t byte = ((cc < 4 ? w0 : w1) >> ((cc & 3) * 8)) & 0xFFu;
              st_shared_v4(bt + sw128_offset((uint32_t)n, (uint32_t)cc), pm1_octet(byte));
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              st_shared_v4(bt + sw128_offset((uint32_t)n, (uint32_t)cc), make_uint4(0, 0, 0, 0));
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_addr(&bar_b_full[s]));
    }
  } else {
    // ---------------- epilogue warps 2 .. 2 + EPI/32: row 32·(warp & 3) + lane
    // of the tile (a warp reaches only its quarter of the tensor-memory
    // lanes).  With EPI = 256 the eight warps form two groups of four (h),
    // each covering the whole tile: group h takes the chunks i ≡ h (mod 2),
    // with accumulator h and output tile h.  The per-chunk chain of waits,
    // fences and barriers of one group then overlaps the other group's,
    // as the chains of two CTAs on one SM do for EPI = 128.
    const int q = warp & 3;
    const int h = EPI == 128 ? 0 : (warp - 2) >> 2;
    constexpr int kGroups = EPI / 128;
    const bool storer = ((threadIdx.x - 64) & 127) == 0;  // first thread of the group issues its stores
    const uint32_t group_bar = EPI == 128 ? 1u : 3u + (uint32_t)h;
    // warps 2-5 load S by themselves through barrier kPrologueBar; with eight
    // epilogue warps the others may already wait at barrier 1 meanwhile
    constexpr uint32_t kPrologueBar = EPI == 128 ? 1 : 2;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    if (kStage && a.s_tma) {
      // S from the staged boxes: row `row` of box j holds ranks 32j .. 32j+31
      // in 16-byte chunks swizzled by (row & 7); four threads share each group
      // of banks, the minimum for a 512-byte warp read
      if (__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_s_full), 0, abort_p, a.err, kDevTimeoutOperand))) {
        for (int j = h; j < s_boxes; j += EPI / 128) {
          float sv[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = ld_shared_v4(w_base + (uint32_t)j * 16384u + sw128_offset((uint32_t)row, (uint32_t)c));
            sv[4 * c] = __uint_as_float(u.x);
            sv[4 * c + 1] = __uint_as_float(u.y);
            sv[4 * c + 2] = __uint_as_float(u.z);
            sv[4 * c + 3] = __uint_as_float(u.w);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              split_bf16x2(sv[16 * half + 2 * jj], sv[16 * half + 2 * jj + 1], hi[jj], lo[jj]);
            tmem_st8(t_shi + lane_off + (uint32_t)(16 * j + 8 * half), hi);
            tmem_st8(t_slo + lane_off + (uint32_t)(16 * j + 8 * half), lo);
          }
        }
        tmem_wait_st();
        tc_fence_before_sync();
        fence_proxy_async_smem();  // the W stream's TMA loads overwrite the staged boxes next
        mbar_arrive(smem_addr(&bar_s_ready));
      }
    } else if (h == 0) {
    // S tile → bf16 hi / lo pairs → tensor memory, 32 ranks at a time.  The
    // tile is read with coalesced loads (eight threads per 128-byte row
    // piece) and staged through the output tiles, which are idle until the
    // first store, with a 144-byte row pitch so that both the staging writes
    // and each thread's read of its own row are free of bank conflicts; the
    // next piece's loads are in flight while the current one is converted
    // (issued after the row read, which keeps the loop free of spills).
    const int et = threadIdx.x - 64;  // 0..127
    float4 nxt[8];
    auto load_piece = [&](int n0) {
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int f = it * 128 + et, pr = f >> 3, c = n0 + (f & 7) * 4;
        const int64_t gr = d0 + pr;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (gr < job.d) {
          const float* src = job.S + gr * job.lds + c;
          if (job.s_vec4 && c + 4 <= a.r) {
            v = __ldg(reinterpret_cast<const float4*>(src));
          } else {
            if (c < a.r) v.x = __ldg(src);
            if (c + 1 < a.r) v.y = __ldg(src + 1);
            if (c + 2 < a.r) v.z = __ldg(src + 2);
            if (c + 3 < a.r) v.w = __ldg(src + 3);
          }
        }
        nxt[it] = v;
      }
    };
    load_piece(0);
    for (int n0 = 0; n0 < a.np; n0 += 32) {
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int f = it * 128 + et;
        st_shared_v4(o_base + (uint32_t)((f >> 3) * 144 + (f & 7) * 16),
                     make_uint4(__float_as_uint(nxt[it].x), __float_as_uint(nxt[it].y), __float_as_uint(nxt[it].z),
                                __float_as_uint(nxt[it].w)));
      }
      named_barrier_sync(kPrologueBar, 128);
      float sv[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 u = ld_shared_v4(o_base + (uint32_t)(row * 144 + j * 16));
        sv[4 * j] = __uint_as_float(u.x);
        sv[4 * j + 1] = __uint_as_float(u.y);
        sv[4 * j + 2] = __uint_as_float(u.z);
        sv[4 * j + 3] = __uint_as_float(u.w);
      }
      named_barrier_sync(kPrologueBar, 128);  // every row read before the next piece lands
      if (n0 + 32 < a.np) load_piece(n0 + 32);
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // 16 ranks = 8 packed columns per store
        uint32_t hi[8], lo[8];
#pragma unroll
        // (scalar conversions here: the packed form, used for the staged
        // boxes above, costs this four-warp kernel 12 bytes of spills)
        for (int j = 0; j < 8; ++j) {
          const float x0 = sv[16 * half + 2 * j], x1 = sv[16 * half + 2 * j + 1];
          const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
          const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
          const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
          hi[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lo[j] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        tmem_st8(t_shi + lane_off + (uint32_t)(n0 / 2 + 8 * half), hi);
        tmem_st8(t_slo + lane_off + (uint32_t)(n0 / 2 + 8 * half), lo);
      }
    }
    tmem_wait_st();
    tc_fence_before_sync();
    mbar_arrive(smem_addr(&bar_s_ready));
    }

    const float cc = a.alpha_eta_dev ? (*a.alpha_eta_dev) * a.inv_sqrt_r : a.c;
    if constexpr (GROUP) {
      if (storer) tmap_acquire(job.tw);  // the storing threads read the map too
    }
    for (int i = h; i < nch; i += kGroups) {
      const int s = i % a.w_stages;
      const int acc = i & 1;  // = h with two groups
      // Wait results are made warp-uniform (the TMEM loads below are
      // warp-collective) and the four warps leave the loop together through
      // a barrier vote, so no thread is ever left waiting at a barrier.
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_w_full[s]), (i / a.w_stages) & 1, abort_p, a.err,
                                                   kDevTimeoutTmaFull));
      constexpr int NCH = 8;  // 16-byte column chunks of the row per thread
      constexpr int ch0 = 0;
      uint4 wv[NCH];
      if (ok) {
        // W row chunk out of shared memory; the slot is released at once
        const uint32_t wt = w_base + s * kWTileBytes;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
          wv[ch] = ld_shared_v4(wt + sw128_offset((uint32_t)row, (uint32_t)(ch0 + ch)));
        // The next TMA load into this slot writes through the async proxy:
        // without a proxy fence these generic reads are not ordered before
        // it (a merge of 196 weights in one launch measured stale rows).
        fence_proxy_async_smem();
        mbar_arrive(smem_addr(&bar_w_empty[s]));
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_acc_full[acc]), (i >> 1) & 1, abort_p, a.err,
                                               kDevTimeoutAccum));
      }
      // W' for this thread's columns of the row, packed as bf16 pairs
      uint32_t out[NCH][4];
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int hh = 0; hh < NCH / 4; ++hh) {
          const int half = ch0 / 4 + hh;  // 32-column half of the chunk
          uint32_t u[2][16];
          tmem_ld16(tmem + lane_off + (uint32_t)(acc * 64 + 32 * half), u[0]);
          tmem_ld16(tmem + lane_off + (uint32_t)(acc * 64 + 32 * half + 16), u[1]);
          tmem_wait_ld();
          if (hh == NCH / 4 - 1) {
            tc_fence_before_sync();
            mbar_arrive(smem_addr(&bar_acc_empty[acc]));
          }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int ch = hh * 4 + c4;
            const uint32_t in[4] = {wv[ch].x, wv[ch].y, wv[ch].z, wv[ch].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float w0 =
                  __uint_as_float(in[e] << 16) - cc * __uint_as_float(u[c4 >> 1][(c4 & 1) * 8 + 2 * e]);
              const float w1 = __uint_as_float(in[e] & 0xFFFF0000u) -
                               cc * __uint_as_float(u[c4 >> 1][(c4 & 1) * 8 + 2 * e + 1]);
              out[ch][e] = bf16x2_rn(w0, w1);
            }
          }
        }
      }
      // The output tile used two chunks ago must have been read by its store
      // (with two groups, the group's own previous store).
      const uint32_t ot = o_base + (uint32_t)(i & 1) * kWTileBytes;
      if (storer) {
        if constexpr (kGroups == 1)
          bulk_wait_group_read1();
        else
          bulk_wait_group_read0();
      }
      if (named_barrier_any(group_bar, 128, !ok)) break;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        st_shared_v4(ot + sw128_offset((uint32_t)row, (uint32_t)(ch0 + ch)),
                     make_uint4(out[ch][0], out[ch][1], out[ch][2], out[ch][3]));
      fence_proxy_async_smem();
      named_barrier_sync(group_bar, 128);
      if (storer) {
        // rows past d and columns past k are clipped by the tensor map
        tma_store_2d(job.tw, ot, (c_begin + i) * 64, (int32_t)d0);
        bulk_commit_group();
      }
    }
    if (storer) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

// Shared-memory and tensor-memory layout of the tensor-core kernel for a rank.
struct TcConfig {
  int np;
  bool two_per_sm;
  uint32_t tmem_cols, b_bytes, smem;
  int b_stages, w_stages;
};

TcConfig tc_config(int r) {
  TcConfig c{};
  c.np = (int)round_up(r, 16);
  // Tensor memory: two 64-column accumulators + S hi / lo (round_up(np, 32) / 2
  // columns each).  Up to np = 128 that is ≤ 256 columns and two CTAs share an
  // SM (≤ 112 KB of shared memory each); above, one CTA per SM.
  c.tmem_cols = c.np <= 128 ? 256u : 512u;
  c.two_per_sm = c.np <= 128;
  // Separate rings: the ±1 tiles (np·128 bytes each) need only run a chunk or
  // two ahead of the MMAs, while the W ring must hold enough bytes in flight
  // to cover the memory latency; W gets whatever the ±1 ring and the two
  // output tiles leave.  The ±1 ring holds three tiles, except two from
  // np = 80 to 128 (two CTAs per SM) and, above, for a given operand
  // (tc_b_stages).  Above np = 128 the builders of the
  // ±1 tiles set the pace of a chunk once two warps issue the MMAs, and a
  // third tile (six W stages instead of eight at np = 256) lets them run
  // ahead: 1-3 % faster in the A/B runs.
  c.b_bytes = (uint32_t)c.np * 128u;
  const uint32_t budget = (c.two_per_sm ? kSmemTwoPerSm : kSmemBudget) - 1024 - 2 * kWTileBytes;
  c.b_stages = (c.b_bytes <= 8192 || !c.two_per_sm) ? 3 : 2;
  c.w_stages = (int)std::min<uint32_t>(kTcMaxWStages, (budget - c.b_stages * c.b_bytes) / kWTileBytes);
  c.smem = c.b_stages * c.b_bytes + c.w_stages * kWTileBytes + 2 * kWTileBytes + 1024;
  return c;
}

// Tiles of the ±1 ring a launch uses.  With two MMA issuers (above np = 128)
// a waiting issuer tells the phases of a stage apart by parity alone, so it
// must never wait on a stage whose previous phase (the other issuer's chunk)
// may still be open: with an odd ring, stage s carries chunks of both
// issuers in turn.  The ±1 builders finish their tiles in chunk order, so an
// issuer that has consumed chunk i - 2 knows chunk i - 3 complete and three
// tiles are safe.  Tiles of a given operand arrive by TMA, whose copies may
// complete out of order; there the ring is even (two tiles), and each stage
// belongs to one issuer.
int tc_b_stages(const TcConfig& c, bool explicit_a) { return (explicit_a && !c.two_per_sm) ? 2 : c.b_stages; }

// Above np = 128 (one CTA per SM, a 128 KB S tile at r = 256) S is staged
// by TMA, all boxes at once, when its rows suit a tensor map (16-byte
// aligned base and row stride) and the boxes fit in the W ring plus the
// output tiles: loaded by threads 32 ranks at a time it took 13 of the
// 49 µs of a CTA.  Up to np = 128 the tile is small and two CTAs share an
// SM; there the W stream starting at once, overlapped with a thread-loaded
// S, measured faster than waiting for a staged S.
bool tc_stage_s(const TcConfig& c, bool s_vec4) { return c.np > 128 && s_vec4 && (c.np + 31) / 32 <= c.w_stages + 2; }

bool s_rows_vec4(const float* S, int64_t lds) {
  return (lds % 4 == 0) && ((reinterpret_cast<uintptr_t>(S) & 15) == 0);
}

}  // namespace

logra_status launch_merge(void* W, int64_t ldw, int64_t d, int64_t k, const float* S, int64_t lds, int r,
                          uint64_t seed, uint32_t stream_id, float alpha_eta, const float* alpha_eta_dev,
                          const void* A, int64_t lda, cudaStream_t st) {
  const double inv_sqrt_r_d = 1.0 / std::sqrt((double)r);
  const float c = (float)((double)alpha_eta * inv_sqrt_r_d);
  const float inv_sqrt_r = (float)inv_sqrt_r_d;
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(W);
  cudaError_t e;
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  const TcConfig cfg = tc_config(r);
  CUtensorMap tw, ta;
  StageMap<256> ts;
  logra_status s = make_tmap_bf16_2d(&tw, W, (uint64_t)k, (uint64_t)d, (uint64_t)ldw * 2, 64, 128);
  if (s != LOGRA_OK) return s;
  if (A) {
    // the given projection: r rows × k columns, tiles of np rows × 64 columns
    s = make_tmap_bf16_2d(&ta, A, (uint64_t)k, (uint64_t)r, (uint64_t)lda * 2, 64, (uint32_t)cfg.np);
    if (s != LOGRA_OK) return s;
  } else {
    ta = tw;  // not read
  }
  MergeTcArgs a{};
  a.d = d;
  a.k = k;
  a.r = r;
  a.np = cfg.np;
  a.num_chunks = (int)((k + 63) / 64);
  const int d_tiles = (int)((d + 127) / 128);
  // Column groups: ~160 CTAs per matrix (a shape-only target), but at least
  // np/16 chunks per CTA.  Each CTA reads its S tile once (128·r·4 bytes)
  // against 128·64·4 bytes of W traffic per chunk, so np/16 chunks keep the
  // S re-reads (one per column group) within a quarter of the W stream and
  // amortise the CTA's prologue; on small matrices (the 1.5B set's k/v is 24
  // chunks wide) the 160-CTA target alone left one chunk per CTA.
  // Concurrent matrices on other streams fill the remaining SMs.  Above
  // np = 128 (one CTA per SM) a column group costs its CTA a prologue (the
  // S tile staged and split into tensor memory: 8-15k cycles at np = 256,
  // with no W streamed meanwhile) and an S re-read, so row tiles are split
  // only while the grid stays within one wave.
  int groups = (160 + d_tiles - 1) / d_tiles;
  if (!cfg.two_per_sm) {
    int sms = 0;
    logra_status q = require_sm103(&sms);
    if (q != LOGRA_OK) return q;
    groups = std::max(1, sms / d_tiles);
  }
  groups = std::max(1, std::min(groups, a.num_chunks));
  a.chunks_per_cta = std::max((a.num_chunks + groups - 1) / groups, std::min(a.num_chunks, std::max(1, a.np / 16)));
  groups = (a.num_chunks + a.chunks_per_cta - 1) / a.chunks_per_cta;
  a.tmem_cols = cfg.tmem_cols;
  a.b_stages = tc_b_stages(cfg, A != nullptr);
  a.w_stages = cfg.w_stages;
  a.c = c;
  a.alpha_eta_dev = alpha_eta_dev;
  a.inv_sqrt_r = inv_sqrt_r;
  a.S = S;
  a.lds = lds;
  a.s_vec4 = s_rows_vec4(S, lds);
  a.W = w;
  a.ldw = ldw;
  a.seed = seed;
  a.stream_id = stream_id;
  a.explicit_a = A ? 1 : 0;
  a.s_tma = tc_stage_s(cfg, a.s_vec4);
  if (a.s_tma) {
    s = make_tmap_f32_2d(&ts.s, S, (uint64_t)r, (uint64_t)d, (uint64_t)lds * 4, 32, 128);
    if (s != LOGRA_OK) return s;
  } else {
    ts.s = tw;  // not read
  }
  a.err = err;
  const dim3 grid((unsigned)d_tiles, (unsigned)groups);
  if (cfg.two_per_sm) {
    e = cudaFuncSetAttribute(merge_tc_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(merge_tc_kernel)");
    merge_tc_kernel<128, false><<<grid, tc_threads(128), cfg.smem, st>>>(tw, ta, StageMap<128>{}, a, GroupRef<false>{});
  } else {
    e = cudaFuncSetAttribute(merge_tc_kernel<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(merge_tc_kernel)");
    merge_tc_kernel<256, false><<<grid, tc_threads(256), cfg.smem, st>>>(tw, ta, ts, a, GroupRef<false>{});
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch merge_tc_kernel");
  return LOGRA_OK;
}

// ---------------------------------------------------------------- merge plan
size_t merge_group_plan_bytes(int n) { return plan_entries_offset(n) + (size_t)n * sizeof(MergeEntry); }

logra_status build_merge_group_plan(int n, const logra_merge_target* tg, int r, void* plan, size_t plan_bytes) {
  std::memset(plan, 0, merge_group_plan_bytes(n));
  uint8_t* base = static_cast<uint8_t*>(plan);
  MergePlanHeader* h = reinterpret_cast<MergePlanHeader*>(base);
  int32_t* cta_begin = reinterpret_cast<int32_t*>(base + kPlanHeaderBytes);
  MergeEntry* ent = reinterpret_cast<MergeEntry*>(base + plan_entries_offset(n));
  const bool explicit_a = n > 0 && tg[0].A != nullptr;
  const TcConfig cfg = tc_config(r);
  h->magic = kPlanMagic;
  h->n = n;
  h->r = r;
  h->explicit_a = explicit_a ? 1 : 0;
  h->path = cfg.two_per_sm ? 1 : 2;
  h->np = cfg.np;
  h->w_stages = cfg.w_stages;
  h->b_stages = tc_b_stages(cfg, explicit_a);
  h->tmem_cols = cfg.tmem_cols;
  h->smem_bytes = cfg.smem;
  // S staged by TMA only when every weight's S allows it (one layout per launch)
  bool all_vec4 = true;
  for (int j = 0; j < n; ++j)
    if (tg[j].d > 0 && tg[j].k > 0) all_vec4 = all_vec4 && s_rows_vec4(tg[j].S, tg[j].lds);
  h->s_tma = tc_stage_s(cfg, all_vec4) ? 1 : 0;
  int64_t total = 0;
  for (int j = 0; j < n; ++j) {
    const logra_merge_target& t = tg[j];
    MergeEntry& e = ent[j];
    cta_begin[j] = (int32_t)total;
    e.W = static_cast<__nv_bfloat16*>(t.W);
    e.ldw = t.ldw;
    e.d = t.d;
    e.k = t.k;
    e.S = t.S;
    e.lds = t.lds;
    e.A = static_cast<const __nv_bfloat16*>(t.A);
    e.lda = t.lda;
    e.seed = t.seed;
    e.stream_id = t.stream_id;
    e.s_vec4 = s_rows_vec4(t.S, t.lds) ? 1 : 0;
    if (t.d == 0 || t.k == 0) continue;  // nothing to merge: no CTAs
    const int d_tiles = (int)((t.d + 127) / 128);
    // One launch covers the set, so a row tile is split only to bound the
    // length of a CTA (and the tail of the launch): at most 32 chunks per
    // CTA, evenly split, and at least np/16 as in the single-weight launch.
    e.num_chunks = (int)((t.k + 63) / 64);
    int groups = (e.num_chunks + 31) / 32;
    e.chunks_per_cta = std::max((e.num_chunks + groups - 1) / groups, std::min(e.num_chunks, std::max(1, cfg.np / 16)));
    e.groups = (e.num_chunks + e.chunks_per_cta - 1) / e.chunks_per_cta;
    logra_status s = make_tmap_bf16_2d(&e.tw, t.W, (uint64_t)t.k, (uint64_t)t.d, (uint64_t)t.ldw * 2, 64, 128);
    if (s != LOGRA_OK) return s;
    if (explicit_a) {
      s = make_tmap_bf16_2d(&e.ta, t.A, (uint64_t)t.k, (uint64_t)r, (uint64_t)t.lda * 2, 64, (uint32_t)cfg.np);
      if (s != LOGRA_OK) return s;
    }
    if (h->s_tma) {
      s = make_tmap_f32_2d(&e.ts, t.S, (uint64_t)r, (uint64_t)t.d, (uint64_t)t.lds * 4, 32, 128);
      if (s != LOGRA_OK) return s;
    }
    e.ctas = d_tiles * e.groups;
    total += e.ctas;
    if (total > 0x7FFFFFFF) return fail(LOGRA_ERR_SHAPE, "merge group: more than 2^31 - 1 CTAs");
  }
  cta_begin[n] = (int32_t)total;
  h->total_ctas = (int32_t)total;
  (void)plan_bytes;
  return LOGRA_OK;
}

logra_status check_merge_group_plan(const void* plan, int* n, int* r) {
  const MergePlanHeader* h = static_cast<const MergePlanHeader*>(plan);
  if (h->magic != kPlanMagic) return fail(LOGRA_ERR_INVALID_ARG, "merge group: not a plan (logra_merge_group_plan)");
  *n = h->n;
  *r = h->r;
  return LOGRA_OK;
}

logra_status launch_merge_group(const void* plan, const void* plan_dev, float alpha_eta, const float* alpha_eta_dev,
                                cudaStream_t st) {
  const MergePlanHeader* h = static_cast<const MergePlanHeader*>(plan);
  if (h->total_ctas == 0) return LOGRA_OK;
  const int r = h->r, n = h->n;
  const double inv_sqrt_r_d = 1.0 / std::sqrt((double)r);
  const float c = (float)((double)alpha_eta * inv_sqrt_r_d);
  const float inv_sqrt_r = (float)inv_sqrt_r_d;
  const uint8_t* pd = static_cast<const uint8_t*>(plan_dev);
  const unsigned grid = (unsigned)h->total_ctas;
  cudaError_t e;
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  MergeTcArgs a{};
  a.r = r;
  a.np = h->np;
  a.tmem_cols = h->tmem_cols;
  a.b_stages = h->b_stages;
  a.w_stages = h->w_stages;
  a.c = c;
  a.alpha_eta_dev = alpha_eta_dev;
  a.inv_sqrt_r = inv_sqrt_r;
  a.explicit_a = h->explicit_a;
  a.s_tma = h->s_tma;
  a.err = err;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  const GroupRef<true> grp{pd, n};
  if (h->path == 1) {
    e = cudaFuncSetAttribute(merge_tc_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)h->smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(merge_tc_kernel)");
    merge_tc_kernel<128, true><<<grid, tc_threads(128), h->smem_bytes, st>>>(unused, unused, StageMap<128>{}, a, grp);
  } else {
    StageMap<256> ts;
    ts.s = unused;
    e = cudaFuncSetAttribute(merge_tc_kernel<256, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)h->smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(merge_tc_kernel)");
    merge_tc_kernel<256, true><<<grid, tc_threads(256), h->smem_bytes, st>>>(unused, unused, ts, a, grp);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch merge_tc_kernel (group)");
  return LOGRA_OK;
}

}  // namespace logra
