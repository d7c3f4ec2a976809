// Sketch accumulation S += dYᵀ (X Aᵀ) on sm_103a tensor cores.
//
// LoGRA summary page, section "草图如何取代完整梯度缓冲": the d×r sketch
// S = G Aᵀ of a d×k weight is accumulated per micro-batch in fp32 by
// projecting the layer inputs before they meet the backward derivatives, so no
// d×k gradient exists at any point.  Here that is two tensor-core passes:
//
//   project:  P = X·(A√r)ᵀ            (T×r, fp32 in tensor memory)
//             P_hi = bf16(P), P_lo = bf16(P − P_hi)  → workspace, stored as Pᵀ
//   contract: S += (1/√r)·(dYᵀ P_hi + dYᵀ P_lo)
//             over split ranges of T; the fp32 partials of the splits are
//             then added in split order by a separate, fully parallel reduce
//             kernel, so the result is bitwise reproducible.
//
// The ±1 tiles of A are never stored in global memory: the projection kernel
// rebuilds each 64-column slab of A in shared memory from the counter-based
// generator while the X tile of the same slab streams in through TMA.
//
// Why the hi/lo split: P carries ~24 significant bits; rounding it once to
// bf16 leaves a relative error near 2⁻⁹ per entry, which shows up as ~1.7e-3
// relative Frobenius error in S on the workloads' shapes, above the 1e-3
// bound.  hi + lo keeps ~16 bits (≈1e-5), at the price of a second MMA per
// step in the contraction.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

constexpr int kTileRows = 128;      // MMA M
constexpr int kSlab = 64;           // K elements per pipeline stage (128 bytes of bf16)
constexpr int kMaxStages = 8;
constexpr uint32_t kSmemBudget = 230400;    // dynamic shared memory per CTA, one CTA per SM
constexpr uint32_t kSmemTwoPerSm = 113664;  // dynamic shared memory per CTA, two CTAs per SM

// ------------------------------------------------------------------ project
// warp 0: TMA, warp 1: MMA, warps 2-9: sign tiles (one rank row per thread),
// warps 2-5 then read the accumulator out (one TMEM lane quarter each).
constexpr int kProjThreads = 320;
constexpr int kGenThreads = 256;

constexpr int kMaxTargets = 4;  // projections sharing one X (q/k/v, gate/up)

struct ProjectArgs {
  int64_t T, k;
  int r, np;
  int ntg;    // targets sharing X; the B tile stacks their sign tiles
  int explicit_a;  // 1: the B tiles come from given bf16 projection operands by TMA (one per target)
  int npt;    // ntg·np rows of the stacked B tile (≤ 512)
  int64_t ldp;
  int num_kb;
  int stages;    // X tiles in flight (with given operands each stage also holds its B tile)
  int b_stages;  // sign tiles built on chip: a ring of their own (given operands: = stages)
  uint32_t tmem_cols;
  int p16;    // 1: write Pᵀ as fp16 blocks scaled per 16-token group (p_hi, p16_half_bytes); 0: bf16 hi + lo
  uint64_t seed[kMaxTargets];
  uint32_t stream_id[kMaxTargets];
  __nv_bfloat16* p_hi[kMaxTargets];
  __nv_bfloat16* p_lo[kMaxTargets];
  unsigned int* err;
};

// The power-of-two scale of a group of 16 consecutive tokens (16 rows of P) in
// the fp16 form: with m the largest |P| of the group, P is stored as
// fp16(P·2^−e) and 2^e is kept, where e = ⌊log₂ m⌋ − 14 puts m in
// [2^14, 2^15): the largest entry keeps all 11 significant bits of fp16,
// entries down to 2^−28·m stay normal, and nothing reaches the fp16 limit
// (65504).  (One scale per 16 tokens instead of per token: the contraction
// then takes one scale per 16-token operand group.)  e is held in [−126, 113] so that 2^e and
// 2^−e are both normal floats; a zero, infinite or NaN maximum gives e = 0 (an
// infinity or NaN then passes through the conversion unchanged).
__device__ __forceinline__ int p16_exponent(float m) {
  if (!(m > 0.f) || !(m <= 3.4028235e38f)) return 0;
  const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  return max(-126, min(113, E - 14));
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// The fp16 form of Pᵀ in the workspace: one block per 64 tokens, each block
// two halves, one per CTA of a contraction pair.  A half is the 64 token
// scales g_t (fp32, 256 bytes; equal within each 16-token group) followed by
// its np/2 rows of Pᵀ, 64 fp16
// tokens per 128-byte row, in the contraction's shared-memory image of its
// operand (K-major, 128-byte swizzle: 16-byte chunk c of local row n stored at
// chunk c ^ (n & 7)).  The contraction then fetches the scales and its operand
// half of a stage with one bulk copy.
__host__ __device__ constexpr uint32_t p16_half_bytes(int np) { return 256u + (uint32_t)np * 64u; }
// MT = 2 (one CTA per SM, at most 256 stacked rows): a CTA covers 256 tokens
// as two 128-row sub-tiles whose MMAs share each B tile, so the B tile moves
// through shared memory once per 256 tokens instead of once per 128.
//
// Operands of targets 1..3 of a shared-input call with given projections.
// They exist only in the MULTI instantiation, so the single-operand and
// on-chip kernels carry no extra parameter block.
template <bool MULTI>
struct ExtraOperands {
  CUtensorMap m[kMaxTargets - 1];
};
template <>
struct ExtraOperands<false> {};

// P16: the epilogue writes the fp16 form of P (the np > 64 plans); compiled
// only into the instantiations that need it, so the bf16 ones keep their
// register budget.
//
// The body runs for the CTA with index `cta` along T; the tensor maps come by
// pointer (kernel parameters, or an entry of a group plan in global memory,
// which GROUP makes the TMA thread acquire before its first use).
template <int MT, bool MULTI, bool P16, bool GROUP>
__device__ __forceinline__ void project_body(const CUtensorMap* tmap_x, const CUtensorMap* tmap_a,
                                             const ExtraOperands<MULTI>& ops, const ProjectArgs& a, int cta) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full_x[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_full_b[kMaxStages];   // sign tiles (on chip only)
  __shared__ __align__(8) uint64_t bar_empty_b[kMaxStages];
  __shared__ __align__(8) uint64_t bar_accum;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  // The X tiles stream through a ring of a.stages slots.  Given operands
  // arrive with them (slot s of the B ring belongs to slot s of the X ring);
  // sign tiles built on chip need no latency hiding and take a short ring of
  // their own, which leaves the shared memory to X tiles in flight.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t x_bytes = kTileRows * 128 * MT;
  const uint32_t b_bytes = (uint32_t)a.npt * 128;
  const uint32_t x_base = smem_addr(smem);
  const uint32_t b_base = x_base + a.stages * x_bytes;
  const bool own_b = !a.explicit_a;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = (int64_t)cta * kTileRows * MT;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&bar_full_x[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
    }
    for (int s = 0; s < a.b_stages; ++s) {
      mbar_init(smem_addr(&bar_full_b[s]), kGenThreads);
      mbar_init(smem_addr(&bar_empty_b[s]), 1);
    }
    mbar_init(smem_addr(&bar_accum), 1);
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

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: X[t0:t0+128, 64·kb : 64·kb+64], and
      // with a given projection also its tile A[0:np, 64·kb : 64·kb+64]
      // (rows past r and columns past k arrive as zeros)
      if constexpr (GROUP) {
        tmap_acquire(tmap_x);
        if (a.explicit_a) tmap_acquire(tmap_a);
      }
      tma_prefetch_desc(tmap_x);
      if (a.explicit_a) {
        tma_prefetch_desc(tmap_a);
        if constexpr (MULTI)
          for (int j = 1; j < a.ntg; ++j) tma_prefetch_desc(&ops.m[j - 1]);
      }
      int issued = 0;
      RingPos rp;
      for (int kb = 0; kb < a.num_kb; ++kb, rp.advance(a.stages)) {
        const int s = rp.s;
        const uint32_t ph = rp.ph;
        if (!mbar_wait(smem_addr(&bar_empty[s]), ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
        mbar_arrive_expect_tx(smem_addr(&bar_full_x[s]), x_bytes + (a.explicit_a ? b_bytes : 0u));
        tma_load_2d(x_base + s * x_bytes, tmap_x, smem_addr(&bar_full_x[s]), kb * kSlab, (int32_t)t0);
        if (a.explicit_a) {
          // target j's tile: rows j·np .. j·np + np of the stacked B stage
          tma_load_2d(b_base + s * b_bytes, tmap_a, smem_addr(&bar_full_x[s]), kb * kSlab, 0);
          if constexpr (MULTI)
            for (int j = 1; j < a.ntg; ++j)
              tma_load_2d(b_base + s * b_bytes + (uint32_t)(j * a.np) * 128u, &ops.m[j - 1], smem_addr(&bar_full_x[s]),
                          kb * kSlab, 0);
        }
        issued = kb + 1;
      }
      // Drain: every issued copy must have landed before the CTA may exit.
      for (int kb = (issued > a.stages ? issued - a.stages : 0); kb < issued; ++kb) {
        const int s = kb % a.stages;
        volatile int no_abort = 0;
        mbar_wait(smem_addr(&bar_full_x[s]), (kb / a.stages) & 1, &no_abort, a.err, kDevTimeoutTeardown);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: P[128 × np] += X_slab · B_slabᵀ
    // The whole warp runs the loop with warp-uniform waits; one elected lane
    // issues.  One MMA covers up to 256 stacked rows; a second one (B rows
    // 256.., D columns 256..) the rest.
    const uint32_t n1 = (uint32_t)min(a.npt, 256), n2 = (uint32_t)(a.npt - (int)n1);
    const uint32_t idesc1 = idesc_bf16_m128(n1, 0, 0), idesc2 = idesc_bf16_m128(n2 > 0 ? n2 : 16, 0, 0);
    // stage-0 descriptors; stage s adds its byte offset >> 4 to the address field
    const uint64_t x0 = sdesc_sw128(x_base, 16, 1024), b0 = sdesc_sw128(b_base, 16, 1024);
    RingPos rp, rb;
    for (int kb = 0; kb < a.num_kb; ++kb, rp.advance(a.stages), rb.advance(a.b_stages)) {
      const int s = rp.s;
      const uint32_t ph = rp.ph;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_full_x[s]), ph, abort_p, a.err, kDevTimeoutTmaFull)))
        break;
      if (own_b &&
          !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_full_b[rb.s]), rb.ph, abort_p, a.err, kDevTimeoutOperand)))
        break;
      tc_fence_after_sync();
      const uint64_t xo = x0 + (uint64_t)((uint32_t)s * (x_bytes >> 4));
      const uint64_t bo = b0 + (uint64_t)((uint32_t)(own_b ? rb.s : s) * (b_bytes >> 4));
      if (n2 > 0) {
#pragma unroll
        for (int ks = 0; ks < kSlab / 16; ++ks) {
          warp_mma_bf16_ss(tmem, xo + (uint64_t)(ks * 2), bo + (uint64_t)(ks * 2), idesc1, (kb | ks) != 0);
          // B rows 256.. start 256·128 bytes further (2048 in 16-byte units)
          warp_mma_bf16_ss(tmem + 256, xo + (uint64_t)(ks * 2), bo + 2048 + (uint64_t)(ks * 2), idesc2,
                           (kb | ks) != 0);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < kSlab / 16; ++ks)
#pragma unroll
          for (int m = 0; m < MT; ++m)  // sub-tile m: X rows 128m.., 16 KB further; D columns m·npt..
            warp_mma_bf16_ss(tmem + (uint32_t)(m * a.npt), xo + (uint64_t)(m * 1024 + ks * 2),
                             bo + (uint64_t)(ks * 2), idesc1, (kb | ks) != 0);
      }
      warp_mma_commit(smem_addr(&bar_empty[s]));
      if (own_b) warp_mma_commit(smem_addr(&bar_empty_b[rb.s]));
    }
    // Signals the epilogue once every MMA issued above has completed.
    warp_mma_commit(smem_addr(&bar_accum));
  } else {
    // ---------------- warps 2..9: sign tiles; warps 2..5 then the epilogue
    // Thread g builds stacked rows g and g + 256: row R is rank R % np of
    // target R / np.
    const int g = threadIdx.x - 64;  // 0..255
    // Per-row constants, fixed for the whole K loop: 0 = no row, 1 = padding
    // rank (zeros), 2 = a rank of target j.
    int kind[2];
    uint32_t rank[2], sid[2];
    uint64_t seed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = g + 256 * h;
      const int j = R / a.np, n = R - j * a.np;
      kind[h] = R >= a.npt ? 0 : (n < a.r ? 2 : 1);
      rank[h] = (uint32_t)n;
      seed[h] = kind[h] == 2 ? a.seed[j] : 0;
      sid[h] = kind[h] == 2 ? a.stream_id[j] : 0;
    }
    uint4 words[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    RingPos rb;
    for (int kb = 0; kb < (own_b ? a.num_kb : 0); ++kb, rb.advance(a.b_stages)) {
      const int s = rb.s;
      if (!mbar_wait(smem_addr(&bar_empty_b[s]), rb.ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
      const uint32_t bt = b_base + s * b_bytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int R = g + 256 * h;
        if (kind[h] != 0) {
          const uint32_t n = rank[h];
          if (kind[h] == 2) {
            // one generator call covers 128 columns = two slabs
            if ((kb & 1) == 0) words[h] = sign_words(seed[h], sid[h], n, (uint32_t)(kb >> 1));
            const uint32_t w0 = (kb & 1) ? words[h].z : words[h].x;
            const uint32_t w1 = (kb & 1) ? words[h].w : words[h].y;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t byte = ((c < 4 ? w0 : w1) >> ((c & 3) * 8)) & 0xFFu;
              st_shared_v4(bt + sw128_offset((uint32_t)R, (uint32_t)c), pm1_octet(byte));
            }
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(bt + sw128_offset((uint32_t)R, (uint32_t)c), make_uint4(0, 0, 0, 0));
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_addr(&bar_full_b[s]));
    }

    // Epilogue: TMEM lane quarter (warp & 3) holds token rows 32·(warp & 3) + lane.
    // Warps 2-5 read sub-tile 0; with two sub-tiles, warps 6-9 (idle once the
    // sign tiles are built) read sub-tile 1 at the same time.
    // (the wait result is made warp-uniform: the TMEM loads are warp-collective)
    const int grp = (warp - 2) >> 2;
    const bool epi = MT == 2 || grp == 0;
    if (epi && __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_accum), 0, abort_p, a.err, kDevTimeoutAccum))) {
      tc_fence_after_sync();
      const int q = warp & 3;
      const int m = MT == 2 ? grp : 0;
      const int64_t t = t0 + m * kTileRows + q * 32 + lane;
      // rows of the last CTA's second sub-tile may lie past the P buffer
      const bool store = MT == 1 || t < a.ldp;
      const uint32_t lane_base = tmem + (uint32_t)(m * a.npt) + ((uint32_t)(q * 32) << 16);
      if constexpr (P16) {
        // fp16 form, per target and 16-token group of this warp: the group's
        // largest |P| (first pass over tensor memory, 16x256b loads whose four
        // threads of a quad share two tokens), then the scaled conversion
        // (second pass).  The fragments of a 16x256b load are the operands of
        // a transposing stmatrix: the blocks are assembled in their global
        // image (p16_half_bytes) in the idle pipeline buffers, and written out
        // below with one bulk copy per block.
        const uint32_t hn = (uint32_t)a.np / 2, hb = p16_half_bytes(a.np);
        const uint32_t blk_bytes = 2u * hb;
        const int tq = lane & 3, tr = lane >> 2;
        for (int tg = 0; tg < a.ntg; ++tg) {
          // target tg's 2·MT blocks, then the next target's
          const uint32_t tstage = x_base + (uint32_t)(tg * 2 * MT) * blk_bytes;
#pragma unroll 1
          for (int gs = 0; gs < 2; ++gs) {
            const uint32_t lb = tmem + (uint32_t)(m * a.npt + tg * a.np) + ((uint32_t)(q * 32 + gs * 16) << 16);
            float m0 = 0.f, m1 = 0.f;  // tokens tr and tr + 8 of the group
            for (int c0 = 0; c0 < a.np; c0 += 32) {
              uint32_t w[4][4];
              const int nb = min(4, (a.np - c0) / 8);
#pragma unroll
              for (int bb = 0; bb < 4; ++bb)
                if (bb < nb) tmem_ld_16x256b(lb + (uint32_t)(c0 + 8 * bb), w[bb]);
              tmem_wait_ld();
#pragma unroll
              for (int bb = 0; bb < 4; ++bb)
                if (bb < nb) {
                  m0 = fmaxf(m0, fmaxf(fabsf(__uint_as_float(w[bb][0])), fabsf(__uint_as_float(w[bb][1]))));
                  m1 = fmaxf(m1, fmaxf(fabsf(__uint_as_float(w[bb][2])), fabsf(__uint_as_float(w[bb][3]))));
                }
            }
            // the group's largest |P| (its 16 tokens are spread over the warp)
            float mg = fmaxf(m0, m1);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
            const int e0 = p16_exponent(mg), e1 = e0;
            const uint64_t inv0 = pack_f2(pow2f(-e0), pow2f(-e0)), inv1 = inv0;
            // block of this group within the CTA, and the group's first token in it
            const uint32_t bl = (uint32_t)(2 * m + (q >> 1));
            const uint32_t tt0 = (uint32_t)(32 * (q & 1) + 16 * gs);
            const uint32_t bstage = tstage + bl * blk_bytes;
            // stmatrix row address of this lane: matrix mi = lane / 8 holds
            // ranks +8·(mi >> 1), tokens +8·(mi & 1); row j = lane % 8 is a rank
            const int mi = lane >> 3, mj = lane & 7;
            const uint32_t chunk = (tt0 >> 3) + (uint32_t)(mi & 1);
            for (int c0 = 0; c0 < a.np; c0 += 16) {
              uint32_t wa[4], wb[4];
              tmem_ld_16x256b(lb + (uint32_t)c0, wa);
              tmem_ld_16x256b(lb + (uint32_t)(c0 + 8), wb);
              tmem_wait_ld();
              const uint32_t n = (uint32_t)(c0 + 8 * (mi >> 1) + mj);
              const uint32_t h = n >= hn ? 1u : 0u, nl = n - h * hn;
              stmatrix_x4_trans(bstage + h * hb + 256u + nl * 128u + ((chunk ^ (nl & 7u)) << 4),
                                half2_scaled(wa[0], wa[1], inv0), half2_scaled(wa[2], wa[3], inv1),
                                half2_scaled(wb[0], wb[1], inv0), half2_scaled(wb[2], wb[3], inv1));
            }
            if (tq == 0) {
              const uint32_t t_a = tt0 + (uint32_t)tr, t_b = t_a + 8u;
              st_shared_f32(bstage + 4u * t_a, pow2f(e0));
              st_shared_f32(bstage + hb + 4u * t_a, pow2f(e0));
              st_shared_f32(bstage + 4u * t_b, pow2f(e1));
              st_shared_f32(bstage + hb + 4u * t_b, pow2f(e1));
            }
          }
        }
      } else {
        // up to four 16-column loads in flight per wait; column c of the
        // accumulator is rank c % np of target c / np (np is a multiple of 16,
        // so a 16-column group never straddles two targets)
        for (int c0 = 0; c0 < a.npt; c0 += 64) {
          uint32_t v[4][16];
          const int nb = min(4, (a.npt - c0) / 16);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
            if (bb < nb) tmem_ld16(lane_base + (uint32_t)(c0 + 16 * bb), v[bb]);
          tmem_wait_ld();
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
            if (bb < nb) {
              const int tg = (c0 + 16 * bb) / a.np, n0 = c0 + 16 * bb - tg * a.np;
              __nv_bfloat16* phi = a.p_hi[tg];
              __nv_bfloat16* plo = a.p_lo[tg];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float x = __uint_as_float(v[bb][j]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
                const size_t off = (size_t)(n0 + j) * (size_t)a.ldp + (size_t)t;
                if (store) {
                  phi[off] = hi;
                  plo[off] = lo;
                }
              }
            }
        }
      }
    }
    if constexpr (P16) {
      // Every epilogue warp meets here (also after a failed wait), then one
      // thread writes the CTA's blocks that lie inside the P buffer (the last
      // CTA's second sub-tile may not), one bulk copy per block.
      if (epi) {
        fence_proxy_async_smem();
        named_barrier_sync(1, MT == 2 ? 256 : 128);
        if (threadIdx.x == 64 && !*abort_p) {
          const uint32_t blk_bytes = 2u * p16_half_bytes(a.np);
          const int64_t b0 = t0 / 64, nblk = a.ldp / 64;
          for (int tg = 0; tg < a.ntg; ++tg) {
            uint8_t* phv = reinterpret_cast<uint8_t*>(a.p_hi[0]);
#pragma unroll
            for (int j = 1; j < kMaxTargets; ++j)
              if (tg == j) phv = reinterpret_cast<uint8_t*>(a.p_hi[j]);
            for (int bl = 0; bl < 2 * MT; ++bl)
              if (b0 + bl < nblk)
                bulk_store(phv + (size_t)(b0 + bl) * blk_bytes, x_base + (uint32_t)(tg * 2 * MT + bl) * blk_bytes,
                           blk_bytes);
          }
          bulk_commit_group();
          bulk_wait_group0();
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (abort_flag) {
      // Make sure no MMA still targets the accumulator before freeing it.
      volatile int no_abort = 0;
      if (lane == 0) mbar_wait(smem_addr(&bar_accum), 0, &no_abort, a.err, kDevTimeoutTeardown);
      __syncwarp();
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

template <int MT, bool MULTI, bool P16>
__global__ void __launch_bounds__(kProjThreads, MT == 1 ? 2 : 1)
    project_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ ExtraOperands<MULTI> ops, const __grid_constant__ ProjectArgs a) {
  project_body<MT, MULTI, P16, false>(&tmap_x, &tmap_a, ops, a, (int)blockIdx.x);
}

// ----------------------------------------------------------------- contract
constexpr int kConThreads = 192;  // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue

struct ContractArgs {
  int64_t d;
  int r, np;
  int mt;  // 128-row sub-tiles of S per CTA (1 or 2); they share each P tile
  int tk;  // tokens per pipeline stage: 64 (P rows of 128 B) or 32 (64 B)
  int num_kb, kb_per_split, splits;
  int stages;
  uint32_t tmem_cols;
  float inv_sqrt_r;
  float* S;
  int64_t lds;
  int s_vec4;  // S rows can be updated with 16-byte accesses
  float* part;
  int64_t dp;
  unsigned int* err;
};

// S += (1/√r)·Σ_s part[s] for every element of S, the split partials added in
// ascending split order (so the result does not depend on which CTA of the
// contraction finished first).  One thread per 4 consecutive columns of a row.
// f: the thread's index over the d·np/4 column quadruples.
__device__ __forceinline__ void reduce_partials_body(const float* __restrict__ part, int splits, int64_t dp, int np,
                                                     int64_t d, int r, float inv_sqrt_r, float* __restrict__ S,
                                                     int64_t lds, int s_vec4, int64_t f) {
  const int q4 = np / 4;
  if (f >= d * q4) return;
  const int64_t row = f / q4;
  const int c = (int)(f % q4) * 4;
  const float4* src = reinterpret_cast<const float4*>(part) + f;
  const size_t stride = (size_t)dp * (size_t)q4;
  float4 acc = __ldcs(src);
#pragma unroll 8
  for (int sp = 1; sp < splits; ++sp) {
    const float4 v = __ldcs(src + (size_t)sp * stride);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  float* dst = S + row * lds + c;
  if (s_vec4 && c + 4 <= r) {
    float4 o = *reinterpret_cast<float4*>(dst);
    o.x += inv_sqrt_r * acc.x;
    o.y += inv_sqrt_r * acc.y;
    o.z += inv_sqrt_r * acc.z;
    o.w += inv_sqrt_r * acc.w;
    *reinterpret_cast<float4*>(dst) = o;
  } else {
    const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c + j < r) dst[j] += inv_sqrt_r * vv[j];
  }
}

__global__ void __launch_bounds__(256)
    reduce_partials_kernel(const float* __restrict__ part, int splits, int64_t dp, int np, int64_t d, int r,
                           float inv_sqrt_r, float* __restrict__ S, int64_t lds, int s_vec4) {
  reduce_partials_body(part, splits, dp, np, d, r, inv_sqrt_r, S, lds, s_vec4,
                       (int64_t)blockIdx.x * blockDim.x + threadIdx.x);
}

// TK: tokens per stage (64 or 32), MT: 128-row sub-tiles per CTA (1 or 2).
// Both are template parameters so that the single thread issuing the MMAs
// runs a fully unrolled loop on precomputed descriptors.
// The body runs for row tile `tile` and split `split`; tensor maps by
// pointer as in project_body.
template <int TK, int MT, bool GROUP>
__device__ __forceinline__ void contract_body(const CUtensorMap* tmap_dy, const CUtensorMap* tmap_phi,
                                              const CUtensorMap* tmap_plo, const ContractArgs& a, int tile,
                                              int split) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_accum;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t sub_bytes = 256u * TK;              // one sub-tile: two 64-column halves of TK tokens
  constexpr uint32_t dy_bytes = sub_bytes * MT;
  const uint32_t p_bytes = (uint32_t)a.np * 2u * TK;     // np rows × TK tokens
  const uint32_t stage_bytes = dy_bytes + 2 * p_bytes;
  const uint32_t base = smem_addr(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t d0 = (int64_t)tile * kTileRows * MT;
  const int kb_begin = split * a.kb_per_split;
  const int kb_end = min(a.num_kb, kb_begin + a.kb_per_split);
  const int nkb = kb_end - kb_begin;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&bar_full[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
    }
    mbar_init(smem_addr(&bar_accum), 1);
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

  if (warp == 0) {
    if (lane == 0) {
      if constexpr (GROUP) {
        tmap_acquire(tmap_dy);
        tmap_acquire(tmap_phi);
        tmap_acquire(tmap_plo);
      }
      tma_prefetch_desc(tmap_dy);
      tma_prefetch_desc(tmap_phi);
      tma_prefetch_desc(tmap_plo);
      int issued = 0;
      RingPos rp;
      for (int i = 0; i < nkb; ++i, rp.advance(a.stages)) {
        const int s = rp.s;
        const uint32_t ph = rp.ph;
        if (!mbar_wait(smem_addr(&bar_empty[s]), ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
        const uint32_t st = base + s * stage_bytes;
        const uint32_t fb = smem_addr(&bar_full[s]);
        const int32_t tk = (kb_begin + i) * TK;
        mbar_arrive_expect_tx(fb, stage_bytes);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          tma_load_2d(st + m * sub_bytes, tmap_dy, fb, (int32_t)(d0 + m * kTileRows), tk);
          tma_load_2d(st + m * sub_bytes + sub_bytes / 2, tmap_dy, fb, (int32_t)(d0 + m * kTileRows) + 64, tk);
        }
        tma_load_2d(st + dy_bytes, tmap_phi, fb, tk, 0);
        tma_load_2d(st + dy_bytes + p_bytes, tmap_plo, fb, tk, 0);
        issued = i + 1;
      }
      for (int i = (issued > a.stages ? issued - a.stages : 0); i < issued; ++i) {
        volatile int no_abort = 0;
        mbar_wait(smem_addr(&bar_full[i % a.stages]), (i / a.stages) & 1, &no_abort, a.err, kDevTimeoutTeardown);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the loop with warp-uniform waits; one elected lane
    // issues.
    // A = dYᵀ tile (M = 128 rows of S, K = tokens): MN-major, two 64-row
    // halves 8 KB apart (LBO), 8-token groups 1 KB apart (SBO).
    // B = Pᵀ tile (N = np, K = tokens): K-major.
    const uint32_t idesc = idesc_bf16_m128((uint32_t)a.np, 1, 0);
    // Descriptors of stage 0; a stage s adds (s·stage_bytes) >> 4 to the
    // start-address field (shared addresses stay below 2^18, so the 14-bit
    // field never carries).
    const uint64_t a0 = sdesc_sw128(base, sub_bytes / 2, 1024);
    const uint64_t h0 = TK == 64 ? sdesc_sw128(base + dy_bytes, 16, 1024) : sdesc_sw64(base + dy_bytes, 512);
    const uint64_t l0 = TK == 64 ? sdesc_sw128(base + dy_bytes + p_bytes, 16, 1024)
                                 : sdesc_sw64(base + dy_bytes + p_bytes, 512);
    const uint32_t step16 = stage_bytes >> 4;
    RingPos rp;
    for (int i = 0; i < nkb; ++i, rp.advance(a.stages)) {
      const int s = rp.s;
      const uint32_t ph = rp.ph;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_full[s]), ph, abort_p, a.err, kDevTimeoutTmaFull)))
        break;
      tc_fence_after_sync();
      const uint64_t off = (uint64_t)((uint32_t)s * step16);
#pragma unroll
      for (int ks = 0; ks < TK / 16; ++ks) {
        const uint64_t bh = h0 + off + (uint64_t)(ks * 2), bl = l0 + off + (uint64_t)(ks * 2);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint64_t ad = a0 + off + (uint64_t)(m * (sub_bytes >> 4) + ks * 128);
          const uint32_t d_tmem = tmem + (uint32_t)(m * a.np);
          warp_mma_bf16_ss(d_tmem, ad, bh, idesc, (i | ks) != 0);
          warp_mma_bf16_ss(d_tmem, ad, bl, idesc, 1);
        }
      }
      warp_mma_commit(smem_addr(&bar_empty[s]));
    }
    warp_mma_commit(smem_addr(&bar_accum));
  } else {
    // ---------------- epilogue (warps 2..5)
    // TMEM lane quarter (warp & 3) holds rows 32·(warp & 3) + lane of the
    // tile.  The accumulator is first staged row-major in shared memory (the
    // pipeline buffers are idle by now), so that every global access below is
    // a coalesced 16-byte stream over the contiguous 128 × np block.
    const int q = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int pitch = a.np + 4;       // floats; the pad spreads rows over banks
    float* stage = reinterpret_cast<float*>(smem);
    // the wait result is made warp-uniform: the TMEM loads are warp-collective
    const bool have =
        nkb > 0 && __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar_accum), 0, abort_p, a.err, kDevTimeoutAccum));
    if (have) tc_fence_after_sync();
    const int q4 = a.np / 4;          // float4 per row
    const int nvec = 128 * q4;        // float4 in one sub-tile
    for (int m = 0; m < MT; ++m) {
      const int64_t r0 = d0 + m * kTileRows;  // first row of S in this sub-tile
      if (m) named_barrier_sync(1, 128);      // the staging buffer is free again
      if (have) {
        float* srow = stage + (q * 32 + lane) * pitch;
        // up to four 16-column loads in flight per wait
        for (int c0 = 0; c0 < a.np; c0 += 64) {
          uint32_t v[4][16];
          const int nb = min(4, (a.np - c0) / 16);
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (b < nb) tmem_ld16(lane_base + (uint32_t)(m * a.np + c0 + 16 * b), v[b]);
          tmem_wait_ld();
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (b < nb) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4*>(srow + c0 + 16 * b + 4 * j) =
                    make_float4(__uint_as_float(v[b][4 * j]), __uint_as_float(v[b][4 * j + 1]),
                                __uint_as_float(v[b][4 * j + 2]), __uint_as_float(v[b][4 * j + 3]));
            }
        }
      }
      named_barrier_sync(1, 128);
      if (a.splits == 1) {
        if (have) {
          for (int f = et; f < nvec; f += 128) {
            const int row = f / q4, c = (f % q4) * 4;
            const int64_t grow = r0 + row;
            if (grow >= a.d) continue;
            const float4 v = *reinterpret_cast<const float4*>(stage + row * pitch + c);
            float* dst = a.S + grow * a.lds + c;
            if (a.s_vec4 && c + 4 <= a.r) {
              float4 o = *reinterpret_cast<float4*>(dst);
              o.x += a.inv_sqrt_r * v.x;
              o.y += a.inv_sqrt_r * v.y;
              o.z += a.inv_sqrt_r * v.z;
              o.w += a.inv_sqrt_r * v.w;
              *reinterpret_cast<float4*>(dst) = o;
            } else {
              const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (c + j < a.r) dst[j] += a.inv_sqrt_r * vv[j];
            }
          }
        }
      } else {
        // partial block of this (split, sub-tile): 128 × np floats, contiguous;
        // the split partials are summed by reduce_partials_kernel afterwards
        float4* pblk =
            reinterpret_cast<float4*>(a.part + ((size_t)split * (size_t)a.dp + (size_t)r0) * (size_t)a.np);
        for (int f = et; f < nvec; f += 128) {
          const int row = f / q4, c = (f % q4) * 4;
          pblk[f] = have ? *reinterpret_cast<const float4*>(stage + row * pitch + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (abort_flag && nkb > 0) {
      volatile int no_abort = 0;
      if (lane == 0) mbar_wait(smem_addr(&bar_accum), 0, &no_abort, a.err, kDevTimeoutTeardown);
      __syncwarp();
    }
    tc_fence_after_sync();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

template <int TK, int MT>
__global__ void __launch_bounds__(kConThreads, 2)
    contract_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_phi,
                    const __grid_constant__ CUtensorMap tmap_plo, const __grid_constant__ ContractArgs a) {
  contract_body<TK, MT, false>(&tmap_dy, &tmap_phi, &tmap_plo, a, (int)blockIdx.x, (int)blockIdx.y);
}

// ------------------------------------------------------------ contract (fp16)
// Above r = 64: S += (1/√r)·dYᵀP with P in fp16 and one MMA per 16 tokens.
//
// The projection stores P row by row (one row per token) as fp16(P·2^−e_t)
// and keeps g_t = 2^e_t (p16_exponent; one value per group of 16 tokens).
// Since dYᵀP = Σ_t dY_tᵀ P_t, moving g_t onto the token's dY row changes
// nothing: S = Σ_t (g_t·dY_t)ᵀ(P_t/g_t).
// kind::f16 MMAs take both operands in one type, so dY (bf16) becomes fp16 as
// well.  A bf16 value has 8 significant bits and fp16 11, so the conversion is
// exact wherever the value lands in fp16's normal range; what fp16 lacks is
// exponent range.  Each row d of the tile therefore carries its own
// power-of-two scale f_d, set from the first nonzero values the row meets so
// that their largest lands in [1, 2): the MMA sees fp16(g_t·dY_td·f_d) and the
// accumulator row holds f_d·S_d, divided out in the epilogue.  When a later
// value of the row would overflow fp16 under f_d, the row's scale is lowered
// to the 2^−⌊log₂ max⌋ of that block of tokens and its accumulator row is
// multiplied by the ratio — exact for a power of two — once every MMA issued
// so far has completed.  Values more than 2^24 below the row's scale lose
// relative precision in fp16's subnormal range; their share of ‖S_d‖ is then
// below 2^−24 of the row's largest term.
//
// The kernel runs as CTA pairs (clusters of two, cta_group::2): a pair owns
// 256 rows of S, 128 per CTA, and every MMA (M = 256, N = np) is issued by
// the even CTA for both.  Each CTA converts and holds the A operand of its own
// rows and keeps its own accumulator rows, while the Pᵀ tile (the B operand)
// is split by N between the two CTAs' shared memory.  Measured on GB300, the
// copy engine's latency caps what one SM can stream; a lone CTA needed about
// 96 bytes per tensor cycle (the full Pᵀ tile for 128 rows), the pair needs 64.
//
// Roles in each CTA (576 threads, one CTA per SM):
//   warp 0     TMA: per stage of 64 tokens, the dY tile [64 tokens × 128 rows]
//              as two 64-row boxes (128-byte swizzle), and with one bulk copy
//              this CTA's half of the stage's Pᵀ block (np/2 rows × 64 tokens,
//              K-major, already in the swizzled image the MMA reads) preceded
//              by its 64 token scales, all on one stage barrier;
//   warp 1     even CTA: the MMAs, D[256 × np] += A·Pᵀ_tile with A (the
//              converted dY of both CTAs) in tensor memory, four K = 16 steps
//              per stage, commits arriving on the barriers of both CTAs;
//              odd CTA: forwards its conversion warps' completion of each step
//              to the even CTA in one remote arrival;
//   warps 2-17 conversion, four warps per tensor-memory lane quarter, in
//              steps of two stages (128 tokens): warp (q, gq, j) owns rows
//              32q + 16gq .. + 15 of stage j of each step: ldmatrix.trans of
//              its bf16 tile, scaling, fp16 packing and tcgen05.st into one of
//              two A buffers of tensor memory (64 columns each, after the
//              accumulator), then one local arrival; then the epilogue.  The
//              two warps of a row group (j = 0, 1) hold the same row scales: a
//              barrier vote per step sends both to the slow path together,
//              where they combine their row maxima through shared memory and
//              reach the same decision.  Four conversion warps per scheduler
//              (instead of two) keep enough independent work in flight:
//              measured on GB300, two left the MMAs waiting on conversion; a
//              variant with eight warps, each converting both stages of its
//              rows (no vote), measured 4 % slower.
// Measured on GB300: an arrival through a shared::cluster address costs the
// arriving thread several hundred cycles even on its own CTA's barrier, so
// every conversion warp arrives locally and only the forwarder crosses CTAs.
// The conversion takes the speculative path: convert under the current row
// scales and look for an infinity among the results (a packed max of the fp16
// magnitudes).  Only a row without a scale that meets nonzero values, or an
// overflow, sends the warp to the slow path that takes the rows' maxima.
// The dY tile crosses shared memory once (TMA write, ldmatrix read) and the
// MMAs read only the P tile from it.
constexpr int kC16Tk = 64;          // tokens per TMA stage
constexpr int kC16MaxStages = 12;
constexpr int kC16Step = 2;         // stages per conversion step
constexpr int kC16ABufs = 2;        // A buffers (one conversion step each)
constexpr uint32_t kC16ACol = 256;  // first tensor-memory column of the A buffers
constexpr uint32_t kC16ABufCols = kC16Step * kC16Tk / 2;  // 64 columns: 128 fp16 tokens per row
constexpr int kC16Threads = 576;
constexpr int kC16Conv = 512;       // conversion threads (warps 2-17)
constexpr int kC16ConvWarps = 16;

struct Contract16Args {
  int64_t d;
  int r, np;
  int num_kb, kb_per_split, splits;
  int stages;
  float inv_sqrt_r;
  float* S;
  int64_t lds;
  int s_vec4;
  float* part;
  int64_t dp;
  const uint8_t* p16;  // Pᵀ blocks of 64 tokens (two halves of p16_half_bytes(np) each)
  unsigned int* err;
};


// 2^−⌊log₂ m⌋ for a positive finite m, held in [2^−126, 2^126].
__device__ __forceinline__ float row_scale_for(float m) {
  const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  return pow2f(max(-126, min(126, -E)));
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Running maximum of fp16 magnitudes, two lanes at once: the magnitude bits
// of the result are max(|acc|, |v|) per half, a NaN in either propagates
// (max.NaN.xorsign.abs.f16x2; the sign bits of the result are not used).
__device__ __forceinline__ uint32_t hmax_abs2(uint32_t acc, uint32_t v) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(v));
  return r;
}

// A bf16 pair (low half: the even token) times its scale g·f (the packed
// operand of mul.f32x2, the same value twice), rounded once to an fp16 pair:
// two instructions to widen, one packed multiply, one packed conversion.
__device__ __forceinline__ uint32_t convert_pair(uint32_t x, uint64_t gf) {
  uint64_t v, p;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(x << 16), "r"(x & 0xFFFF0000u));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(v), "l"(gf));
  uint32_t h;
  asm("{\n\t.reg .f32 a, b;\n\tmov.b64 {a, b}, %1;\n\tcvt.rn.f16x2.f32 %0, b, a;\n\t}" : "=r"(h) : "l"(p));
  return h;
}

// The body runs for row tile `tile` (even on the CTA of rank 0, the next one
// on its peer) and split `split`; the dY tensor map by pointer as in
// project_body.
template <bool GROUP>
__device__ __forceinline__ void contract16_body(const CUtensorMap* tmap_dy, const Contract16Args& a, int tile,
                                                int split) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kC16MaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kC16MaxStages];
  __shared__ __align__(8) uint64_t bar_afull[kC16ABufs];  // even CTA: the pair's A buffers are written
  __shared__ __align__(8) uint64_t bar_afwd[kC16ABufs];   // odd CTA: its own conversion warps are done
  __shared__ __align__(8) uint64_t bar_aempty[kC16ABufs];
  __shared__ __align__(8) uint64_t bar_accum;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float row_max_xch[8][2][16];  // slow path: [row group][stage of the step][row]

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t dy_box = 128u * kC16Tk;   // one 64-row box: TK tokens × 128 bytes
  constexpr uint32_t dy_bytes = 2 * dy_box;
  // stage: dY boxes, 1 KB whose last 256 bytes hold the token scales, then
  // this CTA's Pᵀ half (np/2 rows of 128 bytes), every part 1024-byte aligned
  const uint32_t half_bytes = p16_half_bytes(a.np);
  const uint32_t p_off = dy_bytes + 1024u;
  const uint32_t stage_bytes = p_off + (((uint32_t)a.np * 64u + 1023u) & ~1023u);
  const uint32_t base = smem_addr(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the pair's MMAs
  const int64_t d0 = (int64_t)tile * kTileRows;
  const int kb_begin = split * a.kb_per_split;
  const int kb_end = min(a.num_kb, kb_begin + a.kb_per_split);
  const int nkb = kb_end - kb_begin;
  const int nsteps = (nkb + kC16Step - 1) / kC16Step;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_addr(&bar_full[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
    }
    for (int b = 0; b < kC16ABufs; ++b) {
      // even CTA: one arrival per conversion warp of its own, one from the
      // odd CTA's forwarder; odd CTA: one per conversion warp of its own
      mbar_init(smem_addr(&bar_afull[b]), kC16ConvWarps + 1);
      mbar_init(smem_addr(&bar_afwd[b]), kC16ConvWarps);
      mbar_init(smem_addr(&bar_aempty[b]), 1);
    }
    mbar_init(smem_addr(&bar_accum), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();  // both CTAs' barriers exist before the first arrival from the peer
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      if constexpr (GROUP) tmap_acquire(tmap_dy);
      tma_prefetch_desc(tmap_dy);
      int issued = 0;
      RingPos rp;
      for (int i = 0; i < nkb; ++i, rp.advance(a.stages)) {
        const int s = rp.s;
        const uint32_t ph = rp.ph;
        if (!mbar_wait_sleep(smem_addr(&bar_empty[s]), ph ^ 1, abort_p, a.err, kDevTimeoutStageFree)) break;
        const uint32_t st = base + s * stage_bytes;
        const uint32_t fb = smem_addr(&bar_full[s]);
        const int32_t tk = (kb_begin + i) * kC16Tk;
        mbar_arrive_expect_tx(fb, dy_bytes + half_bytes);
        tma_load_2d(st, tmap_dy, fb, (int32_t)d0, tk);
        tma_load_2d(st + dy_box, tmap_dy, fb, (int32_t)d0 + 64, tk);
        // this CTA's half of the stage's block: scales, then its Pᵀ rows
        bulk_load(st + p_off - 256u, a.p16 + ((size_t)(kb_begin + i) * 2u + rank) * half_bytes, half_bytes, fb);
        issued = i + 1;
      }
      for (int i = (issued > a.stages ? issued - a.stages : 0); i < issued; ++i) {
        volatile int no_abort = 0;
        mbar_wait_sleep(smem_addr(&bar_full[i % a.stages]), (i / a.stages) & 1, &no_abort, a.err, kDevTimeoutTeardown);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
    // The whole warp runs the loop with warp-uniform waits; one elected lane
    // issues.  Per conversion step: wait for the A buffers of both CTAs, then
    // per stage wait for this CTA's Pᵀ half (the peer's half is in place once
    // the peer's conversion warps have arrived: they waited for its stage),
    // issue two MMAs and release the stage in both CTAs; then release the A
    // buffers.
    const uint32_t idesc = idesc_f16_m256((uint32_t)a.np);
    const uint64_t b0 = sdesc_sw128(base + p_off, 16, 1024);
    const uint32_t step16 = stage_bytes >> 4;
    bool ok = true;
    RingPos rp;
    for (int n = 0; n < nsteps && ok; ++n) {
      const int b = n % kC16ABufs;
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_afull[b]), (n / kC16ABufs) & 1, abort_p, a.err,
                                                     kDevTimeoutOperand)))
        break;
      tc_fence_after_sync();
      const int ns = min(kC16Step, nkb - n * kC16Step);
      for (int j = 0; j < ns; ++j, rp.advance(a.stages)) {
        const int i = n * kC16Step + j, s = rp.s;
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_full[s]), rp.ph, abort_p, a.err,
                                                     kDevTimeoutTmaFull))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t bo = b0 + (uint64_t)((uint32_t)s * step16);
        const uint32_t at = tmem + kC16ACol + (uint32_t)b * kC16ABufCols + (uint32_t)(j * (kC16Tk / 2));
#pragma unroll
        for (int ks = 0; ks < kC16Tk / 16; ++ks)
          warp_mma_pair_ts(tmem, at + (uint32_t)(ks * 8), bo + (uint64_t)(ks * 2), idesc, (i | ks) != 0);
        warp_mma_commit_pair(smem_addr(&bar_empty[s]));
      }
      warp_mma_commit_pair(smem_addr(&bar_aempty[b]));
    }
    warp_mma_commit_pair(smem_addr(&bar_accum));
    } else {
      // Odd CTA: forward the completion of its conversion warps' A buffers
      // to the even CTA in one arrival per step (one remote arrival from
      // each warp cost every warp several hundred cycles per step).
      const uint32_t afull0 = map_to_cta(smem_addr(&bar_afull[0]), 0);
      for (int n = 0; n < nsteps; ++n) {
        const int b = n % kC16ABufs;
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_afwd[b]), (n / kC16ABufs) & 1, abort_p, a.err,
                                                     kDevTimeoutOperand)))
          break;
        if (lane == 0) mbar_arrive_remote(afull0 + (uint32_t)(b * 8));
      }
    }
  } else {
    // ---------------- conversion (warps 2..17), then the epilogue
    // Warp (q, gq, jw) owns rows 32q + 16gq .. + 15 of the tile (tensor-memory
    // lanes) in stage jw of each step.  In the ldmatrix fragments of a
    // 16-token group h of a stage, thread t holds rows t/4 (registers 0, 2)
    // and t/4 + 8 (registers 1, 3) of those 16, tokens 16h + 2(t%4) + {0, 1}
    // (registers 0, 1) and 16h + 8 + 2(t%4) + {0, 1} (registers 2, 3), as
    // (even, odd) bf16 pairs: exactly the layout of tcgen05.st.16x128b.x2 for
    // 16 lanes × 8 columns.  Thread t's rows, j = 0 and 1, are 16gq + t/4 + 8j;
    // the quad t & ~3 shares each row.
    const int q = warp & 3, u4 = (warp - 2) >> 2, gq = u4 & 1, jw = u4 >> 1;
    const int grp = q * 2 + gq;               // row group: named barrier 2 + grp
    const int tq = lane & 3, tr = lane >> 2;
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
    const uint32_t lane16 = ((uint32_t)(q * 32 + gq * 16)) << 16;
    // where this warp reports its A buffer: the even CTA's own barrier, or the
    // odd CTA's forwarding barrier (both local)
    const uint32_t abar0 = rank == 0 ? smem_addr(&bar_afull[0]) : smem_addr(&bar_afwd[0]);
    float f[2] = {0.f, 0.f};  // row scales f_d of rows j = 0, 1; 0 = not set yet (the same in both warps of the group)
    bool any_unset = true;    // some row of this group has no scale yet
    bool alive = true;
    // this lane's ldmatrix row address inside a stage, for the token groups h
    uint32_t lm_off[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int token = 16 * h + 8 * (mi >> 1) + mr;
      const int dcol = 32 * q + 16 * gq + 8 * (mi & 1);
      lm_off[h] = (uint32_t)(dcol >> 6) * dy_box + sw128_offset((uint32_t)token, (uint32_t)((dcol & 63) >> 3));
    }
    RingPos rp;  // the ring position of this warp's stage, i = n·kC16Step + jw
    rp.s = jw;
    for (int n = 0; n < nsteps; ++n, rp.advance_by(kC16Step, a.stages)) {
      const int b = n % kC16ABufs;
      const int i = n * kC16Step + jw;  // this warp's stage
      const bool mine = i < nkb;
      uint32_t x[4][4] = {};  // [16-token group h][register]
      float g[4];             // [h]: the scale of token group h
      // (No early exit from this loop: the two warps of a group meet at a named
      // barrier every step, so a warp whose wait failed keeps taking part in
      // the votes, with its work skipped, until the loop ends.)
      if (mine && alive) {
        const int s = rp.s;
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_full[s]), rp.ph, abort_p, a.err,
                                                kDevTimeoutTmaFull)))
          alive = false;
        if (alive) {
          const uint32_t st = base + (uint32_t)s * stage_bytes;
          const uint32_t gs = st + p_off - 256u;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            g[h] = ld_shared_f32(gs + (uint32_t)(16 * h) * 4u);
            ldmatrix_x4_trans(st + lm_off[h], x[h][0], x[h][1], x[h][2], x[h][3]);
          }
        }
      }
      if (!mine || !alive) {
#pragma unroll
        for (int h = 0; h < 4; ++h) g[h] = 0.f;
      }
      // speculative conversion under the current scales (1 for a row without one)
      uint32_t o[4][4];
      uint32_t vmax = 0u, nz_unset = 0u;
      {
        const float f0 = f[0] == 0.f ? 1.f : f[0], f1 = f[1] == 0.f ? 1.f : f[1];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float s0 = g[h] * f0, s1 = g[h] * f1;
          const uint64_t gf0 = pack_f2(s0, s0), gf1 = pack_f2(s1, s1);
#pragma unroll
          for (int rg = 0; rg < 4; ++rg) {
            o[h][rg] = convert_pair(x[h][rg], (rg & 1) ? gf1 : gf0);
            vmax = hmax_abs2(vmax, o[h][rg]);
          }
        }
        if (any_unset) {
#pragma unroll
          for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int rg = 0; rg < 4; ++rg)
              if (f[rg & 1] == 0.f) nz_unset |= x[h][rg] & 0x7FFF7FFFu;
        }
      }
      // an infinity (or NaN) among the results, or a value met by a row without
      // a scale, in either warp of the group (or a failed wait) sends both to
      // the slow path
      const bool slow_w = (vmax & 0x7FFFu) >= 0x7C00u || ((vmax >> 16) & 0x7FFFu) >= 0x7C00u || nz_unset != 0u ||
                          !alive;
      if (named_barrier_any(2 + grp, 64, slow_w)) {
        // ---- slow path: the rows' largest finite |g·dY| over the step (both stages)
        float m[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int rg = 0; rg < 4; ++rg) {
            const float2 xv = bf16x2_to_float2(x[h][rg]);
            const float a0 = fabsf(xv.x * g[h]), a1 = fabsf(xv.y * g[h]);
            if (a0 <= 3.4028235e38f) m[rg & 1] = fmaxf(m[rg & 1], a0);
            if (a1 <= 3.4028235e38f) m[rg & 1] = fmaxf(m[rg & 1], a1);
          }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], 1));
          m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], 2));
          if (tq == 0) row_max_xch[grp][jw][tr + 8 * j] = m[j];
        }
        named_barrier_sync(2 + grp, 64);
#pragma unroll
        for (int j = 0; j < 2; ++j) m[j] = fmaxf(m[j], row_max_xch[grp][jw ^ 1][tr + 8 * j]);
        bool resc = false;
        float rho[2] = {1.f, 1.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (m[j] > 0.f) {
            if (f[j] == 0.f) {
              f[j] = row_scale_for(m[j]);
            } else if (m[j] * f[j] >= 32768.f) {
              const float fn = row_scale_for(m[j]);
              rho[j] = fn / f[j];
              f[j] = fn;
              resc = true;
            }
          }
        }
        any_unset = __any_sync(0xffffffffu, f[0] == 0.f || f[1] == 0.f);
        // Lower the scale of those accumulator rows (the stage-0 warp of the
        // group): wait for every MMA issued so far (those of the steps before
        // this one) to complete, then multiply the 16 rows by their ratio (1
        // for the others).  The MMAs of this step wait for this warp's arrival.
        if (jw == 0 && __any_sync(0xffffffffu, resc) && alive) {
          if (n > 0 && !__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_aempty[(n - 1) % kC16ABufs]),
                                                           ((n - 1) / kC16ABufs) & 1, abort_p, a.err,
                                                           kDevTimeoutAccum)))
            alive = false;
          if (alive) {
            tc_fence_after_sync();
            for (int c0 = 0; c0 < a.np; c0 += 32) {
              uint32_t w[4][4];
              const int nb = min(4, (a.np - c0) / 8);
#pragma unroll
              for (int bb = 0; bb < 4; ++bb)
                if (bb < nb) tmem_ld_16x256b(tmem + lane16 + (uint32_t)(c0 + 8 * bb), w[bb]);
              tmem_wait_ld();
#pragma unroll
              for (int bb = 0; bb < 4; ++bb)
                if (bb < nb) {
#pragma unroll
                  for (int e = 0; e < 4; ++e) w[bb][e] = __float_as_uint(__uint_as_float(w[bb][e]) * rho[e >> 1]);
                  tmem_st_16x256b(tmem + lane16 + (uint32_t)(c0 + 8 * bb), w[bb]);
                }
            }
            tmem_wait_st();
          }
        }
        // reconvert under the new scales
        const float g0 = f[0] == 0.f ? 1.f : f[0], g1 = f[1] == 0.f ? 1.f : f[1];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float s0 = g[h] * g0, s1 = g[h] * g1;
          const uint64_t gf0 = pack_f2(s0, s0), gf1 = pack_f2(s1, s1);
#pragma unroll
          for (int rg = 0; rg < 4; ++rg) o[h][rg] = convert_pair(x[h][rg], (rg & 1) ? gf1 : gf0);
        }
      }
      // fp16 A operand into buffer b (free once the MMAs of the step that used
      // it before have completed): this warp's 16 lanes, stage jw, token group
      // h = columns 32jw + 8h of the buffer
      if (alive && n >= kC16ABufs &&
          !__all_sync(0xffffffffu, mbar_wait_sleep(smem_addr(&bar_aempty[b]), ((n / kC16ABufs) - 1) & 1, abort_p, a.err,
                                              kDevTimeoutStageFree)))
        alive = false;
      if (alive) {
        tc_fence_after_sync();
        if (mine) {
#pragma unroll
          for (int h = 0; h < 4; h += 2)
            tmem_st_16x128b_x4(tmem + lane16 + kC16ACol + (uint32_t)b * kC16ABufCols + (uint32_t)(32 * jw + 8 * h),
                               o[h][0], o[h][1], o[h][2], o[h][3], o[h + 1][0], o[h + 1][1], o[h + 1][2],
                               o[h + 1][3]);
          tmem_wait_st();
        }
        // (the shared-memory reads of the stage completed with the loads that
        // fed the conversion; the stage is refilled only after the MMAs that
        // wait for this arrival)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(abar0 + (uint32_t)(b * 8));
      }
    }

    // ---------------- epilogue: D/f_d staged row-major in shared memory, then
    // coalesced into S (one split) or the split's partial block
    const int et = threadIdx.x - 64;  // 0..511
    const int pitch = a.np + 8;       // floats; rows 8 banks apart
    float* stage = reinterpret_cast<float*>(smem);
    const bool have = alive && nkb > 0 &&
                      __all_sync(0xffffffffu,
                                 mbar_wait_sleep(smem_addr(&bar_accum), 0, abort_p, a.err, kDevTimeoutAccum));
    if (have) tc_fence_after_sync();
    // every stage buffer is idle once the last MMA has completed; the staging
    // below overwrites them, so all eight warps must be past their waits
    named_barrier_sync(1, kC16Conv);
    const int q4 = a.np / 4;
    const int nvec = 128 * q4;
    if (have) {
      const float inv0 = f[0] == 0.f ? 1.f : 1.f / f[0], inv1 = f[1] == 0.f ? 1.f : 1.f / f[1];  // exact
      const int row0 = q * 32 + gq * 16 + (lane >> 2);
      // the two warps of a row group take one half of the columns each
      const int cbeg = jw * (a.np / 2), cend = cbeg + a.np / 2;
      for (int c0 = cbeg; c0 < cend; c0 += 32) {
        uint32_t w[4][4];
        const int nb = min(4, (cend - c0) / 8);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          if (bb < nb) tmem_ld_16x256b(tmem + lane16 + (uint32_t)(c0 + 8 * bb), w[bb]);
        tmem_wait_ld();
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          if (bb < nb) {
            const int c = c0 + 8 * bb + 2 * tq;
            *reinterpret_cast<float2*>(stage + row0 * pitch + c) =
                make_float2(__uint_as_float(w[bb][0]) * inv0, __uint_as_float(w[bb][1]) * inv0);
            *reinterpret_cast<float2*>(stage + (row0 + 8) * pitch + c) =
                make_float2(__uint_as_float(w[bb][2]) * inv1, __uint_as_float(w[bb][3]) * inv1);
          }
      }
    }
    named_barrier_sync(1, kC16Conv);
    if (a.splits == 1) {
      if (have) {
        for (int fi = et; fi < nvec; fi += kC16Conv) {
          const int row = fi / q4, c = (fi % q4) * 4;
          const int64_t grow = d0 + row;
          if (grow >= a.d) continue;
          const float4 vv = *reinterpret_cast<const float4*>(stage + row * pitch + c);
          float* dst = a.S + grow * a.lds + c;
          if (a.s_vec4 && c + 4 <= a.r) {
            float4 ov = *reinterpret_cast<float4*>(dst);
            ov.x += a.inv_sqrt_r * vv.x;
            ov.y += a.inv_sqrt_r * vv.y;
            ov.z += a.inv_sqrt_r * vv.z;
            ov.w += a.inv_sqrt_r * vv.w;
            *reinterpret_cast<float4*>(dst) = ov;
          } else {
            const float va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (c + j < a.r) dst[j] += a.inv_sqrt_r * va[j];
          }
        }
      }
    } else {
      float4* pblk = reinterpret_cast<float4*>(a.part + ((size_t)split * (size_t)a.dp + (size_t)d0) * (size_t)a.np);
      for (int fi = et; fi < nvec; fi += kC16Conv) {
        const int row = fi / q4, c = (fi % q4) * 4;
        pblk[fi] = have ? *reinterpret_cast<const float4*>(stage + row * pitch + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  // No MMA of the pair may still target either CTA's tensor memory when it
  // is freed: the even CTA's MMA warp waits for its last commit after an
  // abort; then both CTAs meet and free the pair's allocation together.
  if (warp == 1 && rank == 0 && abort_flag && nkb > 0) {
    volatile int no_abort = 0;
    if (lane == 0) mbar_wait_sleep(smem_addr(&bar_accum), 0, &no_abort, a.err, kDevTimeoutTeardown);
    __syncwarp();
  }
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, 512);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kC16Threads, 1)
    contract16_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ Contract16Args a) {
  contract16_body<false>(&tmap_dy, a, (int)blockIdx.x, (int)blockIdx.y);
}

uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < (uint32_t)n) c <<= 1;
  return c;
}

// ------------------------------------------------------------ group plan
// A group plan sketches many matrices with one launch per phase
// (logra_sketch_accumulate_group): the projections of all of them, then the
// contractions, then the split reduces.  Layout: a header; for each phase the
// first CTA of every matrix in the phase's launch order (begin[0..n]) and the
// matrix at each position of that order (order[0..n−1]); then one entry per
// matrix with its tensor maps and the arguments of the per-matrix kernels.
// A CTA finds its position with plan_find and its matrix through order.
constexpr uint32_t kSketchPlanMagic = 0x4C475350u;  // "LGSP"
constexpr size_t kSketchPlanHeaderBytes = 128;

struct SketchPlanHeader {
  uint32_t magic;
  int32_t n, r, np, p16;
  int32_t proj_ctas, con_ctas, red_blocks;
  int32_t proj_mt;
  uint32_t proj_smem, con_smem;
  uint64_t ws_bytes;
};
static_assert(sizeof(SketchPlanHeader) <= kSketchPlanHeaderBytes, "plan header");

struct alignas(128) SketchEntry {
  CUtensorMap tx, ta, tdy, tph, tpl;
  ProjectArgs pa;
  ContractArgs ca;      // bf16 contraction (np ≤ 64); the split reduce of both forms
  Contract16Args c16;   // fp16 contraction (np > 64)
  int32_t d_tiles;
  int32_t proj_ctas, con_ctas, red_blocks;
};

__host__ __device__ inline size_t plan_array_bytes(int count) { return ((size_t)count * 4 + 127) / 128 * 128; }
// phase 0: projection, 1: contraction, 2: reduce
__host__ __device__ inline size_t plan_begin_offset(int n, int phase) {
  return kSketchPlanHeaderBytes + (size_t)phase * (plan_array_bytes(n + 1) + plan_array_bytes(n));
}
__host__ __device__ inline size_t plan_order_offset(int n, int phase) {
  return plan_begin_offset(n, phase) + plan_array_bytes(n + 1);
}
__host__ __device__ inline size_t plan_entry_offset(int n) { return plan_begin_offset(n, 3); }

// The entry of this CTA in a phase and the CTA's index among that matrix's CTAs.
__device__ __forceinline__ const SketchEntry* group_entry(const uint8_t* __restrict__ plan, int n, int phase,
                                                          int* local) {
  const int32_t* begin = reinterpret_cast<const int32_t*>(plan + plan_begin_offset(n, phase));
  const int m = plan_find(begin, n);
  const int j = __ldg(reinterpret_cast<const int32_t*>(plan + plan_order_offset(n, phase)) + m);
  *local = (int)blockIdx.x - __ldg(begin + m);
  return reinterpret_cast<const SketchEntry*>(plan + plan_entry_offset(n)) + j;
}

template <int MT, bool P16>
__global__ void __launch_bounds__(kProjThreads, MT == 1 ? 2 : 1)
    project_group_kernel(const uint8_t* __restrict__ plan, int n, unsigned int* err) {
  __shared__ __align__(16) ProjectArgs sa;
  int local;
  const SketchEntry* e = group_entry(plan, n, 0, &local);
  copy_record_to_shared(&sa, &e->pa);
  __syncthreads();
  if (threadIdx.x == 0) sa.err = err;  // the plan holds no device error word
  __syncthreads();
  project_body<MT, false, P16, true>(&e->tx, &e->ta, ExtraOperands<false>{}, sa, local);
}

__global__ void __launch_bounds__(kConThreads, 2)
    contract_group_kernel(const uint8_t* __restrict__ plan, int n, unsigned int* err) {
  __shared__ __align__(16) ContractArgs sa;
  int local;
  const SketchEntry* e = group_entry(plan, n, 1, &local);
  copy_record_to_shared(&sa, &e->ca);
  const int d_tiles = __ldg(&e->d_tiles);
  __syncthreads();
  if (threadIdx.x == 0) sa.err = err;
  __syncthreads();
  contract_body<64, 1, true>(&e->tdy, &e->tph, &e->tpl, sa, local % d_tiles, local / d_tiles);
}

// The CTA pairs of the fp16 contraction: every matrix has an even number of
// CTAs (d_tiles is even) and starts at an even CTA, so the two CTAs of a
// cluster land on one matrix, rank 0 on the even row tile, in one split.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kC16Threads, 1)
    contract16_group_kernel(const uint8_t* __restrict__ plan, int n, unsigned int* err) {
  __shared__ __align__(16) Contract16Args sa;
  int local;
  const SketchEntry* e = group_entry(plan, n, 1, &local);
  copy_record_to_shared(&sa, &e->c16);
  const int d_tiles = __ldg(&e->d_tiles);
  __syncthreads();
  if (threadIdx.x == 0) sa.err = err;
  __syncthreads();
  contract16_body<true>(&e->tdy, sa, local % d_tiles, local / d_tiles);
}

__global__ void __launch_bounds__(256) reduce_group_kernel(const uint8_t* __restrict__ plan, int n) {
  __shared__ __align__(16) ContractArgs sa;
  int local;
  const SketchEntry* e = group_entry(plan, n, 2, &local);
  copy_record_to_shared(&sa, &e->ca);
  __syncthreads();
  reduce_partials_body(sa.part, sa.splits, sa.dp, sa.np, sa.d, sa.r, sa.inv_sqrt_r, sa.S, sa.lds, sa.s_vec4,
                       (int64_t)local * blockDim.x + threadIdx.x);
}

}  // namespace

SketchPlan plan_sketch(int64_t T, int64_t d, int64_t k, int r) {
  SketchPlan p{};
  p.T = T;
  p.d = d;
  p.k = k;
  p.r = r;
  p.np = (int)round_up(r, 16);
  // Above r = 64 the contraction is bound by the tensor pipe rather than by
  // HBM, and P travels as fp16 (11 significant bits, one MMA per step) with a
  // power-of-two scale per token instead of as a bf16 hi + lo pair (two MMAs).
  // Up to r = 64 the step is HBM-bound and keeps the bf16 pair.
  p.p16 = p.np > 64 ? 1 : 0;
  p.mt = 1;
  p.ldp = round_up(T > 0 ? T : 1, kTileRows);
  // the fp16 contraction runs as CTA pairs of two 128-row tiles
  p.dp = round_up(d > 0 ? d : 1, p.p16 ? 2 * kTileRows : kTileRows * p.mt);
  p.d_tiles = (int)(p.dp / (kTileRows * p.mt));
  // Tokens per contraction stage (both forms): 64.
  p.tk = 64;
  p.num_kb_t = (int)((T + p.tk - 1) / p.tk);
  // Split T into ranges whose partial sums are written and read back once,
  // keeping them below half of the dY bytes of the call.  Depends on the
  // shape only, so the summation order never depends on the device.
  // Target ≈ 48 contraction CTAs per matrix when two fit on an SM (r ≤ 64)
  // and ≈ 16 when one does: matrices are sketched several at a time (one
  // grouped launch over a model's matrices, or calls on a few streams), which
  // fill the GPU together, and every split saved is a partial sum that is
  // neither written nor read back (at r = 256 a split of a q projection costs
  // as much HBM traffic as a sixth of its dY).  At r = 256, 16 instead of 32
  // leaves only the 512-row k and v projections of the 7B set split, and took
  // its sketch pass from 18.09 to 17.79 ms per micro-batch.  A lone call on an
  // idle GPU leaves SMs free.
  const int64_t target = p.p16 ? 16 : 48;
  int64_t splits = (target + p.d_tiles - 1) / p.d_tiles;
  const int64_t cap = (T * d * 2) / (2 * p.dp * p.np * 4);
  if (splits > cap) splits = cap;
  if (splits > p.num_kb_t) splits = p.num_kb_t;
  if (splits < 1) splits = 1;
  p.kb_per_split = (int)((p.num_kb_t + splits - 1) / splits);
  if (p.kb_per_split < 1) p.kb_per_split = 1;
  p.splits = p.num_kb_t > 0 ? (int)((p.num_kb_t + p.kb_per_split - 1) / p.kb_per_split) : 1;
  const size_t pbytes = align256((size_t)p.np * (size_t)p.ldp * 2);
  p.off_phi = 0;
  p.off_plo = pbytes;
  // fp16 blocks: ldp/64 blocks of two halves (p16_half_bytes); the bf16 pair: two [np][ldp] arrays
  p.off_part = p.p16 ? align256((size_t)(p.ldp / 64) * 2 * p16_half_bytes(p.np)) : 2 * pbytes;
  const size_t part = p.splits > 1 ? align256((size_t)p.splits * (size_t)p.dp * (size_t)p.np * 4) : 0;
  p.bytes = p.off_part + part;
  return p;
}

namespace {

// Launch shape of the projection for npt stacked rows.  Two CTAs share an SM
// (≤ 112 KB of shared memory, ≤ 256 tensor-memory columns each) whenever an
// X tile and a B tile fit three times, so one CTA's prologue and epilogue
// overlap the other's streaming; otherwise one CTA per SM, which covers 256
// tokens when the stacked rows fit twice in tensor memory.  Sign tiles built
// on chip (own_b) take two B slots and the rest of the budget holds X tiles;
// given operands travel with the X tiles, one B slot per X slot.
struct ProjConfig {
  int mt, stages, b_stages;
  uint32_t tmem_cols, smem;
};
ProjConfig proj_config(int npt, bool own_b) {
  ProjConfig c{};
  const uint32_t b_bytes = (uint32_t)npt * 128u;
  const bool two_per_sm = npt <= 256 && (kSmemTwoPerSm - 1024) / (kTileRows * 128u + b_bytes) >= 3;
  c.mt = !two_per_sm && npt <= 256 ? 2 : 1;
  const uint32_t x_bytes = kTileRows * 128u * (uint32_t)c.mt;
  const uint32_t budget = (two_per_sm ? kSmemTwoPerSm : kSmemBudget) - 1024;
  if (own_b) {
    c.b_stages = 2;
    c.stages = (int)std::min<uint32_t>(kMaxStages, (budget - 2 * b_bytes) / x_bytes);
  } else {
    c.stages = c.b_stages = (int)std::min<uint32_t>(kMaxStages, budget / (x_bytes + b_bytes));
  }
  c.tmem_cols = tmem_cols_for(npt * c.mt);
  c.smem = (uint32_t)c.stages * x_bytes + (uint32_t)c.b_stages * b_bytes + 1024;
  return c;
}
// The fp16 epilogue assembles a CTA's 64-token blocks of every target in the
// pipeline buffers (2·mt blocks of two halves per target).
bool p16_staging_fits(int ntg, int np, const ProjConfig& c) {
  return (size_t)ntg * 2 * c.mt * 2 * p16_half_bytes(np) <= (size_t)c.smem - 1024;
}

int64_t proj_ctas(const SketchPlan& p, const ProjConfig& c) {
  const int64_t rows_per_cta = (int64_t)kTileRows * c.mt;
  return (p.ldp + rows_per_cta - 1) / rows_per_cta;
}

// Arguments of the projection of one target (ntg = 1) whose workspace starts at w.
ProjectArgs project_args(const SketchPlan& p, const ProjConfig& c, uint64_t seed, uint32_t stream_id, bool explicit_a,
                         uint8_t* w, unsigned int* err) {
  ProjectArgs pa{};
  pa.T = p.T;
  pa.k = p.k;
  pa.r = p.r;
  pa.np = p.np;
  pa.ntg = 1;
  pa.explicit_a = explicit_a ? 1 : 0;
  pa.npt = p.np;
  pa.ldp = p.ldp;
  pa.num_kb = (int)((p.k + kSlab - 1) / kSlab);
  pa.p16 = p.p16;
  pa.seed[0] = seed;
  pa.stream_id[0] = stream_id;
  pa.p_hi[0] = reinterpret_cast<__nv_bfloat16*>(w + p.off_phi);
  pa.p_lo[0] = reinterpret_cast<__nv_bfloat16*>(w + p.off_plo);
  pa.stages = c.stages;
  pa.b_stages = c.b_stages;
  pa.tmem_cols = c.tmem_cols;
  pa.err = err;
  return pa;
}

// Arguments and shared memory of the bf16 contraction (np ≤ 64) of one target.
ContractArgs contract_args(const SketchPlan& p, float* S, int64_t lds, uint8_t* w, unsigned int* err,
                           uint32_t* smem) {
  ContractArgs ca{};
  ca.d = p.d;
  ca.r = p.r;
  ca.np = p.np;
  ca.mt = p.mt;
  ca.tk = p.tk;
  ca.num_kb = p.num_kb_t;
  ca.kb_per_split = p.kb_per_split;
  ca.splits = p.splits;
  const uint32_t cstage = 256u * (uint32_t)p.tk * (uint32_t)p.mt + 2u * (uint32_t)p.np * 2u * (uint32_t)p.tk;
  const uint32_t cbudget = p.np <= 64 ? kSmemTwoPerSm : kSmemBudget;
  ca.stages = (int)std::min<uint32_t>(kMaxStages, (cbudget - 1024) / cstage);
  ca.tmem_cols = tmem_cols_for(p.np * p.mt);
  ca.inv_sqrt_r = (float)(1.0 / std::sqrt((double)p.r));
  ca.S = S;
  ca.lds = lds;
  ca.s_vec4 = (lds % 4 == 0) && ((reinterpret_cast<uintptr_t>(S) & 15) == 0);
  ca.part = reinterpret_cast<float*>(w + p.off_part);
  ca.dp = p.dp;
  ca.err = err;
  *smem = ca.stages * cstage + 1024;
  return ca;
}

// Tensor maps of the bf16 contraction: dY (d × T, boxes of 64 rows × tk
// tokens) and the two Pᵀ arrays (np × ldp, boxes of tk tokens × np).
logra_status contract_maps(const SketchPlan& p, const void* dY, int64_t lddy, uint8_t* w, CUtensorMap* tdy,
                           CUtensorMap* tph, CUtensorMap* tpl) {
  const uint32_t pswz = p.tk == 64 ? 128u : 64u;
  logra_status s = make_tmap_bf16_2d(tdy, dY, (uint64_t)p.d, (uint64_t)p.T, (uint64_t)lddy * 2, 64, (uint32_t)p.tk);
  if (s != LOGRA_OK || p.p16) return s;
  s = make_tmap_bf16_2d(tph, w + p.off_phi, (uint64_t)p.ldp, (uint64_t)p.np, (uint64_t)p.ldp * 2, (uint32_t)p.tk,
                        (uint32_t)p.np, pswz);
  if (s != LOGRA_OK) return s;
  return make_tmap_bf16_2d(tpl, w + p.off_plo, (uint64_t)p.ldp, (uint64_t)p.np, (uint64_t)p.ldp * 2, (uint32_t)p.tk,
                           (uint32_t)p.np, pswz);
}

// Projection of one X for ntg targets (their sign tiles stacked in one B
// operand).  plans[j] / ws[j] give each target's workspace layout and base.
// A / lda: one given bf16 projection operand per target, or nullptr for
// signs built on chip.
logra_status launch_projection(int ntg, const SketchPlan* plans, const void* X, int64_t ldx, const uint64_t* seeds,
                               const uint32_t* stream_ids, uint8_t* const* ws, const void* const* A,
                               const int64_t* lda, unsigned int* err, cudaStream_t st) {
  const SketchPlan& p = plans[0];
  const ProjConfig cfg = proj_config(ntg * p.np, A == nullptr);
  const int mt = cfg.mt;
  if (p.p16 && !p16_staging_fits(ntg, p.np, cfg))
    return fail(LOGRA_ERR_UNSUPPORTED, "sketch: the fp16 blocks of a CTA do not fit its shared memory");
  CUtensorMap tx, ta;
  ExtraOperands<true> extra;
  logra_status s =
      make_tmap_bf16_2d(&tx, X, (uint64_t)p.k, (uint64_t)p.T, (uint64_t)ldx * 2, kSlab, (uint32_t)(kTileRows * mt));
  if (s != LOGRA_OK) return s;
  if (A) {
    // the given projections: r rows × k columns each, tiles of np rows × 64 columns
    s = make_tmap_bf16_2d(&ta, A[0], (uint64_t)p.k, (uint64_t)p.r, (uint64_t)lda[0] * 2, kSlab, (uint32_t)p.np);
    if (s != LOGRA_OK) return s;
    for (int j = 1; j < ntg; ++j) {
      s = make_tmap_bf16_2d(&extra.m[j - 1], A[j], (uint64_t)p.k, (uint64_t)p.r, (uint64_t)lda[j] * 2, kSlab,
                            (uint32_t)p.np);
      if (s != LOGRA_OK) return s;
    }
  } else {
    ta = tx;  // not read
  }
  ProjectArgs pa{};
  pa.T = p.T;
  pa.k = p.k;
  pa.r = p.r;
  pa.np = p.np;
  pa.ntg = ntg;
  pa.explicit_a = A ? 1 : 0;
  pa.npt = ntg * p.np;
  pa.ldp = p.ldp;
  pa.num_kb = (int)((p.k + kSlab - 1) / kSlab);
  pa.p16 = p.p16;
  for (int j = 0; j < ntg; ++j) {
    pa.seed[j] = seeds[j];
    pa.stream_id[j] = stream_ids[j];
    pa.p_hi[j] = reinterpret_cast<__nv_bfloat16*>(ws[j] + plans[j].off_phi);
    pa.p_lo[j] = reinterpret_cast<__nv_bfloat16*>(ws[j] + plans[j].off_plo);
  }
  pa.stages = cfg.stages;
  pa.b_stages = cfg.b_stages;
  pa.tmem_cols = cfg.tmem_cols;
  pa.err = err;
  const uint32_t psmem = cfg.smem;
  const unsigned grid = (unsigned)proj_ctas(p, cfg);
  cudaError_t e;
  if (A && ntg > 1) {
    auto kern = p.p16 ? (mt == 2 ? project_kernel<2, true, true> : project_kernel<1, true, true>)
                      : (mt == 2 ? project_kernel<2, true, false> : project_kernel<1, true, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(project_kernel)");
    kern<<<grid, kProjThreads, psmem, st>>>(tx, ta, extra, pa);
  } else {
    auto kern = p.p16 ? (mt == 2 ? project_kernel<2, false, true> : project_kernel<1, false, true>)
                      : (mt == 2 ? project_kernel<2, false, false> : project_kernel<1, false, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(project_kernel)");
    kern<<<grid, kProjThreads, psmem, st>>>(tx, ta, ExtraOperands<false>{}, pa);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch project_kernel");
  return LOGRA_OK;
}

logra_status launch_reduce(const SketchPlan& p, const float* part, float* S, int64_t lds, float inv_sqrt_r, int s_vec4,
                           cudaStream_t st) {
  const int64_t n4 = p.d * (p.np / 4);
  reduce_partials_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(part, p.splits, p.dp, p.np, p.d, p.r,
                                                                      inv_sqrt_r, S, lds, s_vec4);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch reduce_partials_kernel");
  return LOGRA_OK;
}

// Arguments and shared memory of the fp16 contraction (np > 64) of one target
// whose Pᵀ blocks and token scales are in its workspace.
logra_status contract16_args(const SketchPlan& p, float* S, int64_t lds, uint8_t* w, unsigned int* err,
                             Contract16Args* out, uint32_t* smem) {
  Contract16Args ca{};
  ca.d = p.d;
  ca.r = p.r;
  ca.np = p.np;
  ca.num_kb = p.num_kb_t;
  ca.kb_per_split = p.kb_per_split;
  ca.splits = p.splits;
  // dY tile, 1 KB holding the token scales, this CTA's half of the Pᵀ tile
  const uint32_t cstage = 256u * kC16Tk + 1024u + (((uint32_t)p.np * 64u + 1023u) & ~1023u);
  ca.stages = (int)std::min<uint32_t>(kC16MaxStages, (kSmemBudget - 1024) / cstage);
  ca.inv_sqrt_r = (float)(1.0 / std::sqrt((double)p.r));
  ca.S = S;
  ca.lds = lds;
  ca.s_vec4 = (lds % 4 == 0) && ((reinterpret_cast<uintptr_t>(S) & 15) == 0);
  ca.part = reinterpret_cast<float*>(w + p.off_part);
  ca.dp = p.dp;
  ca.p16 = w + p.off_phi;
  ca.err = err;
  // a conversion step holds kC16Step stages while the next one fills
  if (ca.stages < 2 * kC16Step) return fail(LOGRA_ERR_UNSUPPORTED, "sketch: too few contraction stages fit");
  *out = ca;
  *smem = ca.stages * cstage + 1024;
  return LOGRA_OK;
}

// fp16 contraction (np > 64) of one target whose Pᵀ and token scales are in its workspace.
logra_status launch_contraction16(const SketchPlan& p, const void* dY, int64_t lddy, float* S, int64_t lds,
                                  uint8_t* w, unsigned int* err, cudaStream_t st) {
  CUtensorMap tdy;
  logra_status s = make_tmap_bf16_2d(&tdy, dY, (uint64_t)p.d, (uint64_t)p.T, (uint64_t)lddy * 2, 64, kC16Tk);
  if (s != LOGRA_OK) return s;
  Contract16Args ca;
  uint32_t csmem;
  if ((s = contract16_args(p, S, lds, w, err, &ca, &csmem)) != LOGRA_OK) return s;
  cudaError_t e = cudaFuncSetAttribute(contract16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(contract16_kernel)");
  contract16_kernel<<<dim3((unsigned)p.d_tiles, (unsigned)p.splits), kC16Threads, csmem, st>>>(tdy, ca);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch contract16_kernel");
  if (p.splits > 1) return launch_reduce(p, ca.part, S, lds, ca.inv_sqrt_r, ca.s_vec4, st);
  return LOGRA_OK;
}

// Contraction (and split reduce) of one target whose P is in its workspace.
logra_status launch_contraction(const SketchPlan& p, const void* dY, int64_t lddy, float* S, int64_t lds,
                                uint8_t* w, unsigned int* err, cudaStream_t st) {
  if (p.p16) return launch_contraction16(p, dY, lddy, S, lds, w, err, st);
  CUtensorMap tdy, tph, tpl;
  logra_status s = contract_maps(p, dY, lddy, w, &tdy, &tph, &tpl);
  if (s != LOGRA_OK) return s;
  uint32_t csmem;
  const ContractArgs ca = contract_args(p, S, lds, w, err, &csmem);
  auto kern = contract_kernel<64, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(contract_kernel)");
  kern<<<dim3((unsigned)p.d_tiles, (unsigned)p.splits), kConThreads, csmem, st>>>(tdy, tph, tpl, ca);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch contract_kernel");
  if (p.splits > 1) return launch_reduce(p, ca.part, S, lds, ca.inv_sqrt_r, ca.s_vec4, st);
  return LOGRA_OK;
}

}  // namespace

logra_status launch_sketch(const SketchPlan& p, const void* X, int64_t ldx, const void* dY, int64_t lddy,
                           uint64_t seed, uint32_t stream_id, float* S, int64_t lds, void* ws, cudaStream_t st) {
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  logra_status s = launch_projection(1, &p, X, ldx, &seed, &stream_id, &w, nullptr, nullptr, err, st);
  if (s != LOGRA_OK) return s;
  return launch_contraction(p, dY, lddy, S, lds, w, err, st);
}

logra_status launch_sketch_explicit(const SketchPlan& p, const void* X, int64_t ldx, const void* dY, int64_t lddy,
                                    const void* A, int64_t lda, float* S, int64_t lds, void* ws, cudaStream_t st) {
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const uint64_t seed = 0;
  const uint32_t sid = 0;
  logra_status s = launch_projection(1, &p, X, ldx, &seed, &sid, &w, &A, &lda, err, st);
  if (s != LOGRA_OK) return s;
  return launch_contraction(p, dY, lddy, S, lds, w, err, st);
}

size_t shared_x_workspace_bytes(int64_t T, int64_t k, int n, const int64_t* d, int r) {
  size_t total = 0;
  for (int j = 0; j < n; ++j) total += align256(plan_sketch(T, d[j], k, r).bytes);
  return total;
}

logra_status launch_sketch_shared_x(const void* X, int64_t ldx, int64_t T, int64_t k, int n,
                                    const logra_sketch_target* tg, int r, const void* const* A, const int64_t* lda,
                                    void* ws, cudaStream_t st) {
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  SketchPlan plans[kMaxTargets];
  uint8_t* bases[kMaxTargets];
  uint64_t seeds[kMaxTargets];
  uint32_t sids[kMaxTargets];
  uint8_t* w = static_cast<uint8_t*>(ws);
  for (int j = 0; j < n; ++j) {
    plans[j] = plan_sketch(T, tg[j].d, k, r);
    bases[j] = w;
    w += align256(plans[j].bytes);
    seeds[j] = tg[j].seed;
    sids[j] = tg[j].stream_id;
  }
  logra_status s = launch_projection(n, plans, X, ldx, seeds, sids, bases, A, lda, err, st);
  if (s != LOGRA_OK) return s;
  for (int j = 0; j < n; ++j) {
    s = launch_contraction(plans[j], tg[j].dY, tg[j].lddy, tg[j].S, tg[j].lds, bases[j], err, st);
    if (s != LOGRA_OK) return s;
  }
  return LOGRA_OK;
}

// ---------------------------------------------------------------- group plan
size_t sketch_group_plan_bytes(int n) { return plan_entry_offset(n) + (size_t)n * sizeof(SketchEntry); }

namespace {
bool target_empty(const logra_sketch_group_target& t) { return t.T == 0 || t.d == 0 || t.k == 0; }

// Launch order of one phase: positions sorted by decreasing CTA length
// (ties in target order), so that the longest CTAs start first and the
// launch ends on short ones.
void phase_order(int n, const int64_t* len, int32_t* order) {
  std::vector<int32_t> idx((size_t)n);
  for (int j = 0; j < n; ++j) idx[(size_t)j] = j;
  std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return len[a] > len[b]; });
  for (int j = 0; j < n; ++j) order[j] = idx[(size_t)j];
}

// begin[] of one phase in the given order from the CTA count of each target.
logra_status phase_begin(int n, const int32_t* order, const int64_t* ctas, int32_t* begin, int32_t* total) {
  int64_t acc = 0;
  for (int m = 0; m < n; ++m) {
    begin[m] = (int32_t)acc;
    acc += ctas[order[m]];
    if (acc > 0x7FFFFFFF) return fail(LOGRA_ERR_SHAPE, "sketch group: more than 2^31 - 1 CTAs in one launch");
  }
  begin[n] = (int32_t)acc;
  *total = (int32_t)acc;
  return LOGRA_OK;
}
}  // namespace

size_t sketch_group_workspace_bytes(int n, const logra_sketch_group_target* tg, int r) {
  size_t total = 0;
  for (int j = 0; j < n; ++j)
    if (!target_empty(tg[j])) total += align256(plan_sketch(tg[j].T, tg[j].d, tg[j].k, r).bytes);
  return total;
}

logra_status build_sketch_group_plan(int n, const logra_sketch_group_target* tg, int r, void* ws, void* plan) {
  unsigned int* const err = nullptr;  // given to the kernels at launch
  std::memset(plan, 0, sketch_group_plan_bytes(n));
  uint8_t* base = static_cast<uint8_t*>(plan);
  SketchPlanHeader* h = reinterpret_cast<SketchPlanHeader*>(base);
  SketchEntry* ent = reinterpret_cast<SketchEntry*>(base + plan_entry_offset(n));
  const int np = (int)round_up(r, 16);
  // one launch shape (mt) for both kinds of target; the shared memory covers the larger ring layout
  const ProjConfig pc_sign = proj_config(np, true), pc_given = proj_config(np, false);
  const ProjConfig& pc = pc_sign;
  if (np > 64 && (!p16_staging_fits(1, np, pc_sign) || !p16_staging_fits(1, np, pc_given)))
    return fail(LOGRA_ERR_UNSUPPORTED, "sketch group: the fp16 blocks of a CTA do not fit its shared memory");
  h->magic = kSketchPlanMagic;
  h->n = n;
  h->r = r;
  h->np = np;
  h->p16 = np > 64 ? 1 : 0;
  h->proj_mt = pc.mt;
  h->proj_smem = std::max(pc_sign.smem, pc_given.smem);
  std::vector<int64_t> len[3], ctas[3];
  for (int ph = 0; ph < 3; ++ph) {
    len[ph].assign((size_t)n, 0);
    ctas[ph].assign((size_t)n, 0);
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  for (int j = 0; j < n; ++j) {
    const logra_sketch_group_target& t = tg[j];
    SketchEntry& e = ent[j];
    if (target_empty(t)) continue;  // no CTAs, no workspace
    const SketchPlan p = plan_sketch(t.T, t.d, t.k, r);
    logra_status s =
        make_tmap_bf16_2d(&e.tx, t.X, (uint64_t)p.k, (uint64_t)p.T, (uint64_t)t.ldx * 2, kSlab,
                          (uint32_t)(kTileRows * pc.mt));
    if (s != LOGRA_OK) return s;
    if (t.A) {
      s = make_tmap_bf16_2d(&e.ta, t.A, (uint64_t)p.k, (uint64_t)p.r, (uint64_t)t.lda * 2, kSlab, (uint32_t)p.np);
      if (s != LOGRA_OK) return s;
    }
    if ((s = contract_maps(p, t.dY, t.lddy, w, &e.tdy, &e.tph, &e.tpl)) != LOGRA_OK) return s;
    e.pa = project_args(p, t.A ? pc_given : pc_sign, t.seed, t.stream_id, t.A != nullptr, w, err);
    uint32_t csmem = 0;
    e.ca = contract_args(p, t.S, t.lds, w, err, &csmem);
    if (p.p16 && (s = contract16_args(p, t.S, t.lds, w, err, &e.c16, &csmem)) != LOGRA_OK) return s;
    h->con_smem = csmem;  // the same for every target (it depends on np only)
    e.d_tiles = p.d_tiles;
    e.proj_ctas = (int32_t)proj_ctas(p, pc);
    ctas[0][(size_t)j] = e.proj_ctas;
    len[0][(size_t)j] = e.pa.num_kb;
    // (p16: d_tiles is even, so every matrix keeps the CTA pairs aligned)
    e.con_ctas = p.d_tiles * p.splits;
    ctas[1][(size_t)j] = e.con_ctas;
    len[1][(size_t)j] = std::min(p.kb_per_split, p.num_kb_t);
    if (p.splits > 1) {
      e.red_blocks = (int32_t)((p.d * (p.np / 4) + 255) / 256);
      ctas[2][(size_t)j] = e.red_blocks;
      len[2][(size_t)j] = p.splits;
    }
    w += align256(p.bytes);
  }
  h->ws_bytes = (uint64_t)(w - static_cast<uint8_t*>(ws));
  int32_t* totals[3] = {&h->proj_ctas, &h->con_ctas, &h->red_blocks};
  for (int ph = 0; ph < 3; ++ph) {
    int32_t* begin = reinterpret_cast<int32_t*>(base + plan_begin_offset(n, ph));
    int32_t* order = reinterpret_cast<int32_t*>(base + plan_order_offset(n, ph));
    phase_order(n, len[ph].data(), order);
    logra_status s = phase_begin(n, order, ctas[ph].data(), begin, totals[ph]);
    if (s != LOGRA_OK) return s;
  }
  return LOGRA_OK;
}

logra_status check_sketch_group_plan(const void* plan, int* n) {
  const SketchPlanHeader* h = static_cast<const SketchPlanHeader*>(plan);
  if (h->magic != kSketchPlanMagic)
    return fail(LOGRA_ERR_INVALID_ARG, "sketch group: not a plan (logra_sketch_group_plan)");
  *n = h->n;
  return LOGRA_OK;
}

logra_status launch_sketch_group(const void* plan, const void* plan_dev, cudaStream_t st) {
  const SketchPlanHeader* h = static_cast<const SketchPlanHeader*>(plan);
  const uint8_t* pd = static_cast<const uint8_t*>(plan_dev);
  const int n = h->n;
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  cudaError_t e;
  if (h->proj_ctas > 0) {
    auto kern = h->p16 ? (h->proj_mt == 2 ? project_group_kernel<2, true> : project_group_kernel<1, true>)
                       : (h->proj_mt == 2 ? project_group_kernel<2, false> : project_group_kernel<1, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->proj_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(project_group_kernel)");
    kern<<<(unsigned)h->proj_ctas, kProjThreads, h->proj_smem, st>>>(pd, n, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch project_group_kernel");
  }
  if (h->con_ctas > 0 && h->p16) {
    e = cudaFuncSetAttribute(contract16_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)h->con_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(contract16_group_kernel)");
    contract16_group_kernel<<<(unsigned)h->con_ctas, kC16Threads, h->con_smem, st>>>(pd, n, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch contract16_group_kernel");
  } else if (h->con_ctas > 0) {
    e = cudaFuncSetAttribute(contract_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->con_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(contract_group_kernel)");
    contract_group_kernel<<<(unsigned)h->con_ctas, kConThreads, h->con_smem, st>>>(pd, n, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch contract_group_kernel");
  }
  if (h->red_blocks > 0) {
    reduce_group_kernel<<<(unsigned)h->red_blocks, 256, 0, st>>>(pd, n);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "launch reduce_group_kernel");
  }
  return LOGRA_OK;
}

}  // namespace logra
