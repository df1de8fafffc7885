// swiglu_swab_kernel.cuh -- the fused SwiGLU projection for few rows, with
// the weights on the MMA's M side (swapped operands), on CTA pairs (sm_103a).
//
// Computes Y = SiLU(A x W1) (.) (A x W2) (page "Riepilogo Tecnico:
// Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza
// Efficiente di LLM", section "Definizione del Problema") in either weight
// form (section "Metodologia", items 1 and 2) for M <= 128 rows.
//
// With few rows a call is a stream of the weights, and what limits it is how
// much of that stream each SM keeps in flight plus the fixed cost around it.
// Here each CTA pair computes 64 output columns for all (<= 128) rows as the
// transposed product Y^T = W^T A^T:
//   * one tcgen05.mma.cta_group::2 with M = 128 weight rows (64 per CTA: the
//     gate and up rows of this CTA's 32 output columns) and N = the rows of A
//     (padded to 64 or 128, half in each CTA's shared memory), issued by the
//     even CTA;
//   * each CTA streams, per K step of 64, its 64 weight rows (8 KB, taken
//     MN-major straight from the row-major [K,N] weights) and its half of the
//     rows of A (8 KB): 16 KB per step, so the 14 K steps of the Qwen-2.5-0.5B
//     projection (K = 896) are all in flight at once -- one DRAM round trip;
//   * the result lands complete in each CTA's tensor memory (all of K, its 64
//     weight rows, every row of A): no partial sums to exchange, unlike the
//     split-K kernel.  TMEM lanes 0-63 hold the 64 weight rows for the first
//     half of A's rows, lanes 64-127 for the second half;
//   * four epilogue warps read their lanes; the gate and up values of one
//     output column sit in different warps (separate form: rows 0-31 gate,
//     32-63 up) or in neighbouring lanes (interleaved form: row 2j gate,
//     2j+1 up), so warps trade half their values through shared memory (or a
//     lane shuffle), apply y = g * u / (1 + e^-g) in FP32, round to BF16,
//     stage the [rows x 32] block and store it with one TMA store.
// Gate and up values never reach global memory.  One tile per CTA pair: the
// launcher sizes the grid to the output column blocks.
//
// Every wait is bounded as in the other kernels (timeout -> error word, abort
// flag, drain, TMEM freed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace swiglu {

// INTERLEAVED: the weights come as W_fused [K, 2N]; ROWS: rows of A per pair
// (MMA N), 64 or 128.
template <bool INTERLEAVED_, int ROWS_>
struct SwabCfg {
  static constexpr bool INTERLEAVED = INTERLEAVED_;
  static constexpr int ROWS = ROWS_;             // rows of A (MMA N) per pair
  static constexpr int HALF = ROWS / 2;          // rows of A held by each CTA
  static constexpr int COLS = 32;                // output columns per CTA (64 per pair)
  static constexpr int BK = 64;                  // K per stage
  static constexpr int W_BYTES = BK * 2 * COLS * 2;  // 64 weight rows x 64 K: 8 KB
  static constexpr int A_BYTES = HALF * BK * 2;      // HALF rows of A x 64 K
  static constexpr int STAGE_BYTES = W_BYTES + A_BYTES;
  static constexpr int STAGES_FIT = (224 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 16 ? STAGES_FIT : 16;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 3;  // full[S], empty[S], acc_full, drain, spare
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  static constexpr int EPI_WARPS = 4;
  static constexpr int PRODUCER_WARP = 4;
  static constexpr int MMA_WARP = 5;
  static constexpr int THREADS = 32 * 6;
  static constexpr int TMEM_COLS = HALF < 32 ? 32 : HALF;
  // The weight operand (M side, MN-major): separate form, two 32-row boxes
  // (W1's 32 columns, then W2's) with the 64-byte swizzle, 4 KB apart;
  // interleaved form, one 64-row box of W_fused with the 128-byte swizzle.
  static constexpr int W_ROW_BYTES = INTERLEAVED ? 128 : 64;   // one K row of one box
  static constexpr uint32_t W_SWIZZLE = INTERLEAVED ? ptx::SW_128B : ptx::SW_64B;
  static constexpr int W_LBO = INTERLEAVED ? W_BYTES : W_BYTES / 2;
  static constexpr int W_SBO = 8 * W_ROW_BYTES;
  static constexpr int W_KSTEP = 16 * W_ROW_BYTES;
  static constexpr uint32_t IDESC = ptx::idesc_bf16(128, ROWS, true, false);
  // epilogue scratch, reusing the ring once every MMA has completed: the
  // values two warps trade ([32 lanes][HALF/2 + 1] floats, twice, per warp
  // pair) and the BF16 output block [ROWS][32]
  static constexpr int XCH_STRIDE = HALF / 2 + 1;
  static constexpr int XCH_BYTES = 32 * XCH_STRIDE * 4;
  static constexpr int YSTG_OFF = 4 * XCH_BYTES;
  static_assert(ROWS == 64 || ROWS == 128, "rows of A per pair");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(YSTG_OFF + ROWS * COLS * 2 <= BAR_OFF, "epilogue scratch fits the ring");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// One K step of 64 on the pair: four MMAs of K = 16 from stage descriptors
// stepped by immediates (slice j: adesc + j * A_STEP, bdesc + j * B_STEP, in
// 16-byte units); `first` = 1 starts the accumulator.  These MMAs are short
// (64 weight rows per CTA x the rows of A x 16), so the issuing thread's own
// work per MMA matters: two descriptors and a predicate built per MMA would
// take about as long as the MMA itself.
template <int A_STEP, int B_STEP>
__device__ __forceinline__ static void swab_mma_k64(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                                    uint32_t idesc, uint32_t first) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.eq.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %1, %5;\n\t"
      "add.s64 a2, %1, %6;\n\t"
      "add.s64 a3, %1, %7;\n\t"
      "add.s64 b1, %2, %8;\n\t"
      "add.s64 b2, %2, %9;\n\t"
      "add.s64 b3, %2, %10;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a2, b2, %3, t;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(first), "n"(A_STEP), "n"(2 * A_STEP),
      "n"(3 * A_STEP), "n"(B_STEP), "n"(2 * B_STEP), "n"(3 * B_STEP)
      : "memory");
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_swab_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB0,  // W1, or W_fused
                       const __grid_constant__ CUtensorMap tmB1,  // W2 (separate form only)
                       const __grid_constant__ CUtensorMap tmY, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const uint32_t bars = base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::STAGES + s); };
  const uint32_t accf_bar = bars + 8u * (2 * C::STAGES);
  const uint32_t drain_bar = bars + 8u * (2 * C::STAGES + 1);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0 = the pair's leader
  const int pair = static_cast<int>(ptx::cluster_id_x());  // output columns [64 pair, 64 pair + 64)
  const int col0 = pair * 2 * C::COLS + static_cast<int>(rank) * C::COLS;  // this CTA's columns
  const int nk = p.num_k_blk;

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(accf_bar, 1);
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (!C::INTERLEAVED) ptx::prefetch_tmap(&tmB1);
    ptx::prefetch_tmap(&tmY);
  }
  if (warp == C::MMA_WARP) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!wait_bar(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_PRODUCER_EMPTY)) {
          ok = false;
          break;
        }
        const uint32_t sw = base + stage * C::STAGE_BYTES;
        const uint32_t sa = sw + C::W_BYTES;
        const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);
        if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
        if (C::INTERLEAVED) {
          ptx::tma_load_2d_pair(sw, &tmB0, fb, 2 * col0, kb * C::BK);
        } else {
          ptx::tma_load_2d_pair(sw, &tmB0, fb, col0, kb * C::BK);
          ptx::tma_load_2d_pair(sw + C::W_BYTES / 2, &tmB1, fb, col0, kb * C::BK);
        }
        ptx::tma_load_2d_pair(sa, &tmA, fb, kb * C::BK, static_cast<int>(rank) * C::HALF);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        // Consume the MMA-completion arrivals still due on this CTA's "empty"
        // barriers, so no multicast arrive targets this CTA after it exits.
        const uint32_t n = issued < (uint32_t)C::STAGES ? issued : (uint32_t)C::STAGES;
        for (uint32_t i = issued - n; i < issued; ++i)
          wait_quiet(empty_bar(i % C::STAGES), (i / C::STAGES) & 1u, p.timeout_ns);
      } else {
        spin_ns(100000);  // aborted: copies already in flight into this CTA land
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      // Stage 0's descriptors; stage s adds s * STAGE_BYTES (16-byte units).
      // Weights (MMA A, M side): MN-major, boxes W_LBO apart, 8-row K groups
      // W_SBO apart, one MMA's 16 K rows = W_KSTEP bytes; rows of A (MMA B,
      // N side): K-major, 128-byte swizzle, 32 bytes of K per MMA.
      const uint64_t adesc0 = ptx::smem_desc(base, C::W_LBO, C::W_SBO, C::W_SWIZZLE);
      const uint64_t bdesc0 = ptx::smem_desc(base + C::W_BYTES, 16, 1024, ptx::SW_128B);
      static_assert(C::BK == 64, "four MMAs of K = 16 per stage");
      for (int kb = 0; kb < nk; ++kb) {
        if (!wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t off = (stage * C::STAGE_BYTES) >> 4;
        swab_mma_k64<C::W_KSTEP / 16, 32 / 16>(tmem_base, adesc0 + off, bdesc0 + off, C::IDESC,
                                               kb == 0 ? 1u : 0u);
        ptx::mma_commit_pair_mc(empty_bar(stage), 0x3);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::mma_commit_pair_mc(accf_bar, 0x3);
      ptx::mma_commit_pair_mc(drain_bar, 0x1);
      wait_quiet(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-3, both CTAs)
    // Warp q reads TMEM lanes [32q, 32q+32): weight rows 32 (q % 2) + lane,
    // rows of A [HALF (q / 2), HALF (q / 2) + HALF) in columns [0, HALF).
    const int q = warp;
    const int rbase = (q >> 1) * C::HALF;  // first row of A of this warp's half
    bool ok = wait_bar(accf_bar, 0, p.timeout_ns, abort_flag, p.err, WAIT_EPI_ACC_FULL);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    float v[C::HALF];
    if (ok) {
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + 32u * c, r);
        ptx::tmem_wait_ld();
        ptx::reg_fence(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
      }
    }
    // The epilogue's scratch lies in the ring: every MMA has completed (and
    // every copy has landed) once the accumulator barrier has fired.
    __nv_bfloat16 *ystg = reinterpret_cast<__nv_bfloat16 *>(smem + C::YSTG_OFF);
    constexpr int H2 = C::HALF / 2;
    // separate form: warps 2h (gate rows) and 2h + 1 (up rows) hold the same
    // output columns (lane) for the same rows of A; the gate warp finishes
    // rows [0, H2) of the half, the up warp [H2, HALF), each taking the other
    // half of its partner's values through shared memory
    const bool gate = (q & 1) == 0;
    float *xch = reinterpret_cast<float *>(smem) + (q >> 1) * 2 * (C::XCH_BYTES / 4);
    float *to_partner = xch + (gate ? 0 : C::XCH_BYTES / 4);  // gate->up, up->gate
    float *from_partner = xch + (gate ? C::XCH_BYTES / 4 : 0);
    if (!C::INTERLEAVED) {
      if (ok) {
#pragma unroll
        for (int t = 0; t < H2; ++t)
          to_partner[lane * C::XCH_STRIDE + t] = gate ? v[H2 + t] : v[t];
      }
      // the two warps of this half meet (named barrier 1 + half, 64 threads);
      // reached whatever `ok` is, so a warp never waits for a partner that left
      asm volatile("bar.sync %0, 64;" ::"r"(1 + (q >> 1)) : "memory");
    }
    if (ok) {
      if (C::INTERLEAVED) {
        // lanes 2j (gate) and 2j+1 (up) of output column 16 (q % 2) + j: the
        // even lane finishes rows [0, H2) of the half, the odd lane [H2, HALF)
        const bool even = (lane & 1) == 0;
        const int col = 16 * (q & 1) + (lane >> 1);
#pragma unroll
        for (int t = 0; t < H2; ++t) {
          const float mine = even ? v[H2 + t] : v[t];
          const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
          const float y = even ? silu_mul(v[t], other) : silu_mul(other, v[H2 + t]);
          const int row = rbase + (even ? t : H2 + t);
          ystg[row * C::COLS + col] = __float2bfloat16_rn(y);
        }
      } else {
        // the partner's values first, into registers: the output stores below
        // go to the same shared array, so loads interleaved with them would
        // wait for each store in turn
        float o[H2];
#pragma unroll
        for (int t = 0; t < H2; ++t) o[t] = from_partner[lane * C::XCH_STRIDE + t];
#pragma unroll
        for (int t = 0; t < H2; ++t) {
          const float y = gate ? silu_mul(v[t], o[t]) : silu_mul(o[t], v[H2 + t]);
          const int row = rbase + (gate ? t : H2 + t);
          ystg[row * C::COLS + lane] = __float2bfloat16_rn(y);
        }
      }
      ptx::fence_proxy_async_smem();  // generic-proxy writes, read by the TMA store
    }
    ok = __all_sync(0xffffffffu, ok);
    // all four epilogue warps have staged their rows (named barrier 3, 128 threads)
    asm volatile("bar.sync 3, 128;" ::: "memory");
    if (warp == 0 && lane == 0) {
      // one TMA store of the [ROWS x 32] block; rows beyond M and columns
      // beyond N are clipped by the tensor map
      if (ok && col0 < p.N) ptx::tma_store_2d(&tmY, ptx::smem_u32(ystg), col0, 0);
      ptx::bulk_commit();
      ptx::bulk_wait_read<0>();
    }
    __syncwarp();
  }

  // Both CTAs have passed their last use of the pair's resources (the
  // leader has drained its MMAs, each producer has seen every commit aimed at
  // its barriers) before either frees the tensor memory and leaves.  Only the
  // order of execution matters here, so the arrive is relaxed: a release
  // would also wait for this CTA's output stores to reach global memory.
  ptx::tc_fence_before();
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
  asm volatile("barrier.cluster.wait;" ::: "memory");
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace swiglu
