// swiglu_tc2_kernel.cuh -- the CTA-pair (cta_group::2) fused SwiGLU kernel.
//
// Same computation as the one-CTA kernel (page "Riepilogo Tecnico ...
// Inferenza Efficiente di LLM", sections "Definizione del Problema" and
// "Metodologia", items 1 and 2), with one output tile of 256 rows x 128
// columns per pair of CTAs (a 2-CTA cluster on one TPC):
//   * one tcgen05.mma.cta_group::2 M=256 x N=256 x K=16, issued by the even
//     CTA, reads A rows [0,128) from the even CTA's shared memory and rows
//     [128,256) from the odd CTA's, and weight columns [0,128) from the even
//     CTA and [128,256) from the odd CTA.  In the separate form the even CTA
//     therefore loads W1's 128-column block and the odd CTA W2's: each CTA
//     streams A[128 x 64] + one weight block [64 x 128] = 32 KB per K step
//     (48 KB for the one-CTA 128x256 tile), which is what lets the pair reach
//     the tensor pipe's rate from L2;
//   * each CTA's TMEM receives its own 128 rows x 256 columns (gate | up, or
//     the interleaved pairs), double-buffered, so the epilogue is local;
//   * the even CTA owns the "full" barriers (both CTAs' TMA copies count on
//     them) and the "accumulator empty" barriers (all sixteen epilogue warps
//     arrive there); MMA completion is multicast to both CTAs' "empty" and
//     "accumulator full" barriers.
// FP8 E4M3 operands (the page's motivation: quantisation raises tensor-core
// density, section "Definizione del Problema") use tcgen05.mma.kind::f8f6f4
// with K-major weights; the epilogue multiplies the gate and up accumulators
// by sA*sW1 and sA*sW2 before SiLU.
// Unit schedule: with more units than resident pairs the grid holds one
// cluster per unit, and a running pair, after its own unit, cancels clusters
// that have not started yet (cluster launch control) and takes over their
// units.  The units therefore run in about launch order however far the
// pairs drift apart, which keeps the tiles that share A rows and weight
// columns close together in time, and so in L2.  The leader's producer thread
// requests the next unit while the current one loads; the 16-byte response
// lands in both CTAs and every role reads it from a small ring.
// Waits are bounded as in the one-CTA kernel.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace swiglu {

// FP8 = false: BF16 operands, weights MN-major ([K,N] row-major), 64 K per stage.
// FP8 = true : E4M3 operands, weights K-major ([N,K] row-major), 128 K per stage;
//              the epilogue applies the per-tensor scales.
// LINEAR = false: the fused SwiGLU epilogue (MMA N = 256 = 128 gate + 128 up
//                 columns, 128 output columns per tile).
// LINEAR = true : a plain product Z = X W (+ R) with LIN_N output columns per
//                 tile (MMA N = LIN_N = 256 or 128); the weight block of one
//                 tile is split between the two CTAs like the interleaved form.
template <bool INTERLEAVED_, int STAGES_, bool FP8_ = false, bool LINEAR_ = false,
          int LIN_N = 256>
struct PairCfg {
  static constexpr bool LINEAR = LINEAR_;
  static constexpr bool INTERLEAVED = INTERLEAVED_ || LINEAR_;  // one weight matrix
  static constexpr int STAGES = STAGES_;
  static constexpr bool FP8 = FP8_;
  static constexpr int BM = 128;                 // rows per CTA (MMA M = 256 per pair)
  static constexpr int BK = FP8 ? 128 : 64;      // K per stage: 128 bytes of each A row
  static constexpr int MMA_K = FP8 ? 32 : 16;    // K of one MMA instruction (32 bytes)
  static constexpr int MMA_M = 256;
  static constexpr int MMA_N = LINEAR ? LIN_N : 256;  // accumulator columns per tile
  static constexpr int BN = LINEAR ? LIN_N : 128;     // output columns per tile
  static constexpr int A_BYTES = BM * 128;       // 16 KB
  // BF16: MN-major boxes of 64 columns x 64 K-rows (MMA_N/128 of them per
  // CTA); FP8: one K-major box of this CTA's 128 weight rows x 128 K bytes.
  static constexpr int ATOM_BYTES = FP8 ? 128 * 128 : 64 * 128;
  static constexpr int B_ATOMS = FP8 ? 1 : MMA_N / 128;
  static_assert(!(LINEAR && FP8), "linear mode is BF16");
  static_assert(LIN_N == 256 || LIN_N == 128, "linear tile width");
  static constexpr int B_BYTES = B_ATOMS * ATOM_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB per CTA
  static constexpr int EPI_WARPS = 8;
  static constexpr int STG_BYTES = 32 * 64;
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  // unit-schedule responses: a ring of SCHED_D 16-byte slots
  static constexpr int SCHED_D = 4;
  static constexpr int RESP_OFF = STG_OFF + EPI_WARPS * 2 * STG_BYTES;
  static constexpr int BAR_OFF = RESP_OFF + SCHED_D * 16;
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * SCHED_D;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  // readers of every response: both producers, the MMA thread and the
  // epilogue warps of both CTAs
  static constexpr int SCHED_READERS = 2 + 1 + 2 * EPI_WARPS;
  static constexpr int TMEM_COLS = 2 * MMA_N;
  static constexpr int PRODUCER_WARP = EPI_WARPS;
  static constexpr int MMA_WARP = EPI_WARPS + 1;
  static constexpr int THREADS = 32 * (EPI_WARPS + 2);
  static constexpr uint32_t IDESC = FP8 ? ptx::idesc_e4m3(MMA_M, MMA_N, false, false)
                                        : ptx::idesc_bf16(MMA_M, MMA_N, false, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
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
  auto accf_bar = [&](int b) { return bars + 8u * (2 * C::STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * C::STAGES + 4);
  // response slot s: filled (both CTAs) / read by all readers (leader only)
  auto schf_bar = [&](uint32_t s) { return bars + 8u * (2 * C::STAGES + 5 + s); };
  auto sche_bar = [&](uint32_t s) { return bars + 8u * (2 * C::STAGES + 5 + C::SCHED_D + s); };
  auto resp = [&](uint32_t s) { return base + C::RESP_OFF + 16u * s; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile uint32_t *skip_word = tmem_slot + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0 = the pair's leader
  const int cid = static_cast<int>(ptx::cluster_id_x());
  const int ncl = static_cast<int>(ptx::num_clusters_x());

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar(b), 1);
      ptx::mbar_init(acce_bar(b), 2 * C::EPI_WARPS);
    }
    ptx::mbar_init(drain_bar, 1);
    for (uint32_t i = 0; i < (uint32_t)C::SCHED_D; ++i) {
      ptx::mbar_init(schf_bar(i), 1);
      ptx::mbar_init(sche_bar(i), C::SCHED_READERS);
    }
    *abort_flag = 0;
    // Dynamic schedule: while a timeout is recorded, the clusters that start
    // do no work (the leader decides for both CTAs), so a kernel that keeps
    // timing out ends within about one time limit, not one per unit.
    *skip_word = (p.dyn_sched && rank == 0 && *(volatile const uint32_t *)p.err != 0u) ? 1u : 0u;
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(rank == 0 || C::INTERLEAVED ? &tmB0 : &tmB1);
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
  // Everything above overlaps the previous kernel when launched with PDL.
  ptx::grid_launch_dependents();
  if (warp == C::PRODUCER_WARP && lane == 0) {
    // Warm the TMA unit's descriptor cache while the previous kernel ends.
    ptx::tma_prefetch_2d(&tmA, 0, 0);
    ptx::tma_prefetch_2d(rank == 0 || C::INTERLEAVED ? &tmB0 : &tmB1, 0, 0);  // descriptor warm-up
  }
  ptx::grid_dependency_wait();

  // work units: output tiles x K slices (k_splits == 1 unless split-K)
  const int num_tiles = p.num_m_blk * p.num_n_blk * p.k_splits;
  auto unit_coords = [&](int t, int &mb, int &nb, int &ks, int &kb0, int &kb1) {
    ks = t % p.k_splits;
    tile_coords(t / p.k_splits, p, mb, nb);
    kb0 = ks * p.kb_per_split;
    kb1 = min(p.num_k_blk, kb0 + p.kb_per_split);
  };
  // This pair's first unit (-1: none).  Response r of the dynamic schedule
  // (ring slot r % SCHED_D) names the unit after the r-th one.
  const bool dyn = p.dyn_sched != 0;
  const int first_unit =
      dyn && ptx::ld_shared_cluster_u32(ptx::mapa_shared(ptx::smem_u32(tmem_slot + 2), 0)) != 0u
          ? -1
          : cid;
  // The unit after `t`, the r-th unit of this pair; false if a wait gave up.
  // Called by one thread of each reading role.
  auto next_unit = [&](int t, uint32_t r, int &nxt) -> bool {
    if (!dyn) {
      nxt = t + ncl < num_tiles ? t + ncl : -1;
      return true;
    }
    const uint32_t s = r % C::SCHED_D;
    // The response lands through the async proxy with complete_tx on this
    // CTA's own barrier (as a TMA copy does), so a CTA-scope wait sees it.
    if (!wait_bar(schf_bar(s), (r / C::SCHED_D) & 1u, p.timeout_ns, abort_flag, p.err,
                  WAIT_SCHED_FULL))
      return false;
    int x = 0;
    nxt = ptx::clc_response(resp(s), x) ? (x >> 1) : -1;
    // Release the slot.  The decode above consumed the loaded response, so
    // the read is complete before this arrive issues: no fence is needed (a
    // cluster-scope release here cost ~0.6 us per unit on short-K shapes).
    ptx::mbar_arrive_cluster_relaxed(ptx::mapa_shared(sche_bar(s), 0));
    return true;
  };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const CUtensorMap *tmB = (C::INTERLEAVED || rank == 0) ? &tmB0 : &tmB1;
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      // Leader, dynamic schedule: request the unit after the r-th one into
      // slot r % SCHED_D once every reader has released that slot's previous
      // response.  A request follows only a response that named a unit.
      auto request = [&](uint32_t r) -> bool {
        const uint32_t s = r % C::SCHED_D;
        if (!wait_bar(sche_bar(s), ((r / C::SCHED_D) & 1u) ^ 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_SCHED_EMPTY))
          return false;
        // Each CTA's barrier expects the 16 response bytes; the peer's arrive
        // may land before or after the response (the transaction count may
        // go negative in between).
        ptx::mbar_arrive_expect_tx(schf_bar(s), 16);
        ptx::mbar_arrive_expect_tx_cluster_relaxed(ptx::mapa_shared(schf_bar(s), 1), 16);
        ptx::clc_try_cancel_all(resp(s), schf_bar(s));
        return true;
      };
      int t = first_unit;
      for (uint32_t r = 0; ok && t >= 0; ++r) {
        if (dyn && rank == 0 && !request(r)) {
          ok = false;
          break;
        }
        int mb, nb, ks, kb0, kb1;
        unit_coords(t, mb, nb, ks, kb0, kb1);
        const int arow = mb * 2 * C::BM + static_cast<int>(rank) * C::BM;
        // first weight column (BF16, [K,N]) or row (FP8, [N,K]) of this CTA's block
        const int bcol = C::INTERLEAVED ? nb * C::MMA_N + static_cast<int>(rank) * (C::MMA_N / 2)
                                        : nb * C::BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, p.err,
                        WAIT_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);
          if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
          ptx::tma_load_2d_pair(sa, &tmA, fb, kb * C::BK, arow);
          if (C::FP8) {
            ptx::tma_load_2d_pair(sb, tmB, fb, kb * C::BK, bcol);
          } else {
#pragma unroll
            for (int j = 0; j < C::B_ATOMS; ++j)
              ptx::tma_load_2d_pair(sb + j * C::ATOM_BYTES, tmB, fb, bcol + j * 64, kb * C::BK);
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ok = next_unit(t, r, t);
      }
      if (ok) {
        // Consume the MMA-completion arrivals still due on this CTA's "empty"
        // barriers, so no multicast arrive targets this CTA after it exits.
        const uint32_t n = issued < (uint32_t)C::STAGES ? issued : (uint32_t)C::STAGES;
        for (uint32_t i = issued - n; i < issued; ++i)
          wait_quiet(empty_bar(i % C::STAGES), (i / C::STAGES) & 1u, p.timeout_ns);
      } else {
        // Aborted: give copies already in flight into this CTA time to land.
        spin_ns(100000);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
      bool ok = true;
      int t = first_unit;
      for (uint32_t r = 0; ok && t >= 0; ++r) {
        int mb, nb, ks, kb0, kb1;
        unit_coords(t, mb, nb, ks, kb0, kb1);
        if (!wait_bar(acce_bar(abuf), aphase ^ 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_MMA_ACC_EMPTY)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + abuf * C::MMA_N;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / C::MMA_K; ++kk) {
            // A: K-major, 128-byte swizzle; one MMA's K = 32 bytes along the row.
            const uint64_t adesc = ptx::smem_desc(sa + kk * 32, 16, 1024, ptx::SW_128B);
            if (C::FP8) {
              // B: K-major like A.
              const uint64_t bdesc = ptx::smem_desc(sb + kk * 32, 16, 1024, ptx::SW_128B);
              ptx::mma_f8_pair(d, adesc, bdesc, C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
            } else {
              // B: MN-major; 64-column boxes ATOM_BYTES apart, 8-row K groups 1024
              // bytes apart, 16 K-rows = 2048 bytes.
              const uint64_t bdesc =
                  ptx::smem_desc(sb + kk * 2048, C::ATOM_BYTES, 1024, ptx::SW_128B);
              ptx::mma_f16_pair(d, adesc, bdesc, C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_mc(accf_bar(abuf), 0x3);
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1u;
        }
        ok = next_unit(t, r, t);
      }
      ptx::mma_commit_pair_mc(drain_bar, 0x1);
      wait_quiet(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7, both CTAs)
    const int q = warp & 3;   // TMEM lanes [32q, 32q+32)
    const int h = warp >> 2;  // half of the tile's 32-column chunks
    constexpr int NC = C::BN / 32;
    const uint32_t stg_base = base + C::STG_OFF + warp * 2 * C::STG_BYTES;
    float gs = 1.0f, us = 1.0f;
    if (C::FP8) {
      const float sa = *p.sA;
      gs = sa * *p.sW1;
      us = sa * *p.sW2;
    }
    uint32_t abuf = 0, aphase = 0, it = 0;
    int t = first_unit;
    for (uint32_t r = 0; t >= 0; ++r) {
      int mb, nb, ks, kb0, kb1;
      unit_coords(t, mb, nb, ks, kb0, kb1);
      bool ok = wait_bar(accf_bar(abuf), aphase, p.timeout_ns, abort_flag, p.err,
                         WAIT_EPI_ACC_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * C::MMA_N;
      const int row0 = mb * 2 * C::BM + static_cast<int>(rank) * C::BM + q * 32;
      if (C::LINEAR)
        epilogue_tile_linear<C::BN>(tacc, row0, nb * C::BN, h * (NC / 2), (h + 1) * (NC / 2), &tmY,
                                    p, ks, smem, base, stg_base, it, lane,
                                    ptx::mapa_shared(acce_bar(abuf), 0));
      else
        epilogue_tile<C::INTERLEAVED, C::BN, C::FP8>(
            tacc, row0, nb * C::BN, h * (NC / 2), (h + 1) * (NC / 2), &tmY, p.M, p.N, smem, base,
            stg_base, it, lane, ptx::mapa_shared(acce_bar(abuf), 0), gs, us);
      if (++abuf == 2) {
        abuf = 0;
        aphase ^= 1u;
      }
      int nxt = -1;
      ok = lane == 0 ? next_unit(t, r, nxt) : true;
      if (!__all_sync(0xffffffffu, ok)) break;
      t = __shfl_sync(0xffffffffu, nxt, 0);
    }
    // Shared memory must not be released while a store still reads it; the
    // stores' global writes complete before the grid does.
    if (lane == 0) ptx::bulk_wait_read<0>();
    __syncwarp();
  }

  // Both CTAs have passed their last use of the pair's resources (tensor
  // memory, the barriers the other CTA signals, the schedule responses)
  // before either frees the tensor memory and leaves.  Only the order of
  // execution matters here, so the arrive is relaxed: a release would also
  // wait for this CTA's output stores to reach global memory (~0.6 us).
  ptx::tc_fence_before();
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
  asm volatile("barrier.cluster.wait;" ::: "memory");
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace swiglu
