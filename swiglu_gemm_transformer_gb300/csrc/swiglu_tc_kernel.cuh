// swiglu_tc_kernel.cuh -- the one-CTA fused SwiGLU tcgen05 kernel for sm_103a.
//
// Computes Y = SiLU(A x W1) (.) (A x W2) (page "Riepilogo Tecnico:
// Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza
// Efficiente di LLM", section "Definizione del Problema") one 128-row output
// tile at a time, in either weight form the page describes (section
// "Metodologia": two separate weight matrices, item 1, or one interleaved
// W_fused[K,2N], item 2).
//
// GB300 design (the page's kernels target H100 and register accumulators):
//   * persistent CTAs, one per SM, walk the output tiles in a grouped order so
//     that concurrently running tiles share A rows and weight columns in L2;
//   * warp 8 (one thread) streams A[128 x 64] and the weight tile
//     [64 x MMA_N] of every K step into a STAGES-deep shared-memory ring with
//     TMA (128- or 64-byte swizzle), completion counted on mbarriers;
//   * warp 9 (one thread) issues tcgen05.mma.kind::f16 M=128 x N=MMA_N x K=16.
//     The B operand of one MMA holds the gate columns AND the up columns of the
//     tile side by side, so a single instruction produces both accumulators in
//     tensor memory: separate form -> TMEM columns [0,BN) = gate, [BN,2BN) = up;
//     interleaved form -> column 2j = gate j, 2j+1 = up j (the page's
//     PairMulStore pairing, now on adjacent TMEM columns);
//   * the accumulators are double-buffered in TMEM (2 x MMA_N columns) so the
//     epilogue of tile i overlaps the MMAs of tile i+1;
//   * warps 0-7 (the epilogue; warp w reads TMEM lanes 32*(w%4).. and half
//     w/4 of the tile's columns) apply y = g * u / (1 + e^-g) in FP32, round
//     to BF16 (RNE), stage 32x32 blocks in shared memory (64-byte swizzle,
//     bank-conflict free) and write them with TMA stores whose completion
//     overlaps the next block's arithmetic (the compute/store overlap of the
//     page's Kernel-2).
//   Gate and up values never leave the SM.
//
// Programmatic dependent launch: the prologue (barriers, TMEM, descriptor
// prefetch) runs before griddepcontrol.wait, so it overlaps the previous
// kernel on the stream; no global memory is touched before the wait.
//
// Every mbarrier wait is bounded by a time limit.  On expiry the waiting
// thread records SWIGLU_ERR_TIMEOUT in the device error word, raises a CTA
// abort flag so the other roles stop at their next wait, in-flight copies and
// MMAs are drained (again with a limit), TMEM is freed and the CTA returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace swiglu {

// NB_ATOMS weight boxes of ATOM_COLS columns make the MMA's B operand.
//   ATOM_COLS = 64: 128-byte swizzle; ATOM_COLS = 32: 64-byte swizzle.
template <int NB_ATOMS_, int ATOM_COLS_, bool INTERLEAVED_, int STAGES_>
struct TileCfg {
  static constexpr int NB_ATOMS = NB_ATOMS_;
  static constexpr int ATOM_COLS = ATOM_COLS_;
  static constexpr bool INTERLEAVED = INTERLEAVED_;
  static constexpr int STAGES = STAGES_;
  static constexpr int BM = 128;                 // rows per tile (MMA M)
  static constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row of A
  static constexpr int MMA_N = NB_ATOMS * ATOM_COLS;  // gate+up accumulator columns per tile
  static constexpr int BN = MMA_N / 2;           // output columns per tile
  static constexpr int A_BYTES = BM * BK * 2;    // 16 KB
  static constexpr int ROW_BYTES = ATOM_COLS * 2;          // one K-row of a weight box
  static constexpr int ATOM_BYTES = BK * ROW_BYTES;        // one weight box
  static constexpr uint32_t B_SWIZZLE = ATOM_COLS == 64 ? ptx::SW_128B : ptx::SW_64B;
  static constexpr int B_SBO = 8 * ROW_BYTES;              // 8-row K group
  static constexpr int B_KSTEP = 16 * ROW_BYTES;           // 16 K-rows = one MMA's K
  static constexpr int B_BYTES = NB_ATOMS * ATOM_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_WARPS = 8;
  static constexpr int STG_BYTES = 32 * 64;      // a warp's 32 rows x 32 BF16 columns
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + EPI_WARPS * 2 * STG_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;  // full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;  // + slot/flag + alignment slack
  static constexpr int TMEM_COLS = (2 * MMA_N <= 128) ? 128 : (2 * MMA_N <= 256) ? 256 : 512;
  static constexpr int PRODUCER_WARP = EPI_WARPS;
  static constexpr int MMA_WARP = EPI_WARPS + 1;
  static constexpr int THREADS = 32 * (EPI_WARPS + 2);
  static constexpr uint32_t IDESC = ptx::idesc_bf16(BM, MMA_N, false, true);
  static_assert(MMA_N % 16 == 0 && MMA_N >= 64 && MMA_N <= 256, "MMA N");
  static_assert(INTERLEAVED || NB_ATOMS % 2 == 0, "separate form: half the boxes per weight");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
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
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit0 = static_cast<int>(blockIdx.x);
  const int unit_step = static_cast<int>(gridDim.x);

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar(b), 1);
      ptx::mbar_init(acce_bar(b), C::EPI_WARPS);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (!C::INTERLEAVED) ptx::prefetch_tmap(&tmB1);
    ptx::prefetch_tmap(&tmY);
  }
  if (warp == C::MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above overlaps the previous kernel when launched with PDL.
  ptx::grid_launch_dependents();
  if (warp == C::PRODUCER_WARP && lane == 0) {
    // Warm the TMA unit's descriptor cache while the previous kernel ends.
    ptx::tma_prefetch_2d(&tmA, 0, 0);
    ptx::tma_prefetch_2d(&tmB0, 0, 0);
    if (!C::INTERLEAVED) ptx::tma_prefetch_2d(&tmB1, 0, 0);
  }
  const int num_units = p.num_m_blk * p.num_n_blk;
  // The weight boxes of one stage (K step kb of column block nb).
  auto load_w = [&](uint32_t sb, uint32_t fb, int nb, int kb) {
    if (C::INTERLEAVED) {
#pragma unroll
      for (int j = 0; j < C::NB_ATOMS; ++j)
        ptx::tma_load_2d(sb + j * C::ATOM_BYTES, &tmB0, fb, nb * C::MMA_N + j * C::ATOM_COLS,
                         kb * C::BK);
    } else {
#pragma unroll
      for (int j = 0; j < C::NB_ATOMS / 2; ++j) {
        ptx::tma_load_2d(sb + j * C::ATOM_BYTES, &tmB0, fb, nb * C::BN + j * C::ATOM_COLS,
                         kb * C::BK);
        ptx::tma_load_2d(sb + (C::NB_ATOMS / 2 + j) * C::ATOM_BYTES, &tmB1, fb,
                         nb * C::BN + j * C::ATOM_COLS, kb * C::BK);
      }
    }
  };
  // Weights known to be unwritten by earlier work: the first tile's first
  // stages of weight boxes go out before the dependency wait (the stages are
  // fresh, so no empty-barrier wait is needed); their A boxes follow after it.
  uint32_t pre = 0;
  if (warp == C::PRODUCER_WARP && p.w_early && unit0 < num_units) {
    pre = p.num_k_blk < C::STAGES ? p.num_k_blk : C::STAGES;
    if (lane == 0) {
      int mb, nb;
      tile_coords(unit0, p, mb, nb);
      for (uint32_t s = 0; s < pre; ++s) {
        ptx::mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
        load_w(base + s * C::STAGE_BYTES + C::A_BYTES, full_bar(s), nb, (int)s);
      }
    }
    __syncwarp();
  }
  ptx::grid_dependency_wait();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = unit0; ok && t < num_units; t += unit_step) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        for (int kb = 0; kb < p.num_k_blk; ++kb) {
          const bool early = issued < pre;  // weights already on their way
          if (!early && !wait_bar(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, p.err,
                                  WAIT_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          const uint32_t fb = full_bar(stage);
          if (!early) ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmA, fb, kb * C::BK, mb * C::BM);
          if (!early) load_w(sb, fb, nb, kb);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA's shared
        // memory is released: wait for the last min(issued, STAGES) loads.
        const uint32_t n = issued < (uint32_t)C::STAGES ? issued : (uint32_t)C::STAGES;
        for (uint32_t i = issued - n; i < issued; ++i)
          wait_quiet(full_bar(i % C::STAGES), (i / C::STAGES) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
      bool ok = true;
      for (int t = unit0; ok && t < num_units; t += unit_step) {
        if (!wait_bar(acce_bar(abuf), aphase ^ 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_MMA_ACC_EMPTY)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + abuf * C::MMA_N;
        for (int kb = 0; kb < p.num_k_blk; ++kb) {
          if (!wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = base + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            // A: K-major, 128-byte swizzle; 16 K-elements = 32 bytes along the row.
            const uint64_t adesc = ptx::smem_desc(sa + kk * 32, 16, 1024, ptx::SW_128B);
            // B: MN-major; weight boxes ATOM_BYTES apart (LBO), 8-row K groups
            // B_SBO apart, one MMA's 16 K-rows = B_KSTEP bytes.
            const uint64_t bdesc =
                ptx::smem_desc(sb + kk * C::B_KSTEP, C::ATOM_BYTES, C::B_SBO, C::B_SWIZZLE);
            ptx::mma_f16(d, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(empty_bar(stage));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(accf_bar(abuf));
        if (++abuf == 2) {
          abuf = 0;
          aphase ^= 1u;
        }
      }
      // Every MMA this thread issued completes before TMEM can be freed.
      ptx::mma_commit(drain_bar);
      wait_quiet(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
    const int q = warp & 3;   // TMEM lanes [32q, 32q+32) = tile rows [32q, 32q+32)
    const int h = warp >> 2;  // which half of the tile's 32-column chunks
    constexpr int NC = C::BN / 32;
    const int c_begin = NC >= 2 ? h * (NC / 2) : 0;
    const int c_end = NC >= 2 ? (h + 1) * (NC / 2) : (h == 0 ? NC : 0);
    const uint32_t stg_base = base + C::STG_OFF + warp * 2 * C::STG_BYTES;
    uint32_t abuf = 0, aphase = 0, it = 0;
    for (int t = unit0; t < num_units; t += unit_step) {
      int mb, nb;
      tile_coords(t, p, mb, nb);
      bool ok = wait_bar(accf_bar(abuf), aphase, p.timeout_ns, abort_flag, p.err,
                         WAIT_EPI_ACC_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf * C::MMA_N;
      epilogue_tile<C::INTERLEAVED, C::BN>(tacc, mb * C::BM + q * 32, nb * C::BN, c_begin, c_end,
                                           &tmY, p.M, p.N, smem, base, stg_base, it, lane,
                                           acce_bar(abuf));
      if (++abuf == 2) {
        abuf = 0;
        aphase ^= 1u;
      }
    }
    // Shared memory must not be released while a store still reads it; the
    // stores' global writes complete before the grid does.
    if (lane == 0) ptx::bulk_wait_read<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// A kernel whose only wait is on a barrier that nothing ever completes: it
// exercises the bounded-wait failure path (records SWIGLU_ERR_TIMEOUT and
// returns).
__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t *err);

}  // namespace swiglu
