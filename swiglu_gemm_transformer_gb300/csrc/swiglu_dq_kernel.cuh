// swiglu_dq_kernel.cuh -- the fused SwiGLU projection with low-precision
// weights (INT4, MXFP8, NVFP4; A and Y stay BF16) for wide weight matrices.
//
// Computes Y = SiLU(A x W1) (.) (A x W2) (page "Riepilogo Tecnico:
// Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza
// Efficiente di LLM", section "Definizione del Problema"), separate weight
// form (section "Metodologia", item 1), with W1, W2 given as codes and block
// scales (weight_decode.cuh).
//
// One CTA computes one 128 x 128 output tile over all of K.  Wide tiles are
// the point: every CTA reads its 128 rows of A once for 128 output columns
// (256 gate and up columns), so A's bytes per weight byte are half those of a
// 64-column tile -- with 4-bit weights A is otherwise the larger stream.
//   * warp 8 (one thread) streams each K step's A box and the two matrices'
//     code and scale boxes into a STAGES-deep ring (TMA);
//   * warps 0-7 decode each stage's codes into one of three BF16 operand
//     buffers ([64 K x 256] in the 128-byte-swizzled layout), then release the
//     stage's codes (the stage is free once the MMA has also read its A);
//   * warp 9 (one thread) issues tcgen05.mma M=128 x N=256 x K=16, gate and
//     up columns side by side in TMEM (columns [0,128) gate, [128,256) up),
//     and frees the decoded buffer and the A stage through tcgen05.commit;
//   * after the last K step warps 0-7 run the usual epilogue (TMEM loads,
//     SiLU(g) * u in FP32, BF16, TMA stores through staging buffers that
//     reuse the decoded buffers), applying NVFP4's per-tensor scales.
// Every wait is bounded (timeout -> error word, abort flag, drain, TMEM freed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"
#include "weight_decode.cuh"

namespace swiglu {

template <int WF_>
struct DqCfg {
  static constexpr int WF = WF_;
  static constexpr int BM = 128, BK = 64, BN = 128;
  static constexpr int MMA_N = 2 * BN;               // gate + up
  static constexpr int ATOM_COLS = 64;
  static constexpr int ATOM_BYTES = BK * ATOM_COLS * 2;  // 8 KB
  static constexpr int A_BYTES = BM * BK * 2;          // 16 KB
  static constexpr int DEC_BYTES = 4 * ATOM_BYTES;     // one decoded buffer: W1 then W2, 32 KB
  static constexpr int CODE_ROW_BYTES = BN * WFormat<WF>::CODE_BITS / 8;
  static constexpr int RAW_W_BYTES = BK * CODE_ROW_BYTES;
  static constexpr int RAW_S_BYTES = WFormat<WF>::SCALE_ROWS * BN * WFormat<WF>::SCALE_BYTES;
  static constexpr int TMA_BYTES = A_BYTES + 2 * (RAW_W_BYTES + RAW_S_BYTES);
  static constexpr int STAGE_BYTES = (TMA_BYTES + 1023) / 1024 * 1024;
  // Three decoded buffers let the decoders run a stage ahead of the MMA, so
  // the barrier round trips between them overlap work instead of adding to it.
  static constexpr int DEC_BUFS = 3;
  static constexpr int STAGES = WF == WF_MXFP8 ? 3 : 4;
  static constexpr int DEC_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = DEC_OFF + DEC_BUFS * DEC_BYTES;
  // full[S], empty[S], dfull[D], dempty[D], acc_full, drain, spare
  static constexpr int NUM_BARS = 2 * STAGES + 2 * DEC_BUFS + 3;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  static constexpr int EPI_WARPS = 8, PRODUCER_WARP = 8, MMA_WARP = 9, THREADS = 320;
  static constexpr int TMEM_COLS = 256;
  static constexpr int B_SBO = 8 * 128, B_KSTEP = 16 * 128;
  static constexpr int STG_BYTES = 32 * 64;  // a warp's 32 x 32 BF16 staging block
  static constexpr uint32_t IDESC = ptx::idesc_bf16(BM, MMA_N, false, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(EPI_WARPS * 2 * STG_BYTES <= DEC_BUFS * DEC_BYTES, "staging reuses the decoded buffers");
  static_assert(WF != WF_BF16, "a decoded weight format");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_dq_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmC1,  // gate codes
                     const __grid_constant__ CUtensorMap tmC2,  // up codes
                     const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmS1,  // gate scales
                     const __grid_constant__ CUtensorMap tmS2,  // up scales
                     const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const uint32_t bars = base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::STAGES + s); };
  auto dfull_bar = [&](int d) { return bars + 8u * (2 * C::STAGES + d); };
  auto dempty_bar = [&](int d) { return bars + 8u * (2 * C::STAGES + C::DEC_BUFS + d); };
  const uint32_t accf_bar = bars + 8u * (2 * C::STAGES + 2 * C::DEC_BUFS);
  const uint32_t drain_bar = accf_bar + 8u;
  const uint32_t spare_bar = accf_bar + 16u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int mb, nb;
  tile_coords(static_cast<int>(blockIdx.x), p, mb, nb);
  const int nk = p.num_k_blk;
  // Every CTA reads the same A columns; starting each CTA's K loop at a
  // different step spreads those reads over the whole of A instead of
  // sending every SM to the same few L2 lines at the same moment.
  const int k_rot = static_cast<int>((static_cast<int64_t>(blockIdx.x) * nk) / gridDim.x) % (nk > 0 ? nk : 1);
  auto kstep = [&](int i) { return i + k_rot < nk ? i + k_rot : i + k_rot - nk; };

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1 + C::EPI_WARPS);  // the MMA's A and the decoders' codes
    }
    for (int d = 0; d < C::DEC_BUFS; ++d) {
      ptx::mbar_init(dfull_bar(d), C::EPI_WARPS);
      ptx::mbar_init(dempty_bar(d), 1);
    }
    ptx::mbar_init(accf_bar, 1);
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(spare_bar, (1 << 20) - 1);  // the epilogue's release arrivals; nothing waits on it
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmC1);
    ptx::prefetch_tmap(&tmC2);
    ptx::prefetch_tmap(&tmS1);
    ptx::prefetch_tmap(&tmS2);
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
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int kb = kstep(i);
        if (!wait_bar(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_PRODUCER_EMPTY)) {
          ok = false;
          break;
        }
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t r = sa + C::A_BYTES;
        const uint32_t fb = full_bar(stage);
        const int g = C::WF == WF_INT4 ? kb * C::BK / p.w4_group : kb * WFormat<C::WF>::SCALE_ROWS;
        ptx::mbar_arrive_expect_tx(fb, C::TMA_BYTES);
        ptx::tma_load_2d(sa, &tmA, fb, kb * C::BK, mb * C::BM);
        ptx::tma_load_2d(r, &tmC1, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
        ptx::tma_load_2d(r + C::RAW_W_BYTES, &tmC2, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
        ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES, &tmS1, fb, nb * C::BN, g);
        ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES + C::RAW_S_BYTES, &tmS2, fb, nb * C::BN, g);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        const uint32_t n = issued < (uint32_t)C::STAGES ? issued : (uint32_t)C::STAGES;
        for (uint32_t i = issued - n; i < issued; ++i)
          wait_quiet(full_bar(i % C::STAGES), (i / C::STAGES) & 1u, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {  // kb: position in the (rotated) K loop
        const int d = kb % C::DEC_BUFS;
        const uint32_t dphase = static_cast<uint32_t>(kb / C::DEC_BUFS) & 1u;
        if (!wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL) ||
            !wait_bar(dfull_bar(d), dphase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t sb = base + C::DEC_OFF + d * C::DEC_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint64_t adesc = ptx::smem_desc(sa + kk * 32, 16, 1024, ptx::SW_128B);
          const uint64_t bdesc =
              ptx::smem_desc(sb + kk * C::B_KSTEP, C::ATOM_BYTES, C::B_SBO, ptx::SW_128B);
          ptx::mma_f16(tmem_base, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        ptx::mma_commit(empty_bar(stage));  // this stage's A has been read
        ptx::mma_commit(dempty_bar(d));     // and the decoded buffer
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) ptx::mma_commit(accf_bar);
      ptx::mma_commit(drain_bar);
      wait_quiet(drain_bar, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ decode, then epilogue (warps 0-7)
    bool ok = true;
    uint32_t stage = 0, phase = 0;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int d = kb % C::DEC_BUFS;
      const uint32_t dphase = static_cast<uint32_t>(kb / C::DEC_BUFS) & 1u;
      ok = wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL) &&
           wait_bar(dempty_bar(d), dphase ^ 1u, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      uint8_t *st = smem + stage * C::STAGE_BYTES + C::A_BYTES;
      const int t = static_cast<int>(threadIdx.x) >> 7;  // 0: gate, 1: up
      decode_weights<C::WF, C::BN, 128, C::ATOM_BYTES>(
          st + t * C::RAW_W_BYTES, st + 2 * C::RAW_W_BYTES + t * C::RAW_S_BYTES,
          smem + C::DEC_OFF + d * C::DEC_BYTES + t * 2 * C::ATOM_BYTES, threadIdx.x & 127);
      ptx::fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(dfull_bar(d));
        ptx::mbar_arrive(empty_bar(stage));  // this stage's codes have been read
      }
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    ok = ok && wait_bar(accf_bar, 0, p.timeout_ns, abort_flag, p.err, WAIT_EPI_ACC_FULL);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      ptx::tc_fence_after();
      const int q = warp & 3;   // TMEM lanes [32q, 32q+32)
      const int h = warp >> 2;  // 32-column chunks [2h, 2h+2)
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const uint32_t stg_base = base + C::DEC_OFF + warp * 2 * C::STG_BYTES;
      uint32_t it = 0;
      const float gs = C::WF == WF_NVFP4 ? *p.sW1 : 1.0f;
      const float us = C::WF == WF_NVFP4 ? *p.sW2 : 1.0f;
      epilogue_tile<false, C::BN, C::WF == WF_NVFP4>(tacc, mb * C::BM + q * 32, nb * C::BN, 2 * h,
                                                     2 * h + 2, &tmY, p.M, p.N, smem, base,
                                                     stg_base, it, lane, spare_bar, gs, us);
      if (lane == 0) ptx::bulk_wait_read<0>();
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace swiglu
