// swiglu_dq_kernel.cuh -- the fused SwiGLU projection with low-precision
// weights (INT4, MXFP8, NVFP4; A and Y stay BF16) for wide weight matrices.
//
// Computes Y = SiLU(A x W1) (.) (A x W2) (page "Riepilogo Tecnico:
// Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza
// Efficiente di LLM", section "Definizione del Problema"), separate weight
// form (section "Metodologia", item 1), with W1, W2 given as codes and block
// scales (weight_decode.cuh).
//
// One CTA computes one 128 x 128 output tile over all of K (or, for M > 128,
// two 128-row blocks of the same columns: 256 x 128).  Wide tiles are
// the point: every CTA reads its 128 rows of A once for 128 output columns
// (256 gate and up columns), so A's bytes per weight byte are half those of a
// 64-column tile -- with 4-bit weights A is otherwise the larger stream.
//   * warp 8 (one thread) streams each K step's A box(es) into a short ring
//     and warp 10 (one thread) the two matrices' code and scale boxes into a
//     deep one (TMA): the weight stream is small per step, so many steps of
//     it are in flight;
//   * warps 0-7 decode each step's codes into one of two BF16 operand
//     buffers ([64 K x 256] in the 128-byte-swizzled layout) and release the
//     codes slot;
//   * warp 9 (one thread) issues tcgen05.mma M=128 x N=256 x K=16 per row
//     block, gate and up columns side by side in TMEM (block i: columns
//     [256 i, 256 i + 128) gate, [256 i + 128, 256 i + 256) up), and frees the
//     decoded buffer and the A slot through tcgen05.commit;
//   * after the last K step warps 0-7 run the usual epilogue for each row
//     block (TMEM loads, SiLU(g) * u in FP32, BF16, TMA stores through
//     staging buffers that reuse the decoded buffers), applying NVFP4's
//     per-tensor scales.
// Every wait is bounded (timeout -> error word, abort flag, drain, TMEM freed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"
#include "weight_decode.cuh"

namespace swiglu {

// MB_: 128-row blocks of A per CTA (1 or 2).  With two, one decode of each
// weight step feeds the MMAs of both blocks (two accumulators, all 512 TMEM
// columns): the decode, the weight stream and the per-step protocol are shared
// by 256 rows.
template <int WF_, int MB_ = 1>
struct DqCfg {
  static constexpr int WF = WF_;
  static constexpr int MB = MB_;
  static constexpr int BM = 128, BK = 64, BN = 128;
  static constexpr int MMA_N = 2 * BN;               // gate + up
  static constexpr int ATOM_COLS = 64;
  static constexpr int ATOM_BYTES = BK * ATOM_COLS * 2;  // 8 KB
  static constexpr int A_BOX_BYTES = BM * BK * 2;      // one block's A box, 16 KB
  static constexpr int A_BYTES = MB * A_BOX_BYTES;       // one A stage
  static constexpr int DEC_BYTES = 4 * ATOM_BYTES;     // one decoded buffer: W1 then W2, 32 KB
  static constexpr int CODE_ROW_BYTES = BN * WFormat<WF>::CODE_BITS / 8;
  static constexpr int RAW_W_BYTES = BK * CODE_ROW_BYTES;
  static constexpr int RAW_S_BYTES = WFormat<WF>::SCALE_ROWS * BN * WFormat<WF>::SCALE_BYTES;
  static constexpr int RAW_BYTES = 2 * (RAW_W_BYTES + RAW_S_BYTES);  // codes + scales of one K step
  // Two rings: A (from L2, short latency) and the codes (from DRAM, small):
  // the codes ring is as deep as the rest of shared memory allows (about
  // 104 KB, 56 KB with two A blocks), so many K steps of the weight stream
  // are in flight while A and the decode keep pace.
  static constexpr int A_STAGES = 3;
  static constexpr int C_STAGES_RAW = ((MB == 1 ? 104 : 56) * 1024) / RAW_BYTES;
  static constexpr int C_STAGES = C_STAGES_RAW > 16 ? 16 : C_STAGES_RAW;
  static constexpr int DEC_BUFS = 2;
  static constexpr int C_OFF = A_STAGES * A_BYTES;
  static constexpr int DEC_OFF = (C_OFF + C_STAGES * RAW_BYTES + 1023) / 1024 * 1024;
  static constexpr int BAR_OFF = DEC_OFF + DEC_BUFS * DEC_BYTES;
  // a_full[A], a_empty[A], c_full[C], c_empty[C], dfull[D], dempty[D], acc_full, drain, spare
  static constexpr int NUM_BARS = 2 * A_STAGES + 2 * C_STAGES + 2 * DEC_BUFS + 3;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  static constexpr int EPI_WARPS = 8, PRODUCER_WARP = 8, MMA_WARP = 9, CODES_WARP = 10;
  static constexpr int THREADS = 32 * 11;
  static constexpr int TMEM_COLS = 256 * MB;
  // 4-bit codes (INT4, NVFP4) decode as column pairs (c, c + 4): fewer
  // operations; the accumulator columns then carry that order, undone by the
  // epilogue
  static constexpr bool PAIRED = WF == WF_INT4 || WF == WF_NVFP4;
  static constexpr int B_SBO = 8 * 128, B_KSTEP = 16 * 128;
  static constexpr int STG_BYTES = 32 * 64;  // a warp's 32 x 32 BF16 staging block
  static constexpr uint32_t IDESC = ptx::idesc_bf16(BM, MMA_N, false, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(RAW_BYTES % 128 == 0, "codes stages stay 128-byte aligned");
  static_assert(C_STAGES >= (MB == 1 ? 4 : 3), "codes ring depth");
  static_assert(MB == 1 || MB == 2, "one or two 128-row blocks");
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
  auto a_full = [&](int s) { return bars + 8u * s; };
  auto a_empty = [&](int s) { return bars + 8u * (C::A_STAGES + s); };
  auto c_full = [&](int s) { return bars + 8u * (2 * C::A_STAGES + s); };
  auto c_empty = [&](int s) { return bars + 8u * (2 * C::A_STAGES + C::C_STAGES + s); };
  auto dfull_bar = [&](int d) { return bars + 8u * (2 * C::A_STAGES + 2 * C::C_STAGES + d); };
  auto dempty_bar = [&](int d) {
    return bars + 8u * (2 * C::A_STAGES + 2 * C::C_STAGES + C::DEC_BUFS + d);
  };
  const uint32_t accf_bar = bars + 8u * (2 * C::A_STAGES + 2 * C::C_STAGES + 2 * C::DEC_BUFS);
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
    for (int s = 0; s < C::A_STAGES; ++s) {
      ptx::mbar_init(a_full(s), 1);
      ptx::mbar_init(a_empty(s), 1);            // the MMA's commit
    }
    for (int s = 0; s < C::C_STAGES; ++s) {
      ptx::mbar_init(c_full(s), 1);
      ptx::mbar_init(c_empty(s), C::EPI_WARPS);  // every decoding warp
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

  // One ring's producer: waits for a free slot, then `load(slot, barrier, k)`.
  auto produce = [&](int stages, auto full, auto empty, uint32_t bytes, auto load) {
    uint32_t slot = 0, phase = 0, issued = 0;
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      if (!wait_bar(empty(slot), phase ^ 1u, p.timeout_ns, abort_flag, p.err, WAIT_PRODUCER_EMPTY)) {
        ok = false;
        break;
      }
      ptx::mbar_arrive_expect_tx(full(slot), bytes);
      load(static_cast<int>(slot), full(slot), kstep(i));
      ++issued;
      if (++slot == static_cast<uint32_t>(stages)) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {  // let the copies in flight land before shared memory is released
      const uint32_t n = issued < (uint32_t)stages ? issued : (uint32_t)stages;
      for (uint32_t i = issued - n; i < issued; ++i)
        wait_quiet(full(i % stages), (i / stages) & 1u, p.timeout_ns);
    }
  };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ A producer
    if (lane == 0)
      produce(C::A_STAGES, a_full, a_empty, C::A_BYTES, [&](int s, uint32_t fb, int kb) {
#pragma unroll
        for (int i = 0; i < C::MB; ++i)
          ptx::tma_load_2d(base + s * C::A_BYTES + i * C::A_BOX_BYTES, &tmA, fb, kb * C::BK,
                           (mb * C::MB + i) * C::BM);
      });
    __syncwarp();
  } else if (warp == C::CODES_WARP) {
    // ------------------------------------------------------------ codes producer
    if (lane == 0)
      produce(C::C_STAGES, c_full, c_empty, C::RAW_BYTES, [&](int s, uint32_t fb, int kb) {
        const uint32_t r = base + C::C_OFF + s * C::RAW_BYTES;
        const int g = C::WF == WF_INT4 ? kb * C::BK / p.w4_group : kb * WFormat<C::WF>::SCALE_ROWS;
        ptx::tma_load_2d(r, &tmC1, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
        ptx::tma_load_2d(r + C::RAW_W_BYTES, &tmC2, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
        ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES, &tmS1, fb, nb * C::BN, g);
        ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES + C::RAW_S_BYTES, &tmS2, fb, nb * C::BN, g);
      });
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t a = 0, aphase = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {  // kb: position in the (rotated) K loop
        const int d = kb % C::DEC_BUFS;
        const uint32_t dphase = static_cast<uint32_t>(kb / C::DEC_BUFS) & 1u;
        if (!wait_bar(a_full(a), aphase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL) ||
            !wait_bar(dfull_bar(d), dphase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = base + a * C::A_BYTES;
        const uint32_t sb = base + C::DEC_OFF + d * C::DEC_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint64_t bdesc =
              ptx::smem_desc(sb + kk * C::B_KSTEP, C::ATOM_BYTES, C::B_SBO, ptx::SW_128B);
#pragma unroll
          for (int i = 0; i < C::MB; ++i) {  // block i accumulates in columns [256 i, 256 i + 256)
            const uint64_t adesc =
                ptx::smem_desc(sa + i * C::A_BOX_BYTES + kk * 32, 16, 1024, ptx::SW_128B);
            ptx::mma_f16(tmem_base + i * C::MMA_N, adesc, bdesc, C::IDESC,
                         (kb | kk) != 0 ? 1u : 0u);
          }
        }
        ptx::mma_commit(a_empty(a));        // this A stage has been read
        ptx::mma_commit(dempty_bar(d));     // and the decoded buffer
        if (++a == static_cast<uint32_t>(C::A_STAGES)) {
          a = 0;
          aphase ^= 1u;
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
    uint32_t c = 0, cphase = 0;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int d = kb % C::DEC_BUFS;
      const uint32_t dphase = static_cast<uint32_t>(kb / C::DEC_BUFS) & 1u;
      ok = wait_bar(c_full(c), cphase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL) &&
           wait_bar(dempty_bar(d), dphase ^ 1u, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t *st = smem + C::C_OFF + c * C::RAW_BYTES;
      const int t = static_cast<int>(threadIdx.x) >> 7;  // 0: gate, 1: up
      decode_weights<C::WF, C::BN, 128, C::ATOM_BYTES, C::PAIRED>(
          st + t * C::RAW_W_BYTES, st + 2 * C::RAW_W_BYTES + t * C::RAW_S_BYTES,
          smem + C::DEC_OFF + d * C::DEC_BYTES + t * 2 * C::ATOM_BYTES, threadIdx.x & 127);
      ptx::fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(dfull_bar(d));
        ptx::mbar_arrive(c_empty(c));  // this stage's codes have been read
      }
      if (++c == static_cast<uint32_t>(C::C_STAGES)) {
        c = 0;
        cphase ^= 1u;
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
#pragma unroll 1
      for (int i = 0; i < C::MB; ++i) {
        const int row_blk = (mb * C::MB + i) * C::BM;
        if (row_blk >= p.M) break;  // a second block wholly below the matrix
        epilogue_tile<false, C::BN, C::WF == WF_NVFP4, C::PAIRED>(
            tacc + i * C::MMA_N, row_blk + q * 32, nb * C::BN, 2 * h, 2 * h + 2, &tmY, p.M, p.N,
            smem, base, stg_base, it, lane, spare_bar, gs, us);
      }
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
