// swiglu_sk_kernel.cuh -- split-K fused SwiGLU kernel for small M on sm_103a.
//
// Same result as the other kernels, Y = SiLU(A x W1) (.) (A x W2) (page
// "Riepilogo Tecnico: Sovrapposizione delle Attivazioni a Livello di Tile per
// l'Inferenza Efficiente di LLM", section "Definizione del Problema"), in either
// weight form (section "Metodologia", items 1 and 2).
//
// Why a separate kernel: with M <= 128 the call is a stream of the weights
// (2*K*N*2 bytes, 17.4 MB for the Qwen-2.5-0.5B MLP), and what limits it is how
// much of that stream each SM keeps in flight.  A one-CTA tile needs all of A
// (M x K) next to its weight columns, so a 128-row tile of 32 columns on every
// SM holds only 8 of its 14 K steps in shared memory and waits a second DRAM
// round trip for the rest.  Here a CLUSTER OF TWO CTAs computes one 128 x 64
// output tile and each CTA takes half of the K steps:
//   * per CTA: A[128 x K/2] and the tile's 64 gate + 64 up weight columns over
//     K/2 -- half the A bytes of a one-CTA tile, and all of them in flight;
//   * warp 4 streams its K half into a 6-stage ring (TMA, 128-byte swizzle);
//     warp 5 issues tcgen05.mma M=128 x N=128 (gate and up side by side in
//     TMEM, as in the one-CTA kernel) over that half;
//   * the two partial accumulators are summed through distributed shared
//     memory: CTA r keeps output columns [32r, 32r+32) of the tile for all
//     rows.  Eight epilogue warps (four TMEM lane groups x two 16-column
//     halves, so all four SM sub-partitions share the work) each send the
//     peer their partial gate/up sums of 16 of the peer's columns with
//     st.async (16 bytes per store, counted on the mbarrier of the peer's
//     warp that keeps those columns, so each warp can go on as soon as its
//     own 4 KB are in), then wait for the peer's sums of their own 16
//     columns, add them, apply
//     y = g * u / (1 + e^-g) in FP32, round to BF16 and store their 32 bytes
//     of each row directly.  With few rows this epilogue is not hidden behind
//     MMAs, so its length is what the exchange and the activation take.
// Gate and up values never reach global memory.  One tile per cluster (no
// persistent loop): the launcher sizes the grid to two CTAs per output tile.
//
// Every wait is bounded as in the other kernels (timeout -> error word, abort
// flag, drain, TMEM freed).  A CTA leaves only once everything its peer
// sends it has arrived (or, after a timeout, once late stores have had time
// to land), so no store targets a CTA that has left.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"
#include "weight_decode.cuh"

namespace swiglu {

enum : uint32_t { WAIT_SK_RECV = 7 };

// Weight formats of the split-K kernel.  Besides BF16, the weights may arrive
// as low-precision codes with block scales; the epilogue warps, idle during
// the K loop, decode each stage into the BF16 operand layout the MMA reads
// (see the decode functions above the kernel):
//   WF_INT4  : signed 4-bit codes (two per byte along N), BF16 scale per
//              column and group of K rows;
//   WF_MXFP8 : E4M3 codes, E8M0 scale per column and 32 K rows;
//   WF_NVFP4 : E2M1 codes (two per byte along N), E4M3 scale per column and
//              16 K rows, and one FP32 scale per tensor (applied to the
//              gate and up sums before the activation).
template <bool INTERLEAVED_, int WF_ = WF_BF16>
struct SkCfg {
  static constexpr bool INTERLEAVED = INTERLEAVED_;
  static constexpr int WF = WF_;
  static constexpr bool DECODE = WF != WF_BF16;
  // 4-bit codes (INT4, NVFP4) decode as column pairs (c, c + 4); within every
  // 8 accumulator columns the outputs then lie in the order 0 4 1 5 2 6 3 7
  static constexpr bool PAIRED = (WF == WF_INT4 || WF == WF_NVFP4) && !INTERLEAVED_;
  static constexpr int BM = 128;                 // rows per tile (MMA M)
  static constexpr int BK = 64;                  // K per stage
  static constexpr int BN = 64;                  // output columns per tile
  static constexpr int MMA_N = 2 * BN;           // gate + up accumulator columns
  static constexpr int ATOM_COLS = 64;           // one weight box: 64 columns, 128-byte swizzle
  static constexpr int NB_ATOMS = 2;
  static constexpr int A_BYTES = BM * BK * 2;    // 16 KB
  static constexpr int ROW_BYTES = ATOM_COLS * 2;
  static constexpr int ATOM_BYTES = BK * ROW_BYTES;  // 8 KB
  static constexpr int B_SBO = 8 * ROW_BYTES;
  static constexpr int B_KSTEP = 16 * ROW_BYTES;
  static constexpr int B_BYTES = NB_ATOMS * ATOM_BYTES;
  // Decoded formats: per weight matrix a [64 K rows x 64 columns] box of codes
  // and a [SCALE_ROWS x 64] box of scales, behind the A tile and the decoded
  // B tiles of the stage.
  static constexpr int CODE_ROW_BYTES = ATOM_COLS * WFormat<WF>::CODE_BITS / 8;  // per K row
  static constexpr int SCALE_ROWS = WFormat<WF>::SCALE_ROWS;     // per 64 K rows
  static constexpr int SCALE_ELEM = WFormat<WF>::SCALE_BYTES;    // bytes per scale
  static constexpr int RAW_W_BYTES = BK * CODE_ROW_BYTES;
  static constexpr int RAW_S_BYTES = SCALE_ROWS * ATOM_COLS * SCALE_ELEM;
  static constexpr int RAW_OFF = A_BYTES + B_BYTES;
  static constexpr int RAW_BYTES = DECODE ? 2 * (RAW_W_BYTES + RAW_S_BYTES) : 0;
  static constexpr int TMA_BYTES = A_BYTES + (DECODE ? RAW_BYTES : B_BYTES);  // bytes TMA lands per stage
  static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + RAW_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGES = !DECODE ? 6 : WF == WF_MXFP8 ? 4 : 5;
  // Receive buffer: the peer's partial gate and up sums of the 32 output
  // columns this CTA keeps, for all 128 rows: value v (v < 32: gate of kept
  // output v; v >= 32: up of kept output v - 32) of row i at
  // [v / 4][i][v % 4], so a warp's 32 rows read or write 512 contiguous bytes
  // per 16-byte access.
  static constexpr int KEEP = BN / 2;            // output columns kept per CTA
  static constexpr int RECV_OFF = STAGES * STAGE_BYTES;
  static constexpr int RECV_BYTES = BM * 2 * KEEP * 4;  // 32 KB
  static constexpr int BAR_OFF = RECV_OFF + RECV_BYTES;
  // full[S], empty[S], acc_full, drain, decoded[S], recv[EPI_WARPS] (one per receiving warp)
  static constexpr int NUM_BARS = 3 * STAGES + 2 + 8;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  static constexpr int EPI_WARPS = 8;            // 4 TMEM lane groups x 2 column halves
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int THREADS = 32 * 10;
  static constexpr int TMEM_COLS = 128;
  static constexpr uint32_t IDESC = ptx::idesc_bf16(BM, MMA_N, false, true);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!DECODE || !INTERLEAVED, "decoded weight formats: separate form only");
  static_assert(!DECODE || EPI_WARPS == 8, "the decode stage uses the 256 epilogue threads");
};

// This warp's 32 rows x 16 outputs starting at tile output `o0`: gate and up
// partial sums from TMEM (zeros when the CTA had no K steps).
template <class C>
__device__ __forceinline__ static void sk_load16(uint32_t tacc, bool have_acc, int o0,
                                                 float (&g)[16], float (&u)[16]) {
  if (!have_acc) {
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = u[i] = 0.0f;
    return;
  }
  if (C::INTERLEAVED) {  // columns 2o (gate), 2o+1 (up)
    uint32_t v[32];
    ptx::tmem_ld32(tacc + 2 * o0, v);
    ptx::tmem_wait_ld();
    ptx::reg_fence(v);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      g[i] = __uint_as_float(v[2 * i]);
      u[i] = __uint_as_float(v[2 * i + 1]);
    }
  } else {  // columns o (gate), BN + o (up)
    uint32_t a[16], b[16];
    ptx::tmem_ld16(tacc + o0, a);
    ptx::tmem_ld16(tacc + C::BN + o0, b);
    ptx::tmem_wait_ld();
    ptx::reg_fence(a);
    ptx::reg_fence(b);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      g[i] = __uint_as_float(a[i]);
      u[i] = __uint_as_float(b[i]);
    }
  }
}

// Decode one stage's codes of both weight matrices (gate, then up) into the
// two BF16 atoms the MMA reads; threads 0-127 take the gate matrix, 128-255
// the up matrix.
template <class C>
__device__ __forceinline__ static void decode_stage(uint8_t *stage, int tid) {
  const int t = tid >> 7;
  decode_weights<C::WF, 64, 128, C::ATOM_BYTES, C::PAIRED>(
      stage + C::RAW_OFF + t * C::RAW_W_BYTES,
      stage + C::RAW_OFF + 2 * C::RAW_W_BYTES + t * C::RAW_S_BYTES,
      stage + C::A_BYTES + t * C::ATOM_BYTES, tid & 127);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_bf16_sk_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB0,  // W1, or W_fused
                          const __grid_constant__ CUtensorMap tmB1,  // W2 (separate form only)
                          const __grid_constant__ CUtensorMap tmY,
                          const __grid_constant__ CUtensorMap tmS1,  // INT4: gate scales
                          const __grid_constant__ CUtensorMap tmS2,  // INT4: up scales
                          const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const uint32_t bars = base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::STAGES + s); };
  const uint32_t accf_bar = bars + 8u * (2 * C::STAGES);
  const uint32_t drain_bar = bars + 8u * (2 * C::STAGES + 1);
  auto dec_bar = [&](int s) { return bars + 8u * (2 * C::STAGES + 2 + s); };
  // Epilogue warp w receives the peer's partial sums of its rows and columns
  // on its own barrier, so it can finish as soon as its 4 KB are in.
  auto recv_bar = [&](int w) { return bars + 8u * (3 * C::STAGES + 2 + w); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());  // which half of K
  const int peer = rank ^ 1;
  int mb, nb;
  tile_coords(static_cast<int>(ptx::cluster_id_x()), p, mb, nb);
  const int half = (p.num_k_blk + 1) / 2;
  const int kb0 = rank ? half : 0;
  const int kb1 = rank ? p.num_k_blk : half;
  const bool have_acc = kb1 > kb0;
  // Epilogue warps on TMEM lanes (tile rows) [32q, 32q+32) are live when
  // those rows exist; the peer's live warps send what this CTA keeps.
  auto live = [&](int q) { return mb * C::BM + q * 32 < p.M; };

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(accf_bar, 1);
    for (int w = 0; w < C::EPI_WARPS; ++w) ptx::mbar_init(recv_bar(w), 1);
    ptx::mbar_init(drain_bar, 1);
    for (int s = 0; s < C::STAGES; ++s) ptx::mbar_init(dec_bar(s), C::EPI_WARPS);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    // the peer's warp w (same rows and output half) sends warp w 4 KB when its rows exist
    for (int w = 0; w < C::EPI_WARPS; ++w)
      if (live(w & 3)) ptx::mbar_arrive_expect_tx(recv_bar(w), 4096u);
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (!C::INTERLEAVED) ptx::prefetch_tmap(&tmB1);
    if (C::DECODE) {
      ptx::prefetch_tmap(&tmS1);
      ptx::prefetch_tmap(&tmS2);
    }
  }
  if (warp == C::MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // the peer's receive barrier is armed before any store to it
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_launch_dependents();
  auto load_w = [&](uint32_t sb, uint32_t fb, int kb) {
    if (C::DECODE) {  // codes and scales of both weight matrices, behind the BF16 tiles
      const uint32_t r = sb - C::A_BYTES + C::RAW_OFF;
      const int g = C::WF == WF_INT4 ? kb * C::BK / p.w4_group : kb * C::SCALE_ROWS;
      ptx::tma_load_2d(r, &tmB0, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
      ptx::tma_load_2d(r + C::RAW_W_BYTES, &tmB1, fb, nb * C::CODE_ROW_BYTES, kb * C::BK);
      ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES, &tmS1, fb, nb * C::BN, g);
      ptx::tma_load_2d(r + 2 * C::RAW_W_BYTES + C::RAW_S_BYTES, &tmS2, fb, nb * C::BN, g);
    } else if (C::INTERLEAVED) {
      ptx::tma_load_2d(sb, &tmB0, fb, nb * C::MMA_N, kb * C::BK);
      ptx::tma_load_2d(sb + C::ATOM_BYTES, &tmB0, fb, nb * C::MMA_N + C::ATOM_COLS, kb * C::BK);
    } else {
      ptx::tma_load_2d(sb, &tmB0, fb, nb * C::BN, kb * C::BK);
      ptx::tma_load_2d(sb + C::ATOM_BYTES, &tmB1, fb, nb * C::BN, kb * C::BK);
    }
  };
  // Weights known to be unwritten by earlier work: the first stages' weight
  // boxes go out before the dependency wait, their A boxes after it.
  uint32_t pre = 0;
  if (warp == C::PRODUCER_WARP && p.w_early) {
    pre = static_cast<uint32_t>(kb1 - kb0 < C::STAGES ? kb1 - kb0 : C::STAGES);
    if (lane == 0)
      for (uint32_t s = 0; s < pre; ++s) {
        ptx::mbar_arrive_expect_tx(full_bar(s), C::TMA_BYTES);
        load_w(base + s * C::STAGE_BYTES + C::A_BYTES, full_bar(s), kb0 + (int)s);
      }
    __syncwarp();
  }
  ptx::grid_dependency_wait();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        const bool early = issued < pre;  // weights already on their way
        if (!early && !wait_bar(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, p.err,
                                WAIT_PRODUCER_EMPTY)) {
          ok = false;
          break;
        }
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t sb = sa + C::A_BYTES;
        const uint32_t fb = full_bar(stage);
        if (!early) ptx::mbar_arrive_expect_tx(fb, C::TMA_BYTES);
        ptx::tma_load_2d(sa, &tmA, fb, kb * C::BK, mb * C::BM);
        if (!early) load_w(sb, fb, kb);
        ++issued;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        // let the copies in flight land before shared memory is released
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
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(C::DECODE ? dec_bar(stage) : full_bar(stage), phase, p.timeout_ns, abort_flag,
                      p.err, WAIT_MMA_FULL)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint64_t adesc = ptx::smem_desc(sa + kk * 32, 16, 1024, ptx::SW_128B);
          const uint64_t bdesc =
              ptx::smem_desc(sb + kk * C::B_KSTEP, C::ATOM_BYTES, C::B_SBO, ptx::SW_128B);
          ptx::mma_f16(tmem_base, adesc, bdesc, C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
        }
        ptx::mma_commit(empty_bar(stage));
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
    // ------------------------------------------------------------ epilogue (warps 0-7)
    // CTA r keeps tile outputs [32r, 32r+32) for all rows; warp (q, h) owns
    // rows [32q, 32q+32) (its TMEM lanes) and, of both the kept and the sent
    // outputs, the 16 starting at 16h: it sends the peer its partial sums of
    // the peer's 16, then finishes its own 16 with the peer's partial sums.
    const int q = warp & 3;
    const int h = warp >> 2;
    const int row = q * 32 + lane;  // tile row of this thread
    bool ok = true;
    if (C::DECODE) {  // during the K loop: decode each stage's weights for the MMA
      uint32_t stage = 0, phase = 0;
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        ok = wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        decode_stage<C>(smem + stage * C::STAGE_BYTES, static_cast<int>(threadIdx.x));
        ptx::fence_proxy_async_smem();  // generic-proxy writes, read by the MMA (async proxy)
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(dec_bar(stage));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    ok = ok && wait_bar(accf_bar, 0, p.timeout_ns, abort_flag, p.err, WAIT_EPI_ACC_FULL);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    if (ok && live(q)) {
      {  // send: the peer keeps outputs [32 peer, 32 peer + 32)
        float g[16], u[16];
        sk_load16<C>(tacc, have_acc, C::KEEP * peer + 16 * h, g, u);
        const uint32_t recv_local = base + C::RECV_OFF + static_cast<uint32_t>(row) * 16u;
        const uint32_t dst = ptx::mapa_shared(recv_local, static_cast<uint32_t>(peer));
        const uint32_t rbar = ptx::mapa_shared(recv_bar(warp), static_cast<uint32_t>(peer));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // gate values 16h + 4k .. +3 -> group 4h + k; up values -> group 8 + 4h + k
          ptx::st_async_v4(dst + static_cast<uint32_t>((4 * h + k) * C::BM * 16),
                           __float_as_uint(g[4 * k]), __float_as_uint(g[4 * k + 1]),
                           __float_as_uint(g[4 * k + 2]), __float_as_uint(g[4 * k + 3]), rbar);
          ptx::st_async_v4(dst + static_cast<uint32_t>((8 + 4 * h + k) * C::BM * 16),
                           __float_as_uint(u[4 * k]), __float_as_uint(u[4 * k + 1]),
                           __float_as_uint(u[4 * k + 2]), __float_as_uint(u[4 * k + 3]), rbar);
        }
      }
      float g[16], u[16];
      sk_load16<C>(tacc, have_acc, C::KEEP * rank + 16 * h, g, u);
      // wait for the peer's partial sums of the kept outputs
      bool got = true;
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait_cluster(recv_bar(warp), 0)) {
        if (*abort_flag || ptx::globaltimer_ns() - t0 > p.timeout_ns) {
          got = false;
          break;
        }
      }
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        if (lane == 0) {
          *abort_flag = 1;
          if (atomicCAS(p.err, 0u, kErrTimeout) == 0u) atomicExch(p.err + 1, WAIT_SK_RECV);
          __threadfence();
        }
        // stores from a late peer land within microseconds; let them in
        // before this CTA's shared memory is released
        spin_ns(100000);
      } else {
        const float4 *recv = reinterpret_cast<const float4 *>(smem + C::RECV_OFF);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 pg = recv[(4 * h + k) * C::BM + row];
          const float4 pu = recv[(8 + 4 * h + k) * C::BM + row];
          g[4 * k] += pg.x; g[4 * k + 1] += pg.y; g[4 * k + 2] += pg.z; g[4 * k + 3] += pg.w;
          u[4 * k] += pu.x; u[4 * k + 1] += pu.y; u[4 * k + 2] += pu.z; u[4 * k + 3] += pu.w;
        }
        if (C::WF == WF_NVFP4) {  // the per-tensor scales of the gate and up weights
          const float gs = *p.sW1, us = *p.sW2;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            g[i] *= gs;
            u[i] *= us;
          }
        }
        // register holding output column o of these 16
        auto at = [](int o) { return C::PAIRED ? (o & ~7) | ((o & 7) < 4 ? 2 * (o & 7) : 2 * (o & 7) - 7) : o; };
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          packed[i] = pack_bf16x2(silu_mul(g[at(2 * i)], u[at(2 * i)]),
                                  silu_mul(g[at(2 * i + 1)], u[at(2 * i + 1)]));
        // 32 bytes of this row of Y; N is a multiple of 8, so each 16-byte
        // half is wholly inside or wholly outside the matrix
        const int yrow = mb * C::BM + row;
        const int ycol = nb * C::BN + C::KEEP * rank + 16 * h;
        if (yrow < p.M) {
          uint4 *yp = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y) +
                                                static_cast<int64_t>(yrow) * p.N + ycol);
          if (ycol < p.N) yp[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          if (ycol + 8 < p.N) yp[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      }
    }
  }

  // No cluster barrier at the end: a CTA leaves only after its kept warps
  // have received every byte the peer sends it (or have given up and waited
  // for late stores), and a CTA's own stores target only the peer.
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace swiglu
