// swiglu_dqt_kernel.cuh -- INT4, NVFP4 and MXFP8 weights decoded into tensor
// memory, with the weights on the MMA's M side and the tokens on its N side.
//
// Same result as swiglu_fused_w4 (page "Riepilogo Tecnico: Sovrapposizione
// delle Attivazioni a Livello di Tile per l'Inferenza Efficiente di LLM",
// section "Definizione del Problema": INT4 raises tensor-core density; the
// weights are BF16(q * s)), or as swiglu_fused_nvfp4 / swiglu_fused_mxfp8 (the
// formats the GEMM page's benchmark paragraph names), computed as the
// transposed product
//     Y^T[n, t] = SiLU(sum_k W1[k, n] A[t, k]) * (sum_k W2[k, n] A[t, k]).
// For few tokens the call is a stream of 4-bit codes, and the cost of the
// shared-memory decode kernels is the decode's round trip: every K step they
// write the decoded BF16 tile to shared memory, fence it for the async proxy
// and hand it to the MMA.  Here the decoded weights go straight into tensor
// memory, where tcgen05.mma reads its A operand:
//   * one CTA owns 128 weight columns [n0, n0 + 128) of both matrices over all
//     of K, for TOK tokens per pass (MMA M = 128 weight columns, N = TOK);
//   * the codes come K-major (swiglu_pack_w4_kmajor's layout: each column's K
//     codes contiguous, eight per 32-bit word ordered k0 k2 k4 k6 k1 k3 k5 k7
//     from the low nibble), so one shift and one logic operation give a
//     column's BF16 pair (k, k + 1) -- exactly one 32-bit TMEM column of the A
//     operand (row = TMEM lane, two K values per column); MXFP8 codes are
//     bytes, [N, K], two adjacent bytes giving the pair;
//   * sixteen decoding warps: warp w owns TMEM lanes [32 (w % 4), +32) (thread
//     = weight column), decodes W1 (bit 2 of w clear) or W2, and every other
//     K step (bit 3: the step's parity), all 64 K values of it, stored with
//     one tcgen05.st of 32 columns into one of NBUF decoded buffers -- eight
//     warps per step, so each warp's waits, fences and arrives serve twice
//     the decode work of a half step; four warps per SM sub-partition hide
//     each other's latency; warp 16 streams the tokens and
//     warp 18 the codes and scales (TMA, two rings); per K step warp 17 issues
//     four MMAs into the gate accumulator and warp 19 four into the up one;
//   * the epilogue (the sixteen warps again) reads gate and up for its lanes
//     (weight columns) and a quarter of the tokens, applies y = g * u /
//     (1 + e^-g), and stores Y^T's [32 columns x TOK/4 tokens] block as Y's
//     [TOK/4 rows x 32 columns] block with one TMA store.
// More tokens than TOK: the CTA walks token blocks, decoding the codes again
// for each (later passes read them from L2).
// Every wait is bounded as in the other kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"
#include "weight_decode.cuh"

namespace swiglu {

// WF_: WF_INT4 (BF16 scale per column and group of >= 64 K rows), WF_NVFP4
// (E2M1 codes in the same nibble layout, E4M3 scale per column and 16 K
// rows, FP32 scale per tensor applied to the gate and up sums) or WF_MXFP8
// (E4M3 codes, one byte each, [N, K]; E8M0 scale per column and 32 K rows).
template <int TOK_, int WF_ = WF_INT4>
struct DqtCfg {
  static constexpr int TOK = TOK_;              // tokens per pass (MMA N)
  static constexpr int WF = WF_;
  static constexpr bool NV = WF_ == WF_NVFP4;
  static constexpr bool MX = WF_ == WF_MXFP8;
  static constexpr int BW = 128;                // weight columns per CTA (MMA M)
  static constexpr int BK = 64;                 // K per step
  // Two rings: the tokens (from L2, read by the MMA, freed by its commit) and
  // the codes and scales (from DRAM, read by the decoders, freed as soon as
  // they are decoded), so the weight stream runs many steps ahead of the MMAs.
  static constexpr int A_BYTES = TOK * 128;     // tokens [TOK x 64 K], 128-byte swizzle
  static constexpr int A_STAGES = 4;            // = NBUF: stage s holds tokens and decoded buffer s
  static constexpr int ROW_BYTES = MX ? 64 : 32;  // a column's 64 codes
  static constexpr int CODE_BYTES = BW * ROW_BYTES;  // per matrix: 128 columns x 64 codes
  // per matrix and K step: one BF16 scale row (INT4), two E8M0 rows (MXFP8)
  // or four E4M3 rows (NVFP4)
  static constexpr int SCALE_ROWS = NV ? 4 : MX ? 2 : 1;
  static constexpr int SCALE_BYTES = BW * (NV ? 4 : 2);
  // 8.5 KB (INT4), 9 KB (NVFP4), 16.5 KB (MXFP8)
  static constexpr int C_BYTES = 2 * CODE_BYTES + 2 * SCALE_BYTES;
  static constexpr int C_STAGES = MX ? 6 : 12;
  static constexpr int NBUF = 4;                // decoded K steps in TMEM
  static constexpr int BUF_COL0 = 256;          // decoded buffers: columns [256 + 64 b, +64)
  static constexpr int TMEM_COLS = 512;
  static constexpr int C_OFF = A_STAGES * A_BYTES;
  static constexpr int STG_BYTES = (TOK / 4) * 64;  // a warp's [TOK/4 tokens x 32 columns]
  static constexpr int STG_OFF = C_OFF + C_STAGES * C_BYTES;
  static constexpr int BAR_OFF = STG_OFF + 16 * STG_BYTES;
  // full[A], empty[A], cfull[C], cempty[C], accf, acce, drain[2]
  static constexpr int NUM_BARS = 2 * A_STAGES + 2 * C_STAGES + 4;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  // two MMA issuers (gate on warp 17, up on warp 19) on different
  // sub-partitions: each MMA here is only 128 x TOK x 16, short enough that
  // issuing it costs about as much as executing it
  static constexpr int DEC_WARPS = 16, PRODUCER_WARP = 16, MMA_WARP = 17, CODES_WARP = 18,
                       MMA2_WARP = 19;
  static constexpr int DEC_PER_STEP = 8;  // warps decoding one step (the other eight take the next)
  static constexpr int THREADS = 32 * 20;
  static constexpr uint32_t IDESC = ptx::idesc_bf16(128, TOK, false, false);
  static_assert(TOK == 64 || TOK == 128, "tokens per pass");
  static_assert(WF == WF_INT4 || WF == WF_NVFP4 || WF == WF_MXFP8, "weight format");
  // MXFP8 codes arrive with the 64-byte swizzle, whose pattern repeats every 512 bytes
  static_assert(!MX || (C_OFF % 512 == 0 && C_BYTES % 512 == 0 && CODE_BYTES % 512 == 0),
                "swizzled code tiles start on 512-byte boundaries");
  static_assert(2 * TOK <= BUF_COL0 && BUF_COL0 + NBUF * 64 <= TMEM_COLS, "TMEM map");
  static_assert(C_BYTES % 128 == 0 && STG_BYTES % 128 == 0, "128-byte aligned copies");
  static_assert(A_STAGES == NBUF, "one barrier pair per tokens stage and decoded buffer");
  static_assert(C_STAGES % 2 == 0 && NBUF % 2 == 0, "a stage and a buffer serve steps of one parity");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(2 * SMEM_BYTES > 233472, "one CTA per SM (it holds all 512 TMEM columns)");
};

// Half a step: 32 K values of one column from 16 bytes of codes, 16 pairs
// into r[0..15].
__device__ __forceinline__ static void decode_kmajor_int4_half(const uint4 &w, uint32_t s_bits,
                                                               uint32_t *r) {
  const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
  const uint32_t sp = s_bits | (s_bits << 16);
  const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162 *>(&sp);
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = ((words[j] >> (4 * i)) & 0x000F000Fu) ^ 0x43084308u;
      const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&t), k136);
      const __nv_bfloat162 v = __hmul2(q, s2);
      r[4 * j + i] = *reinterpret_cast<const uint32_t *>(&v);
    }
  }
}

// Half a step of NVFP4: 32 K values of one column from 16 bytes of codes
// (words of eight, the pair (k, k + 1) in nibbles i and 4 + i as for INT4),
// with the E4M3 scales of its two 16-row blocks in the low two bytes of
// `s01` (first block low), 16 pairs into r[0..15].  An E2M1 code s e1 e0 m
// with e1 e0 m placed at BF16 bits 8..6 and s at bit 15 is the BF16 number
// E2M1 * 2^-126 (e = 0, m = 1: the subnormal 2^-127); the multiplies by 2^126
// and by the scale are exact (at most 2 + 4 significant bits).
__device__ __forceinline__ static void decode_kmajor_nvfp4_half(const uint4 &w, uint32_t s01,
                                                                uint32_t *r) {
  const float2 sf = e4m3x2_to_float2(s01 & 0xFFFFu);
  const uint32_t sp[2] = {bf16x2_bits(sf.x, sf.x), bf16x2_bits(sf.y, sf.y)};
  const uint32_t k126 = 0x7E807E80u;  // 2^126 in both halves
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = words[j];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // magnitude bits of nibbles i, 4 + i to bits 8..6 and 24..22; sign bits to 15 and 31
      const uint32_t mag = (i == 0 ? x << 6 : i == 1 ? x << 2 : i == 2 ? x >> 2 : x >> 6) & 0x01C001C0u;
      const uint32_t sgn = (i == 0 ? x << 12 : i == 1 ? x << 8 : i == 2 ? x << 4 : x) & 0x80008000u;
      const uint32_t y = mag | sgn;
      const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&y),
                                       *reinterpret_cast<const __nv_bfloat162 *>(&k126));
      const __nv_bfloat162 o = __hmul2(v, *reinterpret_cast<const __nv_bfloat162 *>(&sp[j >> 1]));
      r[4 * j + i] = *reinterpret_cast<const uint32_t *>(&o);
    }
  }
}

// Half a step of MXFP8: 32 K values of one column from 32 bytes of E4M3
// codes (byte i = K row i), all under one E8M0 block scale `p` (2^(e-127) as
// a float), 16 pairs into r[0..15].  E4M3 * 2^(e-127) is exact in FP32 and
// rounded once to BF16, as in the shared-memory decode.
__device__ __forceinline__ static void decode_kmajor_mxfp8_half(const uint4 &lo, const uint4 &hi,
                                                                float p, uint32_t *r) {
  const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f0 = e4m3x2_to_float2(words[j] & 0xFFFFu);
    const float2 f1 = e4m3x2_to_float2(words[j] >> 16);
    r[2 * j] = bf16x2_bits(__fmul_rn(f0.x, p), __fmul_rn(f0.y, p));
    r[2 * j + 1] = bf16x2_bits(__fmul_rn(f1.x, p), __fmul_rn(f1.y, p));
  }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_dqt_kernel(const __grid_constant__ CUtensorMap tmA,   // tokens [M, K] BF16
                      const __grid_constant__ CUtensorMap tmC1,  // gate codes [N, K/2] u8
                      const __grid_constant__ CUtensorMap tmC2,  // up codes
                      const __grid_constant__ CUtensorMap tmY,   // [M, N] BF16
                      const __grid_constant__ CUtensorMap tmS1,  // gate scales [K/G, N] BF16
                      const __grid_constant__ CUtensorMap tmS2,  // up scales
                      const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const uint32_t bars = base + C::BAR_OFF;
  // stage s: the tokens tile and decoded buffer s; full when the tokens have
  // landed and the step's eight decoding warps have stored, empty once both
  // MMA issuers' commits arrive
  auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bars + 8u * (C::A_STAGES + s); };
  auto cfull_bar = [&](uint32_t s) { return bars + 8u * (2 * C::A_STAGES + s); };
  auto cempty_bar = [&](uint32_t s) { return bars + 8u * (2 * C::A_STAGES + C::C_STAGES + s); };
  const uint32_t accf_bar = bars + 8u * (2 * C::A_STAGES + 2 * C::C_STAGES);
  const uint32_t acce_bar = accf_bar + 8u;
  const uint32_t drain_bar = accf_bar + 16u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = static_cast<int>(blockIdx.x) * C::BW;
  const int nk = p.num_k_blk;
  const int nt = p.num_m_blk;  // token blocks of TOK
  // Every CTA reads the same tokens; starting each CTA's K loop at a different
  // step spreads those reads over all of A in L2.
  const int k_rot =
      static_cast<int>((static_cast<int64_t>(blockIdx.x) * nk) / gridDim.x) % (nk > 0 ? nk : 1);
  auto kstep = [&](int i) { return i + k_rot < nk ? i + k_rot : i + k_rot - nk; };

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::A_STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1 + C::DEC_PER_STEP);  // the tokens' expect_tx and the decoders
      ptx::mbar_init(empty_bar(s), 2);                // both MMA issuers' commits
    }
    for (int s = 0; s < C::C_STAGES; ++s) {
      ptx::mbar_init(cfull_bar(s), 1);
      ptx::mbar_init(cempty_bar(s), C::DEC_PER_STEP);  // the step's decoding warps
    }
    ptx::mbar_init(accf_bar, 2);
    ptx::mbar_init(acce_bar, C::DEC_WARPS);
    ptx::mbar_init(drain_bar, 1);
    ptx::mbar_init(drain_bar + 8u, 1);
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

  const int total = nt * nk;  // steps over all token blocks
  // One ring's producer: waits for a free slot, then `load(slot, barrier, g)`
  // for every step g of every token block.
  auto produce = [&](int stages, auto full, auto empty, uint32_t bytes, auto load) {
    uint32_t issued = 0;
    bool ok = true;
    for (int g = 0; g < total; ++g) {
      const uint32_t s = static_cast<uint32_t>(g % stages);
      const uint32_t ph = static_cast<uint32_t>(g / stages) & 1u;
      if (!wait_bar(empty(s), ph ^ 1u, p.timeout_ns, abort_flag, p.err, WAIT_PRODUCER_EMPTY)) {
        ok = false;
        break;
      }
      ptx::mbar_arrive_expect_tx(full(s), bytes);
      load(s, full(s), g);
      ++issued;
    }
    if (!ok) {  // let the copies in flight land before shared memory is released
      const uint32_t n = issued < (uint32_t)stages ? issued : (uint32_t)stages;
      for (uint32_t i = issued - n; i < issued; ++i)
        wait_quiet(full(i % stages), (i / stages) & 1u, p.timeout_ns);
    }
  };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ tokens producer
    if (lane == 0)
      produce(C::A_STAGES, full_bar, empty_bar, C::A_BYTES, [&](uint32_t s, uint32_t fb, int g) {
        ptx::tma_load_2d(base + s * C::A_BYTES, &tmA, fb, kstep(g % nk) * C::BK, (g / nk) * C::TOK);
      });
    __syncwarp();
  } else if (warp == C::CODES_WARP) {
    // ------------------------------------------------------------ codes producer
    if (lane == 0)
      produce(C::C_STAGES, cfull_bar, cempty_bar, C::C_BYTES, [&](uint32_t s, uint32_t fb, int g) {
        const int kb = kstep(g % nk);
        const uint32_t r = base + C::C_OFF + s * C::C_BYTES;
        const int srow = C::WF == WF_INT4 ? kb * C::BK / p.w4_group : kb * C::SCALE_ROWS;
        ptx::tma_load_2d(r, &tmC1, fb, kb * C::ROW_BYTES, n0);
        ptx::tma_load_2d(r + C::CODE_BYTES, &tmC2, fb, kb * C::ROW_BYTES, n0);
        ptx::tma_load_2d(r + 2 * C::CODE_BYTES, &tmS1, fb, n0, srow);
        ptx::tma_load_2d(r + 2 * C::CODE_BYTES + C::SCALE_BYTES, &tmS2, fb, n0, srow);
      });
    __syncwarp();
  } else if (warp == C::MMA_WARP || warp == C::MMA2_WARP) {
    // ------------------------------------------------------------ MMA issuers (gate, up)
    // Counters advance incrementally and an issuer's four MMAs of a step go
    // out as one asm block: each issuer shares its sub-partition with four
    // decoding warps, and its instruction count per step sets how fast it
    // keeps the tensor pipe fed (measured: one issuer for both products
    // 43 us at 7B M = 128, two 34-36 us).
    if (lane == 0) {
      const uint32_t m = warp == C::MMA_WARP ? 0u : 1u;  // 0: gate, 1: up
      const uint64_t desc0 = ptx::smem_desc(base, 16, 1024, ptx::SW_128B);
      uint32_t s = 0, ph = 0;
      int i = 0, tb = 0;
      for (int g = 0; g < total; ++g) {
        // a new token block may overwrite the accumulators once the epilogue
        // has read the previous block's
        if (i == 0 && tb > 0 &&
            !wait_bar(acce_bar, static_cast<uint32_t>(tb - 1) & 1u, p.timeout_ns, abort_flag, p.err,
                      WAIT_MMA_ACC_EMPTY))
          break;
        if (!wait_bar(full_bar(s), ph, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) break;
        ptx::tc_fence_after();
        const uint32_t abuf = tmem_base + C::BUF_COL0 + 64u * s;
        ptx::mma_f16_tmem_a_k64(tmem_base + m * C::TOK, abuf + 32u * m,
                                desc0 + ((s * C::A_BYTES) >> 4), C::IDESC, i == 0 ? 1u : 0u);
        ptx::mma_commit(empty_bar(s));  // tokens and decoded buffer read
        if (i == nk - 1) ptx::mma_commit(accf_bar);
        if (++s == static_cast<uint32_t>(C::A_STAGES)) {
          s = 0;
          ph ^= 1u;
        }
        if (++i == nk) {
          i = 0;
          ++tb;
        }
      }
      ptx::mma_commit(drain_bar + 8u * m);
      wait_quiet(drain_bar + 8u * m, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp < C::DEC_WARPS) {
    // ------------------------------------------------------------ decode, then epilogue (warps 0-15)
    const int q = warp & 3;          // TMEM lanes [32q, 32q + 32): weight columns n0 + 32q + lane
    const int mtx = (warp >> 2) & 1; // decode: 0 = W1 (gate), 1 = W2 (up)
    const int par = warp >> 3;       // decode: the steps g with g % 2 == par
    const int tq = warp >> 2;        // epilogue: tokens [tq TOK/4, (tq + 1) TOK/4)
    const int c = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t stg = base + C::STG_OFF + warp * C::STG_BYTES;
    const float gs = C::NV ? *p.sW1 : 1.0f;  // per-tensor scales of NVFP4 codes
    const float us = C::NV ? *p.sW2 : 1.0f;
    bool ok = true;
    for (int tb = 0; tb < nt && ok; ++tb) {
      for (int i = 0; i < nk; ++i) {
        const int g = tb * nk + i;
        if ((g & 1) != par) continue;
        const uint32_t s = static_cast<uint32_t>(g % C::C_STAGES);
        const uint32_t b = static_cast<uint32_t>(g % C::NBUF);  // = the tokens stage
        ok = wait_bar(cfull_bar(s), static_cast<uint32_t>(g / C::C_STAGES) & 1u, p.timeout_ns,
                      abort_flag, p.err, WAIT_MMA_FULL);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t *st = smem + C::C_OFF + s * C::C_BYTES;
        const uint8_t *sc = st + 2 * C::CODE_BYTES + mtx * C::SCALE_BYTES;
        uint32_t r[32];
        if constexpr (C::MX) {
          // column c's 64 bytes, 16-byte chunk j at chunk j ^ ((c >> 1) & 3) (the
          // 64-byte swizzle: address bits 4-5 ^= bits 7-8), so that the eight
          // lanes of a load phase hit eight different bank groups
          const uint8_t *row = st + mtx * C::CODE_BYTES + c * C::ROW_BYTES;
          const uint32_t sw = static_cast<uint32_t>(c >> 1) & 3u;
          uint4 w[4];
#pragma unroll
          for (uint32_t j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint4 *>(row + ((j ^ sw) << 4));
          const uint32_t e0 = sc[c], e1 = sc[C::BW + c];  // E8M0 of K rows 0-31, 32-63
          decode_kmajor_mxfp8_half(w[0], w[1], __uint_as_float(e0 ? e0 << 23 : 0x00400000u), r);
          decode_kmajor_mxfp8_half(w[2], w[3], __uint_as_float(e1 ? e1 << 23 : 0x00400000u), r + 16);
        } else if constexpr (C::NV) {
          const uint4 *cw = reinterpret_cast<const uint4 *>(st + mtx * C::CODE_BYTES + c * C::ROW_BYTES);
          const uint4 w0 = cw[0], w1 = cw[1];
          // scale rows 0..3 (16 K rows each) at sc + 128 row: column c's byte
          decode_kmajor_nvfp4_half(w0, uint32_t(sc[c]) | (uint32_t(sc[C::BW + c]) << 8), r);
          decode_kmajor_nvfp4_half(w1, uint32_t(sc[2 * C::BW + c]) | (uint32_t(sc[3 * C::BW + c]) << 8),
                                   r + 16);
        } else {
          const uint4 *cw = reinterpret_cast<const uint4 *>(st + mtx * C::CODE_BYTES + c * C::ROW_BYTES);
          const uint4 w0 = cw[0], w1 = cw[1];
          const uint32_t sbits = *reinterpret_cast<const uint16_t *>(sc + c * 2);
          decode_kmajor_int4_half(w0, sbits, r);
          decode_kmajor_int4_half(w1, sbits, r + 16);
        }
        // The codes were consumed by the decode above: release the stage.
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(cempty_bar(s));
        ok = wait_bar(empty_bar(b), (static_cast<uint32_t>(g / C::NBUF) & 1u) ^ 1u, p.timeout_ns,
                      abort_flag, p.err, WAIT_MMA_FULL);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        ptx::tmem_st32(tmem_base + lane_off + C::BUF_COL0 + 64u * b + 32u * mtx, r);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(full_bar(b));
      }
      if (!ok) break;
      // ---- epilogue of token block tb
      ok = wait_bar(accf_bar, static_cast<uint32_t>(tb) & 1u, p.timeout_ns, abort_flag, p.err,
                    WAIT_EPI_ACC_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      constexpr int TPW = C::TOK / 4;  // tokens per warp
      float yv[TPW];                   // this thread's column, one value per token
#pragma unroll
      for (int j = 0; j < TPW / 16; ++j) {
        const int t0 = tq * TPW + 16 * j;
        uint32_t g16[16], u16[16];
        ptx::tmem_ld16(tmem_base + lane_off + t0, g16);
        ptx::tmem_ld16(tmem_base + lane_off + C::TOK + t0, u16);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          yv[16 * j + e] = C::NV ? silu_mul(gs * __uint_as_float(g16[e]), us * __uint_as_float(u16[e]))
                                 : silu_mul(__uint_as_float(g16[e]), __uint_as_float(u16[e]));
      }
      // accumulators read: the next token block's MMAs may start
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acce_bar);
      // the previous block's store must have read the staging block
      if (lane == 0) ptx::bulk_wait_read<0>();
      __syncwarp();
#pragma unroll
      for (int e = 0; e < TPW; ++e) {
        const __nv_bfloat16 v = __float2bfloat16_rn(yv[e]);
        *reinterpret_cast<__nv_bfloat16 *>(smem + (stg - base) + (e * 32 + lane) * 2) = v;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      const int row0 = tb * C::TOK + tq * TPW;
      if (lane == 0 && row0 < p.M && n0 + 32 * q < p.N) {
        ptx::tma_store_2d(&tmY, stg, n0 + 32 * q, row0);
        ptx::bulk_commit();
      }
    }
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

}  // namespace swiglu
