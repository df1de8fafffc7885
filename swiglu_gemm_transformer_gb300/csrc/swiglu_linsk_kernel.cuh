// swiglu_linsk_kernel.cuh -- the down projection for few rows: split-K over a
// cluster, partial sums reduced in distributed shared memory (sm_103a).
//
// Z[M,N] = X[M,K] W[K,N] (+ R[M,N]): the product that ends the MLP block
// whose cost the page's problem statement measures (page "Riepilogo Tecnico:
// Sovrapposizione delle Attivazioni a Livello di Tile per l'Inferenza
// Efficiente di LLM", section "Definizione del Problema"); X is the fused
// projection's output Y.
//
// With few rows (the decode-sized M <= 128 of the Qwen-2.5 MLPs) the product
// has few output tiles: 0.5B's H = 896 output columns are 14 tiles of 64.
// Each 128-row x BN-column tile (BN = 64 or 128) goes to a cluster of CS
// CTAs (CS = 8, 4 or 2), and CTA r multiplies its CS-th of the K steps:
//   * warp 8 streams X[128 x 64] and W[64 x BN] per K step into a
//     STAGES-deep ring (TMA, 128-byte swizzle), warp 9 issues
//     tcgen05.mma M=128 x N=BN (FP32 accumulators in tensor memory);
//   * reduce-scatter over the cluster: CTA r keeps output columns
//     [r KEEP, (r+1) KEEP) of the tile, KEEP = BN / CS.  Eight epilogue
//     warps (four TMEM lane groups x two BN/2-column halves) read their
//     partial sums and send each peer its KEEP columns with st.async
//     (16-byte stores into the peer's shared memory, counted on the
//     mbarrier of the peer's finishing warp for those rows); the warps that
//     hold the kept columns each wait for their rows of the CS - 1 partial
//     tiles sent to this CTA, add them and R in FP32, round to BF16 and store
//     their KEEP columns of each row.
// No workspace, no second kernel: the partial sums never leave the cluster.
// One tile per cluster (no persistent loop); the launcher sizes the grid.
//
// Every wait is bounded as in the other kernels (timeout -> error word, abort
// flag, drain, TMEM freed).  A CTA leaves only once everything its peers send
// it has arrived (or, after a timeout, once late stores have had time to
// land), so no store targets a CTA that has left.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"
#include "tc_common.cuh"

namespace swiglu {

enum : uint32_t { WAIT_LINSK_RECV = 8 };

template <int CS_, int BN_ = 64>
struct LinSkCfg {
  static constexpr int CS = CS_;                 // CTAs per cluster (K slices)
  static constexpr int BM = 128;                 // rows per tile (MMA M)
  static constexpr int BN = BN_;                 // output columns per tile (MMA N)
  static constexpr int BK = 64;                  // K per stage
  static constexpr int KEEP = BN / CS;           // output columns each CTA finishes
  static constexpr int HALF = BN / 2;            // accumulator columns per epilogue warp
  static constexpr int A_BYTES = BM * BK * 2;    // 16 KB
  static constexpr int ATOM_BYTES = BK * 64 * 2; // one 64-column, 128-byte-swizzled weight box
  static constexpr int B_BYTES = BK * BN * 2;    // BN / 64 boxes
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // Receive buffer: the CS - 1 peers' partial sums of the kept columns, for
  // all 128 rows: slot s (sender rank s, or s + 1 at and above this CTA's
  // rank), row i, KEEP floats.
  static constexpr int RECV_BYTES = (CS - 1) * BM * KEEP * 4;
  // as many stages as fit beside it (at most 8)
  static constexpr int STAGES_FIT = (227 * 1024 - RECV_BYTES - 2048) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 8 ? STAGES_FIT : 8;
  static constexpr int RECV_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = RECV_OFF + RECV_BYTES;
  // full[S], empty[S], acc_full, drain, recv[4] (one per TMEM lane group)
  static constexpr int NUM_BARS = 2 * STAGES + 2 + 4;
  static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;
  static constexpr int EPI_WARPS = 8;            // 4 TMEM lane groups x 2 column halves
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int THREADS = 32 * 10;
  static constexpr int TMEM_COLS = BN;
  static constexpr uint32_t IDESC = ptx::idesc_bf16(BM, BN, false, true);
  static_assert(CS == 2 || CS == 4 || CS == 8, "cluster size");
  static_assert(BN == 64 || BN == 128, "tile width");
  static_assert(KEEP % 8 == 0 && HALF % KEEP == 0, "kept columns: whole 16-byte BF16 groups");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    swiglu_linsk_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw);

  const uint32_t bars = base + C::BAR_OFF;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::STAGES + s); };
  const uint32_t accf_bar = bars + 8u * (2 * C::STAGES);
  const uint32_t drain_bar = bars + 8u * (2 * C::STAGES + 1);
  // the finishing warp of lane group q receives its rows' partial sums on its
  // own barrier, so it can go on as soon as they are in
  auto recv_bar = [&](int q) { return bars + 8u * (2 * C::STAGES + 2 + q); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NUM_BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());  // K slice and kept columns
  int mb, nb;
  tile_coords(static_cast<int>(ptx::cluster_id_x()), p, mb, nb);
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.num_k_blk / C::CS);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.num_k_blk / C::CS);
  const bool have_acc = kb1 > kb0;
  // Epilogue warps on TMEM lanes (tile rows) [32q, 32q+32) take part when
  // those rows exist; every peer agrees on which do.
  auto live = [&](int q) { return mb * C::BM + q * 32 < p.M; };
  // per live lane group, each of the CS - 1 peers sends 32 rows x KEEP floats
  const uint32_t recv_bytes = (C::CS - 1) * 32u * C::KEEP * 4u;

  if (warp == C::PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(accf_bar, 1);
    for (int q = 0; q < 4; ++q) ptx::mbar_init(recv_bar(q), 1);
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    for (int q = 0; q < 4; ++q)
      if (live(q)) ptx::mbar_arrive_expect_tx(recv_bar(q), recv_bytes);
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmW);
  }
  if (warp == C::MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // every peer's receive barrier is armed before any store to it
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_launch_dependents();
  // Weights known to be unwritten by earlier work: the first stages' weight
  // boxes go out before the dependency wait, their X boxes after it.
  uint32_t pre = 0;
  if (warp == C::PRODUCER_WARP && p.w_early) {
    pre = static_cast<uint32_t>(kb1 - kb0 < C::STAGES ? kb1 - kb0 : C::STAGES);
    if (lane == 0)
      for (uint32_t s = 0; s < pre; ++s) {
        ptx::mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
        for (int j = 0; j < C::BN / 64; ++j)
          ptx::tma_load_2d(base + s * C::STAGE_BYTES + C::A_BYTES + j * C::ATOM_BYTES, &tmW,
                           full_bar(s), nb * C::BN + 64 * j, (kb0 + static_cast<int>(s)) * C::BK);
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
        const uint32_t fb = full_bar(stage);
        if (!early) ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        ptx::tma_load_2d(sa, &tmX, fb, kb * C::BK, mb * C::BM);
        if (!early)
          for (int j = 0; j < C::BN / 64; ++j)
            ptx::tma_load_2d(sa + C::A_BYTES + j * C::ATOM_BYTES, &tmW, fb, nb * C::BN + 64 * j,
                             kb * C::BK);
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
        if (!wait_bar(full_bar(stage), phase, p.timeout_ns, abort_flag, p.err, WAIT_MMA_FULL)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          // X: K-major, 128-byte swizzle, 16 K-elements = 32 bytes along a row;
          // W: MN-major, 64-column boxes ATOM_BYTES apart, 8-row K groups
          // 1024 bytes apart, one MMA's 16 K-rows = 2048 bytes.
          const uint64_t adesc = ptx::smem_desc(sa + kk * 32, 16, 1024, ptx::SW_128B);
          const uint64_t bdesc = ptx::smem_desc(sb + kk * 2048, C::ATOM_BYTES, 1024, ptx::SW_128B);
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
    // Warp (q, h) owns rows [32q, 32q+32) (its TMEM lanes) and accumulator
    // columns [h HALF, (h+1) HALF), i.e. the column groups g (KEEP wide) with
    // g / (CS/2) == h.  It sends group g to CTA g for every g != rank; the
    // warp whose half holds group `rank` finishes those columns.
    const int q = warp & 3;
    const int h = warp >> 2;
    const int row = q * 32 + lane;  // tile row of this thread
    constexpr int GPH = C::CS / 2;  // column groups per half
    bool ok = wait_bar(accf_bar, 0, p.timeout_ns, abort_flag, p.err, WAIT_EPI_ACC_FULL);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    // After a failed wait this CTA sends nothing, but its peers may still be
    // sending to it: give their stores time to land before it leaves.
    if (!ok && live(q)) spin_ns(100000);
    if (ok && live(q)) {
      float v[C::HALF];
      if (have_acc) {
#pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(C::HALF * h + 32 * c), r);
          ptx::tmem_wait_ld();
          ptx::reg_fence(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < C::HALF; ++i) v[i] = 0.0f;
      }
      float acc[C::KEEP];  // the kept columns' partial sums (warp h == rank / GPH)
#pragma unroll
      for (int i = 0; i < C::KEEP; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < GPH; ++j) {
        const int g = h * GPH + j;
        if (g == rank) {
#pragma unroll
          for (int i = 0; i < C::KEEP; ++i) acc[i] = v[j * C::KEEP + i];
          continue;
        }
        // this CTA's slot in CTA g's receive buffer
        const int slot = rank < g ? rank : rank - 1;
        const uint32_t local =
            base + C::RECV_OFF + static_cast<uint32_t>((slot * C::BM + row) * C::KEEP * 4);
        const uint32_t dst = ptx::mapa_shared(local, static_cast<uint32_t>(g));
        const uint32_t rbar = ptx::mapa_shared(recv_bar(q), static_cast<uint32_t>(g));
#pragma unroll
        for (int k = 0; k < C::KEEP / 4; ++k) {
          const int c = j * C::KEEP + 4 * k;
          ptx::st_async_v4(dst + 16u * k, __float_as_uint(v[c]), __float_as_uint(v[c + 1]),
                           __float_as_uint(v[c + 2]), __float_as_uint(v[c + 3]), rbar);
        }
      }
      if (h == rank / GPH) {
        bool got = true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait_cluster(recv_bar(q), 0)) {
          if (*abort_flag || ptx::globaltimer_ns() - t0 > p.timeout_ns) {
            got = false;
            break;
          }
        }
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          if (lane == 0) {
            *abort_flag = 1;
            if (atomicCAS(p.err, 0u, kErrTimeout) == 0u) atomicExch(p.err + 1, WAIT_LINSK_RECV);
            __threadfence();
          }
          // stores from a late peer land within microseconds; let them in
          // before this CTA's shared memory is released
          spin_ns(100000);
        } else {
          const float4 *recv = reinterpret_cast<const float4 *>(smem + C::RECV_OFF);
#pragma unroll
          for (int s = 0; s < C::CS - 1; ++s) {
#pragma unroll
            for (int k = 0; k < C::KEEP / 4; ++k) {
              const float4 t = recv[(s * C::BM + row) * (C::KEEP / 4) + k];
              acc[4 * k] += t.x;
              acc[4 * k + 1] += t.y;
              acc[4 * k + 2] += t.z;
              acc[4 * k + 3] += t.w;
            }
          }
          const int zrow = mb * C::BM + row;
          const int zcol = nb * C::BN + rank * C::KEEP;
          if (zrow < p.M) {
            const int64_t off = static_cast<int64_t>(zrow) * p.N + zcol;
#pragma unroll
            for (int k = 0; k < C::KEEP / 8; ++k) {
              if (zcol + 8 * k >= p.N) break;  // N is a multiple of 8
              float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
              if (p.R != nullptr) {
                const uint4 rv =
                    *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.R) + off + 8 * k);
                const __nv_bfloat162 *r2 = reinterpret_cast<const __nv_bfloat162 *>(&rv);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f = __bfloat1622float2(r2[i]);
                  r8[2 * i] = f.x;
                  r8[2 * i + 1] = f.y;
                }
              }
              uint4 o;
              o.x = pack_bf16x2(acc[8 * k] + r8[0], acc[8 * k + 1] + r8[1]);
              o.y = pack_bf16x2(acc[8 * k + 2] + r8[2], acc[8 * k + 3] + r8[3]);
              o.z = pack_bf16x2(acc[8 * k + 4] + r8[4], acc[8 * k + 5] + r8[5]);
              o.w = pack_bf16x2(acc[8 * k + 6] + r8[6], acc[8 * k + 7] + r8[7]);
              *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.Y) + off + 8 * k) = o;
            }
          }
        }
      }
    }
  }

  // No cluster barrier at the end: a CTA leaves only after its finishing
  // warps have received every byte its peers send it (or have given up and
  // waited for late stores), and a CTA's own stores target only its peers.
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace swiglu
