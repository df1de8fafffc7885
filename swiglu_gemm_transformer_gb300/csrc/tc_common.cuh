// tc_common.cuh -- pieces shared by the one-CTA and CTA-pair fused SwiGLU
// kernels: launch parameters, bounded mbarrier waits, the tile order, and the
// epilogue that turns a (gate, up) accumulator tile in TMEM into BF16 Y.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace swiglu {

// Where a wait gave up (device error word, second slot).
enum : uint32_t {
  WAIT_PRODUCER_EMPTY = 1,
  WAIT_MMA_FULL = 2,
  WAIT_MMA_ACC_EMPTY = 3,
  WAIT_EPI_ACC_FULL = 4,
  WAIT_DRAIN = 5,
  WAIT_SELFTEST = 6,
  WAIT_SCHED_FULL = 9,   // a pair kernel role waiting for the next unit's response
  WAIT_SCHED_EMPTY = 10, // the pair's scheduler waiting for a response slot
};

constexpr uint32_t kErrTimeout = 5;  // == SWIGLU_ERR_TIMEOUT

struct KParams {
  int32_t M, N, K;
  int32_t num_m_blk, num_n_blk, num_k_blk;
  int32_t group_m;       // grouped raster: this many m-blocks walk the n-blocks together
  // 1: the weights are not written by any earlier work on the stream, so the
  // producer may load the first stages' weight boxes before the dependency
  // wait of programmatic dependent launch (A is always loaded after it).
  int32_t w_early;
  uint64_t timeout_ns;   // limit of every mbarrier wait
  uint32_t *err;         // device error word: [0] = status, [1] = where
  // FP8 operands only: device pointers to the per-tensor scales of A, W1, W2
  // (the gate and up products are scaled by sA*sW1 and sA*sW2).
  const float *sA, *sW1, *sW2;
  // Linear mode only (Z = X W + R): the residual R [M,N] BF16 (or null), and
  // split-K: k_splits slices of kb_per_split K steps each; with k_splits > 1
  // every slice writes FP32 partial sums to ws[slice][M][N] instead of Z.
  const void *R;
  float *ws;
  int32_t k_splits, kb_per_split;
  // Y itself (the split-K small-M kernel stores its few rows directly).
  void *Y;
  // INT4 weights: K rows per scale group (a multiple of 64).
  int32_t w4_group;
  // CTA-pair kernels only: 1 = dynamic unit schedule (the grid holds one
  // cluster per unit and running pairs take over the units of clusters that
  // have not started, through cluster launch control); 0 = static (the grid
  // holds at most one wave and pair c takes units c, c + clusters, ...).
  int32_t dyn_sched;
};

// Bounded wait, slow path.  Returns false on timeout or when another role of
// this CTA already gave up.
__device__ __noinline__ static bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag, uint32_t *err,
                                              uint32_t where) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      if (atomicCAS(err, 0u, kErrTimeout) == 0u) atomicExch(err + 1, where);
      __threadfence();
      return false;
    }
  }
}

__device__ __forceinline__ static bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                volatile int *abort_flag, uint32_t *err,
                                                uint32_t where) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, limit_ns, abort_flag, err, where);
}

// Bounded wait that records nothing (used while draining after an abort).
__device__ __forceinline__ static void wait_quiet(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < limit_ns) {
  }
}

// Spin for `ns` nanoseconds (bounded), letting in-flight copies land.
__device__ __forceinline__ static void spin_ns(uint64_t ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::globaltimer_ns() - t0 < ns) {
  }
}

// Grouped tile order: `group_m` m-blocks walk all n-blocks together, so tiles
// that run at the same time share A rows and weight columns in L2.
__device__ __forceinline__ static void tile_coords(int t, const KParams &p, int &mb, int &nb) {
  const int per_group = p.group_m * p.num_n_blk;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int rows = min(p.group_m, p.num_m_blk - first);
  const int r = t - g * per_group;
  mb = first + r % rows;
  nb = r / rows;
}

// SiLU(g) * u = g * u / (1 + e^-g), FP32: two special-function-unit
// operations (ex2 and the approximate reciprocal inside the fast divide).  A
// variant with one SFU operation and a Newton-Raphson reciprocal on the FMA
// pipe measured 6 % slower on the large-M pair kernel (its extra FMA work
// competes with the epilogue's other arithmetic under the power cap) and no
// faster on the split-K kernel, so this form is used everywhere.
__device__ __forceinline__ static float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ static uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Epilogue of one accumulator tile, for one warp (32 TMEM lanes = 32 rows,
// output chunks [c_begin, c_end) of 32 columns each).
//   tacc      : TMEM address of this warp's lanes at the tile's first column;
//               separate form: columns [0,BN) gate, [BN,2BN) up;
//               interleaved form: column 2j gate j, 2j+1 up j.
//   row0/col0 : Y coordinates of the warp's first row and the tile's first column.
//   stg_base  : this warp's two 2 KB staging buffers (shared::cta address).
//   it        : running staging-buffer counter of this warp.
//   release   : cluster address of the barrier to arrive on once the warp has
//               read the whole accumulator (frees the TMEM buffer for the MMA).
//               The arrive is relaxed: the loads are complete (tcgen05.wait::ld)
//               before it issues, so no release ordering is needed, and a
//               cluster-scope release costs microseconds.
//   gs, us    : scales applied to the gate and up accumulators (SCALED only).
//   PAIRED    : separate form only; within every 8 accumulator columns the
//               output columns lie in the order 0 4 1 5 2 6 3 7 (the order
//               the paired 4-bit weight decode writes), undone here by the
//               choice of registers.
template <bool INTERLEAVED, int BN, bool SCALED = false, bool PAIRED = false>
__device__ __forceinline__ static void epilogue_tile(uint32_t tacc, int row0, int col0,
                                                     int c_begin, int c_end,
                                                     const CUtensorMap *tmY, int M, int N,
                                                     uint8_t *smem, uint32_t smem_base,
                                                     uint32_t stg_base, uint32_t &it, int lane,
                                                     uint32_t release, float gs = 1.0f,
                                                     float us = 1.0f) {
  if (c_begin >= c_end) {  // nothing to read in this tile: release at once
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster_relaxed(release);
    return;
  }
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    uint32_t g[32], u[32];
    if (INTERLEAVED) {
      ptx::tmem_ld32(tacc + c * 64, g);
      ptx::tmem_ld32(tacc + c * 64 + 32, u);
    } else {
      ptx::tmem_ld32(tacc + c * 32, g);
      ptx::tmem_ld32(tacc + BN + c * 32, u);
    }
    ptx::tmem_wait_ld();
    ptx::reg_fence(g);
    ptx::reg_fence(u);
    if (SCALED) {
      // separate form: g = gate columns, u = up columns; interleaved form:
      // even registers are gate columns, odd registers up columns.
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float sg = INTERLEAVED ? ((i & 1) ? us : gs) : gs;
        const float su = INTERLEAVED ? ((i & 1) ? us : gs) : us;
        g[i] = __float_as_uint(__uint_as_float(g[i]) * sg);
        u[i] = __float_as_uint(__uint_as_float(u[i]) * su);
      }
    }
    if (c == c_end - 1) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(release);
    }
    uint32_t packed[16];
    if (INTERLEAVED) {
      // g: columns 64c..64c+31 = (gate, up) pairs of outputs 32c..32c+15;
      // u: the pairs of outputs 32c+16..32c+31.
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        packed[i] =
            pack_bf16x2(silu_mul(__uint_as_float(g[4 * i]), __uint_as_float(g[4 * i + 1])),
                        silu_mul(__uint_as_float(g[4 * i + 2]), __uint_as_float(g[4 * i + 3])));
        packed[8 + i] =
            pack_bf16x2(silu_mul(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1])),
                        silu_mul(__uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3])));
      }
    } else {
      // register holding output column o of the chunk
      auto at = [](int o) { return PAIRED ? (o & ~7) | ((o & 7) < 4 ? 2 * (o & 7) : 2 * (o & 7) - 7) : o; };
#pragma unroll
      for (int i = 0; i < 16; ++i)
        packed[i] = pack_bf16x2(
            silu_mul(__uint_as_float(g[at(2 * i)]), __uint_as_float(u[at(2 * i)])),
            silu_mul(__uint_as_float(g[at(2 * i + 1)]), __uint_as_float(u[at(2 * i + 1)])));
    }
    const int ccol = col0 + c * 32;
    const uint32_t stg = stg_base + (it & 1u) * 2048u;
    // The store issued from this buffer two blocks ago must have finished reading it.
    if (lane == 0) ptx::bulk_wait_read<1>();
    __syncwarp();
    uint4 *rowp = reinterpret_cast<uint4 *>(smem + (stg - smem_base) + lane * 64);
    const int sw = (lane >> 1) & 3;  // 64-byte swizzle: 16-byte chunk i -> i ^ ((row >> 1) & 3)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      rowp[i ^ sw] =
          make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (row0 < M && ccol < N) ptx::tma_store_2d(tmY, stg, ccol, row0);
      ptx::bulk_commit();
    }
    ++it;
  }
}

// Linear-mode epilogue of one accumulator tile for one warp: Z = acc (+ R),
// rounded to BF16 and stored through the staging buffers with TMA (k_splits
// == 1), or the FP32 partial sums written to the workspace slice (k_splits > 1).
template <int BN>
__device__ __forceinline__ static void epilogue_tile_linear(uint32_t tacc, int row0, int col0,
                                                            int c_begin, int c_end,
                                                            const CUtensorMap *tmZ, const KParams &p,
                                                            int split, uint8_t *smem,
                                                            uint32_t smem_base, uint32_t stg_base,
                                                            uint32_t &it, int lane,
                                                            uint32_t release) {
  if (c_begin >= c_end) {
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster_relaxed(release);
    return;
  }
  const int row = row0 + lane;
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const int ccol = col0 + c * 32;
    // residual for this thread's row, 8 columns per 16-byte load (N % 8 == 0)
    uint4 rv[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                   make_uint4(0, 0, 0, 0)};
    if (p.R != nullptr && p.k_splits == 1 && row < p.M) {
      const uint4 *rp = reinterpret_cast<const uint4 *>(
          static_cast<const __nv_bfloat16 *>(p.R) + static_cast<int64_t>(row) * p.N + ccol);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ccol + 8 * j < p.N) rv[j] = __ldg(rp + j);
    }
    uint32_t v[32];
    ptx::tmem_ld32(tacc + c * 32, v);
    ptx::tmem_wait_ld();
    ptx::reg_fence(v);
    if (c == c_end - 1) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster_relaxed(release);
    }
    if (p.k_splits > 1) {
      if (row < p.M) {
        float4 *wp = reinterpret_cast<float4 *>(
            p.ws + (static_cast<int64_t>(split) * p.M + row) * p.N + ccol);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (ccol + 4 * j < p.N)
            wp[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
      }
      continue;
    }
    uint32_t packed[16];
    const __nv_bfloat162 *r2 = reinterpret_cast<const __nv_bfloat162 *>(rv);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 rf = __bfloat1622float2(r2[i]);
      packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]) + rf.x, __uint_as_float(v[2 * i + 1]) + rf.y);
    }
    const uint32_t stg = stg_base + (it & 1u) * 2048u;
    if (lane == 0) ptx::bulk_wait_read<1>();
    __syncwarp();
    uint4 *rowp = reinterpret_cast<uint4 *>(smem + (stg - smem_base) + lane * 64);
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      rowp[i ^ sw] =
          make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (row0 < p.M && ccol < p.N) ptx::tma_store_2d(tmZ, stg, ccol, row0);
      ptx::bulk_commit();
    }
    ++it;
  }
}

}  // namespace swiglu
