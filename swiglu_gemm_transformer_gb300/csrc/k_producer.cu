// k_producer.cu -- the step before the FP8 projection: RMSNorm of the rows of
// X and per-tensor FP8 E4M3 quantisation of the result, producing the A_q and
// s_A that swiglu_fused_fp8 consumes; and the same quantisation without the
// normalisation (for weights).
//
// The page names FP8 quantisation as what raises the tensor cores' density
// (page "Riepilogo Tecnico: Sovrapposizione delle Attivazioni a Livello di
// Tile per l'Inferenza Efficiente di LLM", section "Definizione del
// Problema"); it defines neither step, so these follow the standard ones:
//   a[m,k] = x[m,k] * gamma[k] / sqrt(mean_k x[m,k]^2 + eps)   (RMSNorm)
//   s      = max|a| / 448                 (one scale for the whole tensor)
//   q      = E4M3(a / s)                  (nearest, ties to even, saturating)
// A row whose mean square plus eps is zero normalises to zeros; s = 0 gives
// all-zero codes.
//
// Two passes, because the scale depends on every element.  Rows of up to
// 25600 elements go through the shared-memory kernels further down; these
// loop kernels serve longer rows:
//   1. amax pass: one warp per row reads the row once, accumulating the sum
//      of squares and max|x * gamma|; the row's max|a| is that max times
//      1/rms (a positive factor, so the maximum commutes with the rounding),
//      and the block's largest max|a| / 448 goes to *s with an atomic max on
//      the float's bits (non-negative floats order like their bit patterns).
//      *s is zeroed by a memset before this pass.
//   2. quantise pass (programmatic dependent launch: waits for pass 1 inside
//      the kernel): each warp recomputes its row's 1/rms with the same code
//      as pass 1, then writes codes for 8 elements per lane step.
// HBM traffic: X is read once from HBM and once more from L2 when it fits
// there (129 MB), codes are written once: 3 bytes per element plus gamma.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "launch.h"
#include "swiglu.h"

namespace swiglu {
namespace {

constexpr int kWarps = 8;                  // rows in flight per block
constexpr int kThreads = kWarps * 32;
constexpr float kE4M3Max = 448.0f;         // largest finite E4M3 value

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float f[8]) {
  // BF16 -> FP32 is exact: the 16 bits become the upper half of the float.
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// 1/rms of a row from its sum of squares: correctly rounded division and
// square root, 0 when the denominator is 0 (a zero row with eps = 0).
__device__ __forceinline__ float inv_rms(float ss, int K, float eps) {
  const float d = __fadd_rn(__fdiv_rn(ss, (float)K), eps);
  return d > 0.0f ? __fdiv_rn(1.0f, __fsqrt_rn(d)) : 0.0f;
}

// Two floats to two E4M3 codes (round to nearest even, saturating to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <bool GAMMA>
__device__ __forceinline__ void load_row_vec(const uint4 *x, const uint4 *g, int v, float f[8]) {
  unpack_bf16x8(__ldg(x + v), f);
  if (GAMMA) {
    float gf[8];
    unpack_bf16x8(__ldg(g + v), gf);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], gf[i]);
  }
}

template <bool GAMMA>
__device__ __forceinline__ void load_row_vec_smem(const uint4 *x, const uint4 *g, int v,
                                                  float f[8]) {
  unpack_bf16x8(x[v], f);
  if (GAMMA) {
    float gf[8];
    unpack_bf16x8(__ldg(g + v), gf);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], gf[i]);
  }
}

// Pass 1: *scale_bits = bits of max over rows of (max|a| / 448).
template <bool NORM, bool GAMMA>
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4 *__restrict__ X,
                                                        const uint4 *__restrict__ gamma,
                                                        float eps, int64_t M, int K,
                                                        unsigned int *scale_bits) {
  __shared__ float red[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = K / 8;
  float mx = 0.0f;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < M;
       row += (int64_t)gridDim.x * kWarps) {
    const uint4 *x = X + row * nvec;
    float ss = 0.0f, rm = 0.0f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      float f[8], xf[8];
      unpack_bf16x8(__ldg(x + v), xf);
      if (GAMMA) {
        float gf[8];
        unpack_bf16x8(__ldg(gamma + v), gf);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(xf[i], gf[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = xf[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = __fmaf_rn(xf[i], xf[i], ss);
        rm = fmaxf(rm, fabsf(f[i]));
      }
    }
    rm = warp_max(rm);
    if (NORM) rm = __fmul_rn(rm, inv_rms(warp_sum(ss), K, eps));
    mx = fmaxf(mx, rm);
  }
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) m = fmaxf(m, red[i]);
    atomicMax(scale_bits, __float_as_uint(__fdiv_rn(m, kE4M3Max)));
  }
  // Let the quantise pass get scheduled; it still waits for this grid to
  // finish (griddepcontrol.wait) before it reads the scale.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Pass 2: codes for every element, from the scale pass 1 left in *scale.
template <bool NORM, bool GAMMA>
__global__ void __launch_bounds__(kThreads) quant_kernel(const uint4 *__restrict__ X,
                                                         const uint4 *__restrict__ gamma,
                                                         float eps, int64_t M, int K,
                                                         const float *scale, uint2 *__restrict__ Q) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = K / 8;
  const float s = *reinterpret_cast<const volatile float *>(scale);
  const float rcp = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < M;
       row += (int64_t)gridDim.x * kWarps) {
    const uint4 *x = X + row * nvec;
    uint2 *q = Q + row * nvec;
    float c = rcp;
    if (NORM) {
      float ss = 0.0f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float xf[8];
        unpack_bf16x8(__ldg(x + v), xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = __fmaf_rn(xf[i], xf[i], ss);
      }
      c = __fmul_rn(inv_rms(warp_sum(ss), K, eps), rcp);
    }
    if (c == 0.0f) {   // zero scale or zero row: all codes +0
      for (int v = lane; v < nvec; v += 32) q[v] = make_uint2(0u, 0u);
      continue;
    }
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      load_row_vec<GAMMA>(x, gamma, v, f);
      // Normalised rows: a / s as a * (1/rms) * (1/s), one product.  Without
      // the normalisation x / s is a correctly rounded division, so a
      // quotient that lands exactly on a midpoint between two codes (common:
      // x and max|x| are both BF16 values) rounds to the even code, as the
      // exact value does.
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = NORM ? __fmul_rn(f[i], c) : __fdiv_rn(f[i], s);
      uint2 o;
      o.x = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
      o.y = cvt_e4m3x2(f[4], f[5]) | (cvt_e4m3x2(f[6], f[7]) << 16);
      q[v] = o;
    }
  }
}

// ---- the same two passes with rows staged in shared memory ---------------
//
// Each block takes 4 rows: one thread copies them into shared memory with
// bulk copies (the copy engine moves the whole 4-row tile at once), then each
// warp reads its row from shared memory, once for the sum of squares and once
// more for the maximum (amax pass) or the codes (quantise pass).  With a few
// tens of KB per block, every SM has many rows in flight, which is what a
// read of a few tens of MB needs to run at HBM speed.  The sum of squares
// runs in the same order as in the loop kernels above.
//
// Launch chain, each later kernel with programmatic dependent launch:
//   zero kernel (normal launch: starts after all earlier work has completed)
//   -> amax pass: copies its rows in at once (X and gamma were complete
//      before the zero kernel started), waits for the zero kernel only
//      before its atomic maximum on the scale;
//   -> quantise pass: likewise copies and reduces its rows first and waits
//      for the amax pass only before it reads the scale.

constexpr int kSmemRows = 4;                 // rows per block, one per warp
constexpr int kSmemThreads = kSmemRows * 32;
constexpr int kSmemMaxBytes = 200 * 1024;    // dynamic shared memory budget per block
constexpr uint32_t kWaitProducerLoad = 8;    // where a wait gave up (device error word)

__global__ void zero_scale_kernel(float *s) {
  *s = 0.0f;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bulk-copy this block's rows into shared memory and wait for them (bounded).
__device__ __forceinline__ bool stage_rows(const uint8_t *X, int64_t row0, int nrows, int K,
                                           uint32_t buf, uint32_t bar, uint32_t *err,
                                           uint64_t timeout_ns) {
  if (threadIdx.x == 0) {
    const uint32_t row_bytes = static_cast<uint32_t>(K) * 2u;
    ptx::mbar_arrive_expect_tx(bar, row_bytes * nrows);
    for (int r = 0; r < nrows; ++r)
      ptx::bulk_load(buf + r * row_bytes, X + (row0 + r) * row_bytes, row_bytes, bar);
  }
  const uint64_t t0 = ptx::globaltimer_ns();
  bool ok = true;
  while (!ptx::mbar_try_wait(bar, 0)) {
    if (ptx::globaltimer_ns() - t0 > timeout_ns) {
      ok = false;
      break;
    }
  }
  if (!ok && threadIdx.x == 0 && atomicCAS(err, 0u, kErrTimeout) == 0u)
    atomicExch(err + 1, kWaitProducerLoad);
  return __syncthreads_and(ok) != 0;
}

template <bool NORM, bool GAMMA, bool QUANT>
__global__ void __launch_bounds__(kSmemThreads) rows_smem_kernel(
    const uint8_t *__restrict__ X, const uint4 *__restrict__ gamma, float eps, int64_t M, int K,
    float *scale, uint2 *__restrict__ Q, uint32_t *err, uint64_t timeout_ns) {
  extern __shared__ __align__(16) uint8_t rows_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[kSmemRows];
  if (!QUANT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = K / 8;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kSmemRows;
  const int nrows = static_cast<int>(M - row0 < kSmemRows ? M - row0 : kSmemRows);
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const bool ok = stage_rows(X, row0, nrows, K, ptx::smem_u32(rows_smem), b, err, timeout_ns);
  const bool live = ok && warp < nrows;
  const uint4 *x = reinterpret_cast<const uint4 *>(rows_smem) + warp * nvec;
  float inv = 1.0f;
  if (live && NORM) {
    float ss = 0.0f;
    for (int v = lane; v < nvec; v += 32) {
      float xf[8];
      unpack_bf16x8(x[v], xf);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = __fmaf_rn(xf[j], xf[j], ss);
    }
    inv = inv_rms(warp_sum(ss), K, eps);
  }
  if (!QUANT) {
    float rm = 0.0f;
    if (live) {
      for (int v = lane; v < nvec; v += 32) {
        float f[8];
        load_row_vec_smem<GAMMA>(x, gamma, v, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) rm = fmaxf(rm, fabsf(f[j]));
      }
      rm = warp_max(rm);
      if (NORM) rm = __fmul_rn(rm, inv);
    }
    if (lane == 0) red[warp] = rm;
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the zero kernel has written the scale
    if (threadIdx.x == 0) {
      float m = red[0];
#pragma unroll
      for (int i = 1; i < kSmemRows; ++i) m = fmaxf(m, red[i]);
      atomicMax(reinterpret_cast<unsigned int *>(scale), __float_as_uint(__fdiv_rn(m, kE4M3Max)));
    }
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the amax pass has finished the scale
  if (!live) return;
  const float s = *reinterpret_cast<const volatile float *>(scale);
  const float rcp = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
  const float c = NORM ? __fmul_rn(inv, rcp) : rcp;
  uint2 *q = Q + (row0 + warp) * nvec;
  for (int v = lane; v < nvec; v += 32) {
    if (c == 0.0f) {  // zero scale or zero row: all codes +0
      q[v] = make_uint2(0u, 0u);
      continue;
    }
    float f[8];
    load_row_vec_smem<GAMMA>(x, gamma, v, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = NORM ? __fmul_rn(f[j], c) : __fdiv_rn(f[j], s);
    uint2 o;
    o.x = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
    o.y = cvt_e4m3x2(f[4], f[5]) | (cvt_e4m3x2(f[6], f[7]) << 16);
    q[v] = o;
  }
}

template <bool NORM, bool GAMMA>
cudaError_t launch_rows_smem(const void *X, const uint4 *g, float eps, void *Q, float *s,
                             int64_t M, int K, uint32_t *err, uint64_t timeout_ns,
                             uint64_t ctx_gen, cudaStream_t st) {
  static PerDeviceOnce once;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (once.needed(dev, ctx_gen)) {
    e = cudaFuncSetAttribute(rows_smem_kernel<NORM, GAMMA, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMaxBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(rows_smem_kernel<NORM, GAMMA, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMaxBytes);
    if (e != cudaSuccess) return e;
    once.done(dev, ctx_gen);
  }
  const int64_t blocks = (M + kSmemRows - 1) / kSmemRows;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kSmemRows) * K * 2;
  zero_scale_kernel<<<1, 32, 0, st>>>(s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kSmemThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint8_t *x = static_cast<const uint8_t *>(X);
  uint2 *q = static_cast<uint2 *>(Q);
  e = cudaLaunchKernelEx(&cfg, rows_smem_kernel<NORM, GAMMA, false>, x, g, eps, M, K, s, q, err,
                         timeout_ns);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, rows_smem_kernel<NORM, GAMMA, true>, x, g, eps, M, K, s, q, err,
                            timeout_ns);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

template <bool NORM, bool GAMMA>
cudaError_t launch_producer(const void *X, const void *gamma, float eps, void *Q, float *s,
                            int64_t M, int K, cudaStream_t st) {
  uint32_t *err = nullptr;
  int sms = 0;
  uint64_t timeout_ns = 0, ctx_gen = 0;
  if (device_info(&err, &sms, &timeout_ns, &ctx_gen) != SWIGLU_OK) return cudaErrorUnknown;
  if (M > 0 && int64_t(kSmemRows) * K * 2 <= kSmemMaxBytes)
    return launch_rows_smem<NORM, GAMMA>(X, static_cast<const uint4 *>(gamma), eps, Q, s, M, K,
                                         err, timeout_ns, ctx_gen, st);
  cudaError_t e = cudaMemsetAsync(s, 0, sizeof(float), st);
  if (e != cudaSuccess || M == 0) return e;
  // longer rows: the loop kernels
  // Up to 8 blocks of 8 warps per SM (64 warps, the SM's limit), one warp per
  // row, grid-stride beyond that.
  const int64_t want = (M + kWarps - 1) / kWarps;
  const int grid = (int)std::min<int64_t>(want, (int64_t)sms * 8);
  const uint4 *x = static_cast<const uint4 *>(X);
  const uint4 *g = static_cast<const uint4 *>(gamma);
  amax_kernel<NORM, GAMMA><<<grid, kThreads, 0, st>>>(x, g, eps, M, K,
                                                      reinterpret_cast<unsigned int *>(s));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_kernel<NORM, GAMMA>, x, g, eps, M, K,
                            static_cast<const float *>(s), static_cast<uint2 *>(Q));
}

// X and Q may be null when M = 0 (nothing is read or written but the scale).
int check_common(const void *X, const void *Q, const float *s, int64_t M, int64_t K) {
  if (!s || M < 0 || K <= 0 || (M > 0 && (!X || !Q))) return SWIGLU_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > (int64_t)1 << 30) return SWIGLU_ERR_UNSUPPORTED;
  if (!aligned(X, 16) || !aligned(Q, 16) || !aligned(s, 4)) return SWIGLU_ERR_MISALIGNED;
  return SWIGLU_OK;
}

}  // namespace
}  // namespace swiglu

extern "C" int swiglu_rmsnorm_quant_fp8(const void *X, const void *gamma, float eps, void *Aq,
                                        float *sA, int64_t M, int64_t K, void *stream) {
  using namespace swiglu;
  int rc = check_common(X, Aq, sA, M, K);
  if (rc != SWIGLU_OK) return rc;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return SWIGLU_ERR_INVALID_ARG;
  if (gamma && !aligned(gamma, 16)) return SWIGLU_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = gamma ? launch_producer<true, true>(X, gamma, eps, Aq, sA, M, (int)K, st)
                        : launch_producer<true, false>(X, nullptr, eps, Aq, sA, M, (int)K, st);
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

extern "C" int swiglu_quant_fp8(const void *X, void *Xq, float *s, int64_t M, int64_t K,
                                void *stream) {
  using namespace swiglu;
  int rc = check_common(X, Xq, s, M, K);
  if (rc != SWIGLU_OK) return rc;
  cudaError_t e = launch_producer<false, false>(X, nullptr, 0.0f, Xq, s, M, (int)K,
                                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}
