// k_linear.cu -- the linear (down-projection) instantiations of the CTA-pair
// kernel and the split-K reduction kernel.
#include <algorithm>

#include <cuda_bf16.h>

#include "launch_tc.cuh"
#include "swiglu_linsk_kernel.cuh"

namespace swiglu {

cudaError_t launch_linear(int lin_n, const LaunchArgs &la) {
  return lin_n == 256 ? launch_pair<PairCfg<true, 6, false, true, 256>>(la)
                      : launch_pair<PairCfg<true, 8, false, true, 128>>(la);
}

namespace {

// The split-K cluster down projection: one 128 x BN output tile per cluster
// of CS CTAs (la.p.num_m_blk x la.p.num_n_blk tiles).
template <int CS, int BN>
cudaError_t launch_linsk(const LaunchArgs &la) {
  using C = LinSkCfg<CS, BN>;
  static PerDeviceOnce once;
  auto kern = swiglu_linsk_kernel<C>;
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    once.done(la.device, la.ctx_gen);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  const int64_t tiles = int64_t(la.p.num_m_blk) * la.p.num_n_blk;  // one tile per cluster
  cfg.gridDim = dim3(static_cast<unsigned>(CS * tiles), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.p);
}

}  // namespace

cudaError_t launch_linear_sk(int cs, int bn, const LaunchArgs &la) {
  if (bn == 128) {
    switch (cs) {
      case 2: return launch_linsk<2, 128>(la);
      case 4: return launch_linsk<4, 128>(la);
      case 8: return launch_linsk<8, 128>(la);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (cs) {
    case 2: return launch_linsk<2, 64>(la);
    case 4: return launch_linsk<4, 64>(la);
    case 8: return launch_linsk<8, 64>(la);
    default: return cudaErrorInvalidValue;
  }
}

// Z = BF16(sum_s ws[s] + R): four columns per thread (N is a multiple of 8),
// one pass over the FP32 partial sums; memory-bound, grid-stride, with the
// slices' loads unrolled so they are in flight together.  Launched as a
// programmatic dependent of the linear kernel: its blocks are resident while
// that kernel ends and read the partial sums only after it has completed.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4 *__restrict__ ws,
                                                            int splits, int64_t slice_vec4,
                                                            const uint2 *__restrict__ R,
                                                            uint2 *__restrict__ Z, int64_t n_vec4) {
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (R != nullptr) {
      const uint2 r = __ldg(R + i);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
      acc = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    int s = 0;
    for (; s + 4 <= splits; s += 4) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __ldg(ws + (s + j) * slice_vec4 + i);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
      }
    }
    for (; s < splits; ++s) {
      const float4 v = __ldg(ws + s * slice_vec4 + i);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t *>(&lo);
    o.y = *reinterpret_cast<const uint32_t *>(&hi);
    Z[i] = o;
  }
}

cudaError_t launch_splitk_reduce(const float *ws, int splits, const void *R, void *Z, int64_t M,
                                 int64_t N, int sm_count, cudaStream_t s) {
  const int64_t n_vec4 = M * N / 4;
  if (n_vec4 == 0) return cudaSuccess;
  const int threads = 256;
  const int grid = (int)std::min<int64_t>((n_vec4 + threads - 1) / threads, (int64_t)sm_count * 8);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, reinterpret_cast<const float4 *>(ws),
                            splits, M * N / 4, static_cast<const uint2 *>(R),
                            static_cast<uint2 *>(Z), n_vec4);
}

}  // namespace swiglu
