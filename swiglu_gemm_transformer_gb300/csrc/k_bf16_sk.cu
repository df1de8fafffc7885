// k_bf16_sk.cu -- the split-K cluster kernel for small M, both weight forms.
#include "launch.h"
#include "swiglu_sk_kernel.cuh"

namespace swiglu {
namespace {

template <class C>
cudaError_t launch_sk(const LaunchArgs &la) {
  static PerDeviceOnce once;
  auto kern = swiglu_bf16_sk_kernel<C>;
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    once.done(la.device, la.ctx_gen);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  const int64_t tiles = int64_t(la.p.num_m_blk) * la.p.num_n_blk;  // one tile per cluster
  cfg.gridDim = dim3(static_cast<unsigned>(2 * tiles), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, la.s1, la.s2, la.p);
}

}  // namespace

cudaError_t launch_bf16_sk(bool interleaved, const LaunchArgs &la) {
  return interleaved ? launch_sk<SkCfg<true>>(la) : launch_sk<SkCfg<false>>(la);
}

cudaError_t launch_w4_sk(const LaunchArgs &la) { return launch_sk<SkCfg<false, WF_INT4>>(la); }
cudaError_t launch_mx_sk(bool nvfp4, const LaunchArgs &la) {
  return nvfp4 ? launch_sk<SkCfg<false, WF_NVFP4>>(la) : launch_sk<SkCfg<false, WF_MXFP8>>(la);
}

}  // namespace swiglu
