// k_bf16_swab.cu -- the swapped-operand CTA-pair kernel for few rows, both
// weight forms.
#include "launch.h"
#include "swiglu_swab_kernel.cuh"

namespace swiglu {
namespace {

template <class C>
cudaError_t launch_swab_cfg(const LaunchArgs &la) {
  static PerDeviceOnce once;
  auto kern = swiglu_swab_kernel<C>;
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    once.done(la.device, la.ctx_gen);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * la.p.num_n_blk), 1, 1);  // one pair per 64 columns
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, la.p);
}

}  // namespace

cudaError_t launch_bf16_swab(bool interleaved, int rows, const LaunchArgs &la) {
  if (rows == 64)
    return interleaved ? launch_swab_cfg<SwabCfg<true, 64>>(la) : launch_swab_cfg<SwabCfg<false, 64>>(la);
  return interleaved ? launch_swab_cfg<SwabCfg<true, 128>>(la) : launch_swab_cfg<SwabCfg<false, 128>>(la);
}

}  // namespace swiglu
