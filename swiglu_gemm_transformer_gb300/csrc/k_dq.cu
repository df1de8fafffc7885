// k_dq.cu -- the wide-tile kernel for INT4, MXFP8 and NVFP4 weights.
#include "launch.h"
#include "swiglu_dq_kernel.cuh"

namespace swiglu {
namespace {

template <class C>
cudaError_t launch_dq(const LaunchArgs &la) {
  static PerDeviceOnce once;
  auto kern = swiglu_dq_kernel<C>;
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    once.done(la.device, la.ctx_gen);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int64_t tiles = int64_t(la.p.num_m_blk) * la.p.num_n_blk;  // one tile per CTA
  cfg.gridDim = dim3(static_cast<unsigned>(tiles), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, la.s1, la.s2, la.p);
}

}  // namespace

cudaError_t launch_dq_kernel(int wf, int m_blocks, const LaunchArgs &la) {
  if (m_blocks == 2) {
    switch (wf) {
      case WF_INT4: return launch_dq<DqCfg<WF_INT4, 2>>(la);
      case WF_MXFP8: return launch_dq<DqCfg<WF_MXFP8, 2>>(la);
      case WF_NVFP4: return launch_dq<DqCfg<WF_NVFP4, 2>>(la);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (wf) {
    case WF_INT4: return launch_dq<DqCfg<WF_INT4>>(la);
    case WF_MXFP8: return launch_dq<DqCfg<WF_MXFP8>>(la);
    case WF_NVFP4: return launch_dq<DqCfg<WF_NVFP4>>(la);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swiglu
