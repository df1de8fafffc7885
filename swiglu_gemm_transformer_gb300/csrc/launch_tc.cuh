// launch_tc.cuh -- one launcher per tcgen05 kernel configuration.
#pragma once

#include "launch.h"
#include "swiglu_tc2_kernel.cuh"

namespace swiglu {

// Launch attributes shared by every fused kernel: programmatic dependent
// launch (the prologue may overlap the previous kernel on the stream; the
// kernel waits on griddepcontrol.wait before touching global memory).
inline void pdl_attr(cudaLaunchAttribute &a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}

template <class C>
cudaError_t launch_tc(const LaunchArgs &la) {
  // Per-device one-time set-up: the dynamic shared-memory opt-in.
  static PerDeviceOnce once;
  auto kern = swiglu_bf16_tc_kernel<C>;
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    once.done(la.device, la.ctx_gen);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_attr(attr[0]);
  cfg.gridDim = dim3(la.grid, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, la.p);
}

// CTA-pair kernel: 2-CTA clusters, persistent over as many clusters as can be
// resident at once (queried once per device).
template <class C>
cudaError_t launch_pair(const LaunchArgs &la) {
  static PerDeviceOnce once;
  static int max_clusters[64] = {0};
  auto kern = swiglu_bf16_pair_kernel<C>;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  pdl_attr(attr[1]);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  if (once.needed(la.device, la.ctx_gen)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * 64, 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters[la.device & 63] = n;
    once.done(la.device, la.ctx_gen);
  }
  // work units: output tiles x K slices
  const int64_t tiles =
      int64_t(la.p.num_m_blk) * la.p.num_n_blk * (la.p.k_splits > 1 ? la.p.k_splits : 1);
  const int n = max_clusters[la.device & 63];
  // One wave: one cluster per unit, static.  More units than resident pairs:
  // the dynamic schedule (one cluster per unit, taken over by running pairs)
  // unless turned off; else one wave of pairs walking the units statically.
  KParams p = la.p;
  p.dyn_sched = tiles > n && tiles <= (int64_t(1) << 30) && pair_dynamic_schedule() ? 1 : 0;
  const int64_t clusters = p.dyn_sched ? tiles : (tiles < n ? tiles : n);
  cfg.gridDim = dim3(unsigned(2 * clusters), 1, 1);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, p);
}

}  // namespace swiglu
