// launch_tc.cuh -- one launcher per tcgen05 kernel configuration.
#pragma once

#include <atomic>

#include "launch.h"

namespace swiglu {

template <class C>
cudaError_t launch_tc(const LaunchArgs &la) {
  // The dynamic shared-memory opt-in is a per-device function attribute; set it
  // once per device.
  static std::atomic<uint64_t> configured{0};
  const uint64_t bit = 1ull << (la.device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(swiglu_bf16_tc_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  swiglu_bf16_tc_kernel<C><<<la.grid, C::THREADS, C::SMEM_BYTES, la.stream>>>(la.a, la.b0, la.b1,
                                                                                la.y, la.p);
  return cudaGetLastError();
}

}  // namespace swiglu
