// k_bf16_interleaved.cu -- instantiations of the tcgen05 kernel for the
// interleaved W_fused[K,2N] form.
#include "launch_tc.cuh"
#include "swiglu.h"

namespace swiglu {

cudaError_t launch_bf16_interleaved(int variant, const LaunchArgs &la) {
  switch (variant) {
    case SWIGLU_VARIANT_1SM_N128:
      return launch_tc<TileCfg<4, 64, true, 4>>(la);
    case SWIGLU_VARIANT_1SM_N64:
      return launch_tc<TileCfg<2, 64, true, 6>>(la);
    case SWIGLU_VARIANT_1SM_N32:
      return launch_tc<TileCfg<1, 64, true, 8>>(la);
    case SWIGLU_VARIANT_2SM_N128:
      return launch_pair<PairCfg<true, 6>>(la);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace swiglu
