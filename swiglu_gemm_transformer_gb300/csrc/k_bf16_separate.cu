// k_bf16_separate.cu -- instantiations of the tcgen05 kernel for the separate
// weight form (W1 and W2 as two [K,N] matrices).
#include "launch_tc.cuh"
#include "swiglu.h"

namespace swiglu {

cudaError_t launch_bf16_separate(int variant, const LaunchArgs &la) {
  switch (variant) {
    case SWIGLU_VARIANT_1SM_N128:
      return launch_tc<TileCfg<4, 64, false, 4>>(la);
    case SWIGLU_VARIANT_1SM_N64:
      return launch_tc<TileCfg<2, 64, false, 6>>(la);
    case SWIGLU_VARIANT_1SM_N32:
      return launch_tc<TileCfg<2, 32, false, 8>>(la);
    case SWIGLU_VARIANT_2SM_N128:
      return launch_pair<PairCfg<false, 6>>(la);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace swiglu
