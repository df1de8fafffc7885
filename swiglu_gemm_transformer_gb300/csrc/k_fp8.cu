// k_fp8.cu -- instantiations of the CTA-pair kernel for FP8 E4M3 operands
// (K-major weights, per-tensor scales), and the row-interleave packer for the
// K-major W_fused layout.
#include <algorithm>

#include "launch_tc.cuh"
#include "swiglu.h"

namespace swiglu {

cudaError_t launch_fp8(bool interleaved, const LaunchArgs &la) {
  return interleaved ? launch_pair<PairCfg<true, 6, true>>(la)
                     : launch_pair<PairCfg<false, 6, true>>(la);
}

// W_fused^T[2n, :] = W1^T[n, :] (gate), W_fused^T[2n+1, :] = W2^T[n, :] (up):
// the column interleave of page "Riepilogo Tecnico ...", section "Metodologia",
// item 2, in the K-major ([N,K] row-major) storage of the FP8 weights.  Each
// thread moves one 16-byte vector; rows are K bytes (K a multiple of 16).
__global__ void __launch_bounds__(256) pack_rows_interleaved_u8_kernel(
    const uint4 *__restrict__ w1t, const uint4 *__restrict__ w2t, uint4 *__restrict__ wft,
    int64_t n_rows, int64_t vec_per_row) {
  const int64_t total = 2 * n_rows * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t out_row = i / vec_per_row, v = i - out_row * vec_per_row;
    const int64_t src_row = out_row >> 1;
    const uint4 *src = (out_row & 1) ? w2t : w1t;
    wft[i] = __ldg(src + src_row * vec_per_row + v);
  }
}

cudaError_t launch_pack_rows_interleaved_u8(const void *W1t, const void *W2t, void *Wft,
                                            int64_t N, int64_t K, int sm_count, cudaStream_t s) {
  const int64_t vec_per_row = K / 16;
  const int64_t total = 2 * N * vec_per_row;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int grid = (int)std::min<int64_t>((total + threads - 1) / threads, (int64_t)sm_count * 8);
  pack_rows_interleaved_u8_kernel<<<grid, threads, 0, s>>>(static_cast<const uint4 *>(W1t),
                                                            static_cast<const uint4 *>(W2t),
                                                            static_cast<uint4 *>(Wft), N,
                                                            vec_per_row);
  return cudaGetLastError();
}

}  // namespace swiglu
