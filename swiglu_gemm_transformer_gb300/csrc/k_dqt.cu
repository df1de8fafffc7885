// k_dqt.cu -- INT4, MXFP8 and NVFP4 weights decoded into tensor memory (swiglu_dqt_kernel.cuh),
// and the packer that writes the K-major code layout it reads.
#include "launch.h"
#include "swiglu_dqt_kernel.cuh"

namespace swiglu {
namespace {

template <class C>
cudaError_t launch_dqt_cfg(const LaunchArgs &la) {
  static PerDeviceOnce once;
  auto kern = swiglu_dqt_kernel<C>;
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
  cfg.gridDim = dim3(static_cast<unsigned>(la.p.num_n_blk), 1, 1);  // one CTA per 128 columns
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = la.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, la.a, la.b0, la.b1, la.y, la.s1, la.s2, la.p);
}

// Wk[n][j] (32-bit word j of column n) holds codes k = 8j .. 8j + 7 of column
// n: code 8j + 2i in nibble i and code 8j + 2i + 1 in nibble 4 + i (i < 4),
// so ((word >> 4i) & 0x000F000F) is the pair (k, k + 1) in two 16-bit halves.
// Wq is [K, N/2] bytes with column n in the low nibble of byte n/2 when n is
// even, in the high nibble when odd.  One thread per output word.
__global__ void pack_w4_kmajor_kernel(const uint8_t *__restrict__ Wq, uint32_t *__restrict__ Wk,
                                      int64_t K, int64_t N) {
  const int64_t words_per_col = K / 8;
  const int64_t total = N * words_per_col;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t n = idx / words_per_col, j = idx % words_per_col;
    const uint8_t *src = Wq + (8 * j) * (N / 2) + n / 2;
    const int sh = (n & 1) ? 4 : 0;
    uint32_t w = 0;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t code = (src[kk * (N / 2)] >> sh) & 0xFu;
      const int nib = (kk & 1) ? 4 + kk / 2 : kk / 2;
      w |= code << (4 * nib);
    }
    Wk[idx] = w;
  }
}

}  // namespace

cudaError_t launch_dqt(int tok, int wf, const LaunchArgs &la) {
  if (wf == WF_NVFP4)
    return tok == 64 ? launch_dqt_cfg<DqtCfg<64, WF_NVFP4>>(la) : launch_dqt_cfg<DqtCfg<128, WF_NVFP4>>(la);
  if (wf == WF_MXFP8)
    return tok == 64 ? launch_dqt_cfg<DqtCfg<64, WF_MXFP8>>(la) : launch_dqt_cfg<DqtCfg<128, WF_MXFP8>>(la);
  return tok == 64 ? launch_dqt_cfg<DqtCfg<64>>(la) : launch_dqt_cfg<DqtCfg<128>>(la);
}

cudaError_t launch_pack_w4_kmajor(const void *Wq, void *Wk, int64_t K, int64_t N, int sm_count,
                                  cudaStream_t s) {
  const int64_t total = N * (K / 8);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = int64_t(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_w4_kmajor_kernel<<<unsigned(blocks), 256, 0, s>>>(static_cast<const uint8_t *>(Wq),
                                                          static_cast<uint32_t *>(Wk), K, N);
  return cudaGetLastError();
}

}  // namespace swiglu
