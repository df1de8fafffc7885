// k_misc.cu -- the W_fused packer and the bounded-wait self-test kernel.
#include <algorithm>

#include "launch.h"

namespace swiglu {

// W_fused[k, 2n] = W1[k, n], W_fused[k, 2n+1] = W2[k, n]  (page "Riepilogo
// Tecnico ...", section "Metodologia", item 2).  With N a multiple of 8, eight
// consecutive elements of a W1 row starting at flat index j map to the sixteen
// consecutive W_fused elements starting at 2j, so each thread moves one
// 16-byte vector of W1 and of W2 into two 16-byte vectors of W_fused.
// Memory-bound: 2 x 16 B read, 32 B written per vector, grid-stride.
__global__ void __launch_bounds__(256) pack_interleaved_u16_kernel(const uint4 *__restrict__ w1,
                                                                   const uint4 *__restrict__ w2,
                                                                   uint4 *__restrict__ wf,
                                                                   int64_t n_vec) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = __ldg(w1 + i);
    const uint4 b = __ldg(w2 + i);
    uint4 o0, o1;
    o0.x = (a.x & 0xFFFFu) | (b.x << 16);
    o0.y = (a.x >> 16) | (b.x & 0xFFFF0000u);
    o0.z = (a.y & 0xFFFFu) | (b.y << 16);
    o0.w = (a.y >> 16) | (b.y & 0xFFFF0000u);
    o1.x = (a.z & 0xFFFFu) | (b.z << 16);
    o1.y = (a.z >> 16) | (b.z & 0xFFFF0000u);
    o1.z = (a.w & 0xFFFFu) | (b.w << 16);
    o1.w = (a.w >> 16) | (b.w & 0xFFFF0000u);
    wf[2 * i] = o0;
    wf[2 * i + 1] = o1;
  }
}

cudaError_t launch_pack_interleaved_u16(const void *W1, const void *W2, void *Wf, int64_t n_elems,
                                        int sm_count, cudaStream_t s) {
  const int64_t n_vec = n_elems / 8;
  if (n_vec == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (n_vec + threads - 1) / threads;
  const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count * 8);
  pack_interleaved_u16_kernel<<<grid, threads, 0, s>>>(static_cast<const uint4 *>(W1),
                                                        static_cast<const uint4 *>(W2),
                                                        static_cast<uint4 *>(Wf), n_vec);
  return cudaGetLastError();
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t *err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing arrives on `bar`: phase 0 never completes and the wait gives up.
    wait_bar(b, 0, limit_ns, &abort_flag, err, WAIT_SELFTEST);
  }
  __syncthreads();
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, uint32_t *err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace swiglu
