// launch.h -- internal interface between the C-ABI host code and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "swiglu_tc_kernel.cuh"
#include "tc_common.cuh"

namespace swiglu {

struct LaunchArgs {
  CUtensorMap a, b0, b1, y;
  CUtensorMap s1, s2;  // INT4 weights: the gate and up scale matrices
  KParams p;
  int grid;
  int device;
  // Generation of the device's context the call runs in: it changes when the
  // context is replaced (e.g. after cudaDeviceReset), which drops every
  // function attribute set on the old one.
  uint64_t ctx_gen;
  cudaStream_t stream;
};

// One-time launch set-up per device (function attributes such as the
// dynamic shared-memory opt-in), redone when the device's context changes.
// Objects of this class live in static storage (zero-initialised);
// generations start at 1.
class PerDeviceOnce {
 public:
  bool needed(int device, uint64_t gen) const {
    return gen_[device & 63].load(std::memory_order_acquire) != gen;
  }
  void done(int device, uint64_t gen) { gen_[device & 63].store(gen, std::memory_order_release); }

 private:
  std::atomic<uint64_t> gen_[64];
};

// Tile geometry of each BF16 variant (SWIGLU_VARIANT_*), for host-side planning.
struct VariantGeom {
  int bm, bn, bk;     // output rows, output columns, K per stage (per tile)
  int box_b;          // weight box width (columns) per TMA copy
  int b_swizzle_64;   // 1: weight boxes use the 64-byte swizzle (32-column boxes)
  int box_a;          // A box height (rows) per TMA copy
  int cluster;        // CTAs per tile (1, or 2 for the CTA-pair kernel)
};

VariantGeom variant_geom(int variant, bool interleaved);

cudaError_t launch_bf16_separate(int variant, const LaunchArgs &la);
cudaError_t launch_bf16_interleaved(int variant, const LaunchArgs &la);
cudaError_t launch_bf16_sk(bool interleaved, const LaunchArgs &la);
// rows: 64 or 128 rows of A per CTA pair (M <= rows); la.p.num_n_blk pairs of 64 columns
cudaError_t launch_bf16_swab(bool interleaved, int rows, const LaunchArgs &la);
cudaError_t launch_w4_sk(const LaunchArgs &la);
cudaError_t launch_mx_sk(bool nvfp4, const LaunchArgs &la);
// wf: 1 INT4, 2 MXFP8, 3 NVFP4 (weight_decode.cuh); m_blocks: 128-row blocks
// per CTA (1, or 2 with la.p.num_m_blk counting 256-row blocks)
cudaError_t launch_dq_kernel(int wf, int m_blocks, const LaunchArgs &la);
// INT4, MXFP8 or NVFP4 weights (wf 1, 2, 3) decoded into tensor memory: tok 64
// or 128 tokens per pass; la.p.num_n_blk CTAs of 128 weight columns
cudaError_t launch_dqt(int tok, int wf, const LaunchArgs &la);
cudaError_t launch_pack_w4_kmajor(const void *Wq, void *Wk, int64_t K, int64_t N, int sm_count,
                                  cudaStream_t s);
int device_info(uint32_t **err, int *sm_count, uint64_t *timeout_ns, uint64_t *ctx_gen);
// CTA-pair kernels: whether launches with more units than resident pairs use
// the dynamic unit schedule.
bool pair_dynamic_schedule();
cudaError_t launch_pack_interleaved_u16(const void *W1, const void *W2, void *Wf, int64_t n_elems,
                                        int sm_count, cudaStream_t s);
cudaError_t launch_selftest_wait(uint64_t limit_ns, uint32_t *err, cudaStream_t s);
cudaError_t launch_fp8(bool interleaved, const LaunchArgs &la);
cudaError_t launch_linear(int lin_n, const LaunchArgs &la);
// cs: CTAs per cluster (2, 4 or 8); bn: tile width (64 or 128); la.p tiles are 128 x bn
cudaError_t launch_linear_sk(int cs, int bn, const LaunchArgs &la);
cudaError_t launch_splitk_reduce(const float *ws, int splits, const void *R, void *Z, int64_t M,
                                 int64_t N, int sm_count, cudaStream_t s);
cudaError_t launch_pack_rows_interleaved_u8(const void *W1t, const void *W2t, void *Wft,
                                            int64_t N, int64_t K, int sm_count, cudaStream_t s);

}  // namespace swiglu
