// swiglu_api.cu -- host side of the C ABI declared in include/swiglu.h:
// argument validation, per-device state, TMA tensor-map encoding, variant
// choice and launch.  No entry point allocates device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "swiglu.h"

using namespace swiglu;

// Device error word: [0] = first status recorded by a kernel since the last
// swiglu_device_status(), [1] = which wait gave up.
__device__ uint32_t g_swiglu_err_word[2];

namespace {

struct DeviceState {
  bool ready = false;
  int status = SWIGLU_OK;  // sticky result of the one-time set-up
  int sm_count = 0;
  uint32_t *err = nullptr;
  // The context the set-up was done in (driver context id, 0 if unknown) and
  // its generation number: a new context on the device (after
  // cudaDeviceReset) gets a new generation, and the set-up is redone.
  unsigned long long ctx_id = 0;
  uint64_t gen = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_weights_read_only{0};
// Weight-format kernel: -1 = chosen by shape, 0/1/2 forces one (sweeps, tests).
std::atomic<int> g_weight_kernel_forced{-1};
// Row blocks that walk the column blocks together in the CTA-pair kernels'
// tile order: 0 = the default (8), else the SWIGLU_GROUP_M environment
// variable's value, read once (for tuning sweeps).
std::atomic<int> g_group_m{0};
// Down-projection tile width: 0 = chosen by shape; 128 or 256 forces it (the
// SWIGLU_LINEAR_N environment variable, read once, sets it for tuning sweeps).
std::atomic<int> g_linear_n{0};
// Split-K cluster down projection: -1 = chosen by shape, 0 = never, 2/4/8 =
// that cluster size whenever its grid fits one wave (SWIGLU_LINEAR_SK), and
// 0 = either tile width, 64 or 128 = that one (SWIGLU_LINEAR_SKN); both read
// once, for tuning sweeps.
std::atomic<int> g_linear_sk{-1};
std::atomic<int> g_linear_skn{0};
// CTA-pair kernels with more units than resident pairs: 1 = dynamic unit
// schedule (cluster launch control), 0 = static (swiglu_set_pair_schedule;
// the SWIGLU_PAIR_SCHED=static environment variable, read once, sets 0).
std::atomic<int> g_pair_dyn{1};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
uint64_t g_next_gen = 1;  // guarded by g_mu

void *driver_entry(const char *name, int version) {
  cudaDriverEntryPointQueryResult q;
  void *fn = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return fn;
}

// Process-unique id of the calling thread's current context; 0 when none is
// current or the driver offers no id.
unsigned long long current_ctx_id() {
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current && g_ctx_get_id && g_ctx_current(&c) == CUDA_SUCCESS && c != nullptr &&
      g_ctx_get_id(c, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

int device_state(DeviceState **out, int *dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SWIGLU_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(
        driver_entry("cuTensorMapEncodeTiled", 12000));
    if (!g_encode) return SWIGLU_ERR_CUDA;
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent", 4000));
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId", 12000));
  }
  DeviceState &st = g_dev[dev];
  if (!st.ready || current_ctx_id() != st.ctx_id) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
    // The kernels are built for sm_103a only (arch-specific tcgen05 code).
    if (major != 10 || minor != 3) return SWIGLU_ERR_UNSUPPORTED;
    // (also makes the device's primary context current on this thread)
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&st.err), g_swiglu_err_word) !=
        cudaSuccess) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
    const unsigned long long id = current_ctx_id();
    if (!st.ready || id != st.ctx_id) st.gen = g_next_gen++;
    st.ctx_id = id;
    st.sm_count = sms;
    st.ready = true;
    if (const char *e = std::getenv("SWIGLU_LINEAR_N")) {
      const long v = std::strtol(e, nullptr, 10);
      if (v == 128 || v == 256) g_linear_n.store(int(v), std::memory_order_relaxed);
    }
    if (const char *e = std::getenv("SWIGLU_GROUP_M")) {
      const long v = std::strtol(e, nullptr, 10);
      if (v >= 1 && v <= 4096) g_group_m.store(int(v), std::memory_order_relaxed);
    }
    if (const char *e = std::getenv("SWIGLU_LINEAR_SK")) {
      const long v = std::strtol(e, nullptr, 10);
      if (v == 0 || v == 2 || v == 4 || v == 8) g_linear_sk.store(int(v), std::memory_order_relaxed);
    }
    if (const char *e = std::getenv("SWIGLU_PAIR_SCHED")) {
      if (std::strcmp(e, "static") == 0) g_pair_dyn.store(0, std::memory_order_relaxed);
    }
    if (const char *e = std::getenv("SWIGLU_LINEAR_SKN")) {
      const long v = std::strtol(e, nullptr, 10);
      if (v == 64 || v == 128) g_linear_skn.store(int(v), std::memory_order_relaxed);
    }
  }
  *out = &st;
  *dev_out = dev;
  return SWIGLU_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, uint64_t an, const void *b, uint64_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

int encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
              uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int pair_group_m() {
  const int g = g_group_m.load(std::memory_order_relaxed);
  return g > 0 ? g : 8;
}

// The variants a caller may name (numbers 5-8 are retired and rejected).
bool variant_known(int32_t v) {
  return v == SWIGLU_VARIANT_AUTO || v == SWIGLU_VARIANT_1SM_N128 || v == SWIGLU_VARIANT_1SM_N64 ||
         v == SWIGLU_VARIANT_2SM_N128 || v == SWIGLU_VARIANT_1SM_N32 ||
         v == SWIGLU_VARIANT_1SM_N64_SK2 || v == SWIGLU_VARIANT_2SM_SWAP;
}

// Kernel for the weight formats (INT4, MXFP8, NVFP4): 0 = the split-K
// cluster kernel (64-column tiles; few rows and few columns, so that its
// tiles fill the GPU), 1 = the wide kernel with one 128-row block per CTA,
// 2 = the wide kernel with two (M > 128 and that grid still fills about one
// wave: one decode of each weight step then serves 256 rows).
int weight_kernel(int64_t M, int64_t N, int sm_count) {
  const int forced = g_weight_kernel_forced.load(std::memory_order_relaxed);
  if (forced >= 0) return forced;
  if (M <= 128 && 2 * cdiv(N, 64) <= sm_count) return 0;
  if (M > 128 && 10 * cdiv(M, 256) * cdiv(N, 128) >= 9 * int64_t(sm_count)) return 2;
  return 1;
}


int choose_variant(int64_t M, int64_t N, int64_t K, bool /*interleaved*/, int sm_count) {
  // One 128-row block whose 128x64 tiles, split over two CTAs along K, fill
  // the GPU in one wave: the split-K cluster kernel keeps all of a CTA's
  // bytes in flight (measured 6.8 / 7.3 us against 8.7 / 7.9 us for the best
  // one-CTA tiles at M = 64 / 128, K = 896, N = 4864).
  if (M <= 128 && K >= 128 && 2 * cdiv(N, 64) <= sm_count && 4 * cdiv(N, 64) >= sm_count)
    return SWIGLU_VARIANT_1SM_N64_SK2;
  // Two 128-row blocks of 64-column tiles in one wave (M = 256, N = 4864:
  // 8.4 us against 9.8 us for the CTA-pair tiles).
  if (M <= 256 && cdiv(M, 128) * cdiv(N, 64) <= sm_count) return SWIGLU_VARIANT_1SM_N64;
  // Larger M: one 256x128 tile per CTA pair halves the weight bytes each SM
  // streams per K step (32 KB instead of 48 KB).  This holds for a single
  // wave too (0.5B, M = 512: 9.9 us against 10.1 us for one 128 x 128 tile
  // per SM, measured variant table).
  if (M > 128) return SWIGLU_VARIANT_2SM_N128;
  // Small M (one 128-row block): narrow the tiles until they occupy every SM
  // (the page's Kernel-2 argument: more thread blocks for small batches); a
  // 128-column tile per SM is worth a few idle SMs (7B, M = 128: 148 tiles,
  // 43.6 us against 46.4 us for 296 tiles of 64 columns).
  if (10 * cdiv(N, 128) >= 9 * sm_count) return SWIGLU_VARIANT_1SM_N128;
  if (cdiv(N, 64) >= sm_count) return SWIGLU_VARIANT_1SM_N64;
  return SWIGLU_VARIANT_1SM_N32;
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// The swapped-operand CTA-pair kernel (M <= 128): one pair per 64 output
// columns, A's rows padded to 64 or 128 (half in each CTA of the pair).
int run_bf16_swab(const void *A, const void *B0, const void *B1, void *Y, int64_t M, int64_t N,
                  int64_t K, bool interleaved, DeviceState *st, int dev, cudaStream_t s) {
  if (M > 128) return SWIGLU_ERR_UNSUPPORTED;
  const int rows = M <= 64 ? 64 : 128;
  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int rc = encode_2d(&la.a, BF16, A, K, M, K * 2, 64, rows / 2, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == SWIGLU_OK) {
    if (interleaved) {
      rc = encode_2d(&la.b0, BF16, B0, 2 * N, K, 4 * N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
      la.b1 = la.b0;
    } else {
      rc = encode_2d(&la.b0, BF16, B0, N, K, 2 * N, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
      if (rc == SWIGLU_OK)
        rc = encode_2d(&la.b1, BF16, B1, N, K, 2 * N, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
    }
  }
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, BF16, Y, N, M, 2 * N, 32, rows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  p.num_m_blk = 1;
  p.num_n_blk = int32_t(cdiv(N, 64));
  p.num_k_blk = int32_t(cdiv(K, 64));
  p.group_m = 1;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  p.Y = Y;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  return launch_bf16_swab(interleaved, rows, la) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

int run_bf16(const void *A, const void *B0, const void *B1, void *Y, int64_t M, int64_t N,
             int64_t K, int32_t variant, bool interleaved, void *stream) {
  if (!variant_known(variant)) return SWIGLU_ERR_INVALID_ARG;
  if (variant == SWIGLU_VARIANT_2SM_SWAP && M > 128) return SWIGLU_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || 2 * N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Y) return SWIGLU_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B0 || (!interleaved && !B1))) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y)) return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && (!aligned16(A) || !aligned16(B0) || (!interleaved && !aligned16(B1))))
    return SWIGLU_ERR_MISALIGNED;
  if (N % 8 != 0 || K % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  const uint64_t y_bytes = uint64_t(M) * N * 2, a_bytes = uint64_t(M) * K * 2;
  const uint64_t w_bytes = uint64_t(K) * N * 2 * (interleaved ? 2 : 1);
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, B0, w_bytes) ||
      (!interleaved && overlaps(Y, y_bytes, B1, w_bytes)))
    return SWIGLU_ERR_INVALID_ARG;

  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // every product is zero, and SiLU(0) * 0 = 0
    return cudaMemsetAsync(Y, 0, y_bytes, s) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
  }
  if (variant == SWIGLU_VARIANT_AUTO) variant = choose_variant(M, N, K, interleaved, st->sm_count);
  if (variant == SWIGLU_VARIANT_2SM_SWAP)
    return run_bf16_swab(A, B0, B1, Y, M, N, K, interleaved, st, dev, s);
  const VariantGeom g = variant_geom(variant, interleaved);
  const CUtensorMapSwizzle bsw =
      g.b_swizzle_64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;

  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  rc = encode_2d(&la.a, BF16, A, K, M, K * 2, g.bk, g.box_a, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == SWIGLU_OK) {
    if (interleaved) {
      rc = encode_2d(&la.b0, BF16, B0, 2 * N, K, 4 * N, g.box_b, g.bk, bsw);
      la.b1 = la.b0;
    } else {
      rc = encode_2d(&la.b0, BF16, B0, N, K, 2 * N, g.box_b, g.bk, bsw);
      if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, BF16, B1, N, K, 2 * N, g.box_b, g.bk, bsw);
    }
  }
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, BF16, Y, N, M, 2 * N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != SWIGLU_OK) return rc;

  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  p.num_m_blk = int32_t(cdiv(M, g.bm));
  p.num_n_blk = int32_t(cdiv(N, g.bn));
  p.num_k_blk = int32_t(cdiv(K, g.bk));
  const int gm = g.cluster == 2 ? pair_group_m() : 16;
  p.group_m = p.num_m_blk < gm ? p.num_m_blk : gm;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  p.w_early = g_weights_read_only.load(std::memory_order_relaxed);
  p.Y = Y;
  const int64_t tiles = int64_t(p.num_m_blk) * p.num_n_blk;
  if (tiles > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  la.grid = int(tiles < st->sm_count ? tiles : st->sm_count);  // one-CTA kernels
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  cudaError_t e = variant == SWIGLU_VARIANT_1SM_N64_SK2 ? launch_bf16_sk(interleaved, la)
                  : interleaved ? launch_bf16_interleaved(variant, la)
                                : launch_bf16_separate(variant, la);
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}


// INT4 weights (codes two per byte along N, BF16 scales per column and group
// of G rows along K): the split-K cluster kernel with the decode stage.
int run_w4(const void *A, const void *W1q, const void *S1, const void *W2q, const void *S2,
           void *Y, int64_t M, int64_t N, int64_t K, int64_t G, void *stream) {
  if (M < 0 || N < 0 || K < 0 || G <= 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Y) return SWIGLU_ERR_INVALID_ARG;
  if (G % 64 != 0 || K % G != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (N % 32 != 0 || K % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && (!A || !W1q || !W2q || !S1 || !S2)) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y) || (K > 0 && (!aligned16(A) || !aligned16(W1q) || !aligned16(W2q) ||
                                  !aligned16(S1) || !aligned16(S2))))
    return SWIGLU_ERR_MISALIGNED;
  const uint64_t y_bytes = uint64_t(M) * N * 2, a_bytes = uint64_t(M) * K * 2;
  const uint64_t q_bytes = uint64_t(K) * N / 2, s_bytes = uint64_t(K / G) * N * 2;
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, W1q, q_bytes) ||
      overlaps(Y, y_bytes, W2q, q_bytes) || overlaps(Y, y_bytes, S1, s_bytes) ||
      overlaps(Y, y_bytes, S2, s_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cudaMemsetAsync(Y, 0, y_bytes, s) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;

  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  // Few rows and few output columns: 64-column tiles split along K over CTA
  // pairs; otherwise 128-column tiles, one CTA each over all of K (A read once
  // for twice the weights), with one or two 128-row blocks per CTA.
  const int kern = weight_kernel(M, N, st->sm_count);
  const bool wide = kern != 0;
  const uint32_t cols = wide ? 128 : 64;
  rc = encode_2d(&la.a, BF16, A, K, M, K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.b0, U8, W1q, N / 2, K, N / 2, cols / 2, 64, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, U8, W2q, N / 2, K, N / 2, cols / 2, 64, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.s1, BF16, S1, N, K / G, N * 2, cols, 1, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.s2, BF16, S2, N, K / G, N * 2, cols, 1, NOSW);
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, BF16, Y, N, M, 2 * N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  const int m_blocks = kern == 2 ? 2 : 1;
  p.num_m_blk = int32_t(cdiv(M, 128 * m_blocks));
  p.num_n_blk = int32_t(cdiv(N, cols));
  p.num_k_blk = int32_t(cdiv(K, 64));
  p.group_m = p.num_m_blk < 8 ? p.num_m_blk : 8;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  p.w_early = wide ? 0 : g_weights_read_only.load(std::memory_order_relaxed);
  p.Y = Y;
  p.w4_group = int32_t(G);
  if (int64_t(p.num_m_blk) * p.num_n_blk > kMaxDim / 2) return SWIGLU_ERR_UNSUPPORTED;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  const cudaError_t e = wide ? launch_dq_kernel(1, m_blocks, la) : launch_w4_sk(la);
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

// Weights in a K-major layout, decoded into tensor memory: one CTA per 128
// weight columns, tokens in passes of 64 or 128.  wf 1, INT4: codes [N, K/2]
// (swiglu_pack_w4_kmajor), BF16 scales [K/G, N], G a multiple of 64.  wf 2,
// MXFP8: E4M3 codes [N, K], E8M0 scales [K/32, N].  wf 3, NVFP4: E2M1 codes
// [N, K/2] (swiglu_pack_w4_kmajor), E4M3 scales [K/16, N], per-tensor scales
// g1, g2.  G is read for INT4 only.
int run_kmajor(int wf, const void *A, const void *W1k, const void *S1, const float *g1,
               const void *W2k, const void *S2, const float *g2, void *Y, int64_t M, int64_t N,
               int64_t K, int64_t G, void *stream) {
  const bool nvfp4 = wf == 3, mxfp8 = wf == 2;
  if (M < 0 || N < 0 || K < 0 || G <= 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Y) return SWIGLU_ERR_INVALID_ARG;
  if (wf == 1 ? (G % 64 != 0 || K % G != 0) : K % 64 != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (N % 32 != 0 || K % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && (!A || !W1k || !W2k || !S1 || !S2 || (nvfp4 && (!g1 || !g2))))
    return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y) || (K > 0 && (!aligned16(A) || !aligned16(W1k) || !aligned16(W2k) ||
                                  !aligned16(S1) || !aligned16(S2))))
    return SWIGLU_ERR_MISALIGNED;
  if (nvfp4 && K > 0 &&
      ((reinterpret_cast<uintptr_t>(g1) & 3u) || (reinterpret_cast<uintptr_t>(g2) & 3u)))
    return SWIGLU_ERR_MISALIGNED;
  const uint64_t y_bytes = uint64_t(M) * N * 2, a_bytes = uint64_t(M) * K * 2;
  const uint64_t q_bytes = mxfp8 ? uint64_t(K) * N : uint64_t(K) * N / 2;
  const uint64_t s_bytes = nvfp4 ? uint64_t(K / 16) * N
                           : mxfp8 ? uint64_t(K / 32) * N : uint64_t(K / G) * N * 2;
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, W1k, q_bytes) ||
      overlaps(Y, y_bytes, W2k, q_bytes) || overlaps(Y, y_bytes, S1, s_bytes) ||
      overlaps(Y, y_bytes, S2, s_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cudaMemsetAsync(Y, 0, y_bytes, s) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;

  const int tok = M <= 64 ? 64 : 128;
  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  rc = encode_2d(&la.a, BF16, A, K, M, K * 2, 64, uint32_t(tok), CU_TENSOR_MAP_SWIZZLE_128B);
  if (mxfp8) {   // a column's 64 codes per K step, 64-byte swizzle (the kernel undoes it)
    const auto SW64 = CU_TENSOR_MAP_SWIZZLE_64B;
    if (rc == SWIGLU_OK) rc = encode_2d(&la.b0, U8, W1k, K, N, K, 64, 128, SW64);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, U8, W2k, K, N, K, 64, 128, SW64);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s1, U8, S1, N, K / 32, N, 128, 2, NOSW);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s2, U8, S2, N, K / 32, N, 128, 2, NOSW);
  } else {
    if (rc == SWIGLU_OK) rc = encode_2d(&la.b0, U8, W1k, K / 2, N, K / 2, 32, 128, NOSW);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, U8, W2k, K / 2, N, K / 2, 32, 128, NOSW);
  }
  if (nvfp4) {
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s1, U8, S1, N, K / 16, N, 128, 4, NOSW);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s2, U8, S2, N, K / 16, N, 128, 4, NOSW);
  } else if (!mxfp8) {
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s1, BF16, S1, N, K / G, N * 2, 128, 1, NOSW);
    if (rc == SWIGLU_OK) rc = encode_2d(&la.s2, BF16, S2, N, K / G, N * 2, 128, 1, NOSW);
  }
  if (rc == SWIGLU_OK) rc = encode_2d(&la.y, BF16, Y, N, M, 2 * N, 32, uint32_t(tok / 4), NOSW);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  p.num_m_blk = int32_t(cdiv(M, tok));
  p.num_n_blk = int32_t(cdiv(N, 128));
  p.num_k_blk = int32_t(cdiv(K, 64));
  p.group_m = 1;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  p.Y = Y;
  p.w4_group = int32_t(G);
  p.sW1 = g1;
  p.sW2 = g2;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  return launch_dqt(tok, wf, la) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

// MXFP8 (nvfp4 = false) or NVFP4 (true) weights: the split-K cluster kernel
// with the matching decode stage.  g1, g2: NVFP4 per-tensor scales.
int run_mx(bool nvfp4, const void *A, const void *C1, const void *S1, const float *g1,
           const void *C2, const void *S2, const float *g2, void *Y, int64_t M, int64_t N,
           int64_t K, void *stream) {
  if (M < 0 || N < 0 || K < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Y) return SWIGLU_ERR_INVALID_ARG;
  if (K % 64 != 0) return SWIGLU_ERR_UNSUPPORTED;
  if (N % 32 != 0) return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && (!A || !C1 || !C2 || !S1 || !S2 || (nvfp4 && (!g1 || !g2))))
    return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y) || (K > 0 && (!aligned16(A) || !aligned16(C1) || !aligned16(C2) ||
                                  !aligned16(S1) || !aligned16(S2))))
    return SWIGLU_ERR_MISALIGNED;
  if (nvfp4 && K > 0 &&
      ((reinterpret_cast<uintptr_t>(g1) & 3u) || (reinterpret_cast<uintptr_t>(g2) & 3u)))
    return SWIGLU_ERR_MISALIGNED;
  const int64_t code_pitch = nvfp4 ? N / 2 : N;
  const int64_t blk = nvfp4 ? 16 : 32;
  const uint64_t y_bytes = uint64_t(M) * N * 2, a_bytes = uint64_t(M) * K * 2;
  const uint64_t c_bytes = uint64_t(K) * code_pitch, s_bytes = uint64_t(K / blk) * N;
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, C1, c_bytes) ||
      overlaps(Y, y_bytes, C2, c_bytes) || overlaps(Y, y_bytes, S1, s_bytes) ||
      overlaps(Y, y_bytes, S2, s_bytes))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cudaMemsetAsync(Y, 0, y_bytes, s) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;

  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto NOSW = CU_TENSOR_MAP_SWIZZLE_NONE;
  const int kern = weight_kernel(M, N, st->sm_count);  // as for INT4
  const bool wide = kern != 0;
  const uint32_t cols = wide ? 128 : 64;
  const uint32_t cbox = nvfp4 ? cols / 2 : cols, srows = nvfp4 ? 4 : 2;
  rc = encode_2d(&la.a, BF16, A, K, M, K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.b0, U8, C1, code_pitch, K, code_pitch, cbox, 64, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, U8, C2, code_pitch, K, code_pitch, cbox, 64, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.s1, U8, S1, N, K / blk, N, cols, srows, NOSW);
  if (rc == SWIGLU_OK) rc = encode_2d(&la.s2, U8, S2, N, K / blk, N, cols, srows, NOSW);
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, BF16, Y, N, M, 2 * N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  const int m_blocks = kern == 2 ? 2 : 1;
  p.num_m_blk = int32_t(cdiv(M, 128 * m_blocks));
  p.num_n_blk = int32_t(cdiv(N, cols));
  p.num_k_blk = int32_t(cdiv(K, 64));
  p.group_m = p.num_m_blk < 8 ? p.num_m_blk : 8;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  p.w_early = wide ? 0 : g_weights_read_only.load(std::memory_order_relaxed);
  p.Y = Y;
  p.sW1 = g1;
  p.sW2 = g2;
  if (int64_t(p.num_m_blk) * p.num_n_blk > kMaxDim / 2) return SWIGLU_ERR_UNSUPPORTED;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  const cudaError_t e = wide ? launch_dq_kernel(nvfp4 ? 3 : 2, m_blocks, la) : launch_mx_sk(nvfp4, la);
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

// FP8 E4M3 path: CTA-pair kernel, K-major weights, per-tensor scales.
int run_fp8(const void *A, const void *B0, const void *B1, const float *sA, const float *sW1,
            const float *sW2, void *Y, int64_t M, int64_t N, int64_t K, bool interleaved,
            void *stream) {
  if (M < 0 || N < 0 || K < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || 2 * N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Y) return SWIGLU_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B0 || (!interleaved && !B1) || !sA || !sW1 || !sW2))
    return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Y)) return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && (!aligned16(A) || !aligned16(B0) || (!interleaved && !aligned16(B1))))
    return SWIGLU_ERR_MISALIGNED;
  if (K > 0 && ((reinterpret_cast<uintptr_t>(sA) | reinterpret_cast<uintptr_t>(sW1) |
                 reinterpret_cast<uintptr_t>(sW2)) & 3u))
    return SWIGLU_ERR_MISALIGNED;
  if (N % 8 != 0 || K % 16 != 0) return SWIGLU_ERR_MISALIGNED;
  const uint64_t y_bytes = uint64_t(M) * N * 2, a_bytes = uint64_t(M) * K;
  const uint64_t w_bytes = uint64_t(K) * N * (interleaved ? 2 : 1);
  if (overlaps(Y, y_bytes, A, a_bytes) || overlaps(Y, y_bytes, B0, w_bytes) ||
      (!interleaved && overlaps(Y, y_bytes, B1, w_bytes)))
    return SWIGLU_ERR_INVALID_ARG;

  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return cudaMemsetAsync(Y, 0, y_bytes, s) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;

  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  rc = encode_2d(&la.a, U8, A, K, M, K, 128, 128, SW);
  if (rc == SWIGLU_OK) {
    if (interleaved) {
      rc = encode_2d(&la.b0, U8, B0, K, 2 * N, K, 128, 128, SW);
      la.b1 = la.b0;
    } else {
      rc = encode_2d(&la.b0, U8, B0, K, N, K, 128, 128, SW);
      if (rc == SWIGLU_OK) rc = encode_2d(&la.b1, U8, B1, K, N, K, 128, 128, SW);
    }
  }
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, N, M, 2 * N, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  p.num_m_blk = int32_t(cdiv(M, 256));
  p.num_n_blk = int32_t(cdiv(N, 128));
  p.num_k_blk = int32_t(cdiv(K, 128));
  p.group_m = p.num_m_blk < pair_group_m() ? p.num_m_blk : pair_group_m();
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.sA = sA;
  p.sW1 = sW1;
  p.sW2 = sW2;
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blk;
  if (int64_t(p.num_m_blk) * p.num_n_blk > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  return launch_fp8(interleaved, la) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}


// ---- the down projection: Z = X W (+ R) ----------------------------------------

struct LinearPlan {
  int sk_cs;       // > 0: the split-K cluster kernel with this many CTAs per tile
  int sk_bn;       //      and output tiles of 128 x sk_bn
  int lin_n;       // output columns per CTA-pair tile (256 or 128)
  int k_splits;    // K slices (1 = no split)
  int kb_per;      // 64-deep K steps per slice
  uint64_t ws_bytes;
};

// Cluster size (return value, 0 = not used) and tile width (*bn) of the
// split-K cluster down projection for this shape.  Its 128 x bn tiles, each
// spread over a cluster whose CTAs take one K slice each, must fit one wave.
// In order of preference: 64-column tiles over 8 or 4 CTAs (short K slices,
// many SMs), then 128-column tiles over 4 or 2 (X read by half as many
// tiles), then 64-column tiles over 2.  Clusters of 2 are used only for
// short K (at most 96 steps of 64): with long K the CTA-pair kernel with a
// workspace reduction measured faster (7B, M = 128: 36.8 us against 44.6).
int linear_sk_cluster(int64_t M, int64_t N, int64_t K, int sm_count, int *bn) {
  const int forced = g_linear_sk.load(std::memory_order_relaxed);
  const int forced_n = g_linear_skn.load(std::memory_order_relaxed);
  if (forced == 0) return 0;
  const int64_t nk = cdiv(K, 64);
  static const int kOrder[5][2] = {{8, 64}, {4, 64}, {4, 128}, {2, 128}, {2, 64}};
  for (const auto &o : kOrder) {
    const int cs = o[0], w = o[1];
    if (forced > 0 && cs != forced) continue;
    if (forced_n > 0 && w != forced_n) continue;
    const int64_t tiles = cdiv(M, 128) * cdiv(N, w);
    if (tiles * cs > sm_count || nk < cs) continue;
    if (cs == 2 && forced <= 0 && nk > 96) continue;
    *bn = w;
    return cs;
  }
  return 0;
}

LinearPlan plan_linear(int64_t M, int64_t N, int64_t K, int sm_count) {
  LinearPlan pl;
  pl.sk_bn = 64;
  pl.sk_cs = linear_sk_cluster(M, N, K, sm_count, &pl.sk_bn);
  if (pl.sk_cs > 0) {   // no workspace: the partial sums are reduced in the cluster
    pl.lin_n = pl.sk_bn;
    pl.k_splits = pl.sk_cs;
    pl.kb_per = int(cdiv(cdiv(K, 64), pl.sk_cs));
    pl.ws_bytes = 0;
    return pl;
  }
  const int forced = g_linear_n.load(std::memory_order_relaxed);
  // 256-column tiles (the pair's weight halves of 128 columns, 32 KB per CTA
  // per K step) keep the tensor pipe fed; measured faster than 128 even when
  // the last tile is half empty (N = 896: 50 us vs 70 us at M = 8192).
  // Very few output tiles (small M and N): 128-column tiles give more of them
  // before K is split (0.5B, M = 128: 14.0 us vs 16.7 us).
  if (!forced) pl.lin_n = (N <= 128 || cdiv(M, 256) * cdiv(N, 256) < 8) ? 128 : 256;
  else pl.lin_n = forced;
  const int64_t nk = cdiv(K, 64);
  const int64_t tiles = cdiv(M, 256) * cdiv(N, pl.lin_n);
  const int64_t pairs = sm_count / 2;
  int64_t ks = 1;
  // Few output tiles (small M): split K so that every CTA pair has work; each
  // slice keeps at least four K steps.
  if (tiles * 2 <= pairs) ks = std::min<int64_t>({pairs / tiles, nk / 4, 16});
  if (ks < 2) ks = 1;
  pl.kb_per = int(cdiv(nk, ks));
  pl.k_splits = int(cdiv(nk, pl.kb_per));
  pl.ws_bytes = pl.k_splits > 1 ? uint64_t(pl.k_splits) * M * N * 4 : 0;
  return pl;
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;  // GB300's SM count, for host-only planning without a device
  }
  return sms;
}

int run_linear(const void *X, const void *W, const void *R, void *Z, int64_t M, int64_t N,
               int64_t K, void *ws, uint64_t ws_bytes, void *stream) {
  if (M < 0 || N < 0 || K < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SWIGLU_OK;
  if (!Z || (K > 0 && (!X || !W))) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(Z) || (R && !aligned16(R)) || (K > 0 && (!aligned16(X) || !aligned16(W))))
    return SWIGLU_ERR_MISALIGNED;
  if (N % 8 != 0 || K % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  const uint64_t z_bytes = uint64_t(M) * N * 2;
  if (overlaps(Z, z_bytes, X, uint64_t(M) * K * 2) || overlaps(Z, z_bytes, W, uint64_t(K) * N * 2))
    return SWIGLU_ERR_INVALID_ARG;
  if (R && R != Z && overlaps(Z, z_bytes, R, z_bytes)) return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // Z = R (or zeros)
    cudaError_t e = R ? (R == Z ? cudaSuccess
                                : cudaMemcpyAsync(Z, R, z_bytes, cudaMemcpyDeviceToDevice, s))
                      : cudaMemsetAsync(Z, 0, z_bytes, s);
    return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
  }
  LinearPlan pl = plan_linear(M, N, K, st->sm_count);
  if (pl.sk_cs > 0) {
    LaunchArgs la;
    std::memset(&la, 0, sizeof la);
    const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    rc = encode_2d(&la.a, BF16, X, K, M, K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == SWIGLU_OK)
      rc = encode_2d(&la.b0, BF16, W, N, K, 2 * N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != SWIGLU_OK) return rc;
    KParams &p = la.p;
    p.M = int32_t(M);
    p.N = int32_t(N);
    p.K = int32_t(K);
    p.num_m_blk = int32_t(cdiv(M, 128));
    p.num_n_blk = int32_t(cdiv(N, pl.sk_bn));
    p.num_k_blk = int32_t(cdiv(K, 64));
    p.group_m = p.num_m_blk;
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    p.err = st->err;
    p.R = R;
    p.Y = Z;
    p.k_splits = pl.sk_cs;
    p.kb_per_split = pl.kb_per;
    p.w_early = g_weights_read_only.load(std::memory_order_relaxed);
    la.device = dev;
    la.ctx_gen = st->gen;
    la.stream = s;
    return launch_linear_sk(pl.sk_cs, pl.sk_bn, la) == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
  }
  if (pl.k_splits > 1 &&
      (ws == nullptr || ws_bytes < pl.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 15u) ||
       overlaps(ws, pl.ws_bytes, Z, z_bytes) || overlaps(ws, pl.ws_bytes, X, uint64_t(M) * K * 2))) {
    pl.k_splits = 1;  // no usable workspace: one K slice (correct, fewer busy SMs)
    pl.kb_per = int(cdiv(K, 64));
  }
  LaunchArgs la;
  std::memset(&la, 0, sizeof la);
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  rc = encode_2d(&la.a, BF16, X, K, M, K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.b0, BF16, W, N, K, 2 * N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  la.b1 = la.b0;
  if (rc == SWIGLU_OK)
    rc = encode_2d(&la.y, BF16, Z, N, M, 2 * N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc != SWIGLU_OK) return rc;
  KParams &p = la.p;
  p.M = int32_t(M);
  p.N = int32_t(N);
  p.K = int32_t(K);
  p.num_m_blk = int32_t(cdiv(M, 256));
  p.num_n_blk = int32_t(cdiv(N, pl.lin_n));
  p.num_k_blk = int32_t(cdiv(K, 64));
  p.group_m = p.num_m_blk < pair_group_m() ? p.num_m_blk : pair_group_m();
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.err = st->err;
  p.R = R;
  p.ws = pl.k_splits > 1 ? static_cast<float *>(ws) : nullptr;
  p.k_splits = pl.k_splits;
  p.kb_per_split = pl.kb_per;
  if (int64_t(p.num_m_blk) * p.num_n_blk * p.k_splits > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  la.device = dev;
  la.ctx_gen = st->gen;
  la.stream = s;
  if (launch_linear(pl.lin_n, la) != cudaSuccess) return SWIGLU_ERR_CUDA;
  if (pl.k_splits > 1 &&
      launch_splitk_reduce(p.ws, pl.k_splits, R, Z, M, N, st->sm_count, s) != cudaSuccess)
    return SWIGLU_ERR_CUDA;
  return SWIGLU_OK;
}

uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255u); }

}  // namespace

namespace swiglu {

VariantGeom variant_geom(int variant, bool interleaved) {
  // separate N32: two 32-column boxes (W1, W2); interleaved N32: one 64-column W_fused box
  switch (variant) {
    case SWIGLU_VARIANT_1SM_N64: return {128, 64, 64, 64, 0, 128, 1};
    case SWIGLU_VARIANT_1SM_N32:
      return interleaved ? VariantGeom{128, 32, 64, 64, 0, 128, 1}
                         : VariantGeom{128, 32, 64, 32, 1, 128, 1};
    case SWIGLU_VARIANT_2SM_N128: return {256, 128, 64, 64, 0, 128, 2};
    case SWIGLU_VARIANT_1SM_N64_SK2: return {128, 64, 64, 64, 0, 128, 2};
    case SWIGLU_VARIANT_1SM_N128:
    default: return {128, 128, 64, 64, 0, 128, 1};
  }
}

// This device's error word, SM count, wait limit and context generation, for
// kernels launched from other translation units (per-device set-up on first
// use, redone when the device's context changes).
int device_info(uint32_t **err, int *sm_count, uint64_t *timeout_ns, uint64_t *ctx_gen) {
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  *err = st->err;
  *sm_count = st->sm_count;
  *timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  *ctx_gen = st->gen;
  return SWIGLU_OK;
}

bool pair_dynamic_schedule() { return g_pair_dyn.load(std::memory_order_relaxed) != 0; }

}  // namespace swiglu

extern "C" {

int swiglu_fused(const void *A, const void *W1, const void *W2, void *Y, int64_t M, int64_t N,
                 int64_t K, void *stream) {
  return run_bf16(A, W1, W2, Y, M, N, K, SWIGLU_VARIANT_AUTO, false, stream);
}

int swiglu_fused_ex(const void *A, const void *W1, const void *W2, void *Y, int64_t M, int64_t N,
                    int64_t K, int32_t variant, void *stream) {
  return run_bf16(A, W1, W2, Y, M, N, K, variant, false, stream);
}

int swiglu_fused_interleaved(const void *A, const void *Wfused, void *Y, int64_t M, int64_t N,
                             int64_t K, void *stream) {
  return run_bf16(A, Wfused, nullptr, Y, M, N, K, SWIGLU_VARIANT_AUTO, true, stream);
}

int swiglu_fused_interleaved_ex(const void *A, const void *Wfused, void *Y, int64_t M, int64_t N,
                                int64_t K, int32_t variant, void *stream) {
  return run_bf16(A, Wfused, nullptr, Y, M, N, K, variant, true, stream);
}

int swiglu_pack_interleaved(const void *W1, const void *W2, void *Wfused, int64_t K, int64_t N,
                            void *stream) {
  if (K < 0 || N < 0) return SWIGLU_ERR_INVALID_ARG;
  if (K > kMaxDim || 2 * N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (K == 0 || N == 0) return SWIGLU_OK;
  if (!W1 || !W2 || !Wfused) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wfused)) return SWIGLU_ERR_MISALIGNED;
  if (N % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  const uint64_t w = uint64_t(K) * N * 2;
  if (overlaps(Wfused, 2 * w, W1, w) || overlaps(Wfused, 2 * w, W2, w))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaError_t e = launch_pack_interleaved_u16(W1, W2, Wfused, K * N, st->sm_count,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

int swiglu_fused_fp8(const void *Aq, const void *W1t, const void *W2t, const float *sA,
                     const float *sW1, const float *sW2, void *Y, int64_t M, int64_t N,
                     int64_t K, void *stream) {
  return run_fp8(Aq, W1t, W2t, sA, sW1, sW2, Y, M, N, K, false, stream);
}

int swiglu_fused_interleaved_fp8(const void *Aq, const void *Wfused_t, const float *sA,
                                 const float *sW1, const float *sW2, void *Y, int64_t M,
                                 int64_t N, int64_t K, void *stream) {
  return run_fp8(Aq, Wfused_t, nullptr, sA, sW1, sW2, Y, M, N, K, true, stream);
}

int swiglu_fused_w4(const void *A, const void *W1q, const void *S1, const void *W2q,
                    const void *S2, void *Y, int64_t M, int64_t N, int64_t K, int64_t group,
                    void *stream) {
  return run_w4(A, W1q, S1, W2q, S2, Y, M, N, K, group, stream);
}

int swiglu_pack_w4_kmajor(const void *Wq, void *Wk, int64_t K, int64_t N, void *stream) {
  if (K < 0 || N < 0) return SWIGLU_ERR_INVALID_ARG;
  if (K > kMaxDim || N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (K == 0 || N == 0) return SWIGLU_OK;
  if (!Wq || !Wk) return SWIGLU_ERR_INVALID_ARG;
  if (N % 2 != 0 || K % 8 != 0) return SWIGLU_ERR_MISALIGNED;
  if (!aligned16(Wq) || !aligned16(Wk)) return SWIGLU_ERR_MISALIGNED;
  if (overlaps(Wk, uint64_t(K) * N / 2, Wq, uint64_t(K) * N / 2)) return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  const cudaError_t e =
      launch_pack_w4_kmajor(Wq, Wk, K, N, st->sm_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

int swiglu_fused_w4_kmajor(const void *A, const void *W1k, const void *S1, const void *W2k,
                           const void *S2, void *Y, int64_t M, int64_t N, int64_t K,
                           int64_t group, void *stream) {
  return run_kmajor(1, A, W1k, S1, nullptr, W2k, S2, nullptr, Y, M, N, K, group, stream);
}

int swiglu_fused_mxfp8_kmajor(const void *A, const void *C1k, const void *S1, const void *C2k,
                              const void *S2, void *Y, int64_t M, int64_t N, int64_t K,
                              void *stream) {
  return run_kmajor(2, A, C1k, S1, nullptr, C2k, S2, nullptr, Y, M, N, K, 32, stream);
}

int swiglu_fused_nvfp4_kmajor(const void *A, const void *C1k, const void *S1, const float *g1,
                              const void *C2k, const void *S2, const float *g2, void *Y,
                              int64_t M, int64_t N, int64_t K, void *stream) {
  return run_kmajor(3, A, C1k, S1, g1, C2k, S2, g2, Y, M, N, K, 16, stream);
}

int swiglu_fused_mxfp8(const void *A, const void *C1, const void *S1, const void *C2,
                       const void *S2, void *Y, int64_t M, int64_t N, int64_t K, void *stream) {
  return run_mx(false, A, C1, S1, nullptr, C2, S2, nullptr, Y, M, N, K, stream);
}

int swiglu_fused_nvfp4(const void *A, const void *C1, const void *S1, const float *g1,
                       const void *C2, const void *S2, const float *g2, void *Y, int64_t M,
                       int64_t N, int64_t K, void *stream) {
  return run_mx(true, A, C1, S1, g1, C2, S2, g2, Y, M, N, K, stream);
}

int swiglu_pack_interleaved_fp8(const void *W1t, const void *W2t, void *Wfused_t, int64_t N,
                                int64_t K, void *stream) {
  if (K < 0 || N < 0) return SWIGLU_ERR_INVALID_ARG;
  if (K > kMaxDim || 2 * N > kMaxDim) return SWIGLU_ERR_UNSUPPORTED;
  if (K == 0 || N == 0) return SWIGLU_OK;
  if (!W1t || !W2t || !Wfused_t) return SWIGLU_ERR_INVALID_ARG;
  if (!aligned16(W1t) || !aligned16(W2t) || !aligned16(Wfused_t)) return SWIGLU_ERR_MISALIGNED;
  if (K % 16 != 0) return SWIGLU_ERR_MISALIGNED;
  const uint64_t w = uint64_t(K) * N;
  if (overlaps(Wfused_t, 2 * w, W1t, w) || overlaps(Wfused_t, 2 * w, W2t, w))
    return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaError_t e = launch_pack_rows_interleaved_u8(W1t, W2t, Wfused_t, N, K, st->sm_count,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

uint64_t swiglu_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return plan_linear(M, N, K, device_sm_count()).ws_bytes;
}

int swiglu_linear(const void *X, const void *W, const void *R, void *Z, int64_t M, int64_t N,
                  int64_t K, void *workspace, uint64_t workspace_bytes, void *stream) {
  return run_linear(X, W, R, Z, M, N, K, workspace, workspace_bytes, stream);
}

uint64_t swiglu_mlp_workspace_size(int64_t M, int64_t H, int64_t F) {
  if (M <= 0 || H <= 0 || F <= 0) return 0;
  return align256(uint64_t(M) * F * 2) + swiglu_linear_workspace_size(M, H, F);
}

int swiglu_mlp(const void *A, const void *W1, const void *W2, const void *W3, const void *R,
               void *Z, int64_t M, int64_t H, int64_t F, void *workspace, uint64_t workspace_bytes,
               void *stream) {
  if (M < 0 || H < 0 || F < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M == 0 || H == 0) return SWIGLU_OK;
  if (F == 0) return run_linear(nullptr, nullptr, R, Z, M, H, 0, nullptr, 0, stream);
  const uint64_t y_bytes = align256(uint64_t(M) * F * 2);
  if (!workspace || workspace_bytes < uint64_t(M) * F * 2) return SWIGLU_ERR_INVALID_ARG;
  if (!A || !W3 || !Z) return SWIGLU_ERR_INVALID_ARG;
  if (overlaps(workspace, workspace_bytes, Z, uint64_t(M) * H * 2) ||
      overlaps(workspace, workspace_bytes, A, uint64_t(M) * H * 2) ||
      (R && overlaps(workspace, workspace_bytes, R, uint64_t(M) * H * 2)))
    return SWIGLU_ERR_INVALID_ARG;
  void *Y = workspace;
  int rc = run_bf16(A, W1, W2, Y, M, F, H, SWIGLU_VARIANT_AUTO, false, stream);
  if (rc != SWIGLU_OK) return rc;
  char *rest = static_cast<char *>(workspace) + y_bytes;
  const uint64_t rest_bytes = workspace_bytes > y_bytes ? workspace_bytes - y_bytes : 0;
  return run_linear(Y, W3, R, Z, M, H, F, rest_bytes ? rest : nullptr, rest_bytes, stream);
}

int swiglu_select_variant(int64_t M, int64_t N, int64_t K, int32_t interleaved) {
  if (M < 0 || N < 0 || K < 0) return SWIGLU_VARIANT_AUTO;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 152;  // GB300's SM count, for host-only planning without a device
  }
  return choose_variant(M, N, K, interleaved != 0, sms);
}

int swiglu_select_weight_kernel(int64_t M, int64_t N) {
  if (M < 0 || N < 0) return -1;
  return weight_kernel(M, N, device_sm_count());
}

int swiglu_set_weight_kernel(int32_t kernel) {
  if (kernel < -1 || kernel > 2) return SWIGLU_ERR_INVALID_ARG;
  g_weight_kernel_forced.store(kernel, std::memory_order_relaxed);
  return SWIGLU_OK;
}

int swiglu_set_pair_schedule(int32_t dynamic) {
  if (dynamic != 0 && dynamic != 1) return SWIGLU_ERR_INVALID_ARG;
  g_pair_dyn.store(dynamic, std::memory_order_relaxed);
  return SWIGLU_OK;
}

const char *swiglu_variant_name(int32_t variant) {
  switch (variant) {
    case SWIGLU_VARIANT_AUTO: return "auto";
    case SWIGLU_VARIANT_1SM_N128: return "1sm_n128";
    case SWIGLU_VARIANT_1SM_N64: return "1sm_n64";
    case SWIGLU_VARIANT_2SM_N128: return "2sm_n128";
    case SWIGLU_VARIANT_1SM_N32: return "1sm_n32";
    case SWIGLU_VARIANT_1SM_N64_SK2: return "1sm_n64_sk2";
    case SWIGLU_VARIANT_2SM_SWAP: return "2sm_swap";
    default: return "?";
  }
}

const char *swiglu_status_string(int32_t status) {
  switch (status) {
    case SWIGLU_OK: return "ok";
    case SWIGLU_ERR_INVALID_ARG: return "invalid argument";
    case SWIGLU_ERR_MISALIGNED: return "misaligned pointer or row pitch";
    case SWIGLU_ERR_UNSUPPORTED: return "unsupported device or size";
    case SWIGLU_ERR_CUDA: return "CUDA error";
    case SWIGLU_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int swiglu_device_status(void *stream, uint32_t *detail) {
  if (detail) *detail = 0;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  uint32_t h[2] = {0, 0};
  if (cudaMemcpy(h, st->err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  if (h[0] != 0) {
    const uint32_t z[2] = {0, 0};
    if (cudaMemcpy(st->err, z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
  }
  if (detail) *detail = h[1];
  return h[0] != 0 ? int(h[0]) : SWIGLU_OK;
}

int swiglu_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000000ull) return SWIGLU_ERR_INVALID_ARG;
  g_timeout_ns.store(ns, std::memory_order_relaxed);
  return SWIGLU_OK;
}

int swiglu_set_weights_read_only(int32_t on) {
  if (on != 0 && on != 1) return SWIGLU_ERR_INVALID_ARG;
  g_weights_read_only.store(on, std::memory_order_relaxed);
  return SWIGLU_OK;
}

int swiglu_selftest_wait_timeout(uint32_t timeout_us, void *stream) {
  if (timeout_us < 1 || timeout_us > 1000000u) return SWIGLU_ERR_INVALID_ARG;
  DeviceState *st = nullptr;
  int dev = -1;
  int rc = device_state(&st, &dev);
  if (rc != SWIGLU_OK) return rc;
  cudaError_t e = launch_selftest_wait(uint64_t(timeout_us) * 1000ull, st->err,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SWIGLU_OK : SWIGLU_ERR_CUDA;
}

}  // extern "C"
