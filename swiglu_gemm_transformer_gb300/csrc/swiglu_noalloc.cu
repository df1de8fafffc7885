// swiglu_noalloc.cu -- the MLP block for callers that cannot allocate device
// memory.
//
// swiglu_mlp() needs device scratch for the intermediate Y (and, for small M,
// the split-K partial sums of the down projection) and asks the caller for
// it.  Some callers cannot provide it: code that runs where no allocator is
// available or allowed, such as a plugin handed only the tensors it reads and
// writes, or a runtime whose device memory is planned before it runs and that
// forbids allocations while it executes.  For them this file keeps one fixed
// scratch area inside the library and offers an entry point that needs
// nothing beyond the inputs and the output.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "swiglu.h"

namespace swiglu {
// The device's error word, SM count, wait limit and context generation
// (swiglu_api.cu); the generation changes when the device's context does.
int device_info(uint32_t **err, int *sm_count, uint64_t *timeout_ns, uint64_t *ctx_gen);
}  // namespace swiglu

namespace {

// The scratch area: part of the library's device code, so every GPU the
// library is used on holds it until the process exits.
constexpr uint64_t kScratchBytes = 32ull << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
uint64_t g_scratch_gen[kMaxDevices] = {0};  // context generation the address belongs to

// Device address of the scratch area on the current device.  In host code the
// array's name only stands in for it, so the address is looked up once per
// device (with that device current) and cached; a new context on the device
// (after cudaDeviceReset) reloads the library's device code, so the lookup
// is redone then.
int scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SWIGLU_ERR_UNSUPPORTED;
  uint32_t *err = nullptr;
  int sms = 0;
  uint64_t timeout_ns = 0, gen = 0;
  int rc = swiglu::device_info(&err, &sms, &timeout_ns, &gen);
  if (rc != SWIGLU_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_gen[dev] != gen) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SWIGLU_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_gen[dev] = gen;
  }
  *out = g_scratch_ptr[dev];
  return SWIGLU_OK;
}

}  // namespace

extern "C" uint64_t swiglu_mlp_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" int swiglu_mlp_noalloc(const void *A, const void *W1, const void *W2, const void *W3,
                                  const void *R, void *Z, int64_t M, int64_t H, int64_t F,
                                  void *stream) {
  if (M < 0 || H < 0 || F < 0) return SWIGLU_ERR_INVALID_ARG;
  if (M == 0 || H == 0) return SWIGLU_OK;
  // Y (M x F BF16) must fit in the scratch area; the down projection uses
  // what is left for split-K partial sums when they fit, and otherwise runs
  // without splitting K.  Nothing in the area needs to start at zero: every
  // byte a call reads was written earlier in the same call.
  const uint64_t y_bytes = uint64_t(M) * uint64_t(F) * 2;
  if (y_bytes > kScratchBytes) return SWIGLU_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != SWIGLU_OK) return rc;
  return swiglu_mlp(A, W1, W2, W3, R, Z, M, H, F, scratch, kScratchBytes, stream);
}
