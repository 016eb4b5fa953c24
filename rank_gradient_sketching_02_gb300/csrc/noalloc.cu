// logra_sketch_accumulate_noalloc: the bf16 sketch with its scratch memory in
// a fixed, statically sized device array instead of the library's workspace.
//
// Some callers cannot call cudaMalloc at all: frameworks whose caching
// allocator owns every byte of device memory and forbids side allocations,
// real-time paths that must not block on the driver, and runtimes whose
// device memory is fixed at start-up.  This entry point serves them: it
// allocates nothing, ever.  Its price is a cap on problem size and one
// scratch array shared by every call on a device (see include/logra.h).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace logra {

// Scratch for the projection partials and the swizzled hi/lo image of
// P^T: 32 MiB, held by every GPU that loads the library until the process
// exits.  In host code `g_noalloc_scratch` is only a host-side stand-in for
// the symbol, never a device address; the device address comes from
// cudaGetSymbolAddress below.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_na_mu;
void* g_na_ptr[kMaxDev] = {};
}  // namespace

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
static int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDev) return LOGRA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_na_ptr[dev] = p;
  }
  *out = g_na_ptr[dev];
  return LOGRA_OK;
}

}  // namespace logra

using namespace logra;

extern "C" size_t logra_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int logra_sketch_accumulate_noalloc(const void* X, const void* dY, int64_t n, int64_t d, int64_t k, int r,
                                               uint64_t seed, uint64_t step, float* S, logra_stream_t stream) {
  if (!S || n < 0) return LOGRA_ERR_INVALID_ARG;
  if (d < 1 || k < 1) return LOGRA_ERR_INVALID_ARG;
  if (d % 8 || k % 8 || d > (int64_t(1) << 31) || k > (int64_t(1) << 24)) return LOGRA_ERR_UNSUPPORTED;
  if (r < 32 || r > 512 || r % 32) return LOGRA_ERR_UNSUPPORTED;
  if (n == 0) return LOGRA_OK;
  if (!X || !dY) return LOGRA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(dY) | reinterpret_cast<uintptr_t>(S)) & 15u)
    return LOGRA_ERR_UNSUPPORTED;
  if (sketch_tc_workspace_bytes(n, d, k, r, sm_count()) > kNoAllocScratchBytes) return LOGRA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (int st = noalloc_scratch(&scratch)) return st;
  int st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  return launch_sketch_tc(X, dY, n, d, k, r, step_key(seed, step), inv_sqrt_r(r), S, scratch, nullptr, ctl, stream);
}
