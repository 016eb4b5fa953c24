// Shared device helpers of liblogra: the sign hash, status word, launch checks.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/logra.h"

namespace logra {

// ---------------------------------------------------------------------------
// Sign generator.  SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): the key of
// (seed, step) is the generator's output number step+1 for seed `seed`; word w
// of row i of Sigma is the finaliser applied to key ^ (i << 32 | w).  Bit b of
// that word is the sign of Sigma[i][64 w + b] (set -> -1).  A new key per step
// is the per-step redraw of the projection (academy.dair.ai summary, "Gradient
// sketches"); all microbatches of a step share it.
// ---------------------------------------------------------------------------
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t step_key(uint64_t seed, uint64_t step) {
  return mix64(seed + kGolden * (step + 1));
}

__host__ __device__ __forceinline__ uint64_t sign_word(uint64_t key, uint32_t row, uint32_t word) {
  return mix64(key ^ ((uint64_t(row) << 32) | uint64_t(word)));
}

// fl32(1/sqrt(r)), computed in double and rounded once.
inline float inv_sqrt_r(int r) { return float(1.0 / __builtin_sqrt(double(r))); }

// ---------------------------------------------------------------------------
// Per-device control block: status word and the bounded-wait settings.  It is
// a file-scope __device__ object of the API translation unit; kernels receive
// its device address (taken once per device with cudaGetSymbolAddress).
// ---------------------------------------------------------------------------
struct Control {
  int status;                    // first device-side failure since last read
  int inject_fault;              // test hook: drop one producer arrival
  unsigned long long wait_limit; // clock64 ticks a bounded wait may spin
};

__device__ __forceinline__ void record_status(Control* ctl, int code) {
  atomicCAS(&ctl->status, 0, code);
}

Control* control_block(int* status);                     // current device
// What the host knows about the leading bytes of a workspace being zero
// (the sketch's projection reduce-adds into a zeroed P^T at its start).
// `bytes` holds only for eagerly issued work: once any call on the workspace
// has been captured into a CUDA graph, replays may change it behind the
// host's back, so `captured` is set for good and nothing is trusted again.
struct ZeroTrack {
  std::atomic<size_t> bytes{0};
  std::atomic<bool> captured{false};
  // leading bytes that are zero for certain when the next launch runs
  size_t trusted() const { return captured.load() ? 0 : bytes.load(); }
};
// The per-(device, stream) scratch workspace, grown on demand.  zt (optional)
// receives its ZeroTrack: bytes = 0 after every (re)allocation; users that
// overwrite the workspace set it to 0, the sketch keeps it up to date.  A call
// made while `stream` is capturing marks the workspace as captured.
void* workspace(cudaStream_t stream, size_t bytes, int* status, ZeroTrack** zt = nullptr);
// Forget every workspace's known-zero prefix (after a device-side failure).
void forget_zero_workspaces();
// Zero-initialised counters per (device, stream) for in-kernel last-CTA
// detection; every user leaves them at zero.  Word 0: the apply's update
// pass; from kArrivalBase, kArrivalWords per matrix of a grouped apply: the
// Gram tiles' arrivals (at most 16 x 16 tiles of 32 x 32 for r <= 512).
constexpr int kArrivalBase = 64;
// Words 8 and 9: the dX kernel's tile counter and finished-pair counter.
constexpr int kDgradNextWord = 8;
constexpr int kDgradDoneWord = 9;
constexpr int kArrivalWords = 256;
constexpr int kCounterWords = 4096;
// Gram counts per (device, stream): r x r ints (r <= 512) for each of up to
// eight matrices of a grouped apply, zero when allocated and left zero by
// every apply.
constexpr size_t kGramCountInts = size_t(8) * 512 * 512;
int* gram_counts(cudaStream_t stream, int* status);
unsigned* stream_counter(cudaStream_t stream, int* status);
int sm_count();
// Streams on which the caller issues sketch calls at the same time (logra_set_concurrency).
int concurrency();
int cuda_fail(cudaError_t e);
void count_launch();
// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; remembered per (device, kernel) so repeated calls are free.
cudaError_t ensure_smem(const void* kernel, int bytes);

}  // namespace logra

namespace logra {
// Launch with programmatic stream serialization (see grid_dependency_wait in
// tc.cuh): every kernel launched this way waits for its predecessor's
// completion with griddepcontrol.wait before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same for a kernel whose CTAs run in clusters of `cluster_x` along x
// (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                      unsigned cluster_x, Args... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace logra

// After every kernel launch: count it and surface a launch error.
#define LOGRA_LAUNCHED()                                       \
  do {                                                         \
    ::logra::count_launch();                                   \
    cudaError_t _e = cudaGetLastError();                       \
    if (_e != cudaSuccess) return ::logra::cuda_fail(_e);      \
  } while (0)

#define LOGRA_CUDA_TRY(expr)                                   \
  do {                                                         \
    cudaError_t _e = (expr);                                   \
    if (_e != cudaSuccess) return ::logra::cuda_fail(_e);      \
  } while (0)
