// C ABI of liblogra: argument checks, per-(device, stream) workspace, the
// per-device control block, and the launches behind each logra_* entry point.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace logra {

// Control block of each device that loads this library (status word and the
// bounded-wait settings).  Host code reaches it only through the address
// cudaGetSymbolAddress returns for the current device.
static __device__ Control g_control = {0, 0, 2000000000ull};

static thread_local int t_last_cuda_error = 0;
static std::atomic<int> g_concurrency{1};

// A grouped sketch call shapes its launches for the side streams it uses,
// whatever the process-wide hint says; the override lives for the calling
// thread's issue loop only.
static thread_local int t_hint_override = 0;

int concurrency() {
  return t_hint_override > 0 ? t_hint_override : g_concurrency.load(std::memory_order_relaxed);
}
static std::atomic<unsigned long long> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::mutex g_attr_mu;
static std::map<std::pair<int, const void*>, int> g_attr;

cudaError_t ensure_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  int& have = g_attr[std::make_pair(dev, kernel)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = int(e);
  return LOGRA_ERR_CUDA;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
Control* g_ctl_ptr[kMaxDevices] = {};
std::atomic<int> g_sm_count[kMaxDevices] = {};

struct Buffer {
  void* ptr = nullptr;
  size_t bytes = 0;
  unsigned* counters = nullptr;   // kCounterWords zero-initialised words, never freed while the stream's entry lives
  int* gram = nullptr;            // kGramCountInts Gram counts, zero between applies
  ZeroTrack zero;                 // leading bytes of ptr known to be zero
};
std::map<std::pair<int, cudaStream_t>, Buffer> g_ws;

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (*dev < 0 || *dev >= kMaxDevices) return LOGRA_ERR_NO_DEVICE;
  return LOGRA_OK;
}
}  // namespace

Control* control_block(int* status) {
  int dev;
  if ((*status = current_device(&dev))) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ctl_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_control);
    if (e != cudaSuccess) {
      *status = cuda_fail(e);
      return nullptr;
    }
    g_ctl_ptr[dev] = static_cast<Control*>(p);
  }
  return g_ctl_ptr[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (!n) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

void forget_zero_workspaces() {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_ws) e.second.zero.bytes.store(0);
}

void* workspace(cudaStream_t stream, size_t bytes, int* status, ZeroTrack** zt) {
  *status = LOGRA_OK;
  int dev;
  if ((*status = current_device(&dev))) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
  if (ce != cudaSuccess) {
    *status = cuda_fail(ce);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  Buffer& b = g_ws[std::make_pair(dev, stream)];
  if (cap != cudaStreamCaptureStatusNone) b.zero.captured.store(true);
  if (zt) *zt = &b.zero;
  if (b.bytes < bytes) {
    if (b.ptr) {
      // Work already queued on this stream may still read the old buffer.
      cudaError_t e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaFree(b.ptr);
      b.ptr = nullptr;
      b.bytes = 0;
      if (e != cudaSuccess) {
        *status = cuda_fail(e);
        return nullptr;
      }
    }
    size_t want = bytes < (size_t(1) << 20) ? (size_t(1) << 20) : bytes;
    b.zero.bytes.store(0);
    cudaError_t e = cudaMalloc(&b.ptr, want);
    if (e != cudaSuccess) {
      b.ptr = nullptr;
      *status = cuda_fail(e);
      return nullptr;
    }
    b.bytes = want;
  }
  return b.ptr;
}

int* gram_counts(cudaStream_t stream, int* status) {
  *status = LOGRA_OK;
  int dev;
  if ((*status = current_device(&dev))) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  Buffer& b = g_ws[std::make_pair(dev, stream)];
  if (!b.gram) {
    void* p = nullptr;
    const size_t bytes = kGramCountInts * sizeof(int);
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, bytes, stream);   // ordered before its first user
    if (e != cudaSuccess) {
      if (p) cudaFree(p);
      *status = cuda_fail(e);
      return nullptr;
    }
    b.gram = static_cast<int*>(p);
  }
  return b.gram;
}

unsigned* stream_counter(cudaStream_t stream, int* status) {
  *status = LOGRA_OK;
  int dev;
  if ((*status = current_device(&dev))) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  Buffer& b = g_ws[std::make_pair(dev, stream)];
  if (!b.counters) {
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, kCounterWords * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, kCounterWords * sizeof(unsigned), stream);   // ordered before its first user
    if (e != cudaSuccess) {
      if (p) cudaFree(p);
      *status = cuda_fail(e);
      return nullptr;
    }
    b.counters = static_cast<unsigned*>(p);
  }
  return b.counters;
}

int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint32_t elem_bytes, uint64_t inner,
                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swizzle) {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> encode_fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn.load(std::memory_order_acquire);
  if (!encode) {
    std::lock_guard<std::mutex> lk(g_mu);
    encode = encode_fn.load(std::memory_order_relaxed);
    if (!encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) return cuda_fail(e);
      if (q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(cudaErrorNotSupported);
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      encode_fn.store(encode, std::memory_order_release);
    }
  }
  (void)elem_bytes;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LOGRA_OK : LOGRA_ERR_UNSUPPORTED;
}

}  // namespace logra

using namespace logra;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_rank(int r) { return (r >= 32 && r <= 512 && r % 32 == 0) ? LOGRA_OK : LOGRA_ERR_UNSUPPORTED; }

int check_mat(int64_t d, int64_t k) {
  if (d < 1 || k < 1) return LOGRA_ERR_INVALID_ARG;
  if (d % 8 || k % 8) return LOGRA_ERR_UNSUPPORTED;
  if (d > (int64_t(1) << 31) || k > (int64_t(1) << 24)) return LOGRA_ERR_UNSUPPORTED;
  return LOGRA_OK;
}

}  // namespace

extern "C" {

const char* logra_status_string(int status) {
  switch (status) {
    case LOGRA_OK: return "ok";
    case LOGRA_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or unknown dtype)";
    case LOGRA_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case LOGRA_ERR_CUDA: return "CUDA runtime error";
    case LOGRA_ERR_TIMEOUT: return "a device-side wait gave up";
    case LOGRA_ERR_NO_DEVICE: return "no usable CUDA device";
    default: return "unknown status";
  }
}

int logra_last_cuda_error(void) { return t_last_cuda_error; }

int logra_version(void) { return (1 << 16) | 1; }

uint64_t logra_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int logra_sign_matrix(uint64_t seed, uint64_t step, int r, int64_t k, float* A_out, logra_stream_t stream) {
  if (!A_out || k < 1) return LOGRA_ERR_INVALID_ARG;
  if (check_rank(r) || k > (int64_t(1) << 31)) return LOGRA_ERR_UNSUPPORTED;
  return launch_sign_matrix(step_key(seed, step), r, k, inv_sqrt_r(r), A_out, stream);
}

// Largest token count of one sketch call (the fp32 path runs the bf16 kernels on 4n stacked tokens).
constexpr int64_t kMaxSketchTokens = int64_t(1) << 28;

// fp32 sketch workspace: the bf16 sketch's scratch for 4n tokens, then the
// stacked bf16 planes of X (4n x k) and dY (4n x d).
struct F32SketchLayout {
  size_t x_off, y_off, bytes;
};
static F32SketchLayout f32_sketch_layout(int64_t n, int64_t d, int64_t k, int r) {
  F32SketchLayout L;
  L.x_off = (sketch_tc_workspace_bytes(4 * n, d, k, r, sm_count()) + 255) & ~size_t(255);
  L.y_off = L.x_off + ((size_t(8) * size_t(n) * size_t(k) + 255) & ~size_t(255));
  L.bytes = L.y_off + size_t(8) * size_t(n) * size_t(d);
  return L;
}

size_t logra_sketch_workspace_bytes(int64_t n, int64_t d, int64_t k, int r, int in_dtype) {
  if (n <= 0 || r <= 0 || d <= 0 || k <= 0 || n > kMaxSketchTokens) return 0;
  if (in_dtype == LOGRA_BF16) return sketch_tc_workspace_bytes(n, d, k, r, sm_count());
  return f32_sketch_layout(n, d, k, r).bytes;
}

size_t logra_apply_workspace_bytes(int64_t d, int64_t k, int r) {
  if (d <= 0 || k <= 0 || r <= 0) return 0;
  return apply_workspace_layout(d, k, r).bytes;
}

int logra_reserve_workspace(size_t bytes, logra_stream_t stream) {
  int st;
  workspace(stream, bytes, &st);
  return st;
}

// The bf16 sketch of one microbatch on `stream` (arguments already checked).
static int sketch_bf16_on(const void* X, const void* dY, int64_t n, int64_t d, int64_t k, int r, uint64_t seed,
                          uint64_t step, float* S, cudaStream_t stream) {
  int st;
  ZeroTrack* zero = nullptr;
  void* ws = workspace(stream, logra_sketch_workspace_bytes(n, d, k, r, LOGRA_BF16), &st, &zero);
  if (st) return st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  return launch_sketch_tc(X, dY, n, d, k, r, step_key(seed, step), inv_sqrt_r(r), S, ws, zero, ctl, stream);
}

int logra_sketch_accumulate(const void* X, const void* dY, int in_dtype, int64_t n, int64_t d, int64_t k, int r,
                            uint64_t seed, uint64_t step, float* S, logra_stream_t stream) {
  if (!S || n < 0) return LOGRA_ERR_INVALID_ARG;
  if (in_dtype != LOGRA_F32 && in_dtype != LOGRA_BF16) return LOGRA_ERR_INVALID_ARG;
  if (int st = check_mat(d, k)) return st;
  if (check_rank(r)) return LOGRA_ERR_UNSUPPORTED;
  if (n == 0) return LOGRA_OK;
  if (n > kMaxSketchTokens) return LOGRA_ERR_UNSUPPORTED;
  if (!X || !dY) return LOGRA_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(S)) return LOGRA_ERR_UNSUPPORTED;
  int st;
  ZeroTrack* zero = nullptr;
  void* ws = workspace(stream, logra_sketch_workspace_bytes(n, d, k, r, in_dtype), &st, &zero);
  if (st) return st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  if (in_dtype == LOGRA_BF16)
    return launch_sketch_tc(X, dY, n, d, k, r, step_key(seed, step), inv_sqrt_r(r), S, ws, zero, ctl, stream);
  // fp32: the bf16 planes of X and dY stacked along the tokens, then the bf16
  // sketch of the 4n stacked tokens.  The planes lie past that sketch's own
  // scratch, so nothing from their offset on stays known to be zero.
  const F32SketchLayout F = f32_sketch_layout(n, d, k, r);
  char* base = static_cast<char*>(ws);
  if (zero->bytes.load() > F.x_off) zero->bytes.store(F.x_off);
  if (int e = launch_f32_planes(static_cast<const float*>(X), static_cast<const float*>(dY), n, d, k,
                                base + F.x_off, base + F.y_off, stream))
    return e;
  return launch_sketch_tc(base + F.x_off, base + F.y_off, 4 * n, d, k, r, step_key(seed, step), inv_sqrt_r(r), S,
                          ws, zero, ctl, stream);
}

// Side streams of the grouped sketch, per device: created on first use and kept.
namespace {
constexpr int kSideStreams = 16;
struct SideStreams {
  cudaStream_t s[kSideStreams] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kSideStreams] = {};
  bool ready = false;
};
std::mutex g_side_mu;                 // also serialises the fork/issue/join sequence of a device
SideStreams g_side[kMaxDevices];

int side_streams(SideStreams** out) {
  int dev;
  if (int st = current_device(&dev)) return st;
  SideStreams& sd = g_side[dev];
  if (!sd.ready) {
    cudaError_t e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < kSideStreams; ++i) {
      e = cudaStreamCreateWithFlags(&sd.s[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    sd.ready = true;
  }
  *out = &sd;
  return LOGRA_OK;
}
}  // namespace

int logra_sketch_accumulate_group(const logra_sketch_item* items, int count, int64_t n, int r, uint64_t step,
                                  logra_stream_t stream) {
  if (count < 0 || (count > 0 && !items) || n < 0) return LOGRA_ERR_INVALID_ARG;
  if (check_rank(r) || n > kMaxSketchTokens) return LOGRA_ERR_UNSUPPORTED;
  for (int i = 0; i < count; ++i) {
    const logra_sketch_item& it = items[i];
    if (!it.S) return LOGRA_ERR_INVALID_ARG;
    if (int st = check_mat(it.d, it.k)) return st;
    if (n > 0 && (!it.X || !it.dY)) return LOGRA_ERR_INVALID_ARG;
    if (!aligned16(it.X) || !aligned16(it.dY) || !aligned16(it.S)) return LOGRA_ERR_UNSUPPORTED;
  }
  if (count == 0 || n == 0) return LOGRA_OK;
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStreams* sd = nullptr;
  if (int st = side_streams(&sd)) return st;
  const int ns = count < kSideStreams ? count : kSideStreams;
  LOGRA_CUDA_TRY(cudaEventRecord(sd->fork, stream));
  for (int j = 0; j < ns; ++j) LOGRA_CUDA_TRY(cudaStreamWaitEvent(sd->s[j], sd->fork, 0));
  int first_error = LOGRA_OK;
  t_hint_override = ns;
  for (int i = 0; i < count && first_error == LOGRA_OK; ++i) {
    const logra_sketch_item& it = items[i];
    first_error = sketch_bf16_on(it.X, it.dY, n, it.d, it.k, r, it.seed, step, it.S, sd->s[i % ns]);
  }
  t_hint_override = 0;
  // join every side stream back, also after an error, so that the caller's
  // later work stays ordered after whatever was launched
  for (int j = 0; j < ns; ++j) {
    cudaError_t e = cudaEventRecord(sd->join[j], sd->s[j]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, sd->join[j], 0);
    if (e != cudaSuccess && first_error == LOGRA_OK) first_error = cuda_fail(e);
  }
  return first_error;
}

int logra_linear_backward(const void* X, const void* dY, const void* W, void* dX, int64_t n, int64_t d, int64_t k,
                          int r, uint64_t seed, uint64_t step, float* S, logra_stream_t stream) {
  if (n < 0 || (!dX && !S)) return LOGRA_ERR_INVALID_ARG;
  if (int st = check_mat(d, k)) return st;
  if (S && check_rank(r)) return LOGRA_ERR_UNSUPPORTED;
  if (n > int64_t(INT32_MAX) || (S && n > kMaxSketchTokens)) return LOGRA_ERR_UNSUPPORTED;
  if (n == 0) return LOGRA_OK;
  if (!dY || (dX && !W) || (S && !X)) return LOGRA_ERR_INVALID_ARG;
  if (!aligned16(dY) || (dX && (!aligned16(dX) || !aligned16(W))) || (S && (!aligned16(X) || !aligned16(S))))
    return LOGRA_ERR_UNSUPPORTED;
  if (!dX) return sketch_bf16_on(X, dY, n, d, k, r, seed, step, S, stream);
  int st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  if ((st = launch_dgrad_tc(dY, W, dX, n, d, k, 0, ctl, stream))) return st;
  return S ? sketch_bf16_on(X, dY, n, d, k, r, seed, step, S, stream) : LOGRA_OK;
}

// 1 / (1 - beta2^t): the factor of Adam's bias correction for the t-th
// update; 1 for t == 0 (no correction).  0 when t or beta2 is invalid.
static float bias_scale(float beta2, int64_t t) {
  if (t == 0) return 1.0f;
  if (t < 0 || !(beta2 >= 0.0f) || !(beta2 < 1.0f)) return 0.0f;
  const double den = 1.0 - std::pow(double(beta2), double(t));
  if (!(den > 0.0)) return 0.0f;
  const double f = 1.0 / den;
  return f < 3.0e38 ? float(f) : 0.0f;
}

static int rowadam_common(int mode, float* W, const float* S, float* v, int64_t d, int64_t k, int r, uint64_t seed,
                          uint64_t step, float beta2, float eps, float lr, float c, double* norms_out,
                          uint16_t* W_bf16_out, float* sync_out, int64_t t, logra_stream_t stream) {
  if (!S || !v) return LOGRA_ERR_INVALID_ARG;
  const float vscale = bias_scale(beta2, t);
  if (vscale == 0.0f) return LOGRA_ERR_INVALID_ARG;
  if (mode == 0 && !W) return LOGRA_ERR_INVALID_ARG;
  if (int st = check_mat(d, k)) return st;
  if (check_rank(r)) return LOGRA_ERR_UNSUPPORTED;
  if (!aligned16(S) || !aligned16(v) || (W && !aligned16(W)) || (W_bf16_out && !aligned16(W_bf16_out)) ||
      (sync_out && !aligned16(sync_out)) || (norms_out && !aligned16(norms_out)))
    return LOGRA_ERR_UNSUPPORTED;
  int st;
  ZeroTrack* zero = nullptr;
  char* ws = static_cast<char*>(workspace(stream, logra_apply_workspace_bytes(d, k, r), &st, &zero));
  if (st) return st;
  zero->bytes.store(0);           // the apply overwrites the workspace
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  RowAdamItem it{};
  it.W = W;
  it.Wb = reinterpret_cast<__nv_bfloat16*>(W_bf16_out);
  it.S = S;
  it.v_in = v;
  it.v_out = mode == 0 ? v : nullptr;
  it.sync_out = mode == 0 ? sync_out : nullptr;
  it.d = d;
  it.k = k;
  it.key = step_key(seed, step);
  it.lrc = lr * c;
  it.vscale = vscale;
  it.norms = norms_out;
  it.ws = ws;
  return launch_rowadam(mode, &it, 1, r, beta2, eps, 0, ctl, stream);
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of the largest run of up to kMaxGroup consecutive items (the
// items of one launch group lie side by side, each 256-byte aligned).
static size_t group_workspace_bytes(const logra_apply_item* items, int count, int r) {
  size_t best = 0;
  for (int g = 0; g < count; g += kMaxGroup) {
    size_t sum = 0;
    for (int i = g; i < count && i < g + kMaxGroup; ++i)
      sum += align256(apply_workspace_layout(items[i].d, items[i].k, r).bytes);
    if (sum > best) best = sum;
  }
  return best;
}

int logra_rowadam_apply(float* W, const float* S, float* v, int64_t d, int64_t k, int r, uint64_t seed,
                        uint64_t step, float beta2, float eps, float lr, float c, double* norms_out,
                        logra_stream_t stream) {
  return rowadam_common(0, W, S, v, d, k, r, seed, step, beta2, eps, lr, c, norms_out, nullptr, nullptr, 0, stream);
}

int logra_rowadam_apply_ex(float* W, const float* S, float* v, int64_t d, int64_t k, int r, uint64_t seed,
                           uint64_t step, float beta2, float eps, float lr, float c, double* norms_out,
                           uint16_t* W_bf16_out, float* sync_sketch_out, logra_stream_t stream) {
  return rowadam_common(0, W, S, v, d, k, r, seed, step, beta2, eps, lr, c, norms_out, W_bf16_out, sync_sketch_out,
                        0, stream);
}

int logra_rowadam_apply_bc(float* W, const float* S, float* v, int64_t d, int64_t k, int r, uint64_t seed,
                           uint64_t step, float beta2, float eps, float lr, float c, int64_t t, double* norms_out,
                           uint16_t* W_bf16_out, float* sync_sketch_out, logra_stream_t stream) {
  return rowadam_common(0, W, S, v, d, k, r, seed, step, beta2, eps, lr, c, norms_out, W_bf16_out, sync_sketch_out,
                        t, stream);
}

int logra_rowadam_predict(const float* S, const float* v, int64_t d, int64_t k, int r, uint64_t seed,
                          uint64_t step, float beta2, float eps, float lr, double* norms_out,
                          logra_stream_t stream) {
  return logra_rowadam_predict_bc(S, v, d, k, r, seed, step, beta2, eps, lr, 0, norms_out, stream);
}

int logra_rowadam_predict_bc(const float* S, const float* v, int64_t d, int64_t k, int r, uint64_t seed,
                             uint64_t step, float beta2, float eps, float lr, int64_t t, double* norms_out,
                             logra_stream_t stream) {
  if (!norms_out) return LOGRA_ERR_INVALID_ARG;
  return rowadam_common(1, nullptr, S, const_cast<float*>(v), d, k, r, seed, step, beta2, eps, lr, 1.0f, norms_out,
                        nullptr, nullptr, t, stream);
}

int logra_reconstruct(const float* S, int64_t d, int64_t k, int r, uint64_t seed, uint64_t step, void* dW_out,
                      int out_dtype, int accumulate, logra_stream_t stream) {
  if (!S || !dW_out) return LOGRA_ERR_INVALID_ARG;
  if (out_dtype != LOGRA_F32 && out_dtype != LOGRA_BF16) return LOGRA_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return LOGRA_ERR_INVALID_ARG;
  if (int st = check_mat(d, k)) return st;
  if (check_rank(r)) return LOGRA_ERR_UNSUPPORTED;
  if (!aligned16(S) || !aligned16(dW_out)) return LOGRA_ERR_UNSUPPORTED;
  int st;
  ZeroTrack* zero = nullptr;
  char* ws = static_cast<char*>(workspace(stream, logra_apply_workspace_bytes(d, k, r), &st, &zero));
  if (st) return st;
  zero->bytes.store(0);
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  RowAdamItem it{};
  it.out = dW_out;
  it.vscale = 1.0f;
  it.S = S;
  it.d = d;
  it.k = k;
  it.key = step_key(seed, step);
  it.ws = ws;
  return launch_rowadam(out_dtype == LOGRA_F32 ? 2 : 3, &it, 1, r, 0.f, 0.f, accumulate, ctl, stream);
}

size_t logra_apply_group_workspace_bytes(const logra_apply_item* items, int count, int r) {
  if (!items || count <= 0 || check_rank(r)) return 0;
  for (int i = 0; i < count; ++i)
    if (items[i].d <= 0 || items[i].k <= 0) return 0;
  return group_workspace_bytes(items, count, r);
}

int logra_rowadam_apply_group(const logra_apply_item* items, int count, int r, uint64_t step, float beta2, float eps,
                              logra_stream_t stream) {
  if (count < 0 || (count > 0 && !items)) return LOGRA_ERR_INVALID_ARG;
  if (check_rank(r)) return LOGRA_ERR_UNSUPPORTED;
  for (int i = 0; i < count; ++i) {
    const logra_apply_item& m = items[i];
    if (!m.W || !m.S || !m.v) return LOGRA_ERR_INVALID_ARG;
    if (bias_scale(beta2, m.t) == 0.0f) return LOGRA_ERR_INVALID_ARG;
    if (int st = check_mat(m.d, m.k)) return st;
    if (!aligned16(m.W) || !aligned16(m.S) || !aligned16(m.v) || (m.W_bf16_out && !aligned16(m.W_bf16_out)) ||
        (m.sync_sketch_out && !aligned16(m.sync_sketch_out)) || (m.norms_out && !aligned16(m.norms_out)))
      return LOGRA_ERR_UNSUPPORTED;
  }
  if (count == 0) return LOGRA_OK;
  int st;
  ZeroTrack* zero = nullptr;
  char* ws = static_cast<char*>(workspace(stream, group_workspace_bytes(items, count, r), &st, &zero));
  if (st) return st;
  zero->bytes.store(0);
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  for (int g = 0; g < count; g += kMaxGroup) {
    const int n = count - g < kMaxGroup ? count - g : kMaxGroup;
    RowAdamItem it[kMaxGroup] = {};
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
      const logra_apply_item& m = items[g + i];
      it[i].W = m.W;
      it[i].Wb = reinterpret_cast<__nv_bfloat16*>(m.W_bf16_out);
      it[i].S = m.S;
      it[i].v_in = m.v;
      it[i].v_out = m.v;
      it[i].sync_out = m.sync_sketch_out;
      it[i].d = m.d;
      it[i].k = m.k;
      it[i].key = step_key(m.seed, step);
      it[i].lrc = m.lr * m.c;
      it[i].vscale = bias_scale(beta2, m.t);
      it[i].norms = m.norms_out;
      it[i].ws = ws + off;
      off += align256(apply_workspace_layout(m.d, m.k, r).bytes);
    }
    if (int e = launch_rowadam(0, it, n, r, beta2, eps, 0, ctl, stream)) return e;
  }
  return LOGRA_OK;
}

int logra_get_status(logra_stream_t stream) {
  int st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  LOGRA_CUDA_TRY(cudaStreamSynchronize(stream));
  int code = 0;
  LOGRA_CUDA_TRY(cudaMemcpy(&code, &ctl->status, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  LOGRA_CUDA_TRY(cudaMemcpy(&ctl->status, &zero, sizeof(int), cudaMemcpyHostToDevice));
  if (code != 0) forget_zero_workspaces();   // an aborted kernel may have left scratch dirty
  return code;
}

int logra_set_concurrency(int streams) {
  if (streams < 1 || streams > 64) return LOGRA_ERR_INVALID_ARG;
  g_concurrency.store(streams, std::memory_order_relaxed);
  return LOGRA_OK;
}

int logra_debug_inject(int fault, uint64_t timeout_cycles) {
  int st;
  Control* ctl = control_block(&st);
  if (!ctl) return st;
  const int f = fault ? 1 : 0;
  LOGRA_CUDA_TRY(cudaMemcpy(&ctl->inject_fault, &f, sizeof(int), cudaMemcpyHostToDevice));
  if (timeout_cycles) {
    const unsigned long long t = timeout_cycles;
    LOGRA_CUDA_TRY(cudaMemcpy(&ctl->wait_limit, &t, sizeof(t), cudaMemcpyHostToDevice));
  }
  return LOGRA_OK;
}

}  // extern "C"
