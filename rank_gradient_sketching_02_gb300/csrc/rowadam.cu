// One RowAdam apply (or predict, or reconstruct) as a short sequence of
// launches.
//
// apply / predict (theclarity.today write-up, "What happened": running
// estimates of squared row magnitudes, no first moment):
//   1+2. one launch: S split into bf16 hi + lo, pre-swizzled; and M = Sigma
//      Sigma^T from popcounts of sign words hashed in place (word ranges split
//      over blocks, exact integer atomics), stored as an exact bf16 hi + lo
//      image                                                      (apply_tc.cu)
//   3. row norms on the tensor cores: q_i = S_i M S_i^T = r ||(S A)_i||^2,
//      v_i <- beta2 v_i + (1 - beta2) q_i / (r k), 1/sqrt(v_i + eps),
//      optional sync sketch, ||S||^2 partials                     (mode 4)
//   4. W += -lr c (S A) / (sqrt(r) sqrt(v + eps)), tile by tile   (mode 0; 1 = dW^2 only);
//      its last CTA sums the partials into {||S||^2, ||dW||^2} in a fixed order
// reconstruct: steps 1 (S image only) and 4 with a plain (or accumulating) store epilogue.
#include "common.cuh"
#include "kernels.h"

namespace logra {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

ApplyWorkspace apply_workspace_layout(int64_t d, int64_t k, int r) {
  ApplyWorkspace w{};
  size_t off = 0;
  w.gram_off = off;    off += align256(gram_image_bytes(r));
  w.inv_off = off;     off += align256(size_t(d) * 4);
  w.ssq_off = off;     off += align256(size_t(1024) * 8);
  w.dw2_off = off;     off += align256(size_t(1024) * 8);
  w.img_off = off;     off += align256(s_image_bytes(d, r));
  w.bytes = off;
  return w;
}

int launch_rowadam(int mode, float* W, __nv_bfloat16* Wb, void* out, int accumulate, const float* S,
                   const float* v_in, float* v_out, float* sync_out, int64_t d, int64_t k, int r, uint64_t key,
                   float beta2, float eps, float lrc, double* norms, char* ws, Control* ctl, cudaStream_t s) {
  const ApplyWorkspace WL = apply_workspace_layout(d, k, r);
  float* inv = reinterpret_cast<float*>(ws + WL.inv_off);
  double* ssq = reinterpret_cast<double*>(ws + WL.ssq_off);
  double* dw2 = reinterpret_cast<double*>(ws + WL.dw2_off);
  uint8_t* img = reinterpret_cast<uint8_t*>(ws + WL.img_off);
  uint8_t* mimg = reinterpret_cast<uint8_t*>(ws + WL.gram_off);
  const bool rownorms = (mode == 0 || mode == 1);
  // per-stream zeroed scratch: counters [0] the update pass's finished CTAs,
  // [64..) the Gram tiles' arrivals; the Gram counts
  unsigned* counters = nullptr;
  int* counts = nullptr;
  if (rownorms) {
    int st = 0;
    counters = stream_counter(s, &st);
    if (!st) counts = gram_counts(s, &st);
    if (st) return st;
  }
  if (int st = launch_apply_prep(key, r, k, rownorms, counts, counters ? counters + 64 : nullptr, mimg, S, d, img, s))
    return st;

  ApplyLaunch L{};
  L.d = d; L.k = k; L.r = r; L.key = key; L.neg_lrc = -lrc;
  L.s_img = img; L.m_img = mimg; L.S = S; L.inv = inv; L.beta2 = beta2; L.eps = eps;
  int grid_norm = 0, grid_upd = 0;
  if (rownorms) {
    L.mode = 4;
    L.v_in = v_in;
    L.v_out = v_out;
    L.sync_out = sync_out;
    L.part = ssq;
    if (int st = launch_apply_tc(L, &grid_norm, ctl, s)) return st;
  }
  L.mode = mode;
  L.W = W; L.Wb = Wb; L.out = out; L.accumulate = accumulate;
  L.v_in = nullptr; L.v_out = nullptr; L.sync_out = nullptr;
  L.part = dw2;
  L.norms = norms;   // null for predict without norms: no last-CTA sum
  L.ssq = ssq;
  L.nssq = grid_norm;
  L.counter = counters;
  if (int st = launch_apply_tc(L, &grid_upd, ctl, s)) return st;
  return LOGRA_OK;
}

}  // namespace logra
