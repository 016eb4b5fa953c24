// RowAdam applies (or predicts, or reconstructions) of up to eight matrices
// as one short sequence of launches.
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

static_assert(kArrivalBase + kArrivalWords * kMaxGroup <= kCounterWords, "arrival words of a full group");
static_assert(kGramCountInts >= size_t(kMaxGroup) * 512 * 512, "Gram counts of a full group");

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

int launch_rowadam(int mode, const RowAdamItem* items, int n, int r, float beta2, float eps, int accumulate,
                   Control* ctl, cudaStream_t s) {
  if (n < 1 || n > kMaxGroup) return LOGRA_ERR_INVALID_ARG;
  const bool rownorms = (mode == 0 || mode == 1);
  // per-stream zeroed scratch: counters [0] the update pass's finished CTAs,
  // [kArrivalBase + kArrivalWords i, ...) the Gram tiles' arrivals of matrix i;
  // the Gram counts, r x r per matrix
  unsigned* counters = nullptr;
  int* counts = nullptr;
  if (rownorms) {
    int st = 0;
    counters = stream_counter(s, &st);
    if (!st) counts = gram_counts(s, &st);
    if (st) return st;
  }
  PrepMatLaunch pm[kMaxGroup];
  ApplyLaunch L{};
  L.nm = n;
  L.r = r;
  L.beta2 = beta2;
  L.eps = eps;
  for (int i = 0; i < n; ++i) {
    const RowAdamItem& it = items[i];
    const ApplyWorkspace WL = apply_workspace_layout(it.d, it.k, r);
    uint8_t* img = reinterpret_cast<uint8_t*>(it.ws + WL.img_off);
    uint8_t* mimg = reinterpret_cast<uint8_t*>(it.ws + WL.gram_off);
    pm[i].key = it.key;
    pm[i].d = it.d;
    pm[i].k = it.k;
    pm[i].counts = counts ? counts + size_t(i) * r * r : nullptr;
    pm[i].arrivals = counters ? counters + kArrivalBase + kArrivalWords * i : nullptr;
    pm[i].mimg = mimg;
    pm[i].S = it.S;
    pm[i].img = img;
    ApplyMatLaunch& M = L.m[i];
    M.d = it.d;
    M.k = it.k;
    M.key = it.key;
    M.neg_lrc = -it.lrc;
    M.vscale = it.vscale;
    M.s_img = img;
    M.m_img = mimg;
    M.S = it.S;
    M.inv = reinterpret_cast<float*>(it.ws + WL.inv_off);
  }
  if (int st = launch_apply_prep(pm, n, r, rownorms, s)) return st;

  int grid_norm = 0, grid_upd = 0;
  if (rownorms) {
    L.mode = 4;
    for (int i = 0; i < n; ++i) {
      const ApplyWorkspace WL = apply_workspace_layout(items[i].d, items[i].k, r);
      L.m[i].v_in = items[i].v_in;
      L.m[i].v_out = items[i].v_out;
      L.m[i].sync_out = items[i].sync_out;
      L.m[i].part = reinterpret_cast<double*>(items[i].ws + WL.ssq_off);
    }
    if (int st = launch_apply_tc(L, &grid_norm, ctl, s)) return st;
  }
  L.mode = mode;
  L.accumulate = accumulate;
  L.nssq = grid_norm;
  L.counter = counters;
  for (int i = 0; i < n; ++i) {
    const ApplyWorkspace WL = apply_workspace_layout(items[i].d, items[i].k, r);
    ApplyMatLaunch& M = L.m[i];
    M.W = items[i].W;
    M.Wb = items[i].Wb;
    M.out = items[i].out;
    M.v_in = nullptr;
    M.v_out = nullptr;
    M.sync_out = nullptr;
    M.part = reinterpret_cast<double*>(items[i].ws + WL.dw2_off);
    M.norms = items[i].norms;   // null for predict without norms: no last-CTA sum
    M.ssq = reinterpret_cast<const double*>(items[i].ws + WL.ssq_off);
  }
  return launch_apply_tc(L, &grid_upd, ctl, s);
}

}  // namespace logra
