// Internal launchers of liblogra (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace logra {

struct Control;

struct ApplyWorkspace {
  size_t gram_off, inv_off, ssq_off, dw2_off, img_off, bytes;
};

ApplyWorkspace apply_workspace_layout(int64_t d, int64_t k, int r);

int launch_sign_matrix(uint64_t key, int r, int64_t k, float scale, float* A, cudaStream_t s);
size_t gram_image_bytes(int r);


// fp32 X (n x k) and dY (n x d) -> bf16 planes Xp = [X1; X2; X1; X2] (4n x k) and
// dYp = [dY1; dY1; dY2; dY2] (4n x d), x = x1 + x2 the two-term bf16 split.
int launch_f32_planes(const float* X, const float* dY, int64_t n, int64_t d, int64_t k, void* Xp, void* dYp,
                      cudaStream_t s);

size_t sketch_tc_workspace_bytes(int64_t n, int64_t d, int64_t k, int r, int sms);
struct ZeroTrack;
// zt: what is known about ws being zero (read and updated), or null (nothing)
int launch_sketch_tc(const void* X, const void* dY, int64_t n, int64_t d, int64_t k, int r, uint64_t key,
                     float scale, float* S, void* ws, ZeroTrack* zt, Control* ctl, cudaStream_t s);

// dX = dY W (bf16 in and out) on CTA pairs; max_pairs > 0 caps the grid.
int launch_dgrad_tc(const void* dY, const void* W, void* dX, int64_t n, int64_t d, int64_t k, int max_pairs,
                    Control* ctl, cudaStream_t s);

size_t s_image_bytes(int64_t d, int r);

// Matrices per grouped apply launch.
constexpr int kMaxGroup = 8;

// One matrix of the preparation launch: its S image (A operand of the apply)
// and, when `gram` is set, its Gram image M = Sigma Sigma^T.  counts: r x r
// ints and arrivals: one word per 32 x 32 tile of M, both zero on entry and
// left zero.
struct PrepMatLaunch {
  uint64_t key;
  int64_t d, k;
  int* counts;
  unsigned* arrivals;
  uint8_t* mimg;
  const float* S;
  uint8_t* img;
};
int launch_apply_prep(const PrepMatLaunch* mats, int nm, int r, bool gram, cudaStream_t s);

// The tensor-core kernel behind the apply, over 1..kMaxGroup matrices of one
// rank: mode 0 apply, 1 predict (dW^2 only), 2 rebuild fp32, 3 rebuild bf16,
// 4 row norms (v, 1/sqrt(v+eps), sync sketch, ||S||^2 partials) from the Gram
// image.
struct ApplyMatLaunch {
  float* W;
  __nv_bfloat16* Wb;
  void* out;
  int64_t d, k;
  uint64_t key;
  float neg_lrc;            // -lr c
  float vscale;             // mode 4: the step uses v * vscale (Adam's bias correction), 1 = none
  const uint8_t* s_img;
  const uint8_t* m_img;     // mode 4
  const float* S;           // mode 4
  const float* v_in;        // mode 4
  float* v_out;             // mode 4 (nullable: predict)
  float* inv;               // written by mode 4, read by modes 0 and 1
  float* sync_out;          // mode 4 (nullable)
  double* part;             // per-CTA partials: dW^2 (modes 0, 1) or ||S||^2 (mode 4)
  // modes 0, 1: the last CTA to finish sums the partials into norms[0..1]
  double* norms;            // nullable
  const double* ssq;        // mode 4's ||S||^2 partials
};
struct ApplyLaunch {
  int mode;
  int nm;
  int r;
  float beta2, eps;
  int accumulate;
  int nssq;                 // mode 4's grid (partials per matrix in ssq)
  unsigned* counter;        // per-stream, zero between launches
  ApplyMatLaunch m[kMaxGroup];
};
int launch_apply_tc(const ApplyLaunch& L, int* grid_out, Control* ctl, cudaStream_t s);

// One matrix of launch_rowadam; ws: its own apply_workspace_layout(d, k, r) bytes.
struct RowAdamItem {
  float* W;
  __nv_bfloat16* Wb;
  void* out;
  const float* S;
  const float* v_in;
  float* v_out;
  float* sync_out;
  int64_t d, k;
  uint64_t key;
  float lrc;                // lr c
  float vscale;             // 1 / (1 - beta2^t) for a bias-corrected step, else 1
  double* norms;
  char* ws;
};
// mode 0 apply, 1 predict, 2 reconstruct fp32, 3 reconstruct bf16, over
// 1..kMaxGroup matrices of rank r: three launches (prep, row norms, update)
// for apply and predict, two for reconstruct.
int launch_rowadam(int mode, const RowAdamItem* items, int n, int r, float beta2, float eps, int accumulate,
                   Control* ctl, cudaStream_t s);

}  // namespace logra
