// RowAdam's per-row statistic and the norms, plus the orchestration of one
// apply (theclarity.today write-up, "What happened": running estimates of
// squared row magnitudes, no first moment):
//   rownorm:  q_i = ||(S A)_i||^2 = S_i M S_i^T / r with M = Sigma Sigma^T
//             (exact integers from popcounts), v_i <- beta2 v_i + (1-beta2) q_i/k,
//             inv_i = 1/sqrt(v_i + eps), optional sync sketch, ||S||^2 partials
//   apply:    the tensor-core reconstruct-and-update kernel (apply_tc.cu)
//   norms:    {||S||^2, ||dW||^2} reduced in fp64 in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace logra {

constexpr int kRowsPerNormBlock = 32;

// One block per 32 rows of S.  Thread t owns ranks b = t, t + 256 (< r).
__global__ void __launch_bounds__(256) rownorm_kernel(const float* __restrict__ S, const float* __restrict__ M,
                                                      const float* __restrict__ v_in, float* __restrict__ v_out,
                                                      float* __restrict__ inv_den, double* __restrict__ ssq_part,
                                                      float* __restrict__ sync_out, int64_t d, int64_t k, int r,
                                                      float beta2, float eps, float lrc) {
  extern __shared__ float smem[];
  float* ss = smem;                                  // [32][r]
  __shared__ float red[8][kRowsPerNormBlock];
  __shared__ float qrow[kRowsPerNormBlock];
  const int64_t i0 = int64_t(blockIdx.x) * kRowsPerNormBlock;
  const int rows = int(d - i0 < kRowsPerNormBlock ? d - i0 : kRowsPerNormBlock);
  for (int e = threadIdx.x; e < kRowsPerNormBlock * r; e += blockDim.x) {
    const int rr = e / r;
    ss[e] = rr < rows ? S[(i0 + rr) * r + (e - rr * r)] : 0.f;
  }
  __syncthreads();
  float part[kRowsPerNormBlock];
#pragma unroll
  for (int q = 0; q < kRowsPerNormBlock; ++q) part[q] = 0.f;
  for (int b = threadIdx.x; b < r; b += 256) {
    float t[kRowsPerNormBlock];
#pragma unroll
    for (int q = 0; q < kRowsPerNormBlock; ++q) t[q] = 0.f;
    for (int a = 0; a < r; ++a) {
      const float m = __ldg(M + int64_t(a) * r + b);
#pragma unroll
      for (int q = 0; q < kRowsPerNormBlock; ++q) t[q] = fmaf(ss[q * r + a], m, t[q]);
    }
#pragma unroll
    for (int q = 0; q < kRowsPerNormBlock; ++q) part[q] = fmaf(t[q], ss[q * r + b], part[q]);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < kRowsPerNormBlock; ++q) {
    float x = part[q];
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp][q] = x;
  }
  __syncthreads();
  if (threadIdx.x < kRowsPerNormBlock) {
    float q = 0.f;
    for (int w = 0; w < 8; ++w) q += red[w][threadIdx.x];
    qrow[threadIdx.x] = q;
  }
  __syncthreads();
  if (threadIdx.x < kRowsPerNormBlock && threadIdx.x < rows) {
    const int64_t i = i0 + threadIdx.x;
    const float mean_sq = qrow[threadIdx.x] / (float(r) * float(k));
    const float vn = beta2 * v_in[i] + (1.f - beta2) * mean_sq;
    if (v_out) v_out[i] = vn;
    inv_den[i] = 1.f / sqrtf(vn + eps);
  }
  __syncthreads();
  if (sync_out) {
    for (int e = threadIdx.x; e < rows * r; e += blockDim.x) {
      const int rr = e / r;
      sync_out[(i0 + rr) * r + (e - rr * r)] = -lrc * ss[e] * inv_den[i0 + rr];
    }
  }
  // ||S||^2 partial of this block, fixed order.
  double acc = 0.0;
  for (int e = threadIdx.x; e < rows * r; e += blockDim.x) acc += double(ss[e]) * double(ss[e]);
  __shared__ double dred[256];
  dred[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o; o >>= 1) {
    if (threadIdx.x < o) dred[threadIdx.x] += dred[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) ssq_part[blockIdx.x] = dred[0];
}

// norms[0] = sum ssq_part, norms[1] = sum dw2_part (fixed order, one block).
__global__ void norms_kernel(const double* __restrict__ ssq, int nssq, const double* __restrict__ dw2, int ndw2,
                             double* __restrict__ norms) {
  __shared__ double red[2][256];
  double a = 0.0, b = 0.0;
  for (int e = threadIdx.x; e < nssq; e += 256) a += ssq[e];
  for (int e = threadIdx.x; e < ndw2; e += 256) b += dw2[e];
  red[0][threadIdx.x] = a;
  red[1][threadIdx.x] = b;
  __syncthreads();
  for (int o = 128; o; o >>= 1) {
    if (threadIdx.x < o) {
      red[0][threadIdx.x] += red[0][threadIdx.x + o];
      red[1][threadIdx.x] += red[1][threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    norms[0] = red[0][0];
    norms[1] = red[1][0];
  }
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

ApplyWorkspace apply_workspace_layout(int64_t d, int64_t k, int r) {
  ApplyWorkspace w{};
  const int64_t nw = (k + 63) / 64;
  const int64_t nnorm = (d + kRowsPerNormBlock - 1) / kRowsPerNormBlock;
  size_t off = 0;
  w.words_off = off;   off += align256(size_t(r) * nw * 8);
  w.gram_off = off;    off += align256(size_t(r) * r * 4);
  w.inv_off = off;     off += align256(size_t(d) * 4);
  w.ssq_off = off;     off += align256(size_t(nnorm) * 8);
  w.dw2_off = off;     off += align256(size_t(1024) * 8);
  w.img_off = off;     off += align256(s_image_bytes(d, r));
  w.n_ssq = int(nnorm);
  w.bytes = off;
  return w;
}

// mode 0 apply, 1 predict (norms only), 2 rebuild fp32, 3 rebuild bf16.
int launch_rowadam(int mode, float* W, __nv_bfloat16* Wb, void* out, int accumulate, const float* S,
                   const float* v_in, float* v_out, float* sync_out, int64_t d, int64_t k, int r, uint64_t key,
                   float beta2, float eps, float lrc, double* norms, char* ws, Control* ctl, cudaStream_t s) {
  const ApplyWorkspace L = apply_workspace_layout(d, k, r);
  float* inv = reinterpret_cast<float*>(ws + L.inv_off);
  double* ssq = reinterpret_cast<double*>(ws + L.ssq_off);
  double* dw2 = reinterpret_cast<double*>(ws + L.dw2_off);
  uint8_t* img = reinterpret_cast<uint8_t*>(ws + L.img_off);
  if (mode == 0 || mode == 1) {
    uint64_t* words = reinterpret_cast<uint64_t*>(ws + L.words_off);
    float* M = reinterpret_cast<float*>(ws + L.gram_off);
    if (int st = launch_gram(key, r, k, words, M, s)) return st;
    const size_t sm = size_t(kRowsPerNormBlock) * r * 4;
    LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(rownorm_kernel), int(sm)));
    rownorm_kernel<<<unsigned(L.n_ssq), 256, sm, s>>>(S, M, v_in, v_out, inv, ssq, sync_out, d, k, r, beta2, eps,
                                                       lrc);
    LOGRA_LAUNCHED();
  }
  if (int st = launch_s_image(S, d, r, img, s)) return st;
  int grid = 0;
  if (int st = launch_apply_tc(mode, W, Wb, out, accumulate, d, k, r, key, -lrc, img, inv, dw2, &grid, ctl, s))
    return st;
  if ((mode == 0 || mode == 1) && norms) {
    norms_kernel<<<1, 256, 0, s>>>(ssq, L.n_ssq, dw2, grid, norms);
    LOGRA_LAUNCHED();
  }
  return LOGRA_OK;
}

}  // namespace logra
