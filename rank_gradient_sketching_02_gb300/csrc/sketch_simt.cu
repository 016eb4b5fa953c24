// fp32 CUDA-core sketch: P = X Sigma^T, then S += (dY^T P) / sqrt(r).
// Used for fp32 inputs, where the whole sketch must hold fp32 accuracy.
// (theclarity.today write-up, "Why it matters": S = G A^T with G = dY^T X.)
#include "common.cuh"
#include "kernels.h"

namespace logra {

template <class T> __device__ __forceinline__ float ld_as_f32(const T* p);
template <> __device__ __forceinline__ float ld_as_f32<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_as_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// P[t][b] = sum_j X[t][j] * Sigma[b][j]   (64 tokens x 64 ranks per block,
// 4 x 4 outputs per thread; one sign word per rank row per 64-wide k chunk).
template <class T>
__global__ void __launch_bounds__(256) project_simt_kernel(const T* __restrict__ X, int64_t n, int64_t k,
                                                           int r, uint64_t key, float* __restrict__ P) {
  __shared__ float xs[64][65];
  __shared__ uint64_t ws[64];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t t0 = int64_t(blockIdx.x) * 64;
  const int b0 = blockIdx.y * 64;
  float acc[4][4] = {};
  const int64_t nchunks = (k + 63) / 64;
  for (int64_t c = 0; c < nchunks; ++c) {
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
      const int tt = e >> 6, jj = e & 63;
      const int64_t t = t0 + tt, j = c * 64 + jj;
      xs[tt][jj] = (t < n && j < k) ? ld_as_f32(X + t * k + j) : 0.f;
    }
    if (threadIdx.x < 64) {
      const int b = b0 + threadIdx.x;
      ws[threadIdx.x] = b < r ? sign_word(key, uint32_t(b), uint32_t(c)) : 0ull;
    }
    __syncthreads();
#pragma unroll 8
    for (int jj = 0; jj < 64; ++jj) {
      float xv[4];
      uint32_t sg[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[ty * 4 + i][jj];
#pragma unroll
      for (int q = 0; q < 4; ++q) sg[q] = (uint32_t(ws[tx * 4 + q] >> jj) & 1u) << 31;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] += __uint_as_float(__float_as_uint(xv[i]) ^ sg[q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + ty * 4 + i;
    if (t >= n) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int b = b0 + tx * 4 + q;
      if (b < r) P[t * r + b] = acc[i][q];
    }
  }
}

// S[a][b] += scale * sum_t dY[t][a] * P[t][b]  (64 rows of S x 64 ranks per
// block, 32 tokens per stage).
template <class T>
__global__ void __launch_bounds__(256) accumulate_simt_kernel(const T* __restrict__ dY, const float* __restrict__ P,
                                                              int64_t n, int64_t d, int r, float scale,
                                                              float* __restrict__ S) {
  __shared__ float ds[32][65];
  __shared__ float ps[32][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t a0 = int64_t(blockIdx.x) * 64;
  const int b0 = blockIdx.y * 64;
  float acc[4][4] = {};
  for (int64_t t0 = 0; t0 < n; t0 += 32) {
    for (int e = threadIdx.x; e < 32 * 64; e += 256) {
      const int tt = e >> 6, cc = e & 63;
      const int64_t t = t0 + tt;
      const int64_t a = a0 + cc;
      const int b = b0 + cc;
      ds[tt][cc] = (t < n && a < d) ? ld_as_f32(dY + t * d + a) : 0.f;
      ps[tt][cc] = (t < n && b < r) ? P[t * r + b] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int tt = 0; tt < 32; ++tt) {
      float dv[4], pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) dv[i] = ds[tt][ty * 4 + i];
#pragma unroll
      for (int q = 0; q < 4; ++q) pv[q] = ps[tt][tx * 4 + q];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(dv[i], pv[q], acc[i][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t a = a0 + ty * 4 + i;
    if (a >= d) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int b = b0 + tx * 4 + q;
      // atomic, so that calls into one S may run concurrently on several streams
      if (b < r) atomicAdd(&S[a * r + b], scale * acc[i][q]);
    }
  }
}

template <class T>
static int sketch_simt(const T* X, const T* dY, int64_t n, int64_t d, int64_t k, int r, uint64_t key,
                       float scale, float* S, float* P, cudaStream_t s) {
  dim3 g1(unsigned((n + 63) / 64), unsigned((r + 63) / 64));
  project_simt_kernel<T><<<g1, 256, 0, s>>>(X, n, k, r, key, P);
  LOGRA_LAUNCHED();
  dim3 g2(unsigned((d + 63) / 64), unsigned((r + 63) / 64));
  accumulate_simt_kernel<T><<<g2, 256, 0, s>>>(dY, P, n, d, r, scale, S);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

int launch_sketch_simt(const void* X, const void* dY, int dtype, int64_t n, int64_t d, int64_t k, int r,
                       uint64_t key, float scale, float* S, float* P, cudaStream_t s) {
  if (dtype == LOGRA_F32)
    return sketch_simt(static_cast<const float*>(X), static_cast<const float*>(dY), n, d, k, r, key, scale, S, P, s);
  return sketch_simt(static_cast<const __nv_bfloat16*>(X), static_cast<const __nv_bfloat16*>(dY), n, d, k, r, key,
                     scale, S, P, s);
}

}  // namespace logra
