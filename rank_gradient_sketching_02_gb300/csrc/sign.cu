// Sign-matrix kernels: explicit A (for tests / callers), packed sign words,
// and the integer Gram matrix Sigma Sigma^T used for RowAdam's row norms.
#include "common.cuh"
#include "kernels.h"

namespace logra {

// A[i][j] = +-scale; one thread per element, so stores are coalesced along j.
// The 64 threads that share a word recompute it (a few integer ops each).
__global__ void sign_matrix_kernel(uint64_t key, int r, int64_t k, float scale, float* __restrict__ A) {
  const int64_t total = int64_t(r) * k;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t i = e / k, j = e - i * k;
    const uint64_t w = sign_word(key, uint32_t(i), uint32_t(j >> 6));
    const uint32_t bit = uint32_t(w >> (j & 63)) & 1u;
    A[e] = __uint_as_float(__float_as_uint(scale) ^ (bit << 31));
  }
}

// words[i][w] = sign word of row i, word w (nw = ceil(k / 64)).
__global__ void sign_words_kernel(uint64_t key, int r, int nw, uint64_t* __restrict__ words) {
  const int total = r * nw;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const int i = e / nw, w = e - i * nw;
    words[e] = sign_word(key, uint32_t(i), uint32_t(w));
  }
}

// M[a][b] = sum_j Sigma[a][j] Sigma[b][j] = k - 2 * popcount over the valid bits
// of (word_a XOR word_b).  Exact integers, stored as float (|M| <= k < 2^24).
// 32 x 32 output tile per block; word columns staged through shared memory.
__global__ void gram_kernel(const uint64_t* __restrict__ words, int r, int nw, int64_t k,
                            float* __restrict__ M) {
  __shared__ uint64_t wa[32][33];
  __shared__ uint64_t wb[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32;
  int diff[4] = {0, 0, 0, 0};
  for (int w0 = 0; w0 < nw; w0 += 32) {
    for (int rr = ty; rr < 32; rr += 8) {
      const int w = w0 + tx;
      uint64_t va = 0, vb = 0;
      if (w < nw) {
        uint64_t valid = ~0ull;
        const int64_t rem = k - int64_t(w) * 64;
        if (rem < 64) valid = (1ull << rem) - 1ull;
        va = words[int64_t(a0 + rr) * nw + w] & valid;
        vb = words[int64_t(b0 + rr) * nw + w] & valid;
      }
      wa[rr][tx] = va;
      wb[rr][tx] = vb;
    }
    __syncthreads();
#pragma unroll 4
    for (int w = 0; w < 32; ++w) {
      const uint64_t x = wb[tx][w];
#pragma unroll
      for (int q = 0; q < 4; ++q) diff[q] += __popcll(wa[ty + 8 * q][w] ^ x);
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    M[int64_t(a0 + ty + 8 * q) * r + (b0 + tx)] = float(k - 2 * int64_t(diff[q]));
}

int launch_sign_matrix(uint64_t key, int r, int64_t k, float scale, float* A, cudaStream_t s) {
  const int64_t total = int64_t(r) * k;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = int64_t(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  sign_matrix_kernel<<<unsigned(blocks), threads, 0, s>>>(key, r, k, scale, A);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

int launch_gram(uint64_t key, int r, int64_t k, uint64_t* words, float* M, cudaStream_t s) {
  const int nw = int((k + 63) / 64);
  const int total = r * nw;
  int blocks = (total + 255) / 256;
  if (blocks > sm_count() * 8) blocks = sm_count() * 8;
  sign_words_kernel<<<blocks, 256, 0, s>>>(key, r, nw, words);
  LOGRA_LAUNCHED();
  dim3 grid(r / 32, r / 32);
  gram_kernel<<<grid, 256, 0, s>>>(words, r, nw, k, M);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
