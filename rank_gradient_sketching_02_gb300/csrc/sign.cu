// Sign-matrix kernel: explicit A (for tests / callers).  The in-kernel sign
// tiles and the Gram pass live with the kernels that use them.
#include <cuda_bf16.h>

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

}  // namespace logra
