// Sign-matrix kernels: explicit A (for tests / callers) and the integer Gram
// matrix Sigma Sigma^T used for RowAdam's row norms.
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

// M = Sigma Sigma^T, the B operand of the row-norm GEMM, straight into its
// image: one block per 32 x 32 tile of the padded image extent counts, over
// all sign words of its 64 rows, the bit positions where rows a and b differ
// (no atomics, so no zeroing pass), then M[a][b] = k - 2 * count exactly and
// the exact split M = hi + lo into two bf16 terms (|M| <= k < 2^15, so lo is
// an integer below 2^7 in magnitude).  Image layout per (256-column
// super-tile st, 64-rank chunk c, term): a 32 KB MN-major tile of 4 groups of
// 64 columns x 64 rows of 128 bytes, 16-byte chunk q of row a stored at
// q ^ (a & 7).  Entries outside r x r are zero.
__global__ void __launch_bounds__(256) gram_kernel(const uint64_t* __restrict__ words, int r, int nw, int64_t k,
                                                   uint8_t* __restrict__ img) {
  __shared__ uint64_t wa[32][33];
  __shared__ uint64_t wb[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32;
  int diff[4] = {0, 0, 0, 0};
  if (a0 < r && b0 < r) {                                     // block-uniform
    for (int w0 = 0; w0 < nw; w0 += 32) {
      for (int rr = ty; rr < 32; rr += 8) {
        const int w = w0 + tx;
        uint64_t va = 0, vb = 0;
        if (w < nw) {
          uint64_t valid = ~0ull;
          const int64_t rem = k - int64_t(w) * 64;
          if (rem < 64) valid = (1ull << rem) - 1ull;
          if (a0 + rr < r) va = words[int64_t(a0 + rr) * nw + w] & valid;
          if (b0 + rr < r) vb = words[int64_t(b0 + rr) * nw + w] & valid;
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
  }
  const int nck = (r + 63) / 64;
  const int b = b0 + tx;
  const int st = b >> 8, grp = (b >> 6) & 3, qq = (b >> 3) & 7;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int a = a0 + ty + 8 * q;
    const float m = (a < r && b < r) ? float(k - 2 * int64_t(diff[q])) : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(m);
    const __nv_bfloat16 lo = __float2bfloat16_rn(m - __bfloat162float(hi));
    const int c = a >> 6, a_l = a & 63;
    const size_t off = size_t(grp) * 8192 + size_t(a_l) * 128 + size_t((qq ^ (a_l & 7)) << 4) + size_t(b & 7) * 2;
    uint8_t* t0 = img + (size_t(st) * nck + c) * 2 * 32768;
    *reinterpret_cast<uint16_t*>(t0 + off) = __bfloat16_as_ushort(hi);
    *reinterpret_cast<uint16_t*>(t0 + 32768 + off) = __bfloat16_as_ushort(lo);
  }
}

size_t gram_image_bytes(int r) { return size_t((r + 255) / 256) * ((r + 63) / 64) * 2 * 32768; }

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

int launch_gram(const uint64_t* words, int r, int64_t k, uint8_t* img, cudaStream_t s) {
  const int nw = int((k + 63) / 64);
  const int nck = (r + 63) / 64, nst = (r + 255) / 256;
  dim3 grid(nst * 8, nck * 2);
  gram_kernel<<<grid, 256, 0, s>>>(words, r, nw, k, img);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
