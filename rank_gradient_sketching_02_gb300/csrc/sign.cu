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

// M = Sigma Sigma^T, the B operand of the row-norm GEMM.  Blocks split the
// sign words of each 32 x 32 tile into ranges of at most kGramWords words (many
// small blocks: the pass is latency-bound) and
// add, with exact integer atomics, the number of bit positions where rows a and
// b differ into counts (zeroed by the prep launch).  The last block of a tile
// (a wrapping arrival counter, left at zero) writes its part of the image:
// M[a][b] = k - 2 * count exactly, split into bf16 hi + lo (|M| <= k < 2^15,
// so lo is an integer below 2^7 in magnitude).  Image layout per (256-column
// super-tile st, 64-rank chunk c, term): a 32 KB MN-major tile of 4 groups of
// 64 columns x 64 rows of 128 bytes, 16-byte chunk q of row a stored at
// q ^ (a & 7).  Entries outside r x r are zero.
constexpr int kGramWords = 16;

__global__ void __launch_bounds__(256) gram_kernel(const uint64_t* __restrict__ words, int r, int nw, int64_t k,
                                                   int* __restrict__ counts, unsigned* __restrict__ arrivals,
                                                   uint8_t* __restrict__ img) {
  __shared__ uint64_t wa[32][33];
  __shared__ uint64_t wb[32][33];
  __shared__ unsigned last;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32;
  const bool live = a0 < r && b0 < r;                         // block-uniform
  if (live) {
    const int wbeg = blockIdx.z * kGramWords, wend = min(nw, wbeg + kGramWords);
    int diff[4] = {0, 0, 0, 0};
    for (int w0 = wbeg; w0 < wend; w0 += 32) {
      const int nwr = min(32, wend - w0);
      for (int rr = ty; rr < 32; rr += 8) {
        const int w = w0 + tx;
        uint64_t va = 0, vb = 0;
        if (w < wend) {
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
      for (int w = 0; w < nwr; ++w) {
        const uint64_t x = wb[tx][w];
#pragma unroll
        for (int q = 0; q < 4; ++q) diff[q] += __popcll(wa[ty + 8 * q][w] ^ x);
      }
      __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + ty + 8 * q, b = b0 + tx;
      if (a < r && b < r && diff[q]) atomicAdd(&counts[a * r + b], diff[q]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      last = (atomicInc(&arrivals[blockIdx.y * gridDim.x + blockIdx.x], gridDim.z - 1) == gridDim.z - 1) ? 1u : 0u;
    __syncthreads();
    if (!last) return;
    __threadfence();
  } else if (blockIdx.z != 0) {
    return;                                                   // padding tiles: block z = 0 writes the zeros
  }
  // the tile's image: 32 rows x 4 sixteen-byte chunks x 2 terms, one whole
  // chunk (8 consecutive columns of one row, one term) per thread
  const int nck = (r + 63) / 64;
  const int term = threadIdx.x >> 7, a = a0 + ((threadIdx.x >> 2) & 31), bq = b0 + (threadIdx.x & 3) * 8;
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t two = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int b = bq + 2 * i + h;
      const float m = (a < r && b < r) ? float(k - 2 * int64_t(__ldcg(counts + a * r + b))) : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(m);
      const __nv_bfloat16 v = term ? __float2bfloat16_rn(m - __bfloat162float(hi)) : hi;
      two |= uint32_t(__bfloat16_as_ushort(v)) << (16 * h);
    }
    packed[i] = two;
  }
  const int st = bq >> 8, grp = (bq >> 6) & 3, q = (bq >> 3) & 7;
  const int c = a >> 6, a_l = a & 63;
  uint8_t* tile = img + ((size_t(st) * nck + c) * 2 + term) * 32768;
  *reinterpret_cast<uint4*>(tile + grp * 8192 + a_l * 128 + ((q ^ (a_l & 7)) << 4)) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
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

int launch_gram(const uint64_t* words, int r, int64_t k, int* counts, unsigned* arrivals, uint8_t* img,
                cudaStream_t s) {
  const int nw = int((k + 63) / 64);
  const int nck = (r + 63) / 64, nst = (r + 255) / 256;
  dim3 grid(nst * 8, nck * 2, (nw + kGramWords - 1) / kGramWords);
  gram_kernel<<<grid, 256, 0, s>>>(words, r, nw, k, counts, arrivals, img);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
