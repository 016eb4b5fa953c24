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

// counts[a][b] += number of valid bit positions where rows a and b of Sigma
// differ, over one range of 32 words; then M[a][b] = sum_j Sigma[a][j] Sigma[b][j]
// = k - 2 counts[a][b] exactly.  32 x 32 output tile per block, word ranges
// over blockIdx.z, integer atomics (exact, so the order does not matter).
__global__ void gram_count_kernel(const uint64_t* __restrict__ words, int r, int nw, int64_t k,
                                  int* __restrict__ counts) {
  __shared__ uint64_t wa[32][33];
  __shared__ uint64_t wb[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32, w0 = blockIdx.z * 32;
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
  int diff[4] = {0, 0, 0, 0};
#pragma unroll 4
  for (int w = 0; w < 32; ++w) {
    const uint64_t x = wb[tx][w];
#pragma unroll
    for (int q = 0; q < 4; ++q) diff[q] += __popcll(wa[ty + 8 * q][w] ^ x);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) atomicAdd(&counts[(a0 + ty + 8 * q) * r + (b0 + tx)], diff[q]);
}

// M as the B operand of the row-norm GEMM: exact split M = hi + lo into two
// bf16 terms (|M| <= k < 2^15, so lo is an integer below 2^7 in magnitude),
// laid out per (256-column super-tile st, 64-rank chunk c, term) as a 32 KB
// MN-major tile: 4 groups of 64 columns x 64 rows of 128 bytes, 16-byte chunk
// q of row a stored at q ^ (a & 7).  Entries outside r x r are zero.
__global__ void gram_image_kernel(const int* __restrict__ counts, int r, int64_t k, uint8_t* __restrict__ img) {
  const int nck = (r + 63) / 64, nst = (r + 255) / 256;
  const int64_t total = int64_t(nst) * nck * 2 * 2048;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int q = int(e & 7);
    const int a_l = int((e >> 3) & 63);
    const int grp = int((e >> 9) & 3);
    const int64_t t = e >> 11;                 // (st, c, term)
    const int term = int(t & 1);
    const int c = int((t >> 1) % nck);
    const int st = int((t >> 1) / nck);
    const int a = c * 64 + a_l;
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t two = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = st * 256 + grp * 64 + q * 8 + 2 * i + h;
        float v = 0.f;
        if (a < r && b < r) {
          const float m = float(k - 2 * int64_t(counts[a * r + b]));
          const float hi = __bfloat162float(__float2bfloat16_rn(m));
          v = term == 0 ? hi : m - hi;
        }
        two |= uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v))) << (16 * h);
      }
      packed[i] = two;
    }
    uint8_t* tile = img + size_t(t) * 32768;
    *reinterpret_cast<uint4*>(tile + grp * 8192 + a_l * 128 + ((q ^ (a_l & 7)) << 4)) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
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

int launch_gram(uint64_t key, int r, int64_t k, uint64_t* words, int* counts, uint8_t* img, cudaStream_t s) {
  const int nw = int((k + 63) / 64);
  const int total = r * nw;
  int blocks = (total + 255) / 256;
  if (blocks > sm_count() * 8) blocks = sm_count() * 8;
  sign_words_kernel<<<blocks, 256, 0, s>>>(key, r, nw, words);
  LOGRA_LAUNCHED();
  LOGRA_CUDA_TRY(cudaMemsetAsync(counts, 0, size_t(r) * r * sizeof(int), s));
  dim3 grid(r / 32, r / 32, (nw + 31) / 32);
  gram_count_kernel<<<grid, 256, 0, s>>>(words, r, nw, k, counts);
  LOGRA_LAUNCHED();
  const int64_t itotal = int64_t(gram_image_bytes(r)) / 16;
  int iblocks = int((itotal + 255) / 256);
  if (iblocks > sm_count() * 4) iblocks = sm_count() * 4;
  gram_image_kernel<<<iblocks, 256, 0, s>>>(counts, r, k, img);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
