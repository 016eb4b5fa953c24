// fp32 inputs of the sketch, split into bf16 planes for the tensor-core path.
//
// The sketch is S += dY^T (X A^T) (theclarity.today write-up, "Why it
// matters": S = G A^T with G = dY^T X).  For fp32 X and dY each element is
// split into two bf16 terms, x = x1 + x2 + e with x1 = RN_bf16(x) and
// x2 = RN_bf16(x - x1), where x - x1 is exact in fp32 and |e| <= u^2 |x| =
// 2^-16 |x| for bf16's unit roundoff u = 2^-8 (about 2.5e-6 |x| root-mean-
// square): the two-term splitting of Henry, Tang & Heinecke, "Leveraging the
// bfloat16 Artificial Intelligence Datatype For Higher-Precision
// Computations", ARITH 2019.  Stacking the planes along the token axis,
//
//   X' = [X1; X2; X1; X2],   dY' = [dY1; dY1; dY2; dY2]   (4n rows each),
//
// makes the bf16 sketch of the 4n stacked tokens equal to
// (dY1 + dY2)^T ((X1 + X2) A^T): all four cross terms of the two expansions,
// so the fp32 sketch runs on the same tcgen05 kernels as the bf16 one; with
// the projection's two-term image of P the sketch comes within about 4e-6 of
// the exact one in practice, under the 1e-5 bound.  Inputs must be finite with
// magnitude below bf16's largest finite value (about 3.39e38).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace logra {

// two fp32 values -> their leading bf16 terms (hi) and the bf16 of the exact remainders (lo)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// One float4 of X or dY per iteration; each row of a plane sits at the same
// offset as its source row, plane p of a tensor n rows further on.  Rows are
// whole float4s (k, d multiples of 8), so no float4 straddles two rows.
__global__ void __launch_bounds__(256) f32_planes_kernel(const float4* __restrict__ X, const float4* __restrict__ dY,
                                                         int64_t nx, int64_t ny, uint2* __restrict__ Xp,
                                                         uint2* __restrict__ dYp) {
  const int64_t total = nx + ny;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const bool is_x = i < nx;
    const int64_t j = is_x ? i : i - nx;
    const float4 v = is_x ? __ldcs(X + j) : __ldcs(dY + j);
    uint2 hi, lo;
    split2(v.x, v.y, hi.x, lo.x);
    split2(v.z, v.w, hi.y, lo.y);
    if (is_x) {                       // [X1; X2; X1; X2]
      Xp[j] = hi;
      Xp[j + nx] = lo;
      Xp[j + 2 * nx] = hi;
      Xp[j + 3 * nx] = lo;
    } else {                          // [dY1; dY1; dY2; dY2]
      dYp[j] = hi;
      dYp[j + ny] = hi;
      dYp[j + 2 * ny] = lo;
      dYp[j + 3 * ny] = lo;
    }
  }
}

int launch_f32_planes(const float* X, const float* dY, int64_t n, int64_t d, int64_t k, void* Xp, void* dYp,
                      cudaStream_t s) {
  const int64_t nx = n * (k / 4), ny = n * (d / 4);
  const int threads = 256;
  int64_t blocks = (nx + ny + threads - 1) / threads;
  const int64_t cap = int64_t(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  f32_planes_kernel<<<unsigned(blocks), threads, 0, s>>>(reinterpret_cast<const float4*>(X),
                                                         reinterpret_cast<const float4*>(dY), nx, ny,
                                                         static_cast<uint2*>(Xp), static_cast<uint2*>(dYp));
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
