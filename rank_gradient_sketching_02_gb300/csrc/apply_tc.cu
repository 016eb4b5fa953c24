// Tensor-core reconstruct-and-update (tcgen05 + TMEM + TMA), and the row norms
// that RowAdam needs before it.
//
//   for each 128-row block of W and each 256-column super-tile:
//     D[128 x 256] = S_rows (hi + lo bf16, two MMAs) * Sigma[:, cols]   (TMEM)
//   epilogue, 32 columns at a time, thread = row:
//     apply    W_ij += f_i D_ij  with f_i = -lr c / (sqrt(r) sqrt(v_i + eps)),
//              optional bf16 copy of W, sum of (f_i D_ij)^2
//     predict  only the sum of squares
//     rebuild  out_ij (+)= D_ij / sqrt(r)   (fp32 or bf16 output)
//   row norms (mode 4): D = S_rows * M with M = Sigma Sigma^T (exact integers,
//     split hi + lo), q_i = sum_b D_ib S_ib = r ||(S A)_i||^2, then
//     v_i <- beta2 v_i + (1 - beta2) q_i / (r k), 1/sqrt(v_i + eps), the
//     optional sync sketch and ||S||^2 partials.
//
// Ghat = S A is formed tile by tile and consumed in the same kernel, so the
// d x k reconstruction never reaches memory (theclarity.today write-up, "Why
// it matters": the full-size estimate exists only when the update is
// applied).  RowAdam keeps one squared-row-magnitude statistic per row and no
// first moment (same write-up, "What happened"); mode 4 updates it from the
// exact row norms before the update pass uses it.
//
// Operands: A = the row block of S, pre-split into bf16 hi/lo and pre-swizzled
// (one bulk copy per 32-wide rank chunk); B = Sigma rows of that chunk for the
// super-tile's 256 columns, MN-major, generated in shared memory from the sign
// hash (mode 4: the M image by bulk copy).  W moves in by TMA in 128 x 32
// sub-tiles through a 3-stage ring whose stages are released as soon as the
// epilogue warps have read them; two epilogue groups take alternate sub-tiles
// and each warp writes its updated 32-row slice (and its bf16 copy) to its
// group's staging and stores it by TMA on its own, the store draining while the
// other group works on the next sub-tile.
//
// Roles: warp 0 = A (and mode-4 B) producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..5 and 11..14 = two epilogue groups (TMEM lane quadrant = warp % 4),
// warps 6..9 = sign-tile generators, warp 10 = W tile producer.  TMEM holds two 256-column
// accumulators so the epilogue of one super-tile overlaps the MMAs of the next.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace logra {

using namespace tc;

namespace {

constexpr int kRows = 128;        // MMA M: rows of W per block
constexpr int kCols = 256;        // MMA N: columns per super-tile
// Ranks per K chunk.  A chunk of 32 ranks (16 KB of S image, 16 KB of sign
// tile) lets four stages fit where two 64-rank stages did: the producers then
// have three chunks of MMA time, not one, to refill a stage (bulk copy from L2
// plus sign generation), which at r = 512 held the MMAs back.
constexpr int kRc = 32;
constexpr int kARow = kRc * 2;    // bytes per row of an A chunk (64: SWIZZLE_64B, K-major)
constexpr int kSub = 32;          // epilogue sub-tile width (columns)
constexpr int kAbStages = 4;      // A/B stages of the update and rebuild passes
constexpr int kAbStagesNorm = 4;  // row norms: four 48 KB stages (S chunk + M hi + M lo) in the A/B, W ring and staging space
constexpr int kWStages = 3;
constexpr uint32_t kABytes = 2 * kRows * kARow; // hi + lo: 16 KB
constexpr uint32_t kBBytes = kRc * kCols * 2;   // 32 ranks x 256 columns bf16: 16 KB
constexpr uint32_t kWBytes = kRows * kSub * 4;  // fp32 sub-tile: 16 KB
constexpr uint32_t kHBytes = kRows * kSub * 2;  // bf16 sub-tile: 8 KB

struct ApplyShared {
  uint64_t ab_full[kAbStagesNorm], gen_full[kAbStagesNorm], ab_empty[kAbStagesNorm];
  uint64_t w_full[kWStages], w_empty[kWStages];
  uint64_t tmem_full[2], tmem_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int flag;
  double red[kMaxGroup][8];   // per matrix, per epilogue warp: this CTA's partial sum
};

constexpr size_t kApplySmem = 1024 + kAbStages * (kABytes + kBBytes) + kWStages * kWBytes + 2 * kWBytes + 2 * kHBytes +
                              sizeof(ApplyShared) + 64;

// Named barrier of the eight epilogue warps (warp-aligned, so reconverged first).
__device__ __forceinline__ void epi_sync() {
  __syncwarp();
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

}  // namespace

// One matrix of a launch.
struct ApplyMat {
  int64_t d, k;
  int nsuper;                 // super-tiles per row block (columns of W; mode 4: of M)
  int units;                  // modes 0-3: row blocks x super-tiles; mode 4: row blocks
  uint64_t key;
  float neg_lrc_scale;        // -lr c / sqrt(r)   (apply, predict)
  float neg_lrc;              // -lr c             (mode 4 sync sketch)
  float vscale;               // mode 4: 1 / (1 - beta2^t) with Adam's bias correction, else 1
  int write_bf16;             // apply: also store the bf16 copy
  const uint8_t* s_image;     // [row block][rank chunk][hi | lo][128 rows][128 B]
  const uint8_t* m_image;     // [super-tile][rank chunk][hi, lo][32 KB]
  const float* S;
  const float* v_in;
  float* v_out;
  float* inv;                 // d values 1/sqrt(v_i + eps)
  float* sync_out;
  double* part;               // one per CTA
  double* norms;              // modes 0, 1 (nullable): {||S||^2, ||dW||^2} from the last CTA
  const double* ssq;          // mode 4's ||S||^2 partials
};

// A launch over up to kMaxGroup matrices of the same rank: their work units
// (row block x super-tile; mode 4: row block) are numbered one matrix after
// another and dealt round robin to the persistent CTAs, so small matrices
// share the machine with large ones instead of each paying its own fill and
// tail.  Passed as one __grid_constant__ parameter block (about 5 KB).
struct ApplyArgs {
  CUtensorMap tm[kMaxGroup][4];   // fp32 load (128 rows), bf16 load, fp32 store (32 rows), bf16 store
  ApplyMat m[kMaxGroup];
  int ustart[kMaxGroup + 1];      // first unit of each matrix; ustart[nm] = all units
  int nm;
  int r;
  int inner;                  // super-tiles per unit: 1, or nsuper in mode 4
  int nck;                    // rank chunks of kRc
  float scale;                // 1 / sqrt(r)       (rebuild)
  float beta2, eps;
  int accumulate;             // rebuild: add into the output
  int nssq;                   // mode 4's grid: partials per matrix in ssq
  unsigned* counter;          // CTAs finished, wrapping to 0 after the last one (null: no norms)
};

// Matrix of unit u (units are numbered matrix by matrix).
__device__ __forceinline__ int mat_of(const ApplyArgs& A, int u) {
  int m = 0;
  while (m + 1 < A.nm && u >= A.ustart[m + 1]) ++m;
  return m;
}

template <int MODE>
__global__ void __launch_bounds__(480, 1)
    apply_tc_kernel(const __grid_constant__ ApplyArgs A, Control* ctl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* ab = base;                                              // [stage][A 32 KB | B 32 KB]
  uint8_t* wr = ab + kAbStages * (kABytes + kBBytes);              // [stage][16 KB] W sub-tiles in
  uint8_t* sb32 = wr + kWStages * kWBytes;                         // 2 x 16 KB fp32 staging out
  uint8_t* hb = sb32 + 2 * kWBytes;                                // 2 x 8 KB bf16 staging out
  ApplyShared* sh = reinterpret_cast<ApplyShared*>(hb + 2 * kHBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = ctl->wait_limit;
  constexpr bool kNorm = (MODE == 4);
  constexpr int AS = kNorm ? kAbStagesNorm : kAbStages;   // mode 4 uses no W ring or staging
  // a stage holds one rank chunk of the S image and its B operand: the sign
  // tile, or (mode 4) both terms of the Gram image, so each S chunk loads once
  constexpr uint32_t kStageB = kNorm ? kABytes + 2 * kBBytes : kABytes + kBBytes;
  const int nchunks = A.nck;
  const int units = A.ustart[A.nm];
  const bool load_in = (MODE == 0) || ((MODE == 2 || MODE == 3) && A.accumulate);

  if (threadIdx.x == 0) {
    for (int s = 0; s < AS; ++s) {
      mbar_init(&sh->ab_full[s], 1);
      mbar_init(&sh->gen_full[s], 4);
      mbar_init(&sh->ab_empty[s], 1);
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&sh->w_full[s], 1);
      mbar_init(&sh->w_empty[s], 4);   // one release per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->tmem_full[b], 1);
      mbar_init(&sh->tmem_empty[b], kNorm ? 4 : 8);   // every active epilogue warp
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    for (int i = 0; i < kMaxGroup * 8; ++i) sh->red[i / 8][i % 8] = 0.0;
    fence_mbar_init();
    for (int mi = 0; mi < A.nm; ++mi) {
      if (MODE == 0 || MODE == 2) {
        prefetch_tmap(&A.tm[mi][0]);
        prefetch_tmap(&A.tm[mi][2]);
      }
      if ((MODE == 0 && A.m[mi].write_bf16) || MODE == 3) {
        prefetch_tmap(&A.tm[mi][1]);
        prefetch_tmap(&A.tm[mi][3]);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();      // the S image, Gram image and row factors come from the launches before

  if (warp == 0) {
    // ------------------------------------------------------------------ A producer (S hi/lo chunks; mode 4: + M)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int mi = mat_of(A, u), lu = u - A.ustart[mi];
        const ApplyMat& M = A.m[mi];
        for (int t = 0; t < A.inner; ++t) {
          const int rb = kNorm ? lu : lu / M.nsuper;
          const int st = kNorm ? t : lu % M.nsuper;
          for (int c = 0; c < nchunks; ++c) {
            if (!wait_or_abort(sh, &sh->ab_empty[stage], phase ^ 1u, limit, ctl)) goto a_done;
            uint8_t* dst = ab + stage * kStageB;
            if (inject && c == 0) {
              inject = 0;
            } else {
              mbar_arrive_expect_tx(&sh->ab_full[stage], kNorm ? kStageB : kABytes);
              bulk_load(dst, M.s_image + (size_t(rb) * A.nck + c) * kABytes, kABytes, &sh->ab_full[stage]);
              if (kNorm)   // M_hi and M_lo of this chunk are adjacent in the image
                bulk_load(dst + kABytes, M.m_image + (size_t(st) * A.nck + c) * 2 * kBBytes, 2 * kBBytes,
                          &sh->ab_full[stage]);
            }
            if (++stage == AS) { stage = 0; phase ^= 1u; }
          }
        }
      }
    a_done:
      for (int s = 0; s < AS; ++s) mbar_wait(&sh->ab_full[s], (s < stage) ? phase : (phase ^ 1u), limit);
      // and the MMA commits' last arrivals on the ring land before the CTA can leave
      for (int s = 0; s < AS; ++s) {
        const bool aborted = *reinterpret_cast<volatile int*>(&sh->abort) != 0;
        mbar_wait(&sh->ab_empty[s], (s < stage) ? phase : (phase ^ 1u), aborted ? limit / 64 + 1 : limit);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ W tile producer
    if (lane == 0 && load_in) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t bytes = (MODE == 3) ? kHBytes : kWBytes;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int mi = mat_of(A, u), lu = u - A.ustart[mi];
        const CUtensorMap* map = &A.tm[mi][MODE == 3 ? 1 : 0];
        const int rb = lu / A.m[mi].nsuper, st = lu % A.m[mi].nsuper;
        for (int s = 0; s < kCols / kSub; ++s) {
          const int64_t col0 = int64_t(st) * kCols + s * kSub;
          if (col0 >= A.m[mi].k) break;
          if (!wait_or_abort(sh, &sh->w_empty[stage], phase ^ 1u, limit, ctl)) goto w_done;
          mbar_arrive_expect_tx(&sh->w_full[stage], bytes);
          tma_load_2d(wr + stage * kWBytes, map, &sh->w_full[stage], int32_t(col0), rb * kRows);
          if (++stage == kWStages) { stage = 0; phase ^= 1u; }
        }
      }
    w_done:
      for (int s = 0; s < kWStages; ++s) mbar_wait(&sh->w_full[s], (s < stage) ? phase : (phase ^ 1u), limit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tph[2] = {0, 0};
      int buf = 0;
      const uint32_t idesc = idesc_bf16(kRows, kCols, 0, 1);
      // stage-0 descriptors, advanced by adds of the 16-byte-unit address field
      const uint64_t adesc0 = smem_desc(smem_addr(ab), 16, 8 * kARow, kSw64);
      const uint64_t bdesc0 = smem_desc(smem_addr(ab + kABytes), kRc * 128, 1024, kSw128);
      for (int u = blockIdx.x; u < units && !sh->abort; u += gridDim.x) {
        for (int t = 0; t < A.inner; ++t) {
          if (!wait_or_abort(sh, &sh->tmem_empty[buf], tph[buf] ^ 1u, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint32_t dt = tmem + uint32_t(buf * kCols);
          for (int c = 0; c < nchunks; ++c) {
            if (!wait_or_abort(sh, &sh->ab_full[stage], phase, limit, ctl)) goto mma_done;
            if (!kNorm && !wait_or_abort(sh, &sh->gen_full[stage], phase, limit, ctl)) goto mma_done;
            tc_fence_after();
            const uint64_t ad = adesc0 + uint64_t(uint32_t(stage) * (kStageB >> 4));
            const uint64_t bd = bdesc0 + uint64_t(uint32_t(stage) * (kStageB >> 4));
            const int ksteps = min(kRc, A.r - c * kRc) / 16;
            for (int ks = 0; ks < ksteps; ++ks) {
              const uint64_t a_hi = ad + uint64_t(2 * ks), a_lo = a_hi + uint64_t((kRows * kARow) >> 4);
              const uint64_t b = bd + uint64_t(ks * (2048 >> 4));
              mma_bf16(dt, a_hi, b, idesc, (c | ks) ? 1u : 0u);
              mma_bf16(dt, a_lo, b, idesc, 1u);
              if (kNorm) {                                   // the M_lo term
                const uint64_t bl = b + uint64_t(kBBytes >> 4);
                mma_bf16(dt, a_hi, bl, idesc, 1u);
                mma_bf16(dt, a_lo, bl, idesc, 1u);
              }
            }
            mma_commit(&sh->ab_empty[stage]);
            if (++stage == AS) { stage = 0; phase ^= 1u; }
          }
          mma_commit(&sh->tmem_full[buf]);
          tph[buf] ^= 1u;
          buf ^= 1;
        }
      }
    mma_done:
      mma_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else if (warp < 6 || warp >= 11) {
    // ------------------------------------------------------------------ epilogue
    // Two groups of four warps (2..5 and 11..14), each covering the four TMEM
    // lane quadrants, take alternate 32-column sub-tiles (row norms: group 0
    // only), so two warps per scheduler share the per-sub-tile work.
    const int grp = warp >= 11 ? 1 : 0;
    const int ngrp = kNorm ? 1 : 2;
    const int quad = warp & 3;
    const int row_l = quad * 32 + lane;                  // row within the block = TMEM lane
    const int eidx = grp * 4 + (grp ? warp - 11 : warp - 2);
    const int et = eidx * 32 + lane;                     // 0..255
    uint32_t tph[2] = {0, 0};
    int buf = 0;
    int wstage = 0;
    uint32_t wphase = 0;
    double acc_cta = 0.0;   // the current matrix's dW^2 (modes 0, 1) or ||S||^2 (mode 4)
    int cur = -1;           // the matrix acc_cta belongs to
    bool aborted = false;
    // the warp's partial of one matrix, summed over its lanes in a fixed order
    auto flush = [&]() {
      for (int o = 16; o; o >>= 1) acc_cta += __shfl_xor_sync(0xffffffffu, acc_cta, o);
      if (lane == 0 && cur >= 0) sh->red[cur][eidx] = acc_cta;
      acc_cta = 0.0;
    };
    for (int u = blockIdx.x; u < units && !aborted && grp < ngrp; u += gridDim.x) {
      const int mi = mat_of(A, u), lu = u - A.ustart[mi];
      const ApplyMat& M = A.m[mi];
      if (mi != cur) {    // units come in increasing order, so a matrix's units are contiguous here
        flush();
        cur = mi;
      }
      const int rb = kNorm ? lu : lu / M.nsuper;
      const int64_t row = int64_t(rb) * kRows + row_l;
      const bool row_ok = row < M.d;
      double q = 0.0;                                    // mode 4: S_i M S_i^T over the row
      for (int t = 0; t < A.inner && !aborted; ++t) {
        const int st = kNorm ? t : lu % M.nsuper;
        // row norms: the first S slice is fetched while the MMAs still run
        float4 snext[8];
        if (MODE == 4 && row_ok) {
          const float4* sp = reinterpret_cast<const float4*>(M.S + row * A.r + int64_t(st) * kCols);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) snext[q4] = sp[q4];
        }
        if (!warp_wait(sh, &sh->tmem_full[buf], tph[buf], limit, ctl)) { aborted = true; break; }
        tph[buf] ^= 1u;
        tc_fence_after();
        float f = 0.f;
        if (MODE == 0 || MODE == 1) f = row_ok ? M.neg_lrc_scale * M.inv[row] : 0.f;
        else f = A.scale;
        const int64_t ncols_total = kNorm ? int64_t(A.r) : M.k;
        for (int s = 0; s < kCols / kSub; ++s) {
          const int64_t col0 = int64_t(st) * kCols + s * kSub;
          if (col0 >= ncols_total) break;
          if ((s & (ngrp - 1)) != grp) {
            // the other group's sub-tile: keep this warp's place in the W ring
            if (load_in) {
              if (++wstage == kWStages) { wstage = 0; wphase ^= 1u; }
            }
            continue;
          }
          uint32_t g[32];
          tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + uint32_t(buf * kCols + s * kSub), g);
          tmem_ld_wait();
          const int ncol = int(ncols_total - col0 < kSub ? ncols_total - col0 : kSub);
          if (MODE == 4) {
            if (row_ok) {
              // this slice of S was fetched one sub-tile ahead; fetch the next one
              float4 scur[8];
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) scur[q4] = snext[q4];
              if (col0 + kSub < ncols_total && s + 1 < kCols / kSub) {
                const float4* sp = reinterpret_cast<const float4*>(M.S + row * A.r + col0 + kSub);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) snext[q4] = sp[q4];
              }
              float dot = 0.f, ss = 0.f;
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const float4 sv = scur[q4];
                dot = fmaf(__uint_as_float(g[4 * q4 + 0]), sv.x, dot);
                dot = fmaf(__uint_as_float(g[4 * q4 + 1]), sv.y, dot);
                dot = fmaf(__uint_as_float(g[4 * q4 + 2]), sv.z, dot);
                dot = fmaf(__uint_as_float(g[4 * q4 + 3]), sv.w, dot);
                ss = fmaf(sv.x, sv.x, fmaf(sv.y, sv.y, fmaf(sv.z, sv.z, fmaf(sv.w, sv.w, ss))));
              }
              q += double(dot);
              acc_cta += double(ss);
            }
            continue;
          }
          if (MODE == 1) {
            float acc = 0.f;
            if (row_ok) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float dw = f * __uint_as_float(g[j]);
                if (j < ncol) acc = fmaf(dw, dw, acc);
              }
            }
            acc_cta += double(acc);
            continue;
          }
          const uint8_t* wt = wr + wstage * kWBytes;
          uint8_t* st = sb32 + grp * kWBytes;                   // one staging buffer per group
          uint8_t* ht = hb + grp * kHBytes;
          // W comes in through the ring and leaves through separate staging, so
          // a ring stage is released as soon as the warps have read it and the
          // whole ring stays available for loads in flight
          float4 w[8];
          uint4 wb[4];
          if (load_in) {
            if (!warp_wait(sh, &sh->w_full[wstage], wphase, limit, ctl)) { aborted = true; break; }
            if (MODE == 0 || MODE == 2) {
              // fp32 sub-tile, 128-byte rows, 16-byte chunk q at q ^ (row & 7)
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                w[q4] = *reinterpret_cast<const float4*>(wt + row_l * 128 + ((q4 ^ (row_l & 7)) << 4));
            } else {
              // bf16 sub-tile, 64-byte rows, 16-byte chunk h at h ^ ((row >> 1) & 3)
#pragma unroll
              for (int h = 0; h < 4; ++h)
                wb[h] = *reinterpret_cast<const uint4*>(wt + row_l * 64 + ((h ^ ((row_l >> 1) & 3)) << 4));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->w_empty[wstage]);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) w[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int h = 0; h < 4; ++h) wb[h] = make_uint4(0, 0, 0, 0);
          }
          // the group's previous stores have read the staging buffers (they had
          // the other group's sub-tile worth of time; usually no wait)
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
          if (MODE == 0 || MODE == 2) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float d0 = f * __uint_as_float(g[4 * q4 + 0]), d1 = f * __uint_as_float(g[4 * q4 + 1]);
              const float d2 = f * __uint_as_float(g[4 * q4 + 2]), d3 = f * __uint_as_float(g[4 * q4 + 3]);
              if (MODE == 0) {
                if (4 * q4 + 0 < ncol) acc[0] = fmaf(d0, d0, acc[0]);
                if (4 * q4 + 1 < ncol) acc[1] = fmaf(d1, d1, acc[1]);
                if (4 * q4 + 2 < ncol) acc[2] = fmaf(d2, d2, acc[2]);
                if (4 * q4 + 3 < ncol) acc[3] = fmaf(d3, d3, acc[3]);
              }
              w[q4].x += d0; w[q4].y += d1; w[q4].z += d2; w[q4].w += d3;
            }
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(st + row_l * 128 + ((q4 ^ (row_l & 7)) << 4)) = w[q4];
            if (MODE == 0 && M.write_bf16) {
              // bf16 staging: 64-byte rows, 16-byte chunk h at h ^ ((row >> 1) & 3)
#pragma unroll
              for (int h = 0; h < 4; ++h)
                *reinterpret_cast<uint4*>(ht + row_l * 64 + ((h ^ ((row_l >> 1) & 3)) << 4)) =
                    make_uint4(pack_bf16x2(w[2 * h].x, w[2 * h].y), pack_bf16x2(w[2 * h].z, w[2 * h].w),
                               pack_bf16x2(w[2 * h + 1].x, w[2 * h + 1].y), pack_bf16x2(w[2 * h + 1].z, w[2 * h + 1].w));
            }
            if (MODE == 0 && row_ok) acc_cta += double((acc[0] + acc[1]) + (acc[2] + acc[3]));
          } else {
            // MODE 3: bf16 output sub-tile (64-byte rows) in the staging buffer
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int off = (h ^ ((row_l >> 1) & 3)) << 4;
              const uint32_t iw[4] = {wb[h].x, wb[h].y, wb[h].z, wb[h].w};
              uint32_t ow[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(iw[e] << 16) + f * __uint_as_float(g[8 * h + 2 * e]);
                const float hi = __uint_as_float(iw[e] & 0xFFFF0000u) + f * __uint_as_float(g[8 * h + 2 * e + 1]);
                ow[e] = pack_bf16x2(lo, hi);
              }
              *reinterpret_cast<uint4*>(ht + row_l * 64 + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
          }
          // each warp stores its own 32-row slice, so the four epilogue warps
          // run decoupled and a slice's store overlaps the warp's next sub-tile
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int32_t r0 = rb * kRows + quad * 32;
            if (MODE == 0 || MODE == 2) tma_store_2d(&A.tm[mi][2], st + quad * (32 * 128), int32_t(col0), r0);
            if ((MODE == 0 && M.write_bf16) || MODE == 3) tma_store_2d(&A.tm[mi][3], ht + quad * (32 * 64), int32_t(col0), r0);
            bulk_commit();          // in flight until the group's next sub-tile
          }
          __syncwarp();
          if (load_in) {
            if (++wstage == kWStages) { wstage = 0; wphase ^= 1u; }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->tmem_empty[buf]);
        buf ^= 1;
      }
      if (MODE == 4 && !aborted && row_ok) {
        const float mean_sq = float(q) / (float(A.r) * float(M.k));
        const float vn = A.beta2 * M.v_in[row] + (1.f - A.beta2) * mean_sq;
        if (M.v_out) M.v_out[row] = vn;
        const float inv = 1.f / sqrtf(vn * M.vscale + A.eps);   // vscale == 1: exactly vn + eps
        M.inv[row] = inv;
        if (M.sync_out) {
          const float fs = M.neg_lrc * inv;
          const float4* sp = reinterpret_cast<const float4*>(M.S + row * A.r);
          float4* op = reinterpret_cast<float4*>(M.sync_out + row * A.r);
          for (int b = 0; b < A.r / 4; ++b) {
            const float4 sv = sp[b];
            op[b] = make_float4(fs * sv.x, fs * sv.y, fs * sv.z, fs * sv.w);
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    flush();
    epi_sync();
    // this CTA's partial of each matrix (zero for one it had no unit of), fixed order
    if ((MODE == 0 || MODE == 1 || MODE == 4) && et < A.nm) {
      const double* rd = sh->red[et];
      A.m[et].part[blockIdx.x] = ((rd[0] + rd[1]) + (rd[2] + rd[3])) + ((rd[4] + rd[5]) + (rd[6] + rd[7]));
    }
    if ((MODE == 0 || MODE == 1) && A.counter && warp == 2) {
      // The last CTA to finish sums every CTA's partials (and mode 4's) of
      // each matrix in a fixed order: deterministic, and no reduction launch.
      __threadfence();    // by every lane that wrote a partial
      __syncwarp();
      unsigned prev = 0;
      if (lane == 0) prev = atomicInc(A.counter, gridDim.x - 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == gridDim.x - 1) {
        __threadfence();
        for (int mi = 0; mi < A.nm; ++mi) {
          const ApplyMat& M = A.m[mi];
          if (!M.norms) continue;
          double a = 0.0, b = 0.0;
          for (int i = lane; i < A.nssq; i += 32) a += __ldcg(M.ssq + i);
          for (int i = lane; i < int(gridDim.x); i += 32) b += __ldcg(M.part + i);
          for (int o = 16; o; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            b += __shfl_xor_sync(0xffffffffu, b, o);
          }
          if (lane == 0) {
            M.norms[0] = a;
            M.norms[1] = b;
          }
        }
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ sign-tile generators (MN-major)
    if (!kNorm) {
      const int gtid = threadIdx.x - 192;
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int mi = mat_of(A, u);
        const int st = (u - A.ustart[mi]) % A.m[mi].nsuper;
        const uint64_t key = A.m[mi].key;
        for (int c = 0; c < nchunks; ++c) {
          if (!warp_wait(sh, &sh->ab_empty[stage], phase ^ 1u, limit, ctl)) goto gen_done;
          uint8_t* bt = ab + stage * kStageB + kABytes;
          // 4 groups of 64 columns x kRc rank rows; row = one sign word (64 columns)
          for (int e = gtid; e < 4 * kRc; e += 128) {
            const int grp = e / kRc, a_l = e % kRc;
            const int a = c * kRc + a_l;
            const uint64_t w = a < A.r ? sign_word(key, uint32_t(a), uint32_t(st * (kCols / 64) + grp)) : 0ull;
            uint8_t* rowp = bt + grp * (kRc * 128) + a_l * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(rowp + ((q ^ (a_l & 7)) << 4)) = signs8_to_bf16(uint32_t(w >> (8 * q)) & 0xFFu);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->gen_full[stage]);
          if (++stage == AS) { stage = 0; phase ^= 1u; }
        }
      }
    gen_done:;
    }
  }

  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// S image for the A operand: rows split into bf16 hi + lo, 32-rank chunks of
// 64-byte rows (the SWIZZLE_64B K-major layout), 16-byte unit q of row i
// stored at q ^ ((i >> 1) & 3).  Element e is one (row, chunk, 8-rank group).
__device__ __forceinline__ void s_image_elem(const float* __restrict__ S, int64_t d, int r, int nchunks,
                                             uint8_t* __restrict__ img, int64_t e) {
  const int q = int(e & 3);
  const int c = int((e >> 2) % nchunks);
  const int64_t row = (e >> 2) / nchunks;
  // r is a multiple of 32: the 8 ranks of an element are all inside or all outside
  float v[8];
  if (row < d && c * kRc + q * 8 < r) {
    const float4* src = reinterpret_cast<const float4*>(S + row * r + c * kRc + q * 8);
    const float4 x = __ldg(src), y = __ldg(src + 1);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
    hi[i] = uint32_t(__bfloat16_as_ushort(h0)) | (uint32_t(__bfloat16_as_ushort(h1)) << 16);
    lo[i] = uint32_t(__bfloat16_as_ushort(l0)) | (uint32_t(__bfloat16_as_ushort(l1)) << 16);
  }
  const int64_t rb = row / kRows;
  const int rl = int(row % kRows);
  uint8_t* chunk = img + (size_t(rb) * nchunks + c) * kABytes;
  const int off = rl * kARow + ((q ^ ((rl >> 1) & 3)) << 4);
  *reinterpret_cast<uint4*>(chunk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(chunk + kRows * kARow + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// One block of the Gram pass: M = Sigma Sigma^T, the B operand of the
// row-norm GEMM.  Block (bx, by, bz) takes the 32 x 32 tile (rows a0 = 32 by,
// columns b0 = 32 bx) and sign words [64 bz, 64 bz + 64): it hashes the words
// of its 64 rows itself and counts, for each (a, b), the bit positions where
// rows a and b differ.  M is symmetric: only tiles on or above the diagonal
// are counted, and each one above it also writes the mirrored tile's image.  When one block covers all words of the tile (k <= 4096)
// the counts stay in shared memory; otherwise every block adds its counts,
// with exact integer atomics, into `counts`, and the last block of the tile (a
// wrapping arrival counter, left at zero) reads them back and sets them to
// zero for the next apply.  That block writes its part of the image,
// M[a][b] = k - 2 * count, split into bf16 hi + lo: exact while |M| <= k <
// 2^17 (hi keeps 8 significant bits, so the integer M - hi is at most 2^8 in
// magnitude and fits lo's 8 bits); for larger k, lo rounds, an error below
// 2^-16 of the entry.  Image layout per
// (256-column super-tile st, 32-rank chunk c, term): a 16 KB MN-major tile of
// 4 groups of 64 columns x 32 rows of 128 bytes, 16-byte chunk q of row a
// stored at q ^ (a & 7).  Entries outside r x r are zero.
constexpr int kGramWords = 64;

__device__ __forceinline__ void gram_block(uint64_t key, int r, int nw, int64_t k, int* __restrict__ counts,
                                           unsigned* __restrict__ arrivals, uint8_t* __restrict__ mimg, int bx,
                                           int by, int bz, int gx, int gz) {
  __shared__ uint64_t wa[32][kGramWords + 1];
  __shared__ uint64_t wb[32][kGramWords + 1];
  __shared__ int cnt[32][33];
  __shared__ unsigned last;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int a0 = by * 32, b0 = bx * 32;
  const bool live = a0 < r && b0 < r;                         // block-uniform
  if (live && bx < by) return;                                // below the diagonal: its mirror writes it
  if (live) {
    const int wbeg = bz * kGramWords, nwr = min(kGramWords, nw - wbeg);
    for (int e = threadIdx.x; e < 2 * 32 * kGramWords; e += blockDim.x) {
      const int side = e / (32 * kGramWords), rr = (e / kGramWords) % 32, w = e % kGramWords;
      const int row = (side ? b0 : a0) + rr;
      uint64_t v = 0;
      if (w < nwr && row < r) {
        v = sign_word(key, uint32_t(row), uint32_t(wbeg + w));
        const int64_t rem = k - int64_t(wbeg + w) * 64;
        if (rem < 64) v &= (1ull << rem) - 1ull;
      }
      (side ? wb : wa)[rr][w] = v;
    }
    cta_sync();
    int diff[4] = {0, 0, 0, 0};
    for (int w = 0; w < nwr; ++w) {
      const uint64_t x = wb[tx][w];
#pragma unroll
      for (int q = 0; q < 4; ++q) diff[q] += __popcll(wa[ty + 8 * q][w] ^ x);
    }
    if (gz == 1) {
#pragma unroll
      for (int q = 0; q < 4; ++q) cnt[ty + 8 * q][tx] = diff[q];
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int a = a0 + ty + 8 * q, b = b0 + tx;
        if (a < r && b < r && diff[q]) atomicAdd(&counts[a * r + b], diff[q]);
      }
      __threadfence();
      cta_sync();
      if (threadIdx.x == 0) last = (atomicInc(&arrivals[by * gx + bx], gz - 1) == gz - 1) ? 1u : 0u;
      cta_sync();
      if (!last) return;
      __threadfence();
      // the tile's counts, read back and left at zero
      for (int e = threadIdx.x; e < 32 * 32; e += blockDim.x) {
        const int a = a0 + e / 32, b = b0 + e % 32;
        int v = 0;
        if (a < r && b < r) {
          v = __ldcg(counts + a * r + b);
          counts[a * r + b] = 0;
        }
        cnt[e / 32][e % 32] = v;
      }
    }
    cta_sync();
  } else if (bz != 0) {
    return;                                                   // padding tiles: block z = 0 writes the zeros
  }
  // the tile's image (and, above the diagonal, the mirrored tile's): 32 rows
  // x 4 sixteen-byte chunks x 2 terms, one whole chunk (8 consecutive
  // columns of one row, one term) per thread
  const int nck = (r + kRc - 1) / kRc;
  for (int mirror = 0; mirror < ((live && bx > by) ? 2 : 1); ++mirror) {
    const int ra = mirror ? b0 : a0, cb = mirror ? a0 : b0;  // image rows / columns of this tile
    const int term = threadIdx.x >> 7, a = ra + ((threadIdx.x >> 2) & 31), bq = cb + (threadIdx.x & 3) * 8;
    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t two = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = bq + 2 * i + h;
        const int n = (a < r && b < r) ? (mirror ? cnt[b - a0][a - b0] : cnt[a - a0][b - b0]) : 0;
        const float m = (a < r && b < r) ? float(k - 2 * int64_t(n)) : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(m);
        const __nv_bfloat16 v = term ? __float2bfloat16_rn(m - __bfloat162float(hi)) : hi;
        two |= uint32_t(__bfloat16_as_ushort(v)) << (16 * h);
      }
      packed[i] = two;
    }
    const int st = bq >> 8, grp = (bq >> 6) & 3, q = (bq >> 3) & 7;
    const int c = a / kRc, a_l = a % kRc;
    uint8_t* tile = mimg + ((size_t(st) * nck + c) * 2 + term) * kBBytes;
    *reinterpret_cast<uint4*>(tile + grp * (kRc * 128) + a_l * 128 + ((q ^ (a_l & 7)) << 4)) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

// The preparation of a group of applies in one launch: the first ngram blocks
// run the Gram passes of all matrices (when asked), the rest build their S
// images with a grid-stride loop over each matrix in turn.
struct PrepMat {
  uint64_t key;
  int64_t d, k;
  int nw, gz;                 // sign words per row; Gram blocks along the words
  int gram0;                  // first Gram block of this matrix
  int* counts;                // r x r, zero on entry and left zero
  unsigned* arrivals;         // one word per 32 x 32 tile of M, zero on entry and left zero
  uint8_t* mimg;
  const float* S;
  uint8_t* img;
};
struct PrepArgs {
  PrepMat m[kMaxGroup];
  int nm, r, nck, gx, gy, ngram;
};

__global__ void __launch_bounds__(256) apply_prep_kernel(const __grid_constant__ PrepArgs P) {
  grid_dependency_wait();      // S comes from the sketch calls before
  const int b = blockIdx.x;
  if (b < P.ngram) {
    int mi = 0;
    while (mi + 1 < P.nm && b >= P.m[mi + 1].gram0) ++mi;
    const PrepMat& M = P.m[mi];
    const int g = b - M.gram0;
    gram_block(M.key, P.r, M.nw, M.k, M.counts, M.arrivals, M.mimg, g % P.gx, (g / P.gx) % P.gy,
               g / (P.gx * P.gy), P.gx, M.gz);
    return;
  }
  const int64_t nb = int64_t(gridDim.x) - P.ngram;
  for (int mi = 0; mi < P.nm; ++mi) {
    const PrepMat& M = P.m[mi];
    const int64_t total = ((M.d + kRows - 1) / kRows) * kRows * P.nck * (kRc / 8);
    for (int64_t e = (int64_t(b) - P.ngram) * blockDim.x + threadIdx.x; e < total; e += nb * blockDim.x)
      s_image_elem(M.S, M.d, P.r, P.nck, M.img, e);
  }
}

size_t gram_image_bytes(int r) { return size_t((r + kCols - 1) / kCols) * ((r + kRc - 1) / kRc) * 2 * kBBytes; }

size_t s_image_bytes(int64_t d, int r) {
  const int64_t rb = (d + kRows - 1) / kRows;
  const int nchunks = (r + kRc - 1) / kRc;
  return size_t(rb) * nchunks * kABytes;
}

int launch_apply_prep(const PrepMatLaunch* mats, int nm, int r, bool gram, cudaStream_t s) {
  if (nm < 1 || nm > kMaxGroup) return LOGRA_ERR_INVALID_ARG;
  PrepArgs P{};
  P.nm = nm;
  P.r = r;
  P.nck = (r + kRc - 1) / kRc;
  P.gx = gram ? ((r + 255) / 256) * 8 : 0;
  P.gy = gram ? ((r + kRc - 1) / kRc) * (kRc / 32) : 0;
  int64_t total = 0, ngram = 0;
  for (int i = 0; i < nm; ++i) {
    PrepMat& M = P.m[i];
    M.key = mats[i].key;
    M.d = mats[i].d;
    M.k = mats[i].k;
    M.nw = int((M.k + 63) / 64);
    M.gz = gram ? (M.nw + kGramWords - 1) / kGramWords : 0;
    M.gram0 = int(ngram);
    M.counts = mats[i].counts;
    M.arrivals = mats[i].arrivals;
    M.mimg = mats[i].mimg;
    M.S = mats[i].S;
    M.img = mats[i].img;
    ngram += int64_t(P.gx) * P.gy * M.gz;
    total += ((M.d + kRows - 1) / kRows) * kRows * P.nck * (kRc / 8);
  }
  if (ngram > (int64_t(1) << 30)) return LOGRA_ERR_UNSUPPORTED;
  P.ngram = int(ngram);
  int64_t blocks = (total + 255) / 256;
  if (blocks > int64_t(sm_count()) * 8) blocks = int64_t(sm_count()) * 8;
  if (blocks < 1) blocks = 1;
  LOGRA_CUDA_TRY(launch_overlapped(apply_prep_kernel, dim3(unsigned(blocks + ngram)), dim3(256), size_t(0), s, P));
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

int launch_apply_tc(const ApplyLaunch& L, int* grid_out, Control* ctl, cudaStream_t s) {
  const int sms = sm_count();
  const int mode = L.mode;
  if (L.nm < 1 || L.nm > kMaxGroup) return LOGRA_ERR_INVALID_ARG;
  ApplyArgs A{};
  A.nm = L.nm;
  A.r = L.r;
  A.nck = (L.r + kRc - 1) / kRc;
  A.inner = mode == 4 ? (L.r + kCols - 1) / kCols : 1;
  A.scale = inv_sqrt_r(L.r);
  A.beta2 = L.beta2;
  A.eps = L.eps;
  A.accumulate = L.accumulate;
  A.nssq = L.nssq;
  A.counter = nullptr;
  int64_t units = 0;
  for (int i = 0; i < L.nm; ++i) {
    const ApplyMatLaunch& X = L.m[i];
    ApplyMat& M = A.m[i];
    M.d = X.d;
    M.k = X.k;
    const int64_t rbs = (X.d + kRows - 1) / kRows;
    M.nsuper = mode == 4 ? A.inner : int((X.k + kCols - 1) / kCols);
    M.units = int(mode == 4 ? rbs : rbs * M.nsuper);
    M.key = X.key;
    M.neg_lrc = X.neg_lrc;
    M.neg_lrc_scale = X.neg_lrc * A.scale;
    M.vscale = X.vscale;
    M.write_bf16 = (mode == 0 && X.Wb) ? 1 : 0;
    M.s_image = X.s_img;
    M.m_image = X.m_img;
    M.S = X.S;
    M.v_in = X.v_in;
    M.v_out = X.v_out;
    M.inv = X.inv;
    M.sync_out = X.sync_out;
    M.part = X.part;
    M.norms = (mode == 0 || mode == 1) ? X.norms : nullptr;
    M.ssq = X.ssq;
    if (M.norms) A.counter = L.counter;
    A.ustart[i] = int(units);
    units += M.units;
    // loads move 128-row sub-tiles; each epilogue warp stores its own 32-row slice
    if (mode == 0 || mode == 2) {
      const void* p = mode == 0 ? static_cast<const void*>(X.W) : X.out;
      if (int st = make_tmap_2d(&A.tm[i][0], p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, uint64_t(X.k), uint64_t(X.d),
                                uint64_t(X.k) * 4, kSub, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
      if (int st = make_tmap_2d(&A.tm[i][2], p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, uint64_t(X.k), uint64_t(X.d),
                                uint64_t(X.k) * 4, kSub, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
    }
    if ((mode == 0 && X.Wb) || mode == 3) {
      const void* p = mode == 0 ? static_cast<const void*>(X.Wb) : X.out;
      if (int st = make_tmap_2d(&A.tm[i][1], p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(X.k), uint64_t(X.d),
                                uint64_t(X.k) * 2, kSub, kRows, CU_TENSOR_MAP_SWIZZLE_64B))
        return st;
      if (int st = make_tmap_2d(&A.tm[i][3], p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(X.k), uint64_t(X.d),
                                uint64_t(X.k) * 2, kSub, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return st;
    }
  }
  if (units > (int64_t(1) << 30)) return LOGRA_ERR_UNSUPPORTED;
  A.ustart[L.nm] = int(units);
  const int grid = units < sms ? int(units) : sms;
  *grid_out = grid;
  auto run = [&](auto kern) -> int {
    LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(kern), int(kApplySmem)));
    LOGRA_CUDA_TRY(launch_overlapped(kern, dim3(grid), dim3(480), size_t(kApplySmem), s, A, ctl));
    LOGRA_LAUNCHED();
    return LOGRA_OK;
  };
  switch (mode) {
    case 0: return run(apply_tc_kernel<0>);
    case 1: return run(apply_tc_kernel<1>);
    case 2: return run(apply_tc_kernel<2>);
    case 3: return run(apply_tc_kernel<3>);
    default: return run(apply_tc_kernel<4>);
  }
}

}  // namespace logra
