// Tensor-core sketch for bf16 inputs (tcgen05 + TMEM + TMA), three launches:
//
//   project   P_s^T = Sigma X_s^T for a k-range s  (D[128 tokens x r] in TMEM;
//             A = X tile by TMA, B = Sigma tile generated in shared memory
//             from the sign hash; k split over s for occupancy)
//   split     P^T (the k-splits summed by fp32 reductions into one buffer)
//             stored as a two-term bf16 expansion
//             P^T = hi + lo, written pre-swizzled in 32-token chunks so the
//             next kernel loads one chunk with a single bulk copy
//   accumulate S += (P^T dY)^T / sqrt(r): D[r x N d-columns] in TMEM with
//             A = P^T chunk (hi and lo, two MMAs into one accumulator),
//             B = dY tile (MN-major, TMA), tokens split over units; each unit
//             adds its tile into S with TMA tensor reduce-adds (fp32).
//
// (theclarity.today write-up, "Why it matters": S = G A^T is accumulated during
// backpropagation and G is never formed; academy.dair.ai summary: the random-
// sign projection is redrawn per step and shared by the step's microbatches.)
//
// The operand streamed from HBM (X, dY) and the other operand (the generated
// sign tile, the L2-resident P^T image) move through separate shared-memory
// rings, so the HBM stream gets the deep ring its latency needs.
//
// Roles per CTA: warp 0 = producer of the first ring, warp 1 = TMEM owner +
// MMA issuer, warps 2..5 = epilogue (TMEM lane quadrant = warp % 4), warps
// 6..15 except 9 and 13 = sign-tile generators (project; the two skipped warps
// share the MMA warp's scheduler) / warp 6 = dY producer (accumulate).
// Every wait is bounded; a wait that runs out records LOGRA_ERR_TIMEOUT in the
// control block and the CTA drains and exits.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace logra {

using namespace tc;

namespace {

constexpr int kTok = 128;      // tokens per project tile (MMA M)
constexpr int kKc = 64;        // k per project stage (one sign word per row)
constexpr int kChunk = 32;     // tokens per accumulate stage / image chunk
constexpr int kMaxStages = 16;
constexpr int kSmemBudget = 227 * 1024 - 1024 - 512;
constexpr int kStageTile = 32 * 32 * 4;        // one epilogue warp's fp32 staging tile
constexpr int kStagingBytes = 4 * 2 * kStageTile;   // 4 epilogue warps x 2 tiles

struct SketchShape {
  int64_t n, d, k;
  int r, r_pad;                // r_pad: r rounded up to 128 (accumulate M blocks)
  int n_pad;                   // n rounded up to kChunk
  int tiles, tgroup, groups;  // project: 128-token tiles, tiles per unit, tile groups
  int splits, chunks_per_split, nchunks;             // project k-splits
  int ntile_n, dtiles, tsplits, tchunks_per_split;   // accumulate
  int x_stages, g_stages;      // project rings: X tiles, sign tiles
  int a_stages, b_stages;      // accumulate rings: P^T chunks, dY tiles
};

struct Shared {
  uint64_t s_full[kMaxStages], s_empty[kMaxStages];   // streamed operand (X / dY)
  uint64_t o_full[kMaxStages], o_empty[kMaxStages];   // other operand (sign tile / P^T chunk)
  uint64_t tmem_full[2], tmem_empty[4], drain;     // tmem_empty: one per accumulator block
  uint2 nib[16];                                       // 4 sign bits -> 4 bf16 +-1
  uint32_t tmem_base;
  int abort;
};

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) { stage = 0; phase ^= 1u; }
  }
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Copies still in flight land before the CTA exits: wait (bounded) for the
// last phase issued on every stage of a ring; phases already consumed pass.
__device__ __forceinline__ void drain_ring(uint64_t* full, const Ring& rg, int n, unsigned long long limit) {
  for (int s = 0; s < n; ++s) mbar_wait(&full[s], (s < rg.stage) ? rg.phase : (rg.phase ^ 1u), limit);
}

}  // namespace

// ============================================================================ project
// Sigma tile for k-chunk c: rows b < r of 128 bytes (64 bf16 +-1), K-major,
// 128-byte swizzle (16-byte chunk q of row b stored at chunk q ^ (b & 7)).
__device__ __forceinline__ void gen_sigma_kmajor(uint8_t* tile, const uint2* nib, uint64_t key, int r, int c, int tid,
                                                 int nthr) {
  for (int b = tid; b < r; b += nthr) {
    const uint64_t w = sign_word(key, uint32_t(b), uint32_t(c));
    const uint32_t lo = uint32_t(w), hi = uint32_t(w >> 32);
    uint8_t* row = tile + size_t(b) * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t byte = ((q < 4 ? lo : hi) >> (8 * (q & 3))) & 0xFFu;
      const uint2 a = nib[byte & 15u], bb = nib[byte >> 4];
      *reinterpret_cast<uint4*>(row + ((q ^ (b & 7)) << 4)) = make_uint4(a.x, a.y, bb.x, bb.y);
    }
  }
}

// One unit = (group of `tgroup` 128-token tiles, k-split): each generated sign
// tile feeds the MMAs of every token tile of the group, so the generation cost
// per MMA falls with the group size.  The epilogue stages 32 x 32 fp32 tiles in
// shared memory and hands them to TMA: a plain tensor store when k is not split,
// a tensor reduce-add (performed by the TMA unit and L2) into the zeroed P^T
// buffer when it is.
__global__ void __launch_bounds__(512, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_p,
                      SketchShape sh_, uint64_t key, Control* ctl) {
  extern __shared__ uint8_t smem_raw[];
  const SketchShape& P = sh_;
  uint8_t* base = align1024(smem_raw);
  const int XS = P.x_stages, GS = P.g_stages, T = P.tgroup;
  const uint32_t x_bytes = uint32_t(T) * kTok * 128;
  const uint32_t g_bytes = uint32_t(P.r) * 128;
  uint8_t* x_tiles = base;
  uint8_t* g_tiles = base + size_t(XS) * x_bytes;
  uint8_t* staging = g_tiles + size_t(GS) * g_bytes;
  Shared* sh = reinterpret_cast<Shared*>(staging + kStagingBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = ctl->wait_limit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->s_empty[s], 1);
    }
    for (int s = 0; s < GS; ++s) {
      mbar_init(&sh->o_full[s], 8);
      mbar_init(&sh->o_empty[s], 1);
    }
    mbar_init(&sh->tmem_full[0], 1);
    for (int t = 0; t < 4; ++t) mbar_init(&sh->tmem_empty[t], 4);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_p);
  }
  if (threadIdx.x < 16) {
    const uint4 v = signs8_to_bf16(threadIdx.x);       // elements 0..3 of the nibble in .x, .y
    sh->nib[threadIdx.x] = make_uint2(v.x, v.y);
  }
  // one accumulator of acc_cols (>= r) columns per token tile of the group
  uint32_t acc_cols = 32;
  while (acc_cols < uint32_t(P.r)) acc_cols <<= 1;
  uint32_t tmem_cols = 32;
  while (tmem_cols < acc_cols * uint32_t(T)) tmem_cols <<= 1;
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int units = P.groups * P.splits;

  if (warp == 0) {
    // ---------------------------------------------------------------- X tile producer (T tiles per stage)
    if (lane == 0) {
      Ring xr;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int grp = u % P.groups, split = u / P.groups;
        const int c0 = split * P.chunks_per_split;
        const int c1 = min(P.nchunks, c0 + P.chunks_per_split);
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->s_empty[xr.stage], xr.phase ^ 1u, limit, ctl)) goto producer_done;
          if (inject && c == c0 + 1) {
            inject = 0;                      // test hook: this stage never fills
          } else {
            uint8_t* dst = x_tiles + size_t(xr.stage) * x_bytes;
            mbar_arrive_expect_tx(&sh->s_full[xr.stage], x_bytes);
            for (int t = 0; t < T; ++t)
              tma_load_2d(dst + t * (kTok * 128), &tmap_x, &sh->s_full[xr.stage], c * kKc, (grp * T + t) * kTok);
          }
          xr.next(XS);
        }
      }
    producer_done:
      drain_ring(sh->s_full, xr, XS, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      Ring xr, gr;
      uint32_t tphase = 0;
      const int nparts = P.r > 256 ? 2 : 1;
      const int npart = P.r / nparts;
      const uint32_t idesc = idesc_bf16(128, uint32_t(npart), 0, 0);
      for (int u = blockIdx.x; u < units && !sh->abort; u += gridDim.x) {
        const int split = u / P.groups;
        const int c0 = split * P.chunks_per_split;
        const int c1 = min(P.nchunks, c0 + P.chunks_per_split);
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->s_full[xr.stage], xr.phase, limit, ctl)) goto mma_done;
          if (!wait_or_abort(sh, &sh->o_full[gr.stage], gr.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint32_t a0 = smem_addr(x_tiles + size_t(xr.stage) * x_bytes);
          const uint32_t b0 = smem_addr(g_tiles + size_t(gr.stage) * g_bytes);
#pragma unroll
          for (int ks = 0; ks < kKc / 16; ++ks) {
            for (int t = 0; t < T; ++t) {
              if (c == c0 && ks == 0) {
                // accumulator t is free once the epilogue has drained it
                if (!wait_or_abort(sh, &sh->tmem_empty[t], tphase ^ 1u, limit, ctl)) goto mma_done;
                tc_fence_after();
              }
              const uint64_t ad = smem_desc(a0 + t * (kTok * 128) + ks * 32, 16, 1024, kSw128);
              for (int p = 0; p < nparts; ++p) {
                const uint64_t bd = smem_desc(b0 + uint32_t(p * npart) * 128 + ks * 32, 16, 1024, kSw128);
                mma_bf16(tmem + uint32_t(t) * acc_cols + uint32_t(p * npart), ad, bd, idesc,
                         (c == c0 && ks == 0) ? 0u : 1u);
              }
            }
          }
          mma_commit(&sh->s_empty[xr.stage]);
          mma_commit(&sh->o_empty[gr.stage]);
          xr.next(XS);
          gr.next(GS);
        }
        mma_commit(&sh->tmem_full[0]);
        tphase ^= 1u;
      }
    mma_done:
      mma_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- epilogue: TMEM -> smem -> TMA into P^T
    const int quad = warp & 3;
    float* stg = reinterpret_cast<float*>(staging + (warp - 2) * 2 * kStageTile);
    uint32_t tphase = 0;
    int sb = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int grp = u % P.groups;
      if (!warp_wait(sh, &sh->tmem_full[0], tphase, limit, ctl)) break;
      tphase ^= 1u;
      tc_fence_after();
      for (int t = 0; t < T; ++t) {
        const int x0 = (grp * T + t) * kTok + quad * 32;   // first token of this warp's lanes
        for (int c = 0; c < P.r; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + uint32_t(t) * acc_cols + (uint32_t(quad * 32) << 16) + uint32_t(c), v);
          tmem_ld_wait();
          // staging tile [32 ranks][32 tokens]: lane = token, so each row store is one 128-byte line
          float* tile = stg + sb * (32 * 32);
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[j * 32 + lane] = __uint_as_float(v[j]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (x0 < P.n_pad) {
              if (P.splits == 1) tma_store_2d(&tmap_p, tile, x0, c);
              else tma_reduce_add_2d(&tmap_p, tile, x0, c);
            }
            bulk_commit();
            bulk_wait_read_1();      // the other staging tile is free again
          }
          __syncwarp();
          sb ^= 1;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->tmem_empty[t]);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else if (warp != 9 && warp != 13) {
    // ---------------------------------------------------------------- sign-tile generators (8 warps)
    // Warps 9 and 13 stay idle so that no generator shares the MMA warp's
    // scheduler (warp % 4 == 1): the single issuing thread keeps its issue slots.
    const int gtid = (warp - 6 - (warp > 9) - (warp > 13)) * 32 + lane;
    Ring gr;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int split = u / P.groups;
      const int c0 = split * P.chunks_per_split;
      const int c1 = min(P.nchunks, c0 + P.chunks_per_split);
      for (int c = c0; c < c1; ++c) {
        if (!warp_wait(sh, &sh->o_empty[gr.stage], gr.phase ^ 1u, limit, ctl)) goto gen_done;
        gen_sigma_kmajor(g_tiles + size_t(gr.stage) * g_bytes, sh->nib, key, P.r, c, gtid, 256);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->o_full[gr.stage]);
        gr.next(GS);
      }
    }
  gen_done:;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ============================================================================ split
// image[c][row][128 B]: tokens 32c..32c+31 of P^T row `row`; bytes 0..63 hold
// the bf16 "hi" terms, 64..127 the "lo" terms, 16-byte chunk q stored at
// q ^ (row & 7).  Rows >= r and tokens >= n are zero.
__global__ void __launch_bounds__(256) split_kernel(const float* __restrict__ ppart, SketchShape P,
                                                    uint8_t* __restrict__ image) {
  const int64_t total = int64_t(P.n_pad / kChunk) * P.r_pad * 4;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total; e += int64_t(gridDim.x) * blockDim.x) {
    const int g = int(e & 3);
    const int64_t rowc = e >> 2;
    const int row = int(rowc % P.r_pad);
    const int64_t c = rowc / P.r_pad;
    const int64_t t0 = c * kChunk + g * 8;
    float p[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (row < P.r) {
      const float4* src = reinterpret_cast<const float4*>(ppart + int64_t(row) * P.n_pad + t0);
      const float4 x0 = src[0], x1 = src[1];
      p[0] = x0.x; p[1] = x0.y; p[2] = x0.z; p[3] = x0.w;
      p[4] = x1.x; p[5] = x1.y; p[6] = x1.z; p[7] = x1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (t0 + i >= P.n) p[i] = 0.f;
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(p[2 * i]), h1 = __float2bfloat16_rn(p[2 * i + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(p[2 * i] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(p[2 * i + 1] - __bfloat162float(h1));
      hi[i] = uint32_t(__bfloat16_as_ushort(h0)) | (uint32_t(__bfloat16_as_ushort(h1)) << 16);
      lo[i] = uint32_t(__bfloat16_as_ushort(l0)) | (uint32_t(__bfloat16_as_ushort(l1)) << 16);
    }
    uint8_t* rowp = image + (c * P.r_pad + row) * 128;
    *reinterpret_cast<uint4*>(rowp + ((g ^ (row & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(rowp + (((g + 4) ^ (row & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// ============================================================================ accumulate
__global__ void __launch_bounds__(352, 1)
    accumulate_tc_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_s,
                         SketchShape sh_, const uint8_t* __restrict__ image, float scale, Control* ctl) {
  extern __shared__ uint8_t smem_raw[];
  const SketchShape& P = sh_;
  uint8_t* base = align1024(smem_raw);
  const int AS = P.a_stages, BS = P.b_stages;
  const int N = P.ntile_n;
  const uint32_t a_bytes = uint32_t(P.r_pad) * 128;
  const uint32_t b_bytes = uint32_t(N) * kChunk * 2;
  uint8_t* a_tiles = base;
  uint8_t* b_tiles = base + size_t(AS) * a_bytes;
  uint8_t* staging = b_tiles + size_t(BS) * b_bytes;
  Shared* sh = reinterpret_cast<Shared*>(staging + kStagingBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = ctl->wait_limit;
  const int mblocks = P.r_pad / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < BS; ++s) {
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->s_empty[s], 1);
    }
    for (int s = 0; s < AS; ++s) {
      mbar_init(&sh->o_full[s], 1);
      mbar_init(&sh->o_empty[s], 1);
    }
    mbar_init(&sh->tmem_full[0], 1);
    for (int m = 0; m < 4; ++m) mbar_init(&sh->tmem_empty[m], 8);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_dy);
  }
  uint32_t tmem_cols = 32;
  while (tmem_cols < uint32_t(mblocks * N)) tmem_cols <<= 1;
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int units = P.dtiles * P.tsplits;
  const int nchunks = P.n_pad / kChunk;

  if (warp == 0) {
    // ---------------------------------------------------------------- P^T chunk producer (L2)
    if (lane == 0) {
      Ring ar;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int ts = u / P.dtiles;
        const int c0 = ts * P.tchunks_per_split, c1 = min(nchunks, c0 + P.tchunks_per_split);
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->o_empty[ar.stage], ar.phase ^ 1u, limit, ctl)) goto a_done;
          if (inject && c == c0 + 1) {
            inject = 0;
          } else {
            mbar_arrive_expect_tx(&sh->o_full[ar.stage], a_bytes);
            bulk_load(a_tiles + size_t(ar.stage) * a_bytes, image + size_t(c) * a_bytes, a_bytes,
                      &sh->o_full[ar.stage]);
          }
          ar.next(AS);
        }
      }
    a_done:
      drain_ring(sh->o_full, ar, AS, limit);
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------------- dY tile producer (HBM)
    if (lane == 0) {
      Ring br;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int dt = u % P.dtiles, ts = u / P.dtiles;
        const int c0 = ts * P.tchunks_per_split, c1 = min(nchunks, c0 + P.tchunks_per_split);
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->s_empty[br.stage], br.phase ^ 1u, limit, ctl)) goto b_done;
          uint8_t* st = b_tiles + size_t(br.stage) * b_bytes;
          mbar_arrive_expect_tx(&sh->s_full[br.stage], b_bytes);
          for (int j = 0; j < N / 64; ++j)
            tma_load_2d(st + j * (kChunk * 128), &tmap_dy, &sh->s_full[br.stage], dt * N + j * 64, c * kChunk);
          br.next(BS);
        }
      }
    b_done:
      drain_ring(sh->s_full, br, BS, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      Ring ar, br;
      uint32_t tphase = 0;
      const uint32_t idesc = idesc_bf16(128, uint32_t(N), 0, 1);
      for (int u = blockIdx.x; u < units && !sh->abort; u += gridDim.x) {
        const int ts = u / P.dtiles;
        const int c0 = ts * P.tchunks_per_split, c1 = min(nchunks, c0 + P.tchunks_per_split);
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->o_full[ar.stage], ar.phase, limit, ctl)) goto mma_done;
          if (!wait_or_abort(sh, &sh->s_full[br.stage], br.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint32_t a0 = smem_addr(a_tiles + size_t(ar.stage) * a_bytes);
          const uint32_t b0 = smem_addr(b_tiles + size_t(br.stage) * b_bytes);
#pragma unroll
          for (int ks = 0; ks < kChunk / 16; ++ks) {
            const uint64_t bd = smem_desc(b0 + ks * 2048, kChunk * 128, 1024, kSw128);
            for (int m = 0; m < mblocks; ++m) {
              if (c == c0 && ks == 0) {
                // M block m of the accumulator is free once the epilogue drained it
                if (!wait_or_abort(sh, &sh->tmem_empty[m], tphase ^ 1u, limit, ctl)) goto mma_done;
                tc_fence_after();
              }
              const uint32_t am = a0 + m * (128 * 128) + ks * 32;
              mma_bf16(tmem + uint32_t(m * N), smem_desc(am, 16, 1024, kSw128), bd, idesc, (c == c0 && ks == 0) ? 0u : 1u);
              mma_bf16(tmem + uint32_t(m * N), smem_desc(am + 64, 16, 1024, kSw128), bd, idesc, 1u);
            }
          }
          mma_commit(&sh->o_empty[ar.stage]);
          mma_commit(&sh->s_empty[br.stage]);
          ar.next(AS);
          br.next(BS);
        }
        mma_commit(&sh->tmem_full[0]);
        tphase ^= 1u;
      }
    mma_done:
      mma_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else if ((warp >= 2 && warp < 6) || (warp >= 7 && warp < 11)) {
    // ---------------------------------------------------------------- epilogue: TMEM -> smem -> TMA reduce-add into S
    // Two groups of four warps (2..5 and 7..10) cover all four TMEM lane
    // quadrants each; group g drains columns [g N/2, (g+1) N/2) of every M
    // block, so an accumulator is free again after half the drain time.
    const int quad = warp & 3;
    const int grp = warp >= 7 ? 1 : 0;
    const int eidx = grp * 4 + (warp - (grp ? 7 : 2));
    float* tile = reinterpret_cast<float*>(staging + eidx * kStageTile);
    const int cbeg = grp * (N / 2), cend = cbeg + N / 2;
    uint32_t tphase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int dt = u % P.dtiles;
      if (!warp_wait(sh, &sh->tmem_full[0], tphase, limit, ctl)) break;
      tphase ^= 1u;
      tc_fence_after();
      for (int m = 0; m < mblocks; ++m) {
        const int r0 = m * 128 + quad * 32;              // first rank of this warp's lanes
        for (int c = cbeg; c < cend; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + uint32_t(m * N + c), v);
          tmem_ld_wait();
          // staging tile [32 d-rows][32 ranks] = a box of S (d x r, row-major); lane = rank
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[j * 32 + lane] = __uint_as_float(v[j]) * scale;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int64_t d0 = int64_t(dt) * N + c;
            if (r0 < P.r && d0 < P.d) tma_reduce_add_2d(&tmap_s, tile, r0, int32_t(d0));
            bulk_commit();
            bulk_wait_read_all();    // the staging tile is free again
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->tmem_empty[m]);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ============================================================================ host side
static int ceil_div(int64_t a, int64_t b) { return int((a + b - 1) / b); }

// Pick the number of splits of the contraction for `tiles` tiles over `sms`
// SMs: the best fraction of busy SMs in the last wave, each split keeping at
// least min_chunks chunks.
static int pick_splits(int tiles, int sms, int nchunks, int min_chunks, int max_splits) {
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= max_splits; ++s) {
    if (s > 1 && ceil_div(nchunks, s) < min_chunks) break;
    const int per = ceil_div(nchunks, s);
    const int real = ceil_div(nchunks, per);
    const int units = tiles * real;
    const int waves = ceil_div(units, sms);
    const double eff = double(units) / double(waves * sms);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = real;
    }
  }
  return best;
}

static SketchShape plan(int64_t n, int64_t d, int64_t k, int r, int sms) {
  SketchShape P{};
  P.n = n; P.d = d; P.k = k; P.r = r;
  P.r_pad = ceil_div(r, 128) * 128;
  P.n_pad = ceil_div(n, kChunk) * kChunk;
  P.tiles = ceil_div(n, kTok);
  // two token tiles share each generated sign tile when their accumulators fit TMEM together
  P.tgroup = (r <= 256 && P.tiles > 1) ? 2 : 1;
  P.groups = ceil_div(P.tiles, P.tgroup);
  P.nchunks = ceil_div(k, kKc);
  P.splits = pick_splits(P.groups, sms, P.nchunks, 8, 12);
  P.chunks_per_split = ceil_div(P.nchunks, P.splits);
  P.splits = ceil_div(P.nchunks, P.chunks_per_split);
  P.ntile_n = (P.r_pad <= 256) ? 256 : 128;
  P.dtiles = ceil_div(d, P.ntile_n);
  const int tchunks = P.n_pad / kChunk;
  P.tsplits = pick_splits(P.dtiles, sms, tchunks, 8, 16);
  P.tchunks_per_split = ceil_div(tchunks, P.tsplits);
  P.tsplits = ceil_div(tchunks, P.tchunks_per_split);
  // project: two sign-tile stages, the rest of shared memory for X tiles
  P.g_stages = 2;
  P.x_stages = (kSmemBudget - kStagingBytes - 2 * r * 128) / (P.tgroup * kTok * 128);
  if (P.x_stages > kMaxStages) P.x_stages = kMaxStages;
  // accumulate: P^T chunks come from L2 (three stages), dY from HBM (the rest)
  const int a_bytes = P.r_pad * 128, b_bytes = P.ntile_n * kChunk * 2;
  P.a_stages = P.r_pad >= 512 ? 2 : 3;
  P.b_stages = (kSmemBudget - kStagingBytes - P.a_stages * a_bytes) / b_bytes;
  if (P.b_stages > kMaxStages) P.b_stages = kMaxStages;
  return P;
}

static int proj_smem_bytes(const SketchShape& P) {
  return 1024 + P.x_stages * P.tgroup * kTok * 128 + P.g_stages * P.r * 128 + kStagingBytes + int(sizeof(Shared));
}

static int acc_smem_bytes(const SketchShape& P) {
  return 1024 + P.a_stages * P.r_pad * 128 + P.b_stages * P.ntile_n * kChunk * 2 + kStagingBytes +
         int(sizeof(Shared));
}

size_t sketch_tc_workspace_bytes(int64_t n, int64_t d, int64_t k, int r, int sms) {
  const SketchShape P = plan(n, d, k, r, sms);
  const size_t part = size_t(P.r) * P.n_pad * 4;
  const size_t img = size_t(P.n_pad) * P.r_pad * 4;
  return ((part + 1023) & ~size_t(1023)) + img;
}

int launch_sketch_tc(const void* X, const void* dY, int64_t n, int64_t d, int64_t k, int r, uint64_t key,
                     float scale, float* S, void* ws, Control* ctl, cudaStream_t s) {
  const int sms = sm_count();
  const SketchShape P = plan(n, d, k, r, sms);
  float* ppart = static_cast<float*>(ws);
  const size_t part = size_t(P.r) * P.n_pad * 4;
  uint8_t* image = static_cast<uint8_t*>(ws) + ((part + 1023) & ~size_t(1023));

  CUtensorMap tx, tdy, tp, ts;
  if (int st = make_tmap_2d(&tx, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(k), uint64_t(n), uint64_t(k) * 2,
                            kKc, kTok, CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  if (int st = make_tmap_2d(&tdy, dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(d), uint64_t(n), uint64_t(d) * 2,
                            64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  // P^T (r x n_pad fp32) and S (d x r fp32) in 32 x 32 boxes for the epilogues' TMA store / reduce-add
  if (int st = make_tmap_2d(&tp, ppart, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, uint64_t(P.n_pad), uint64_t(r),
                            uint64_t(P.n_pad) * 4, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return st;
  if (int st = make_tmap_2d(&ts, S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, uint64_t(r), uint64_t(d), uint64_t(r) * 4,
                            32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return st;

  const int proj_smem = proj_smem_bytes(P);
  LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(project_tc_kernel), proj_smem));
  const int punits = P.groups * P.splits;
  if (P.splits > 1) LOGRA_CUDA_TRY(cudaMemsetAsync(ppart, 0, part, s));   // the k-splits reduce-add into it
  project_tc_kernel<<<punits < sms ? punits : sms, 512, proj_smem, s>>>(tx, tp, P, key, ctl);
  LOGRA_LAUNCHED();

  const int64_t stotal = int64_t(P.n_pad / kChunk) * P.r_pad * 4;
  int sblocks = int((stotal + 255) / 256);
  if (sblocks > sms * 8) sblocks = sms * 8;
  split_kernel<<<sblocks, 256, 0, s>>>(ppart, P, image);
  LOGRA_LAUNCHED();

  const int acc_smem = acc_smem_bytes(P);
  LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(accumulate_tc_kernel), acc_smem));
  const int aunits = P.dtiles * P.tsplits;
  accumulate_tc_kernel<<<aunits < sms ? aunits : sms, 352, acc_smem, s>>>(tdy, ts, P, image, scale, ctl);
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
