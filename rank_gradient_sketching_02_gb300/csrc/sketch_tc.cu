// Tensor-core sketch for bf16 inputs (tcgen05 + TMEM + TMA), three launches:
//
//   project   P^T partial sums = Sigma X^T over a k-chunk range per segment
//             (D[128 tokens x r] in TMEM per token tile, two token tiles per
//             generated sign tile; A = X tile by TMA, B = Sigma tile generated
//             in shared memory from the sign hash); segments covering a whole
//             k range store, the others reduce-add into the P^T buffer (kept
//             at zero between calls); when every segment covers a whole k
//             range the epilogue writes the split's image itself and the
//             split is not launched
//   split     P^T stored as a two-term bf16 expansion P^T = hi + lo, written
//             pre-swizzled in 32-token chunks so the next kernel loads one
//             chunk with a single bulk copy
//   accumulate S += (P^T dY)^T / sqrt(r): D[r x N d-columns] in TMEM with
//             A = P^T chunk (hi and lo, two MMAs into one accumulator),
//             B = dY tile (MN-major, TMA); each segment adds its tile into S
//             with TMA tensor reduce-adds (fp32); the epilogue warps first
//             set the consumed P^T back to zero for the next call.
//
// The three kernels are launched with programmatic stream serialization and
// wait for their predecessor (griddepcontrol.wait) after their prologue.
//
// Both tensor-core kernels split their work stream-K style: every CTA takes an
// equal contiguous range of the flattened (tile, chunk) space (SegIter), which
// falls into segments at tile boundaries; every segment ends in one drain.
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
// MMA issuer (one thread; its descriptors are built once per ring and advanced
// by adds), warps 2..5 = epilogue (TMEM lane quadrant = warp % 4; the
// accumulate adds a second group, warps 7..10), warps 6..15 except 9 and 13 =
// sign-tile generators (project; the two skipped warps share the MMA warp's
// scheduler) / warp 6 = dY producer (accumulate).
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
  int nchunks;                 // project k-chunks per token group
  int proj_ctas, proj_partial; // project grid; some segment covers only part of the k range
  int ntile_n, dtiles, acc_ctas;   // accumulate: d tile width, d tiles, grid
  int x_stages, g_stages;      // project rings: X tiles, sign tiles
  int a_stages, b_stages;      // accumulate rings: P^T chunks, dY tiles
  // accumulate on CTA pairs (r_pad 256 or 512): rank blocks of 256 and d blocks
  // of 256 per pair tile (prb * pdb = 2, or 1 for narrow d on one stream), pair tiles along d, pairs (clusters)
  int pair, prb, pdb, pdtiles, pairs;
  int direct;                  // every projection segment covers the whole k range: the projection
                               // writes the accumulate's hi/lo image itself and the split is skipped
};

struct Shared {
  uint64_t s_full[kMaxStages], s_empty[kMaxStages];   // streamed operand (X / dY)
  uint64_t o_full[kMaxStages], o_empty[kMaxStages];   // other operand (sign tile / P^T chunk)
  uint64_t tmem_full[2], tmem_empty[4], drain;     // tmem_empty: one per accumulator block
  uint2 nib[16];                                       // 4 sign bits -> 4 bf16 +-1
  uint32_t tmem_base;
  int abort;
};

// Stream-K work split: the flattened (tile, chunk) space of `total` chunks,
// `per` chunks per tile, is cut into gridDim.x equal contiguous ranges, one per
// CTA.  A CTA's range falls into segments at tile boundaries; every segment
// ends with one accumulator drain.  Equal ranges keep the CTAs busy to the end,
// and because the ranges start at different offsets within a tile, the drains
// of different CTAs are spread over the run instead of landing together.
struct SegIter {
  int64_t f, f1;
  int per;
  __device__ __forceinline__ SegIter(int64_t total, int per_) : per(per_) {
    f = total * blockIdx.x / gridDim.x;
    f1 = total * (blockIdx.x + 1) / gridDim.x;
  }
  // range number `idx` of `count` (e.g. one per CTA pair)
  __device__ __forceinline__ SegIter(int64_t total, int per_, int idx, int count) : per(per_) {
    f = total * idx / count;
    f1 = total * (idx + 1) / count;
  }
  __device__ __forceinline__ bool next(int& tile, int& c0, int& c1) {
    if (f >= f1) return false;
    tile = int(f / per);
    c0 = int(f - int64_t(tile) * per);
    const int64_t rem = f1 - f;
    c1 = (rem < int64_t(per - c0)) ? c0 + int(rem) : per;
    f += c1 - c0;
    return true;
  }
};

// The MMA issuer is a single thread, so per-MMA work on it is latency it
// cannot hide.  Descriptors are built once per ring and advanced by plain adds
// of the 16-byte-unit start-address field (all of shared memory lies below
// 256 KB, so the field never carries), inside fully unrolled bodies.

// Projection, one k chunk: T token tiles x NP parts of r, kKc / 16 k steps.
// Each accumulator takes its k steps back to back: a single-CTA MMA stream
// into one accumulator runs at ~7550 FLOP/clk (M128 N256 K16), one that
// alternates between two accumulators at ~6540.
template <int T, int NP>
__device__ __forceinline__ void project_chunk_mmas(uint32_t acc0, uint32_t acc_cols, uint32_t npart, uint64_t ad,
                                                   uint64_t bd, uint32_t idesc, uint32_t first) {
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int ks = 0; ks < kKc / 16; ++ks)
        mma_bf16(acc0 + uint32_t(t) * acc_cols + uint32_t(p) * npart,
                 ad + uint64_t(t * ((kTok * 128) >> 4) + 2 * ks), bd + uint64_t(p * (npart * 8) + 2 * ks), idesc,
                 ks ? 1u : first);
}

// Accumulate, one token chunk: MB M blocks of r, hi and lo terms, kChunk / 16 steps.
template <int MB>
__device__ __forceinline__ void accumulate_chunk_mmas(uint32_t acc0, uint32_t N, uint64_t ad, uint64_t bd,
                                                      uint32_t idesc, uint32_t first) {
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int ks = 0; ks < kChunk / 16; ++ks) {
      const uint64_t bk = bd + uint64_t(ks * (2048 >> 4));
      const uint64_t am = ad + uint64_t(m * ((128 * 128) >> 4) + 2 * ks);
      mma_bf16(acc0 + uint32_t(m) * N, am, bk, idesc, ks ? 1u : first);
      mma_bf16(acc0 + uint32_t(m) * N, am + 4, bk, idesc, 1u);   // lo term: bytes 64..127 of each row
    }
}

// Accumulate on a CTA pair, one token chunk: RB rank blocks x DB d blocks of
// M256 x N256 accumulators (TMEM columns (rb * DB + db) * 256), hi and lo terms.
// A: this CTA's 128 rows of each rank block, 16 KB apart; B: this CTA's 128
// d-columns of each d block, two 64-column boxes of kChunk tokens, 8 KB apart.
template <int RB, int DB>
__device__ __forceinline__ void accumulate_pair_mmas(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                                     uint32_t first) {
#pragma unroll
  for (int rb = 0; rb < RB; ++rb)
#pragma unroll
    for (int db = 0; db < DB; ++db) {
      const uint32_t acc = tmem + uint32_t((rb * DB + db) * 256);
#pragma unroll
      for (int ks = 0; ks < kChunk / 16; ++ks) {
        const uint64_t am = ad + uint64_t(rb * (16384 >> 4) + 2 * ks);
        const uint64_t bk = bd + uint64_t(db * ((2 * kChunk * 128) >> 4) + ks * (2048 >> 4));
        mma_bf16_pair(acc, am, bk, idesc, ks ? 1u : first);
        mma_bf16_pair(acc, am + 4, bk, idesc, 1u);     // lo term: bytes 64..127 of each row
      }
    }
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

// Direct image drain of one segment's accumulators (whole k range): this
// warp's 32 tokens of token tile t are one 32-token image chunk, whose rows
// (one per rank: hi bf16 of the 32 tokens at bytes 0..63, lo at 64..127,
// 16-byte chunk q at q ^ (row & 7)) go straight from registers to global
// memory.  Lane = token; two ranks at a time, lanes exchange with their
// neighbour so that the even lane stores the hi and lo words of tokens
// (t, t + 1) for the first rank and the odd lane those for the second: each
// warp store fills half of two 128-byte rows, whole sectors.  Rows from r up to
// r_pad are zero.  Only the blocks b = t * (r_pad / 32) + j0 / 32 with
// b % nslots == slot are drained, so that several warps of one TMEM lane
// quadrant can share the work.  The image is read by the accumulate's bulk
// copies in a later kernel.
__device__ __forceinline__ void drain_image_blocks(uint32_t acc_tile0, uint32_t acc_cols, int T, int quad, int grp,
                                                   const SketchShape& P, uint8_t* __restrict__ image, int slot,
                                                   int nslots, int lane) {
  const int nchunk32 = P.n_pad / kChunk;
  const int t2 = lane & ~1;
  const int odd = lane & 1;
  const int nb = P.r_pad / 32;
  const uint32_t hi_q = uint32_t(t2 >> 3), lo_q = 4u + uint32_t(t2 >> 3), in_q = uint32_t(t2 & 7) << 1;
  for (int t = 0; t < T; ++t) {
    const uint32_t acc = acc_tile0 + uint32_t(t) * acc_cols + (uint32_t(quad * 32) << 16);
    const int ci = ((grp * T + t) * kTok + quad * 32) / kChunk;
    if (ci >= nchunk32) continue;
    for (int jb = 0; jb < nb; ++jb) {
      if ((t * nb + jb) % nslots != slot) continue;
      const int j0 = jb * 32;
      uint32_t v[32];
      if (j0 < P.r) {
        tmem_ld32(acc + uint32_t(j0), v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      uint8_t* rows = image + (size_t(ci) * P.r_pad + j0) * 128;
#pragma unroll
      for (int jj = 0; jj < 32; jj += 2) {
        const float p0 = __uint_as_float(v[jj]), p1 = __uint_as_float(v[jj + 1]);
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);             // .x = rank jj, .y = rank jj + 1
        const uint32_t hu = *reinterpret_cast<const uint32_t*>(&h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(p0 - __uint_as_float(hu << 16),
                                                       p1 - __uint_as_float(hu & 0xFFFF0000u));
        const uint32_t lu = *reinterpret_cast<const uint32_t*>(&l);
        const uint32_t oh = __shfl_xor_sync(0xffffffffu, hu, 1), ol = __shfl_xor_sync(0xffffffffu, lu, 1);
        // even lane: rank jj of tokens (t2, t2 + 1); odd lane: rank jj + 1 of the same tokens
        const uint32_t wh = odd ? __byte_perm(oh, hu, 0x7632) : __byte_perm(hu, oh, 0x5410);
        const uint32_t wl = odd ? __byte_perm(ol, lu, 0x7632) : __byte_perm(lu, ol, 0x5410);
        const uint32_t row = uint32_t(jj + odd);
        uint8_t* rp = rows + row * 128u + in_q;
        *reinterpret_cast<uint32_t*>(rp + ((hi_q ^ (row & 7u)) << 4)) = wh;
        *reinterpret_cast<uint32_t*>(rp + ((lo_q ^ (row & 7u)) << 4)) = wl;
      }
    }
  }
}

// A segment is (group of `tgroup` 128-token tiles, k-chunk range): each
// generated sign tile feeds the MMAs of every token tile of the group, so the
// generation cost per MMA falls with the group size.  The epilogue stages
// 32 x 32 fp32 tiles in shared memory and hands them to TMA: a plain tensor
// store when the segment covers the whole k range, else a tensor reduce-add
// (performed by the TMA unit and L2) into the zeroed P^T buffer; when every
// segment covers a whole k range (P.direct) it stores the accumulate's hi/lo
// image rows from registers instead (drain_image_blocks).  When two
// groups' accumulators fit TMEM together, consecutive segments alternate
// between them, so the drain of one overlaps the MMAs of the next.
__global__ void __launch_bounds__(512, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_p,
                      SketchShape sh_, uint64_t key, uint8_t* __restrict__ image, Control* ctl) {
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
  // one accumulator of acc_cols (>= r) columns per token tile of the group,
  // and nacc (1 or 2) such sets used by alternate segments
  uint32_t acc_cols = 32;
  while (acc_cols < uint32_t(P.r)) acc_cols <<= 1;
  const int nacc = (acc_cols * uint32_t(T) * 2u <= 512u) ? 2 : 1;
  uint32_t tmem_cols = 32;
  while (tmem_cols < acc_cols * uint32_t(T * nacc)) tmem_cols <<= 1;
  const int64_t total = int64_t(P.groups) * P.nchunks;
  // The image drain of a CTA's only segment is shared by 12 warps (3 per TMEM
  // lane quadrant: the epilogue warp and two of warps 6..13, free by then).
  const bool extra_drain = P.direct;

  if (threadIdx.x == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->s_empty[s], 1);
    }
    for (int s = 0; s < GS; ++s) {
      mbar_init(&sh->o_full[s], 8);
      mbar_init(&sh->o_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) mbar_init(&sh->tmem_full[a], 1);
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
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();      // the previous call's kernels still use P^T until they complete
  int grp, c0, c1;

  if (warp == 0) {
    // ---------------------------------------------------------------- X tile producer (T tiles per stage)
    if (lane == 0) {
      Ring xr;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      SegIter it(total, P.nchunks);
      while (it.next(grp, c0, c1)) {
        for (int c = c0; c < c1; ++c) {
          if (!spin_or_abort<false>(sh, &sh->s_empty[xr.stage], xr.phase ^ 1u, limit, ctl)) goto producer_done;
          if (inject) {
            inject = 0;                      // test hook: this CTA's first stage never fills
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
      drain_empties(sh, sh->s_empty, xr, XS, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      Ring xr, gr;
      const int nparts = P.r > 256 ? 2 : 1;
      const int npart = P.r / nparts;
      const uint32_t idesc = idesc_bf16(128, uint32_t(npart), 0, 0);
      const uint64_t xdesc0 = smem_desc(smem_addr(x_tiles), 16, 1024, kSw128);
      const uint64_t gdesc0 = smem_desc(smem_addr(g_tiles), 16, 1024, kSw128);
      SegIter it(total, P.nchunks);
      for (int seg = 0; !sh->abort && it.next(grp, c0, c1); ++seg) {
        const int ab = seg & (nacc - 1);
        const uint32_t uphase = uint32_t(seg / nacc) & 1u;
        const uint32_t acc0 = tmem + uint32_t(ab * T) * acc_cols;
        // the accumulators of this set are free once the epilogue has drained them
        for (int t = 0; t < T; ++t)
          if (!wait_or_abort(sh, &sh->tmem_empty[ab * T + t], uphase ^ 1u, limit, ctl)) goto mma_done;
        tc_fence_after();
        for (int c = c0; c < c1; ++c) {
          if (!spin_or_abort<false>(sh, &sh->s_full[xr.stage], xr.phase, limit, ctl)) goto mma_done;
          if (!spin_or_abort<false>(sh, &sh->o_full[gr.stage], gr.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint64_t ad = xdesc0 + uint64_t(uint32_t(xr.stage) * (x_bytes >> 4));
          const uint64_t bd = gdesc0 + uint64_t(uint32_t(gr.stage) * (g_bytes >> 4));
          const uint32_t first = (c == c0) ? 0u : 1u;
          if (T == 2)
            project_chunk_mmas<2, 1>(acc0, acc_cols, uint32_t(npart), ad, bd, idesc, first);
          else if (nparts == 1)
            project_chunk_mmas<1, 1>(acc0, acc_cols, uint32_t(npart), ad, bd, idesc, first);
          else
            project_chunk_mmas<1, 2>(acc0, acc_cols, uint32_t(npart), ad, bd, idesc, first);
          mma_commit(&sh->s_empty[xr.stage]);
          mma_commit(&sh->o_empty[gr.stage]);
          xr.next(XS);
          gr.next(GS);
        }
        mma_commit(&sh->tmem_full[ab]);
      }
    mma_done:
      mma_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- epilogue: TMEM -> P^T (smem + TMA) or image
    const int quad = warp & 3;
    float* stg = reinterpret_cast<float*>(staging + (warp - 2) * 2 * kStageTile);
    int sb = 0;
    SegIter it(total, P.nchunks);
    for (int seg = 0; it.next(grp, c0, c1); ++seg) {
      const int ab = seg & (nacc - 1);
      const uint32_t uphase = uint32_t(seg / nacc) & 1u;
      const bool whole = (c0 == 0 && c1 == P.nchunks);
      if (!warp_wait(sh, &sh->tmem_full[ab], uphase, limit, ctl)) break;
      tc_fence_after();
      if (P.direct) {
        // Whole k range: P^T is final here, so the accumulate's image is written directly.
        // When this is the CTA's only segment, the idle generator warps share the drain
        // (extra_drain).  Only then: they wait on tmem_full with the parity of the segment
        // they drain, which identifies the phase only while no earlier phase is pending.
        SegIter peek = it;
        int g2, d0, d1;
        const bool only = seg == 0 && !peek.next(g2, d0, d1);
        drain_image_blocks(tmem + uint32_t(ab * T) * acc_cols, acc_cols, T, quad, grp, P, image, 0,
                           (only && extra_drain) ? 3 : 1, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          for (int t = 0; t < T; ++t) mbar_arrive(&sh->tmem_empty[ab * T + t]);
        continue;
      }
      for (int t = 0; t < T; ++t) {
        const uint32_t acc = tmem + uint32_t(ab * T + t) * acc_cols;
        const int x0 = (grp * T + t) * kTok + quad * 32;   // first token of this warp's lanes
        for (int c = 0; c < P.r; c += 32) {
          uint32_t v[32];
          tmem_ld32(acc + (uint32_t(quad * 32) << 16) + uint32_t(c), v);
          tmem_ld_wait();
          // staging tile [32 ranks][32 tokens]: lane = token, so each row store is one 128-byte line
          float* tile = stg + sb * (32 * 32);
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[j * 32 + lane] = __uint_as_float(v[j]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (x0 < P.n_pad) {
              if (whole) tma_store_2d(&tmap_p, tile, x0, c);
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
        if (lane == 0) mbar_arrive(&sh->tmem_empty[ab * T + t]);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    if (warp != 9 && warp != 13) {
      // -------------------------------------------------------------- sign-tile generators (8 warps)
      // Warps 9 and 13 stay idle so that no generator shares the MMA warp's
      // scheduler (warp % 4 == 1): the single issuing thread keeps its issue slots.
      const int gtid = (warp - 6 - (warp > 9) - (warp > 13)) * 32 + lane;
      Ring gr;
      SegIter it(total, P.nchunks);
      while (it.next(grp, c0, c1)) {
        for (int c = c0; c < c1; ++c) {
          // polling: a generator that sleeps through the stage's release delays the MMAs
          // (the down projection under the hint 327 -> 309 us)
          if (!warp_spin_wait(sh, &sh->o_empty[gr.stage], gr.phase ^ 1u, limit, ctl)) goto gen_done;
          gen_sigma_kmajor(g_tiles + size_t(gr.stage) * g_bytes, sh->nib, key, P.r, c, gtid, 256);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->o_full[gr.stage]);
          gr.next(GS);
        }
      }
    gen_done:
      // the MMA commits' last arrivals on the sign ring land before the CTA can leave
      if (gtid == 0) drain_empties(sh, sh->o_empty, gr, GS, limit);
    }
    if (extra_drain && warp < 14 && !*reinterpret_cast<volatile int*>(&sh->abort)) {
      // -------------------------------------------------------------- share the final segment's image drain
      SegIter it(total, P.nchunks);
      int nseg = 0, fg = 0;
      while (it.next(grp, c0, c1)) {
        ++nseg;
        fg = grp;
      }
      if (nseg == 1) {              // the CTA's only segment: accumulator set 0, first phase
        const int ab = 0;
        const uint32_t uphase = 0u;
        if (warp_wait(sh, &sh->tmem_full[ab], uphase, limit, ctl)) {
          tc_fence_after();
          drain_image_blocks(tmem + uint32_t(ab * T) * acc_cols, acc_cols, T, warp & 3, fg, P, image,
                             warp < 10 ? 1 : 2, 3, lane);
          tc_fence_before();
        }
      }
    }
  }

  tc_fence_before();
  cta_sync();
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
  grid_dependency_wait();      // P^T comes from the projection just before
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
// A segment is (d tile of N columns, token-chunk range).  When two segments'
// accumulators fit TMEM together (r <= 128), consecutive segments alternate
// between them so the drain of one overlaps the MMAs of the next.
__global__ void __launch_bounds__(352, 1)
    accumulate_tc_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_s,
                         SketchShape sh_, const uint8_t* __restrict__ image, float scale, float4* pzero,
                         int64_t pzero_n, Control* ctl) {
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
  const int nacc = (mblocks * N * 2 <= 512) ? 2 : 1;
  const int nchunks = P.n_pad / kChunk;
  const int64_t total = int64_t(P.dtiles) * nchunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < BS; ++s) {
      mbar_init(&sh->s_full[s], 1);
      mbar_init(&sh->s_empty[s], 1);
    }
    for (int s = 0; s < AS; ++s) {
      mbar_init(&sh->o_full[s], 1);
      mbar_init(&sh->o_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) mbar_init(&sh->tmem_full[a], 1);
    for (int m = 0; m < 4; ++m) mbar_init(&sh->tmem_empty[m], 8);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_dy);
  }
  uint32_t tmem_cols = 32;
  while (tmem_cols < uint32_t(nacc * mblocks * N)) tmem_cols <<= 1;
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();      // the image comes from the split just before, S from earlier calls
  int dt, c0, c1;

  if (warp == 0) {
    // ---------------------------------------------------------------- P^T chunk producer (L2)
    if (lane == 0) {
      Ring ar;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      SegIter it(total, nchunks);
      while (it.next(dt, c0, c1)) {
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort(sh, &sh->o_empty[ar.stage], ar.phase ^ 1u, limit, ctl)) goto a_done;
          if (inject) {
            inject = 0;                      // test hook: this CTA's first stage never fills
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
      drain_empties(sh, sh->o_empty, ar, AS, limit);
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------------- dY tile producer (HBM)
    if (lane == 0) {
      Ring br;
      SegIter it(total, nchunks);
      while (it.next(dt, c0, c1)) {
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
      drain_empties(sh, sh->s_empty, br, BS, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      Ring ar, br;
      const uint32_t idesc = idesc_bf16(128, uint32_t(N), 0, 1);
      const uint64_t adesc0 = smem_desc(smem_addr(a_tiles), 16, 1024, kSw128);
      const uint64_t bdesc0 = smem_desc(smem_addr(b_tiles), kChunk * 128, 1024, kSw128);
      SegIter it(total, nchunks);
      for (int seg = 0; !sh->abort && it.next(dt, c0, c1); ++seg) {
        const int ab = seg & (nacc - 1);
        const uint32_t uphase = uint32_t(seg / nacc) & 1u;
        const uint32_t acc0 = tmem + uint32_t(ab * mblocks * N);
        // the M blocks of this accumulator set are free once the epilogue drained them
        for (int m = 0; m < mblocks; ++m)
          if (!wait_or_abort(sh, &sh->tmem_empty[ab * mblocks + m], uphase ^ 1u, limit, ctl)) goto mma_done;
        tc_fence_after();
        for (int c = c0; c < c1; ++c) {
          if (!spin_or_abort<false>(sh, &sh->o_full[ar.stage], ar.phase, limit, ctl)) goto mma_done;
          if (!spin_or_abort<false>(sh, &sh->s_full[br.stage], br.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint64_t ad = adesc0 + uint64_t(uint32_t(ar.stage) * (a_bytes >> 4));
          const uint64_t bd = bdesc0 + uint64_t(uint32_t(br.stage) * (b_bytes >> 4));
          const uint32_t first = (c == c0) ? 0u : 1u;
          if (mblocks == 1)
            accumulate_chunk_mmas<1>(acc0, uint32_t(N), ad, bd, idesc, first);
          else if (mblocks == 2)
            accumulate_chunk_mmas<2>(acc0, uint32_t(N), ad, bd, idesc, first);
          else
            accumulate_chunk_mmas<4>(acc0, uint32_t(N), ad, bd, idesc, first);
          mma_commit(&sh->o_empty[ar.stage]);
          mma_commit(&sh->s_empty[br.stage]);
          ar.next(AS);
          br.next(BS);
        }
        mma_commit(&sh->tmem_full[ab]);
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
    // The split has consumed this call's P^T: set it back to zero for the next
    // call's projection (its partial segments reduce-add into it) while this
    // warp still waits for its first accumulator.
    if (pzero) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int64_t i = int64_t(blockIdx.x) * 256 + eidx * 32 + lane; i < pzero_n; i += int64_t(gridDim.x) * 256)
        pzero[i] = z;
    }
    SegIter it(total, nchunks);
    for (int seg = 0; it.next(dt, c0, c1); ++seg) {
      const int ab = seg & (nacc - 1);
      const uint32_t uphase = uint32_t(seg / nacc) & 1u;
      if (!warp_wait(sh, &sh->tmem_full[ab], uphase, limit, ctl)) break;
      tc_fence_after();
      for (int m = 0; m < mblocks; ++m) {
        const int r0 = m * 128 + quad * 32;              // first rank of this warp's lanes
        const uint32_t acc = tmem + uint32_t((ab * mblocks + m) * N);
        for (int c = cbeg; c < cend; c += 32) {
          uint32_t v[32];
          tmem_ld32(acc + (uint32_t(quad * 32) << 16) + uint32_t(c), v);
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
        if (lane == 0) mbar_arrive(&sh->tmem_empty[ab * mblocks + m]);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ============================================================================ accumulate on CTA pairs
// For r_pad = 256 or 512.  The MMAs of a pair tile run on two CTAs of a cluster
// (tcgen05 cta_group::2, M = 256 ranks across the pair): each CTA holds only
// its own half of every operand (its 128 ranks of each 256-rank block of the
// P^T chunk, its 128 d-columns of each 256-column block of the dY tile), and
// the hardware hands the B halves across the pair.  A pair tile is
// 256 prb ranks x 256 pdb d-columns with prb * pdb = 2 (1 for narrow matrices on
// one stream), so each CTA's TMEM holds two 128 x 256 fp32 accumulators (one
// when prb * pdb = 1; 512 columns are allocated either way); per 32-token chunk a
// CTA takes in 32 KB (prb 1) or 40 KB (prb 2) of operands for 1024 MMA cycles,
// against 48 KB (r_pad 256) or 72 KB (r_pad 512) on a single CTA, which is
// what limits the single-CTA kernel (operand ingest, not the tensor pipe).
//
// Protocol: the even CTA (leader) issues every MMA.  Both CTAs' producers load
// into their own shared memory and signal the LEADER's full barriers
// (cta_group::2 tensor copies); the leader's producers post the expected bytes
// of both halves.  The leader's commits arrive on both CTAs' empty and
// accumulator-full barriers (multicast); both CTAs' epilogue warps drain their
// own TMEM lanes and arrive on the leader's accumulator-empty barrier.  Every
// wait is bounded; a cluster barrier precedes the first cross-CTA signal and
// the TMEM release, so neither CTA leaves while the other may still use it.
__global__ void __launch_bounds__(352, 1)
    accumulate_pair_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_s,
                           const __grid_constant__ CUtensorMap tmap_img, SketchShape sh_, float scale, float4* pzero,
                           int64_t pzero_n, Control* ctl) {
  extern __shared__ uint8_t smem_raw[];
  const SketchShape& P = sh_;
  uint8_t* base = align1024(smem_raw);
  const int AS = P.a_stages, BS = P.b_stages;
  const int RB = P.prb, DB = P.pdb;
  const uint32_t a_bytes = uint32_t(RB) * 128 * 128;           // 128 ranks per rank block, 32 tokens hi + lo
  const uint32_t b_bytes = uint32_t(DB) * 2 * kChunk * 128;    // 128 d-columns per d block, 32 tokens
  uint8_t* a_tiles = base;
  uint8_t* b_tiles = base + size_t(AS) * a_bytes;
  uint8_t* staging = b_tiles + size_t(BS) * b_bytes;
  Shared* sh = reinterpret_cast<Shared*>(staging + 2 * kStagingBytes);   // two staging tiles per epilogue warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = ctl->wait_limit;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;
  const int pair = int(cluster_id_x()), npairs = int(cluster_count_x());
  const int nchunks = P.n_pad / kChunk;
  const int64_t total = int64_t(P.pdtiles) * nchunks;
  const int pdt = DB * 256;
  constexpr uint32_t kTmemCols = 512;

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
    mbar_init(&sh->tmem_empty[0], 16);     // the 8 epilogue warps of each CTA of the pair
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_dy);
    prefetch_tmap(&tmap_img);
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cta_sync();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();      // the image comes from the split just before, S from earlier calls
  int dt, c0, c1;

  if (warp == 0) {
    // ---------------------------------------------------------------- P^T chunk producer (L2)
    if (lane == 0) {
      Ring ar;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      SegIter it(total, nchunks, pair, npairs);
      while (it.next(dt, c0, c1)) {
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort_cluster(sh, &sh->o_empty[ar.stage], ar.phase ^ 1u, limit, ctl)) goto a_done;
          if (inject) {
            inject = 0;                      // test hook: this pair's first stage never fills
          } else {
            const uint32_t full = mapa_shared(smem_addr(&sh->o_full[ar.stage]), 0);
            if (leader) mbar_arrive_expect_tx(&sh->o_full[ar.stage], 2 * a_bytes);
            for (int rb = 0; rb < RB; ++rb)
              tma_load_2d_pair(a_tiles + size_t(ar.stage) * a_bytes + rb * 16384, &tmap_img, full, 0,
                               c * P.r_pad + rb * 256 + int(cta) * 128);
          }
          ar.next(AS);
        }
      }
    a_done:
      // the peer's copies complete on the leader's barriers: the leader waits for both halves
      if (leader) drain_ring(sh->o_full, ar, AS, limit);
      drain_empties(sh, sh->o_empty, ar, AS, limit);
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------------- dY tile producer (HBM)
    if (lane == 0) {
      Ring br;
      SegIter it(total, nchunks, pair, npairs);
      while (it.next(dt, c0, c1)) {
        for (int c = c0; c < c1; ++c) {
          if (!wait_or_abort_cluster(sh, &sh->s_empty[br.stage], br.phase ^ 1u, limit, ctl)) goto b_done;
          const uint32_t full = mapa_shared(smem_addr(&sh->s_full[br.stage]), 0);
          if (leader) mbar_arrive_expect_tx(&sh->s_full[br.stage], 2 * b_bytes);
          uint8_t* st = b_tiles + size_t(br.stage) * b_bytes;
          for (int db = 0; db < DB; ++db)
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(st + (db * 2 + h) * (kChunk * 128), &tmap_dy, full,
                               dt * pdt + db * 256 + int(cta) * 128 + h * 64, c * kChunk);
          br.next(BS);
        }
      }
    b_done:
      if (leader) drain_ring(sh->s_full, br, BS, limit);
      drain_empties(sh, sh->s_empty, br, BS, limit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader only)
    if (lane == 0 && leader) {
      Ring ar, br;
      const uint32_t idesc = idesc_bf16(256, 256, 0, 1);
      const uint64_t adesc0 = smem_desc(smem_addr(a_tiles), 16, 1024, kSw128);
      const uint64_t bdesc0 = smem_desc(smem_addr(b_tiles), kChunk * 128, 1024, kSw128);
      SegIter it(total, nchunks, pair, npairs);
      for (int seg = 0; !sh->abort && it.next(dt, c0, c1); ++seg) {
        // both CTAs have drained the accumulators of the previous segment
        if (!wait_or_abort_cluster(sh, &sh->tmem_empty[0], (uint32_t(seg) & 1u) ^ 1u, limit, ctl)) goto mma_done;
        tc_fence_after();
        for (int c = c0; c < c1; ++c) {
          if (!spin_or_abort<true>(sh, &sh->o_full[ar.stage], ar.phase, limit, ctl)) goto mma_done;
          if (!spin_or_abort<true>(sh, &sh->s_full[br.stage], br.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint64_t ad = adesc0 + uint64_t(uint32_t(ar.stage) * (a_bytes >> 4));
          const uint64_t bd = bdesc0 + uint64_t(uint32_t(br.stage) * (b_bytes >> 4));
          const uint32_t first = (c == c0) ? 0u : 1u;
          if (RB == 1 && DB == 2)
            accumulate_pair_mmas<1, 2>(tmem, ad, bd, idesc, first);
          else if (RB == 2)
            accumulate_pair_mmas<2, 1>(tmem, ad, bd, idesc, first);
          else
            accumulate_pair_mmas<1, 1>(tmem, ad, bd, idesc, first);
          mma_commit_pair(&sh->o_empty[ar.stage], 3);
          mma_commit_pair(&sh->s_empty[br.stage], 3);
          ar.next(AS);
          br.next(BS);
        }
        mma_commit_pair(&sh->tmem_full[0], 3);
      }
    mma_done:
      mma_commit_pair(&sh->drain, 1);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else if ((warp >= 2 && warp < 6) || (warp >= 7 && warp < 11)) {
    // ---------------------------------------------------------------- epilogue: TMEM -> smem -> TMA reduce-add into S
    // Two groups of four warps cover all four TMEM lane quadrants each; group g
    // drains columns [128 g, 128 g + 128) of both accumulators.
    const int quad = warp & 3;
    const int grp = warp >= 7 ? 1 : 0;
    const int eidx = grp * 4 + (warp - (grp ? 7 : 2));
    float* tile0 = reinterpret_cast<float*>(staging + eidx * 2 * kStageTile);
    int sb = 0;
    const uint32_t empty_leader = mapa_shared(smem_addr(&sh->tmem_empty[0]), 0);
    // the split has consumed this call's P^T: set it back to zero for the next call
    if (pzero) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int64_t i = int64_t(blockIdx.x) * 256 + eidx * 32 + lane; i < pzero_n; i += int64_t(gridDim.x) * 256)
        pzero[i] = z;
    }
    SegIter it(total, nchunks, pair, npairs);
    for (int seg = 0; it.next(dt, c0, c1); ++seg) {
      if (!warp_wait_cluster(sh, &sh->tmem_full[0], uint32_t(seg) & 1u, limit, ctl)) break;
      tc_fence_after();
      for (int a = 0; a < RB * DB; ++a) {
        const int rb = a / DB, db = a - (a / DB) * DB;
        const int r0 = rb * 256 + int(cta) * 128 + quad * 32;     // first rank of this warp's lanes
        for (int c = grp * 128; c < grp * 128 + 128; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + (uint32_t(quad * 32) << 16) + uint32_t(a * 256 + c), v);
          tmem_ld_wait();
          float* tile = tile0 + sb * (32 * 32);
          // staging tile [32 d-rows][32 ranks] = a box of S (d x r, row-major); lane = rank
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[j * 32 + lane] = __uint_as_float(v[j]) * scale;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int64_t d0 = int64_t(dt) * pdt + db * 256 + c;
            if (r0 < P.r && d0 < P.d) tma_reduce_add_2d(&tmap_s, tile, r0, int32_t(d0));
            bulk_commit();
            bulk_wait_read_1();      // the other staging tile is free again
          }
          __syncwarp();
          sb ^= 1;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&sh->tmem_empty[0]);
        else mbar_arrive_cluster(empty_leader);
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cta_sync();
  cluster_sync();              // the leader's MMAs are done with this CTA's memory; no more signals
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ============================================================================ host side
static int ceil_div(int64_t a, int64_t b) { return int((a + b - 1) / b); }

// Stream-K grid for `total` chunks: every SM gets an equal share unless that
// would leave a CTA fewer than `min_chunks` chunks to amortise its drain.
static int stream_k_ctas(int64_t total, int sms, int min_chunks) {
  int64_t g = (total + min_chunks - 1) / min_chunks;
  if (g > sms) g = sms;
  return g < 1 ? 1 : int(g);
}

// The grid for `hint` streams issuing calls at once: longer ranges
// (hint_min_chunks) leave SMs to the other streams and reduce fewer partial
// sums, but a call never drops below its fair share of the SMs (sms / hint)
// unless its one-stream grid is already smaller.
static int stream_k_ctas_hinted(int64_t total, int sms, int min_chunks, int hint_min_chunks, int hint) {
  const int base = stream_k_ctas(total, sms, min_chunks);
  if (hint <= 1) return base;
  const int wide = stream_k_ctas(total, sms, hint_min_chunks);
  const int fair = sms / hint > 1 ? sms / hint : 1;
  const int floor_ctas = base < fair ? base : fair;
  return wide > floor_ctas ? wide : floor_ctas;
}

// A stream-K grid of `base` CTAs over `tiles` tiles of `per` chunks each,
// replaced by tiles * s CTAs (s dividing `per`, as many as fit in `base`) when
// that keeps at least num/den of them: every CTA's range is then 1/s of one
// tile, a single segment with a single drain, instead of straddling two.
static int tile_aligned_ctas(int64_t tiles, int per, int base, int num, int den) {
  int64_t best = 0;
  for (int64_t s = 1; tiles * s <= base && s <= per; ++s)
    if (per % s == 0) best = tiles * s;
  return (best > 0 && best * den >= int64_t(base) * num) ? int(best) : base;
}

// True when some CTA's range starts or ends inside a tile, i.e. some segment
// covers only part of that tile's chunks.
static bool has_partial_segment(int64_t total, int per, int ctas) {
  for (int b = 0; b <= ctas; ++b)
    if ((total * b / ctas) % per != 0) return true;
  return false;
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
  const int64_t ptotal = int64_t(P.groups) * P.nchunks;
  // With calls on several streams, the projection runs on one CTA per token
  // group over the whole k range (no partial sums: plain stores, no reduction
  // at the end) unless that is fewer CTAs than a stream's fair share of the SMs,
  // in which case the groups' k ranges are split evenly over the fair share.
  // The projection then takes a quarter of the SM-time of its all-SM form
  // (most of which is spent on the end-of-kernel L2 reduction of 152 CTAs'
  // partial sums) and leaves the other SMs to the other streams' accumulates:
  // 28-layer 7B step on 8 streams 797.9 -> 825.2 TFLOP/s, as a graph 806 -> 848.
  const int hint = concurrency();
  if (hint > 1) {
    const int fair = sms / hint > 1 ? sms / hint : 1;
    int c = P.groups > fair ? P.groups : fair;
    if (int64_t(c) > ptotal) c = int(ptotal);
    P.proj_ctas = c < sms ? c : sms;
  } else {
    // (ranges of whole fractions of a group's k range when that keeps 80% of the
    // CTAs: one partial-sum drain per CTA)
    P.proj_ctas = tile_aligned_ctas(P.groups, P.nchunks, stream_k_ctas(ptotal, sms, 8), 4, 5);
  }
  P.proj_partial = has_partial_segment(ptotal, P.nchunks, P.proj_ctas) ? 1 : 0;
  P.direct = P.proj_partial ? 0 : 1;
  P.ntile_n = (P.r_pad <= 256) ? 256 : 128;
  P.dtiles = ceil_div(d, P.ntile_n);
  const int tchunks = P.n_pad / kChunk;
  P.pair = (P.r_pad == 256 || P.r_pad == 512) && sms >= 2 ? 1 : 0;
  if (P.pair) {
    P.prb = P.r_pad / 256;
    // Pair tiles are 256 ranks x 512 d-columns (two accumulators per CTA) at
    // r_pad 256, except for narrow matrices (d <= 4096) on one stream, where
    // tiles one d block wide (one accumulator) give twice the tiles to spread
    // over the SMs: one-stream sketch +1.4%.  Under the concurrency hint the
    // wide tiles win (28-layer step 920 against 880 TFLOP/s with narrow ones).
    P.pdb = (P.prb == 1 && hint <= 1 && d <= 4096) ? 1 : 2 / P.prb;
    P.pdtiles = ceil_div(d, P.pdb * 256);
    P.pairs = stream_k_ctas_hinted(int64_t(P.pdtiles) * tchunks, sms / 2, 12, 12 * hint, hint);
    // Prefer a pair count that cuts every tile into equal parts: each pair's
    // range is then one segment, with one drain of its accumulators instead of
    // two.  On one stream only when it keeps 90% of the pairs; under the
    // concurrency hint (SM-time counts) when it keeps half.
    P.pairs = hint > 1 ? tile_aligned_ctas(P.pdtiles, tchunks, P.pairs, 1, 2)
                       : tile_aligned_ctas(P.pdtiles, tchunks, P.pairs, 9, 10);
  }
  // With sketch calls running on several streams at once, each accumulate takes
  // fewer, longer CTA ranges: SMs stay free for the other streams' kernels and
  // fewer partial S tiles are reduced in L2 (4 streams, 27B layers: +1.6% on
  // the step; one stream keeps every SM busy)
  if (P.pair) {
    P.acc_ctas = 2 * P.pairs;
  } else {
    const int base = stream_k_ctas_hinted(int64_t(P.dtiles) * tchunks, sms, 12, 12 * hint, hint);
    P.acc_ctas = hint > 1 ? tile_aligned_ctas(P.dtiles, tchunks, base, 1, 2) : tile_aligned_ctas(P.dtiles, tchunks, base, 9, 10);
  }
  // project: three sign-tile stages when three X stages still fit beside
  // them (the generators then have a whole chunk of MMA time of slack), else
  // two; the rest of shared memory for X tiles
  const int x_bytes = P.tgroup * kTok * 128;
  P.g_stages = (kSmemBudget - kStagingBytes - 3 * r * 128) / x_bytes >= 3 ? 3 : 2;
  P.x_stages = (kSmemBudget - kStagingBytes - P.g_stages * r * 128) / x_bytes;
  if (P.x_stages > kMaxStages) P.x_stages = kMaxStages;
  // accumulate: P^T chunks come from L2 (three stages), dY from HBM (the rest)
  const int a_bytes = P.pair ? P.prb * 128 * 128 : P.r_pad * 128;
  const int b_bytes = P.pair ? P.pdb * 2 * kChunk * 128 : P.ntile_n * kChunk * 2;
  P.a_stages = (P.r_pad >= 512 && !P.pair) ? 2 : 3;
  // (the pair kernel's epilogue warps double-buffer their staging: 64 KB instead of 32;
  // its drains then overlap the TMA reads of one tile with filling the next, +0.7% on the step)
  P.b_stages = (kSmemBudget - (P.pair ? 2 : 1) * kStagingBytes - P.a_stages * a_bytes) / b_bytes;
  if (P.b_stages > kMaxStages) P.b_stages = kMaxStages;
  return P;
}

static int proj_smem_bytes(const SketchShape& P) {
  return 1024 + P.x_stages * P.tgroup * kTok * 128 + P.g_stages * P.r * 128 + kStagingBytes + int(sizeof(Shared));
}

static int acc_smem_bytes(const SketchShape& P) {
  if (P.pair)
    return 1024 + P.a_stages * P.prb * 128 * 128 + P.b_stages * P.pdb * 2 * kChunk * 128 + 2 * kStagingBytes +
           int(sizeof(Shared));
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
                     float scale, float* S, void* ws, ZeroTrack* zt, Control* ctl, cudaStream_t s) {
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
  // Segments with a partial k range reduce-add into P^T, so it starts at zero:
  // each call's accumulate leaves its P^T at zero for the next, and `zt`
  // (null: unknown) says how many leading workspace bytes are zero for
  // certain; only a larger P^T, other use of the workspace, a call that did
  // not complete, or any stream capture on the workspace needs a memset.
  // Nothing is known while these launches are outstanding: `bytes` is set
  // again only once all three have been issued.
  const bool tracked = zt && !zt->captured.load();
  const bool trusted = tracked && zt->trusted() >= part;
  // With every segment covering the whole k range the projection writes the
  // image itself: the fp32 P^T region is left untouched, so what is known to be
  // zero there stays known (up to where the image begins), and no split runs.
  const size_t img_off = (part + 1023) & ~size_t(1023);
  const size_t keep = (P.direct && tracked) ? zt->trusted() : 0;
  if (zt) zt->bytes.store(0);
  if (P.proj_partial && !trusted) LOGRA_CUDA_TRY(cudaMemsetAsync(ppart, 0, part, s));
  LOGRA_CUDA_TRY(launch_overlapped(project_tc_kernel, dim3(P.proj_ctas), dim3(512), size_t(proj_smem), s, tx, tp, P,
                                   key, image, ctl));
  LOGRA_LAUNCHED();

  if (!P.direct) {
    const int64_t stotal = int64_t(P.n_pad / kChunk) * P.r_pad * 4;
    int sblocks = int((stotal + 255) / 256);
    if (sblocks > sms * 8) sblocks = sms * 8;
    LOGRA_CUDA_TRY(launch_overlapped(split_kernel, dim3(sblocks), dim3(256), size_t(0), s,
                                     static_cast<const float*>(ppart), P, image));
    LOGRA_LAUNCHED();
  }

  const int acc_smem = acc_smem_bytes(P);
  float4* pzero = (tracked && !P.direct) ? reinterpret_cast<float4*>(ppart) : nullptr;
  if (P.pair) {
    // the P^T image as a 2-D bf16 tensor of 128-byte rows (r_pad rows per 32-token chunk),
    // already swizzled in memory, loaded in boxes of 128 rows
    CUtensorMap timg;
    if (int st = make_tmap_2d(&timg, image, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64,
                              uint64_t(P.n_pad / kChunk) * uint64_t(P.r_pad), 128, 64, 128,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
      return st;
    LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(accumulate_pair_kernel), acc_smem));
    LOGRA_CUDA_TRY(launch_overlapped_cluster(accumulate_pair_kernel, dim3(P.acc_ctas), dim3(352), size_t(acc_smem), s,
                                             2u, tdy, ts, timg, P, scale, pzero, int64_t(part / 16), ctl));
  } else {
    LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(accumulate_tc_kernel), acc_smem));
    LOGRA_CUDA_TRY(launch_overlapped(accumulate_tc_kernel, dim3(P.acc_ctas), dim3(352), size_t(acc_smem), s, tdy, ts,
                                     P, static_cast<const uint8_t*>(image), scale, pzero, int64_t(part / 16), ctl));
  }
  LOGRA_LAUNCHED();
  // known zero now: this call's P^T region, and nothing past it (the image follows it)
  if (tracked) zt->bytes.store(P.direct ? (keep < img_off ? keep : img_off) : part);
  return LOGRA_OK;
}

}  // namespace logra
