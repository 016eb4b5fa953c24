// Input gradient of a Linear layer, dX = dY W (bf16 operands, fp32
// accumulation in TMEM, bf16 result), on CTA pairs with tcgen05 and TMA.
//
// This is the half of a Linear layer's backward pass that LoGRA leaves as it
// is; the other half, the d x k weight gradient dY^T X, is what the method
// never forms: the sketch S += dY^T (X A^T) takes its place (theclarity.today
// write-up, "Why it matters"; academy.dair.ai summary, "Gradient sketches": no
// full gradient buffer is kept).  logra_linear_backward issues both halves.
//
// Pair tile: 256 tokens x 256 k-columns.  M = 256 tokens across the pair (128
// per CTA), N = 256 k-columns (each CTA holds its 128 of them in shared memory;
// the hardware hands the B halves across the pair), K = d in stages of 64:
//   A = dY tile, 128 tokens x 64 d, K-major (d contiguous), 128-byte swizzle;
//   B = W tile, 64 d x 128 k, MN-major (k contiguous): two 64-column boxes.
// Per stage a CTA takes in 32 KB of operands for 512 MMA cycles of the pair.
// Each CTA's TMEM holds two 128 x 256 fp32 accumulators (512 columns): the
// epilogue drains one tile while the MMAs fill the next.  Epilogue: TMEM ->
// registers -> bf16 (round to nearest even) -> shared memory (swizzled) -> TMA
// store; the store clips rows past n and columns past k.  Tiles are taken in
// raster order from a per-stream counter by whichever pair is free; the
// grouped raster lets the pairs at work at one time share dY rows and W
// columns through L2, and pairs that start late, behind other kernels, just
// take fewer tiles.
//
// Roles per CTA (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// (in the even CTA) the MMA issuer, warps 2..5 = epilogue (TMEM lane quadrant
// = warp % 4).  The protocol is the sketch accumulate's: both CTAs' copies
// complete on the leader's full barriers, the leader's commits arrive on both
// CTAs' empty and accumulator-full barriers, both CTAs' epilogue warps arrive
// on the leader's accumulator-empty barriers.  Every wait is bounded.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace logra {

using namespace tc;

namespace {

constexpr int kDgTok = 128;                       // tokens per CTA (pair tile M = 256)
constexpr int kDgCols = 256;                      // k-columns per pair tile (MMA N)
constexpr int kDgK = 64;                          // d per stage
constexpr int kDgABytes = kDgTok * 128;           // 128 tokens x 64 d bf16
constexpr int kDgBBytes = 2 * kDgK * 128;         // 64 d x 128 k bf16, two 64-column boxes
constexpr int kDgStageBytes = kDgABytes + kDgBBytes;
constexpr int kDgMaxStages = 8;
constexpr int kDgOutTile = 32 * 128;              // one bf16 staging tile: 32 tokens x 64 columns
constexpr int kDgStaging = 4 * 4 * kDgOutTile;    // 4 epilogue warps x the 4 column blocks of a tile
constexpr int kDgGroupM = 8;                      // token tiles per raster group
constexpr int kDgSmemBudget = 227 * 1024 - 1024 - 512;

struct DgradShape {
  int64_t n, d, k;
  int mtiles, ntiles, kchunks, stages;
};

// Tile t -> (token tile, column tile), grouped raster: token tiles in groups
// of kDgGroupM, column tiles outer, token tiles inner within a group.  The
// pairs at work at one time (consecutive t) then cover about a square of
// tiles, so the dY rows and W columns they read are shared through L2: a wave
// of 76 tiles (one per pair) reads ~8 token tiles' dY and ~10 column tiles' W
// per d stage instead of one token tile's and all 74 column tiles' (k = 18944).
__device__ __forceinline__ void dgrad_tile(const DgradShape& P, unsigned t, int& mt, int& nt) {
  const unsigned per_group = unsigned(kDgGroupM) * unsigned(P.ntiles);
  const int g = int(t / per_group);
  const int first = g * kDgGroupM;
  const int gsz = P.mtiles - first < kDgGroupM ? P.mtiles - first : kDgGroupM;
  const int local = int(t - unsigned(g) * per_group);
  mt = first + local % gsz;
  nt = local / gsz;
}

// Tile slots between the pair's scheduler and the tile index's readers: the
// leader's MMA thread, the peer's producer, the 4 epilogue warps of each CTA.
constexpr int kDgTileSlots = 4;
constexpr int kDgTileReaders = 1 + 1 + 4 + 4;

struct DgShared {
  uint64_t full[kDgMaxStages], empty[kDgMaxStages];
  uint64_t tmem_full[2], tmem_empty[2], drain;
  uint64_t tile_full[kDgTileSlots], tile_empty[kDgTileSlots];
  int tile_id[kDgTileSlots];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ uint32_t pack_bf16x2_rn(uint32_t a, uint32_t b) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(a)))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(b)))) << 16);
}

}  // namespace

__global__ void __launch_bounds__(192, 1)
    dgrad_pair_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_dx, DgradShape P, unsigned* sched, Control* ctl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  const int NS = P.stages;
  uint8_t* stages = base;
  uint8_t* staging = base + size_t(NS) * kDgStageBytes;
  DgShared* sh = reinterpret_cast<DgShared*>(staging + kDgStaging);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = ctl->wait_limit;
  const uint32_t cta = cluster_ctarank();
  const bool leader = cta == 0;
  const int npairs = int(cluster_count_x());
  const unsigned tiles = unsigned(P.mtiles) * unsigned(P.ntiles);
  constexpr uint32_t kTmemCols = 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tmem_full[a], 1);
      mbar_init(&sh->tmem_empty[a], 8);    // the 4 epilogue warps of each CTA of the pair
    }
    for (int q = 0; q < kDgTileSlots; ++q) {
      mbar_init(&sh->tile_full[q], 1);
      mbar_init(&sh->tile_empty[q], kDgTileReaders);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_dy);
    prefetch_tmap(&tmap_w);
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
  grid_dependency_wait();      // dY and W come from earlier work on the stream

  if (warp == 0) {
    // ---------------------------------------------------------------- tile scheduler + TMA producer
    // The leader's thread takes the pair's next tile from the stream's tile
    // counter and posts its index into both CTAs' tile slots; the peer's
    // producer reads it there.  Pairs that start late (SMs busy with other
    // kernels) simply take fewer tiles.
    if (lane == 0) {
      Ring rg;
      int inject = ctl->inject_fault && blockIdx.x == 0;
      for (int j = 0;; ++j) {
        const int q = j & (kDgTileSlots - 1);
        const uint32_t ph = uint32_t(j / kDgTileSlots) & 1u;
        unsigned t;
        if (leader) {
          if (!wait_or_abort_cluster(sh, &sh->tile_empty[q], ph ^ 1u, limit, ctl)) break;
          t = atomicAdd(&sched[kDgradNextWord], 1u);
          sh->tile_id[q] = int(t < tiles ? t : tiles);
          st_shared_cluster_u32(mapa_shared(smem_addr(&sh->tile_id[q]), 1), t < tiles ? t : tiles);
          mbar_arrive(&sh->tile_full[q]);
          mbar_arrive_cluster(mapa_shared(smem_addr(&sh->tile_full[q]), 1));
        } else {
          if (!wait_or_abort_cluster(sh, &sh->tile_full[q], ph, limit, ctl)) break;
          t = unsigned(*reinterpret_cast<volatile int*>(&sh->tile_id[q]));
          mbar_arrive_cluster(mapa_shared(smem_addr(&sh->tile_empty[q]), 0));
        }
        if (t >= tiles) break;
        int mt, nt;
        dgrad_tile(P, t, mt, nt);
        const int tok0 = mt * (2 * kDgTok) + int(cta) * kDgTok;
        const int col0 = nt * kDgCols + int(cta) * (kDgCols / 2);
        for (int c = 0; c < P.kchunks; ++c) {
          if (!wait_or_abort_cluster(sh, &sh->empty[rg.stage], rg.phase ^ 1u, limit, ctl)) goto p_done;
          if (inject) {
            inject = 0;                      // test hook: the first stage never fills
          } else {
            const uint32_t full = mapa_shared(smem_addr(&sh->full[rg.stage]), 0);
            if (leader) mbar_arrive_expect_tx(&sh->full[rg.stage], 2 * kDgStageBytes);
            uint8_t* st = stages + size_t(rg.stage) * kDgStageBytes;
            tma_load_2d_pair(st, &tmap_dy, full, c * kDgK, tok0);
            tma_load_2d_pair(st + kDgABytes, &tmap_w, full, col0, c * kDgK);
            tma_load_2d_pair(st + kDgABytes + kDgK * 128, &tmap_w, full, col0 + 64, c * kDgK);
          }
          rg.next(NS);
        }
      }
    p_done:
      drain_empties(sh, sh->empty, rg, NS, limit);
      if (leader) {
        drain_ring(sh->full, rg, NS, limit);
        // Every pair has taken its last index from the tile counter before it
        // counts itself finished; the last pair to finish sets both counters
        // back to zero for the next launch on the stream.
        __threadfence();
        if (atomicInc(&sched[kDgradDoneWord], unsigned(npairs - 1)) == unsigned(npairs - 1)) {
          __threadfence();
          atomicExch(&sched[kDgradNextWord], 0u);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader only)
    if (lane == 0 && leader) {
      Ring rg;
      const uint32_t idesc = idesc_bf16(256, kDgCols, 0, 1);
      const uint64_t adesc0 = smem_desc(smem_addr(stages), 16, 1024, kSw128);
      const uint64_t bdesc0 = smem_desc(smem_addr(stages + kDgABytes), kDgK * 128, 1024, kSw128);
      for (int j = 0; !sh->abort; ++j) {
        const int q = j & (kDgTileSlots - 1);
        if (!wait_or_abort(sh, &sh->tile_full[q], uint32_t(j / kDgTileSlots) & 1u, limit, ctl)) goto mma_done;
        const unsigned t = unsigned(*reinterpret_cast<volatile int*>(&sh->tile_id[q]));
        mbar_arrive(&sh->tile_empty[q]);
        if (t >= tiles) break;
        const int acc = j & 1;
        // both CTAs have drained this accumulator's previous tile
        if (!wait_or_abort_cluster(sh, &sh->tmem_empty[acc], (uint32_t(j >> 1) & 1u) ^ 1u, limit, ctl))
          goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(acc * kDgCols);
        for (int c = 0; c < P.kchunks; ++c) {
          if (!spin_or_abort<true>(sh, &sh->full[rg.stage], rg.phase, limit, ctl)) goto mma_done;
          tc_fence_after();
          const uint64_t ad = adesc0 + uint64_t(uint32_t(rg.stage) * (kDgStageBytes >> 4));
          const uint64_t bd = bdesc0 + uint64_t(uint32_t(rg.stage) * (kDgStageBytes >> 4));
#pragma unroll
          for (int ks = 0; ks < kDgK / 16; ++ks)
            mma_bf16_pair(d_tmem, ad + uint64_t(2 * ks), bd + uint64_t(ks * (2048 >> 4)), idesc,
                          (c | ks) ? 1u : 0u);
          mma_commit_pair(&sh->empty[rg.stage], 3);
          rg.next(NS);
        }
        mma_commit_pair(&sh->tmem_full[acc], 3);
      }
    mma_done:
      mma_commit_pair(&sh->drain, 1);
      mbar_wait(&sh->drain, 0, limit);
    }
  } else {
    // ---------------------------------------------------------------- epilogue: TMEM -> bf16 -> smem -> TMA store
    const int quad = warp & 3;
    uint8_t* tile0 = staging + (warp - 2) * 4 * kDgOutTile;
    for (int j = 0;; ++j) {
      const int q = j & (kDgTileSlots - 1);
      if (!warp_wait_cluster(sh, &sh->tile_full[q], uint32_t(j / kDgTileSlots) & 1u, limit, ctl)) break;
      const unsigned t = unsigned(*reinterpret_cast<volatile int*>(&sh->tile_id[q]));
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&sh->tile_empty[q]);
        else mbar_arrive_cluster(mapa_shared(smem_addr(&sh->tile_empty[q]), 0));
      }
      if (t >= tiles) break;
      const int acc = j & 1;
      if (!warp_wait_cluster(sh, &sh->tmem_full[acc], uint32_t(j >> 1) & 1u, limit, ctl)) break;
      tc_fence_after();
      int mt, nt;
      dgrad_tile(P, t, mt, nt);
      const int64_t tok0 = int64_t(mt) * (2 * kDgTok) + int(cta) * kDgTok + quad * 32;
      // the previous tile's stores have long been issued: their staging tiles are free
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      for (int cb = 0; cb < kDgCols / 64; ++cb) {
        uint32_t v0[32], v1[32];
        const uint32_t taddr = tmem + (uint32_t(quad * 32) << 16) + uint32_t(acc * kDgCols + cb * 64);
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 32, v1);
        tmem_ld_wait();
        // this lane's token row: 64 columns = 128 bytes, 16-byte chunk c at c ^ (lane & 7)
        uint8_t* row = tile0 + cb * kDgOutTile + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* v = c < 4 ? v0 : v1;
          const int e = (c & 3) * 8;
          *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16x2_rn(v[e], v[e + 1]), pack_bf16x2_rn(v[e + 2], v[e + 3]),
                         pack_bf16x2_rn(v[e + 4], v[e + 5]), pack_bf16x2_rn(v[e + 6], v[e + 7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int64_t c0 = int64_t(nt) * kDgCols + cb * 64;
          if (tok0 < P.n && c0 < P.k)
            tma_store_2d(&tmap_dx, tile0 + cb * kDgOutTile, int32_t(c0), int32_t(tok0));
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&sh->tmem_empty[acc]);
        else mbar_arrive_cluster(mapa_shared(smem_addr(&sh->tmem_empty[acc]), 0));
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
static DgradShape dgrad_plan(int64_t n, int64_t d, int64_t k) {
  DgradShape P{};
  P.n = n; P.d = d; P.k = k;
  P.mtiles = int((n + 2 * kDgTok - 1) / (2 * kDgTok));
  P.ntiles = int((k + kDgCols - 1) / kDgCols);
  P.kchunks = int((d + kDgK - 1) / kDgK);
  P.stages = (kDgSmemBudget - kDgStaging - int(sizeof(DgShared))) / kDgStageBytes;
  if (P.stages > kDgMaxStages) P.stages = kDgMaxStages;
  return P;
}

static int dgrad_pairs(int64_t tiles, int max_pairs) {
  int pairs = sm_count() / 2;
  if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
  if (int64_t(pairs) > tiles) pairs = int(tiles);
  return pairs < 1 ? 1 : pairs;
}

int launch_dgrad_tc(const void* dY, const void* W, void* dX, int64_t n, int64_t d, int64_t k, int max_pairs,
                    Control* ctl, cudaStream_t s) {
  const DgradShape P = dgrad_plan(n, d, k);
  CUtensorMap tdy, tw, tdx;
  if (int st = make_tmap_2d(&tdy, dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(d), uint64_t(n), uint64_t(d) * 2,
                            kDgK, kDgTok, CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  if (int st = make_tmap_2d(&tw, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(k), uint64_t(d), uint64_t(k) * 2,
                            64, kDgK, CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  if (int st = make_tmap_2d(&tdx, dX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, uint64_t(k), uint64_t(n), uint64_t(k) * 2,
                            64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return st;
  const int64_t tiles = int64_t(P.mtiles) * P.ntiles;
  if (tiles >= (int64_t(1) << 31)) return LOGRA_ERR_UNSUPPORTED;    // 32-bit tile counter
  int st = LOGRA_OK;
  unsigned* sched = stream_counter(s, &st);
  if (!sched) return st;
  const int pairs = dgrad_pairs(tiles, max_pairs);
  const int smem = 1024 + P.stages * kDgStageBytes + kDgStaging + int(sizeof(DgShared));
  LOGRA_CUDA_TRY(ensure_smem(reinterpret_cast<const void*>(dgrad_pair_kernel), smem));
  LOGRA_CUDA_TRY(launch_overlapped_cluster(dgrad_pair_kernel, dim3(2 * pairs), dim3(192), size_t(smem), s, 2u, tdy,
                                           tw, tdx, P, sched, ctl));
  LOGRA_LAUNCHED();
  return LOGRA_OK;
}

}  // namespace logra
