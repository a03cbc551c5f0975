// Block-scaled FP4 x FP4 GEMM on the 5th-generation tensor cores (sm_103a):
// D[m][n] = sum_k A[m][k] * B[n][k], A and B packed E2M1 (K-major rows),
// one E4M3 scale per 16 K-elements on both sides, FP32 accumulation in
// tensor memory.
//
// A persistent CTA (one per SM) computes 128 x 256 tiles in turn with six
// warps:
//   warp 0 lane 0  TMA producer: A box 128 rows x 128 B and B box 256 rows x
//                  128 B (SWIZZLE_128B) plus the 512 B scale chunks of the
//                  stage, into a 4-deep shared-memory ring (mbarrier
//                  full/empty pairs);
//   warp 1         allocates 512 tensor-memory columns and, converged (one
//                  elected lane), issues four tcgen05.mma kind::mxf4nvf4
//                  (K = 64 each) per stage and a commit that frees the stage;
//   warps 2-5      copy each stage's scale chunks from shared memory into
//                  tensor memory with tcgen05.st (each warp its own lane
//                  quarter: the 32-row chunks are replicated in all four),
//                  then, once per tile, run the epilogue: each reads its 32
//                  accumulator lanes (tcgen05.ld 32x32b) and hands rows of
//                  FP32 to the epilogue functor.
// The tensor cores accept an MMA about every hundred cycles and a scale copy
// (tcgen05.cp) every seventy to a hundred from one issuing thread, so keeping
// the copies off the MMA warp and issuing from a converged warp lets the
// four MMAs of a stage (about 390 cycles of FP4 work at 128 x 256 x 256)
// keep the tensor pipe busy.
// Tensor memory: columns [0, 256) accumulator; from 256, per ring slot, 16
// columns of A scales (4 K-groups x 4) and 32 of B scales (4 K-groups x 2
// row tiles x 4).  A 512-byte scale chunk (128 rows x 4 K-blocks, byte
// (r%32)*16 + (r/32)*4 + b) lands in 4 columns: lane r%32, column r/32, byte
// b -- the layout the MMA reads for row r.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 256;  // K elements per stage (128 bytes per row)
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kStageA = kGemmBM * kGemmBK / 2;              // 16 KB
constexpr uint32_t kStageB = kGemmBN * kGemmBK / 2;              // 32 KB
constexpr uint32_t kStageSFA = (kGemmBM / 128) * 4 * kChunkBytes;  // 2 KB
constexpr uint32_t kStageSFB = (kGemmBN / 128) * 4 * kChunkBytes;  // 4 KB
constexpr uint32_t kStageBytes = kStageA + kStageB + kStageSFA + kStageSFB;
constexpr uint32_t kGemmSmem = kGemmStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert((3 * kGemmStages + 2) * 8 + 4 <= 256, "barrier block");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSF = 256;
constexpr uint32_t kTmemSFPerSlot = 48;

struct GemmTile {
  int m_tile, n_tile;   // tile coordinates (units of 128 A rows, 256 B rows)
  int a_row0;           // first A row of this tile (multiple of 128)
  int b_row0;           // first B row (multiple of 256)
  const uint8_t* a_sf;  // scale chunks of A's 128-row tile (K-group 0)
  const uint8_t* b_sf0; // scale chunks of B's first 128-row tile (K-group 0)
  const uint8_t* b_sf1; // ... second 128-row tile
  bool valid;
};

// Persistent tile loop.  CTA b computes tiles b, b + gridDim.x, ... of
// [0, n_tiles) until tile_of(idx) reports an invalid tile (valid tiles form
// a prefix of the index range).  One global stage counter runs across tiles,
// so the producer fills the ring with the next tile's stages while the
// current tile's epilogue runs; the MMA warp starts a tile only after the
// epilogue warps have read the previous accumulator out of tensor memory
// (mbarrier accfree).  Tile source: functor `tile_of(idx) -> GemmTile`;
// epilogue: functor `epi(tmem_row, row_in_tile, tile)`, called once per
// epilogue thread and tile, after the tile's accumulator is complete;
// tmem_row addresses this thread's accumulator row (add a column offset and
// read it with tmem_ld32).
template <class TileOf, class Epi>
__device__ __forceinline__ void gemm_fp4_persistent(const CUtensorMap* map_a, const CUtensorMap* map_b, int K,
                                                    uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                    const Epi& epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGemmStages * kStageBytes);
  uint64_t* empty = full + kGemmStages;
  uint64_t* done = empty + kGemmStages;
  uint64_t* accfree = done + 1;
  uint64_t* sfready = accfree + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfready + kGemmStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= n_tiles || !tile_of((int)blockIdx.x).valid) return;
  const int nk = K / kGemmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], 4);
    }
    mbar_init(done, 1);
    mbar_init(accfree, 4);
    fence_mbar_init();
    tma_prefetch_desc(map_a);
    tma_prefetch_desc(map_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * kStageBytes + kStageA; };
  auto stage_sfa = [&](int s) { return smem + s * kStageBytes + kStageA + kStageB; };
  auto stage_sfb = [&](int s) { return smem + s * kStageBytes + kStageA + kStageB + kStageSFA; };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        const GemmTile t = tile_of(idx);
        if (!t.valid) break;
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % kGemmStages, round = g / kGemmStages;
          if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], kStageBytes);
          tma_load_2d(stage_a(slot), map_a, s * (kGemmBK / 2), t.a_row0, &full[slot]);
          tma_load_2d(stage_b(slot), map_b, s * (kGemmBK / 2), t.b_row0, &full[slot]);
          bulk_load(stage_sfa(slot), t.a_sf + (size_t)(4 * s) * kChunkBytes, kStageSFA, &full[slot]);
          bulk_load(stage_sfb(slot), t.b_sf0 + (size_t)(4 * s) * kChunkBytes, kStageSFB / 2, &full[slot]);
          bulk_load(stage_sfb(slot) + kStageSFB / 2, t.b_sf1 + (size_t)(4 * s) * kChunkBytes, kStageSFB / 2,
                    &full[slot]);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    const uint32_t idesc = idesc_mxf4nvf4(kGemmBM, kGemmBN, false);
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!tile_of(idx).valid) break;
      // the previous tile's accumulator has been read out
      if (it > 0 && !__all_sync(0xffffffffu, mbar_wait(accfree, (it - 1) & 1, err, 16u))) break;
      tc_fence_after();
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % kGemmStages, round = g / kGemmStages;
        bool w = mbar_wait(&full[slot], round & 1, err, 2u);
        w = w && mbar_wait(&sfready[slot], round & 1, err, 2u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_a = tmem + kTmemSF + slot * kTmemSFPerSlot;
        const uint32_t sf_b = sf_a + 16;
        const uint64_t da = smem_desc(smem_u32(stage_a(slot)), 16, 1024, kLayoutSW128);
        const uint64_t db = smem_desc(smem_u32(stage_b(slot)), 16, 1024, kLayoutSW128);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K step of 64 = 32 bytes = 2 descriptor units
          mma_nvf4_warp(tmem, da + 2 * k, db + 2 * k, idesc, sf_a + 4 * k, sf_b + 8 * k, s > 0 || k > 0);
        mma_commit_warp(&empty[slot]);
      }
      if (ok) mma_commit_warp(done);
    }
  } else {
    // scale chunks -> tensor memory (this warp's lane quarter), stage by
    // stage, then the tile's epilogue
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      const GemmTile t = tile_of(idx);
      if (!t.valid) break;
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % kGemmStages, round = g / kGemmStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], round & 1, err, 8u))) {
          ok = false;
          break;
        }
        uint32_t r[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 u = *reinterpret_cast<const uint4*>(stage_sfa(slot) + k * kChunkBytes + lane * 16);
          r[4 * k] = u.x;
          r[4 * k + 1] = u.y;
          r[4 * k + 2] = u.z;
          r[4 * k + 3] = u.w;
        }
        const uint32_t col = tmem + lane_base + kTmemSF + slot * kTmemSFPerSlot;
        tmem_st16(col, r);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // B: K-groups 2h, 2h+1, each both row tiles
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int k = 2 * h + kk;
            const uint4 u0 = *reinterpret_cast<const uint4*>(stage_sfb(slot) + k * kChunkBytes + lane * 16);
            const uint4 u1 =
                *reinterpret_cast<const uint4*>(stage_sfb(slot) + kStageSFB / 2 + k * kChunkBytes + lane * 16);
            r[8 * kk] = u0.x;
            r[8 * kk + 1] = u0.y;
            r[8 * kk + 2] = u0.z;
            r[8 * kk + 3] = u0.w;
            r[8 * kk + 4] = u1.x;
            r[8 * kk + 5] = u1.y;
            r[8 * kk + 6] = u1.z;
            r[8 * kk + 7] = u1.w;
          }
          tmem_st16(col + 16 + 16 * h, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[slot]);
      }
      if (!ok) break;
      // epilogue: every warp reads its 32 lanes (rows) of the accumulator
      if (!__all_sync(0xffffffffu, mbar_wait(done, it & 1, err, 4u))) break;
      tc_fence_after();
      epi(tmem + lane_base, row, t);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accfree);
    }
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace moe_fp4
