// Block-scaled FP4 x FP4 GEMM on the 5th-generation tensor cores (sm_103a):
// D[m][n] = sum_k A[m][k] * B[n][k], A and B packed E2M1 (K-major rows),
// one E4M3 scale per 16 K-elements on both sides, FP32 accumulation in
// tensor memory.
//
// One CTA computes a 128 x 256 tile:
//   warp 0 lane 0  TMA producer: A box 128 rows x 128 B and B box 256 rows x
//                  128 B (SWIZZLE_128B) plus the 512 B scale chunks of the
//                  stage, into a 4-deep shared-memory ring (mbarrier
//                  full/empty pairs);
//   warp 1         allocates 512 tensor-memory columns; lane 0 issues per
//                  stage the scale-factor copies (tcgen05.cp 32x128b.warpx4)
//                  and four tcgen05.mma kind::mxf4nvf4 (K = 64 each), then a
//                  commit that frees the stage;
//   warps 0-3      epilogue: each reads its 32 accumulator lanes
//                  (tcgen05.ld 32x32b) and hands rows of FP32 to the
//                  epilogue functor.
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
constexpr int kGemmThreads = 128;
constexpr uint32_t kStageA = kGemmBM * kGemmBK / 2;              // 16 KB
constexpr uint32_t kStageB = kGemmBN * kGemmBK / 2;              // 32 KB
constexpr uint32_t kStageSFA = (kGemmBM / 128) * 4 * kChunkBytes;  // 2 KB
constexpr uint32_t kStageSFB = (kGemmBN / 128) * 4 * kChunkBytes;  // 4 KB
constexpr uint32_t kStageBytes = kStageA + kStageB + kStageSFA + kStageSFB;
constexpr uint32_t kGemmSmem = kGemmStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSF = 256;
constexpr uint32_t kTmemSFPerSlot = 48;

struct GemmTile {
  int a_row0;        // first A row of this tile (multiple of 128)
  int b_row0;        // first B row (multiple of 256)
  const uint8_t* a_sf;  // scale chunks of A's 128-row tile (K-group 0)
  const uint8_t* b_sf0; // scale chunks of B's first 128-row tile (K-group 0)
  const uint8_t* b_sf1; // ... second 128-row tile
  bool valid;
};

// Generic tile body.  Tile source: functor `tile_of() -> GemmTile`;
// epilogue: functor `epi(tmem_row, row_in_tile, tile)` called once per
// thread after the accumulator is complete; tmem_row addresses this thread's
// accumulator row (add a column offset and read it with tmem_ld32).
template <class TileOf, class Epi>
__device__ __forceinline__ void gemm_fp4_tile(const CUtensorMap* map_a, const CUtensorMap* map_b, int K,
                                              uint32_t* err, const TileOf& tile_of, const Epi& epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGemmStages * kStageBytes);
  uint64_t* empty = full + kGemmStages;
  uint64_t* done = empty + kGemmStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GemmTile t = tile_of();
  if (!t.valid) return;
  const int nk = K / kGemmBK;
  const int KG = K / 64;  // 4-block groups per row (NVFP4: 16-element blocks)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    tma_prefetch_desc(map_a);
    tma_prefetch_desc(map_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * kStageBytes + kStageA; };
  auto stage_sfa = [&](int s) { return smem + s * kStageBytes + kStageA + kStageB; };
  auto stage_sfb = [&](int s) { return smem + s * kStageBytes + kStageA + kStageB + kStageSFA; };

  if (warp == 0 && lane == 0) {
    // producer
    for (int s = 0; s < nk; ++s) {
      const int slot = s % kGemmStages, round = s / kGemmStages;
      if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) break;
      mbar_arrive_expect_tx(&full[slot], kStageBytes);
      tma_load_2d(stage_a(slot), map_a, s * (kGemmBK / 2), t.a_row0, &full[slot]);
      tma_load_2d(stage_b(slot), map_b, s * (kGemmBK / 2), t.b_row0, &full[slot]);
      bulk_load(stage_sfa(slot), t.a_sf + (size_t)(4 * s) * kChunkBytes, kStageSFA, &full[slot]);
      bulk_load(stage_sfb(slot), t.b_sf0 + (size_t)(4 * s) * kChunkBytes, kStageSFB / 2, &full[slot]);
      bulk_load(stage_sfb(slot) + kStageSFB / 2, t.b_sf1 + (size_t)(4 * s) * kChunkBytes, kStageSFB / 2,
                &full[slot]);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_mxf4nvf4(kGemmBM, kGemmBN, false);
    for (int s = 0; s < nk; ++s) {
      const int slot = s % kGemmStages, round = s / kGemmStages;
      if (!mbar_wait(&full[slot], round & 1, err, 2u)) break;
      tc_fence_after();
      const uint32_t sf_a = tmem + kTmemSF + slot * kTmemSFPerSlot;
      const uint32_t sf_b = sf_a + 16;
      const uint32_t sa = smem_u32(stage_sfa(slot)), sb = smem_u32(stage_sfb(slot));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sf_copy(sf_a + 4 * k, smem_desc(sa + k * kChunkBytes, 128, 128, kLayoutNone));
        sf_copy(sf_b + 8 * k, smem_desc(sb + k * kChunkBytes, 128, 128, kLayoutNone));
        sf_copy(sf_b + 8 * k + 4, smem_desc(sb + kStageSFB / 2 + k * kChunkBytes, 128, 128, kLayoutNone));
      }
      const uint32_t a0 = smem_u32(stage_a(slot)), b0 = smem_u32(stage_b(slot));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mma_nvf4(tmem, smem_desc(a0 + 32 * k, 16, 1024, kLayoutSW128), smem_desc(b0 + 32 * k, 16, 1024, kLayoutSW128),
                 idesc, sf_a + 4 * k, sf_b + 8 * k, s > 0 || k > 0);
      }
      mma_commit(&empty[slot]);
    }
    mma_commit(done);
  }
  __syncwarp();

  // epilogue: every warp reads its 32 lanes (rows) of the accumulator
  mbar_wait(done, 0, err, 4u);
  __syncwarp();
  tc_fence_after();
  const int row = (warp & 3) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  epi(tmem + lane_base, row, t);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  (void)KG;
}

}  // namespace moe_fp4
