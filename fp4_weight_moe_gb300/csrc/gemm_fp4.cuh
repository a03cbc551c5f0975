// Block-scaled FP4 x FP4 GEMM on the 5th-generation tensor cores (sm_103a):
// D[m][n] = sum_k A[m][k] * B[n][k], A and B packed E2M1 (K-major rows),
// one E4M3 scale per 16 K-elements on both sides, FP32 accumulation in
// tensor memory.
//
// A persistent CTA (one per SM) computes 128 x BN tiles in turn (BN = 256,
// or 128 with two accumulators) with ten warps:
//   warp 0 lane 0  TMA producer: A box 128 rows x 128 B and B box BN rows x
//                  128 B (SWIZZLE_128B) plus the 512 B scale chunks of the
//                  stage, into a shared-memory ring (mbarrier full/empty);
//   warp 1         allocates 512 tensor-memory columns and, converged (one
//                  elected lane), issues four tcgen05.mma kind::mxf4nvf4
//                  (K = 64 each) per stage and a commit that frees the stage;
//   warps 2-5      copy each stage's scale chunks from shared memory into
//                  tensor memory with tcgen05.st (each warp its own lane
//                  quarter: the 32-row chunks are replicated in all four);
//   warps 6-9      the epilogue: once per tile each reads its 32 accumulator
//                  lanes (tcgen05.ld 32x32b) and hands rows of FP32 to the
//                  epilogue functor.
// The tensor cores accept an MMA about every hundred cycles and a scale copy
// (tcgen05.cp) every seventy to a hundred from one issuing thread, so keeping
// the copies off the MMA warp and issuing from a converged warp lets the
// four MMAs of a stage keep the tensor pipe busy.  With BN = 128 the two
// accumulators alternate between tiles, so a tile's epilogue (FC2's
// reductions into the token accumulator) runs beside the next tile's MMAs.
// Tensor memory: accumulators from column 0 (BN columns each); after them,
// per ring slot, 16 columns of A scales (4 K-groups x 4) and 16 x BN/128 of
// B scales (4 K-groups x BN/128 row tiles x 4).  A 512-byte scale chunk (128
// rows x 4 K-blocks, byte (r%32)*16 + (r/32)*4 + b) lands in 4 columns: lane
// r%32, column r/32, byte b -- the layout the MMA reads for row r.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

// The four K = 64 MMAs of a full 256-K stage from one elected lane of a
// converged warp: A and B descriptors advance by 2 units (32 bytes), the
// scale columns by 4 (A) and sfb_step (B); the first accumulates iff
// `accumulate` (the others always).
__device__ __forceinline__ void mma_nvf4_warp_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa, uint32_t sfb, uint32_t sfb_step, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q, e;\n\tsetp.ne.u32 p, %16, 0;\n\tsetp.eq.u32 q, %16, %16;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %5, %9, [%10], [%13], p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %2, %6, %9, [%11], [%14], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %3, %7, %9, [%12], [%15], q;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %4, %8, %9, [%17], [%18], q;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(a_desc + 2), "l"(a_desc + 4), "l"(a_desc + 6), "l"(b_desc), "l"(b_desc + 2),
        "l"(b_desc + 4), "l"(b_desc + 6), "r"(idesc), "r"(sfa), "r"(sfa + 4), "r"(sfa + 8), "r"(sfb),
        "r"(sfb + sfb_step), "r"(sfb + 2 * sfb_step), "r"(accumulate ? 1u : 0u), "r"(sfa + 12), "r"(sfb + 3 * sfb_step)
      : "memory");
}

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;  // the default tile width (FC1, test GEMM)
constexpr int kGemmBK = 256;  // K elements per stage (128 bytes per row)
constexpr int kGemmThreads = 320;
constexpr uint32_t kTmemCols = 512;

template <int BN>
struct GemmCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int kAcc = BN == 256 ? 1 : 2;                        // accumulator buffers
  static constexpr uint32_t kStageA = kGemmBM * kGemmBK / 2;            // 16 KB
  static constexpr uint32_t kStageB = BN * kGemmBK / 2;                 // 32 or 16 KB
  static constexpr uint32_t kStageSFA = 4 * kChunkBytes;                // 2 KB
  static constexpr uint32_t kStageSFB = (BN / 128) * 4 * kChunkBytes;   // 4 or 2 KB
  static constexpr uint32_t kStageBytes = kStageA + kStageB + kStageSFA + kStageSFB;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t kTmemSF = kAcc * BN;                        // 256 either way
  static constexpr uint32_t kSFPerSlot = 16 + 16 * (BN / 128);
  static_assert(kTmemSF + kStages * kSFPerSlot <= kTmemCols, "tensor memory");
  static_assert((3 * kStages + 4) * 8 + 4 <= 256, "barrier block");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};
constexpr uint32_t kGemmSmem = GemmCfg<256>::kSmem;

struct GemmTile {
  int m_tile, n_tile;   // tile coordinates (units of 128 A rows, BN B rows)
  int a_row0;           // first A row of this tile (multiple of 128)
  int b_row0;           // first B row (multiple of BN)
  const uint8_t* a_sf;  // scale chunks of A's 128-row tile (K-group 0)
  const uint8_t* b_sf0; // scale chunks of B's first 128-row tile (K-group 0)
  const uint8_t* b_sf1; // ... second 128-row tile (BN = 256)
  bool valid;
};

// Persistent tile loop.  CTA b computes tiles b, b + gridDim.x, ... of
// [0, n_tiles) until tile_of(idx) reports an invalid tile (valid tiles form
// a prefix of the index range).  One global stage counter runs across tiles,
// so the producer fills the ring with the next tile's stages while a tile's
// epilogue runs; the MMA warp starts a tile in an accumulator only after the
// epilogue warps have read that accumulator's previous tile out of tensor
// memory (mbarrier accfree).  Tile source: functor `tile_of(idx) ->
// GemmTile`; epilogue: functor `epi(tmem_row, row_in_tile, tile)`, called
// once per epilogue thread and tile, after the tile's accumulator is
// complete; tmem_row addresses this thread's accumulator row (add a column
// offset below BN and read it with tmem_ld32).  K is a multiple of 64; a
// last stage shorter than 256 loads (zero-filled by the tensor maps) and
// multiplies only its valid 64-K groups, and copies only their scale
// chunks.  Launch with kGemmThreads threads and GemmCfg<BN>::kSmem bytes of
// dynamic shared memory.
template <int BN, class TileOf, class Epi>
__device__ __forceinline__ void gemm_fp4_persistent(const CUtensorMap* map_a, const CUtensorMap* map_b, int K,
                                                    uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                    const Epi& epi) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages, NA = Cfg::kAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* sfready = empty + S;
  uint64_t* done = sfready + S;      // [NA]
  uint64_t* accfree = done + 2;      // [NA]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfree + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= n_tiles || !tile_of((int)blockIdx.x).valid) return;
  const int nk = (K + kGemmBK - 1) / kGemmBK;
  // 64-K groups of stage s (4, fewer in a ragged last stage)
  auto groups = [&](int s) { return s + 1 < nk ? 4 : K / 64 - 4 * (nk - 1); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], 4);
    }
    for (int b = 0; b < NA; ++b) {
      mbar_init(&done[b], 1);
      mbar_init(&accfree[b], 4);
    }
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

  auto stage_a = [&](int s) { return smem + s * Cfg::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA; };
  auto stage_sfa = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB; };
  auto stage_sfb = [&](int s) {
    return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB + Cfg::kStageSFA;
  };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      GemmTile t = tile_of(blockIdx.x);
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        if (!t.valid) break;
        // the next tile's parameters load while this tile's stages issue
        GemmTile tn;
        tn.valid = false;
        if (idx + (int)gridDim.x < n_tiles) tn = tile_of(idx + (int)gridDim.x);
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % S, round = g / S;
          if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
            ok = false;
            break;
          }
          const uint32_t sfb = (uint32_t)groups(s) * kChunkBytes;  // scale bytes of one 128-row tile
          mbar_arrive_expect_tx(&full[slot], Cfg::kStageA + Cfg::kStageB + (1 + BN / 128) * sfb);
          tma_load_2d(stage_a(slot), map_a, s * (kGemmBK / 2), t.a_row0, &full[slot]);
          tma_load_2d(stage_b(slot), map_b, s * (kGemmBK / 2), t.b_row0, &full[slot]);
          bulk_load(stage_sfa(slot), t.a_sf + (size_t)(4 * s) * kChunkBytes, sfb, &full[slot]);
          bulk_load(stage_sfb(slot), t.b_sf0 + (size_t)(4 * s) * kChunkBytes, sfb, &full[slot]);
          if (BN == 256)
            bulk_load(stage_sfb(slot) + 4 * kChunkBytes, t.b_sf1 + (size_t)(4 * s) * kChunkBytes, sfb, &full[slot]);
        }
        t = tn;
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    const uint32_t idesc = idesc_mxf4nvf4(kGemmBM, BN, false);
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!tile_of(idx).valid) break;
      const int ab = it % NA, use = it / NA;
      // this accumulator's previous tile has been read out
      if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&accfree[ab], (use - 1) & 1, err, 16u))) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(ab * BN);
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % S, round = g / S;
        // the scale warps arrive on sfready only after they saw the stage's
        // TMA complete (full), so sfready alone orders the MMAs after both
        const bool w = mbar_wait(&sfready[slot], round & 1, err, 2u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sf_a = tmem + Cfg::kTmemSF + slot * Cfg::kSFPerSlot;
        const uint32_t sf_b = sf_a + 16;
        const uint64_t da = smem_desc(smem_u32(stage_a(slot)), 16, 1024, kLayoutSW128);
        const uint64_t db = smem_desc(smem_u32(stage_b(slot)), 16, 1024, kLayoutSW128);
        const int ng = groups(s);
        if (ng == 4) {
          mma_nvf4_warp_x4(acc, da, db, idesc, sf_a, sf_b, 4 * (BN / 128), s > 0);
        } else {
          for (int k = 0; k < ng; ++k)  // K step of 64 = 32 bytes = 2 descriptor units
            mma_nvf4_warp(acc, da + 2 * k, db + 2 * k, idesc, sf_a + 4 * k, sf_b + 4 * (BN / 128) * k,
                          s > 0 || k > 0);
        }
        mma_commit_warp(&empty[slot]);
      }
      if (ok) mma_commit_warp(&done[ab]);
    }
  } else if (warp < 6) {
    // scale chunks -> tensor memory (this warp's lane quarter), stage by stage
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int g = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
      if (!tile_of(idx).valid) break;
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % S, round = g / S;
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
        const uint32_t col = tmem + lane_base + Cfg::kTmemSF + slot * Cfg::kSFPerSlot;
        tmem_st16(col, r);
        if (BN == 128) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 u = *reinterpret_cast<const uint4*>(stage_sfb(slot) + k * kChunkBytes + lane * 16);
            r[4 * k] = u.x;
            r[4 * k + 1] = u.y;
            r[4 * k + 2] = u.z;
            r[4 * k + 3] = u.w;
          }
          tmem_st16(col + 16, r);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // B: K-groups 2h, 2h+1, each both row tiles
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const int k = 2 * h + kk;
              const uint4 u0 = *reinterpret_cast<const uint4*>(stage_sfb(slot) + k * kChunkBytes + lane * 16);
              const uint4 u1 = *reinterpret_cast<const uint4*>(stage_sfb(slot) + 4 * kChunkBytes + k * kChunkBytes +
                                                               lane * 16);
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
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[slot]);
      }
    }
  } else {
    // epilogue: every warp reads its 32 lanes (rows) of the tile's accumulator
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;
    int it = 0;
    for (int idx = blockIdx.x; idx < n_tiles; idx += gridDim.x, ++it) {
      const GemmTile t = tile_of(idx);
      if (!t.valid) break;
      const int ab = it % NA, use = it / NA;
      if (!__all_sync(0xffffffffu, mbar_wait(&done[ab], use & 1, err, 4u))) break;
      tc_fence_after();
      epi(tmem + lane_base + (uint32_t)(ab * BN), row, t);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accfree[ab]);
    }
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace moe_fp4
