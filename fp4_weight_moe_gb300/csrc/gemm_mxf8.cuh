// MXFP8 activations against MXFP4 weights on the 5th-generation tensor cores
// (sm_103a): D[m][n] = sum_k A[m][k] * W[n][k] with A E4M3 (K-major rows, one
// UE8M0 scale per 32 K-elements) and W E2M1 (K-major packed rows), FP32
// accumulation in tensor memory, tcgen05.mma kind::mxf8f6f4 with
// scale_vec::1X.  No instruction touches a weight nibble: the tensor map
// unpacks the E2M1 rows into the 16-byte-group layout the MMA reads 4-bit
// operands in, and the weights' resident scales (E4M3 powers of two per 16
// elements, both halves of an MXFP4 32-block equal) become the UE8M0 scale
// per 32 that the MMA takes, exactly, on their way into tensor memory.
//
// A persistent CTA (one per SM) computes 128 x BN tiles in turn with ten
// warps:
//   warp 0 lane 0  TMA producer: per 128-K stage the A box (128 rows x 128
//                  B, SWIZZLE_128B), the unpacked W box (BN rows x 128 B)
//                  and the stage's scale chunks (A: one 512 B UE8M0 chunk;
//                  W: the two E4M3 chunks of the stage per 128 rows);
//   warp 1         allocates 512 tensor-memory columns and, converged,
//                  issues four tcgen05.mma (K = 32 each, the scale byte
//                  picked by the scale-factor id) per stage and a commit
//                  that frees the stage;
//   warps 2-5      write each stage's scales into tensor memory (tcgen05.st,
//                  each warp its lane quarter), W's converted to UE8M0;
//   warps 6-9      the epilogue, as in the FP4 engine (two accumulators
//                  alternate between tiles when BN = 128).
// Tensor memory: accumulators from column 0; after them, per ring slot, 4
// columns of A scales and 4 x BN / 128 of W scales.  A 512-byte chunk (128
// rows x 4 scale bytes, byte (r%32)*16 + (r/32)*4 + b) lands in 4 columns:
// lane r%32, column r/32, byte b = the 32-block of the stage, which MMA b of
// the stage selects with its scale-factor id.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

constexpr int kMxBM = 128;
constexpr int kMxBK = 128;  // K elements per stage
constexpr int kMxThreads = 320;

template <int BN>
struct MxCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int kAcc = BN == 256 ? 1 : 2;
  static constexpr uint32_t kStageA = kMxBM * kMxBK;       // 16 KB of E4M3
  static constexpr uint32_t kStageB = BN * kMxBK;          // unpacked E2M1: 128 B per row in shared memory
  static constexpr uint32_t kTxB = BN * kMxBK / 2;         // ... of which the copy counts the packed bytes
  static constexpr uint32_t kStageSFA = kChunkBytes;       // UE8M0
  static constexpr uint32_t kStageSFB = (BN / 128) * 2 * kChunkBytes;  // E4M3, two 64-K chunks per 128 rows
  static constexpr uint32_t kStageBytes = (kStageA + kStageB + kStageSFA + kStageSFB + 1023) / 1024 * 1024;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t kTmemSF = kAcc * BN;  // 256 either way
  static constexpr uint32_t kSFPerSlot = 4 + 4 * (BN / 128);
  static_assert(kTmemSF + kStages * kSFPerSlot <= 512, "tensor memory");
  static_assert((3 * kStages + 4) * 8 + 4 <= 256, "barrier block");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4: A E4M3 (format 0),
// B E2M1 (format 5), both K-major, M x N, UE8M0 scales (bit 23), scale-factor
// ids (the byte of each 32-bit scale column) for B at bits 4-5 and for A at
// bits 29-30.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3_e2m1(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (0u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mxf8_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.u32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Store 4 (8) consecutive b32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// UE8M0 bytes of four E4M3 powers of two (one per byte; 0 -> 0: a flushed
// block, read as 2^-127, which leaves its products below the FP32 sums'
// resolution), without branches: a normal 2^(E - 7) (byte E << 3) gives E +
// 120; a subnormal 2^-9, 2^-8, 2^-7 (bytes 1, 2, 4) gives 118, 119, 120 by a
// byte lookup on its low three bits.
__device__ __forceinline__ uint32_t ue8m0_x4(uint32_t w) {
  const uint32_t hi = (w >> 3) & 0x1F1F1F1Fu;                                 // E per byte
  const uint32_t normal = (((hi + 0x7F7F7F7Fu) & 0x80808080u) >> 7) * 0xFFu;  // 0xFF where E > 0
  const uint32_t sub = w & 0x07070707u;                                       // subnormal code (0 if normal)
  const uint32_t sel = (sub & 0xFu) | ((sub >> 4) & 0xF0u) | ((sub >> 8) & 0xF00u) | ((sub >> 12) & 0xF000u);
  return ((hi + 0x78787878u) & normal) | __byte_perm(0x00777600u, 0x00000078u, sel);
}
// Four UE8M0 scales of one 128-K stage from the E4M3 words of its two 64-K
// chunks (bytes = 16-element blocks; each 32-block takes its first half's).
__device__ __forceinline__ uint32_t ue8m0_word(uint32_t c0, uint32_t c1) {
  return ue8m0_x4(__byte_perm(c0, c1, 0x6420));
}

struct MxTile {
  int m_tile, n_tile;   // tile coordinates (units of 128 A rows, BN W rows)
  int a_row0;           // first A row (multiple of 128)
  int b_row0;           // first W row
  const uint8_t* a_sf;  // A's UE8M0 chunk of stage 0 (one chunk per stage)
  const uint8_t* b_sf0; // W's E4M3 chunk of 64-K group 0, first 128 rows (two groups per stage)
  const uint8_t* b_sf1; // ... second 128 rows (BN = 256)
  bool valid;
};

// Persistent tile loop over [0, n_tiles) (valid tiles form a prefix), one
// global stage counter across tiles; K a multiple of 128.  map_a: E4M3 rows
// as bytes, box 128 rows x 128 B, SWIZZLE_128B; map_w: E2M1 rows unpacked
// (make_e2m1_unpacked_map), box BN rows x 128 elements.  Epilogue functor
// `epi(tmem_row, row_in_tile, tile)` as for gemm_fp4_persistent.  Launch with
// kMxThreads threads and MxCfg<BN>::kSmem bytes of dynamic shared memory.
template <int BN, class TileOf, class Epi>
__device__ __forceinline__ void gemm_mxf8_persistent(const CUtensorMap* map_a, const CUtensorMap* map_w, int K,
                                                     uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                     const Epi& epi) {
  using Cfg = MxCfg<BN>;
  constexpr int S = Cfg::kStages, NA = Cfg::kAcc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* sfready = empty + S;
  uint64_t* done = sfready + S;  // [NA]
  uint64_t* accfree = done + 2;  // [NA]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfree + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= n_tiles || !tile_of((int)blockIdx.x).valid) return;
  const int nk = K / kMxBK;

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
    tma_prefetch_desc(map_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * Cfg::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA; };
  auto stage_sfa = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB; };
  auto stage_sfb = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB + Cfg::kStageSFA; };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        const MxTile t = tile_of(idx);
        if (!t.valid) break;
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % S, round = g / S;
          if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], Cfg::kStageA + Cfg::kTxB + Cfg::kStageSFA + Cfg::kStageSFB);
          tma_load_2d(stage_a(slot), map_a, s * kMxBK, t.a_row0, &full[slot]);
          tma_load_2d(stage_b(slot), map_w, s * kMxBK, t.b_row0, &full[slot]);
          bulk_load(stage_sfa(slot), t.a_sf + (size_t)s * kChunkBytes, kChunkBytes, &full[slot]);
          bulk_load(stage_sfb(slot), t.b_sf0 + (size_t)(2 * s) * kChunkBytes, 2 * kChunkBytes, &full[slot]);
          if (BN == 256)
            bulk_load(stage_sfb(slot) + 2 * kChunkBytes, t.b_sf1 + (size_t)(2 * s) * kChunkBytes, 2 * kChunkBytes,
                      &full[slot]);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!tile_of(idx).valid) break;
      const int ab = it % NA, use = it / NA;
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
        const uint32_t sf_b = sf_a + 4;
        const uint64_t da = smem_desc(smem_u32(stage_a(slot)), 16, 1024, kLayoutSW128);
        const uint64_t db = smem_desc(smem_u32(stage_b(slot)), 16, 1024, kLayoutSW128);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K step of 32 = 32 bytes = 2 descriptor units (both operands)
          mma_mxf8_warp(acc, da + 2 * k, db + 2 * k, idesc_mxf8_e4m3_e2m1(kMxBM, BN, (uint32_t)k), sf_a, sf_b,
                        s > 0 || k > 0);
        mma_commit_warp(&empty[slot]);
      }
      if (ok) mma_commit_warp(&done[ab]);
    }
  } else if (warp < 6) {
    // scales -> tensor memory (this warp's lane quarter), stage by stage
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
        const uint32_t col = tmem + lane_base + Cfg::kTmemSF + slot * Cfg::kSFPerSlot;
        {
          const uint4 u = *reinterpret_cast<const uint4*>(stage_sfa(slot) + lane * 16);
          const uint32_t r[4] = {u.x, u.y, u.z, u.w};
          tmem_st4(col, r);
        }
        uint32_t r[4 * (BN / 128)];
#pragma unroll
        for (int q = 0; q < BN / 128; ++q) {
          const uint8_t* c = stage_sfb(slot) + q * 2 * kChunkBytes;
          const uint4 u0 = *reinterpret_cast<const uint4*>(c + lane * 16);
          const uint4 u1 = *reinterpret_cast<const uint4*>(c + kChunkBytes + lane * 16);
          r[4 * q + 0] = ue8m0_word(u0.x, u1.x);
          r[4 * q + 1] = ue8m0_word(u0.y, u1.y);
          r[4 * q + 2] = ue8m0_word(u0.z, u1.z);
          r[4 * q + 3] = ue8m0_word(u0.w, u1.w);
        }
        if constexpr (BN == 128) {
          const uint32_t rr[4] = {r[0], r[1], r[2], r[3]};
          tmem_st4(col + 4, rr);
        } else {
          const uint32_t rr[8] = {r[0], r[1], r[2], r[3], r[4], r[5], r[6], r[7]};
          tmem_st8(col + 4, rr);
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
      const MxTile t = tile_of(idx);
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
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace moe_fp4
