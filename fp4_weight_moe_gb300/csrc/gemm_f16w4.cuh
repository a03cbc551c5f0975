// FP4 weights against 16-bit activations on the FP16 tensor cores (sm_103a):
// D[m][n] = sum_k A[m][k] * W[n][k], A FP16 (K-major rows), W packed E2M1
// (K-major rows, low nibble = even k) with one E4M3 scale per 16 K-elements
// in the resident 512-byte chunk layout, FP32 accumulation in tensor memory
// (tcgen05.mma kind::f16 with FP16 operands).
//
// The weights are decoded to FP16 in shared memory on the CUDA cores: the
// hardware conversion of an E2M1 pair to FP16 (exact), times the block's
// E4M3 scale in FP16 (exact: the product has at most six significant bits
// and lies in [2^-10, 2688]).  Callers keep A exact in FP16 by scaling each
// BF16 row by a power of two (max |a| in [2^14, 2^15)) and undoing it in the
// epilogue: a BF16 value is then exact in FP16 unless it lies more than
// 2^31 below its row's largest magnitude.
//
// A persistent CTA (one per SM) computes 128 x BN tiles in turn with
// 6 + kHwDecWarps warps:
//   warp 0 lane 0  TMA producer: per 64-K stage the A box (128 rows x 128 B,
//                  SWIZZLE_128B), the raw weight box (BN rows x 32 B) and the
//                  stage's scale chunks (BN / 128 of 512 B) into the load
//                  ring;
//   warp 1         allocates 2 x BN tensor-memory columns (two accumulators)
//                  and, converged, issues four tcgen05.mma kind::f16 (K = 16
//                  each) per stage and commits that free the load stage and
//                  the decoded stage;
//   decode warps   (kHwDecWarps) turn a loaded stage's E2M1 bytes into FP16
//                  weights in the decoded ring, half a row (32 elements, two scale blocks) per
//                  work unit, written in the 128-byte-swizzled K-major layout
//                  the MMA reads: chunk c (8 elements) of row n at
//                  n * 128 + ((c ^ (n % 8)) << 4);
//   4 epilogue warps  each reads its 32 accumulator lanes and hands them to
//                  the epilogue functor; the two accumulators alternate
//                  between tiles, so a tile's epilogue runs beside the next
//                  tile's MMAs.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

constexpr int kHwBM = 128;
constexpr int kHwBK = 64;  // K elements per stage (128 bytes of FP16 per A row)
constexpr int kHwDecWarps = 8;
constexpr int kHwThreads = 32 * (2 + kHwDecWarps + 4);

// Shared memory: a ring of kStages load stages (A box, raw weight box and
// scale chunks, filled by TMA) and a ring of kBStages decoded-weight stages
// (FP16, written by the decode warps), so that the loads run further ahead
// than the decoded weights need to.
template <int BN>
struct HwCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr uint32_t kStageA = kHwBM * kHwBK * 2;  // 16 KB
  static constexpr uint32_t kStageRaw = BN * kHwBK / 2;   // E2M1 bytes as loaded
  static constexpr uint32_t kStageSF = (BN / 128) * kChunkBytes;
  // (each stage starts 1024-byte aligned: the swizzled tiles need it)
  static constexpr uint32_t kStageBytes = (kStageA + kStageRaw + kStageSF + 1023) / 1024 * 1024;
  static constexpr uint32_t kStageB = BN * kHwBK * 2;     // decoded FP16 weights
  static constexpr int kBStages = 3;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kLoadBudget = 227u * 1024u - 1024u - kBarBytes - kBStages * kStageB;
  static constexpr int kStages = kLoadBudget / kStageBytes > 8 ? 8 : (int)(kLoadBudget / kStageBytes);
  static constexpr uint32_t kSmem = kStages * kStageBytes + kBStages * kStageB + 1024 /*align*/ + kBarBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static_assert(kStages >= 3, "load ring depth");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(2 * (kStages + kBStages + 2) * 8 + 4 <= (int)kBarBytes, "barrier block");
};

// Instruction descriptor of tcgen05.mma kind::f16: FP16 A and B (format 0),
// both K-major, FP32 accumulator (format 1), M x N tile.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.u32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// E4M3 scale byte -> FP16 pair (both halves), exact.
__device__ __forceinline__ uint32_t e4m3_scale_f16x2(uint32_t sb) {
  uint32_t s2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"((uint16_t)(sb | (sb << 8))));
  return s2;
}

// Eight E2M1 values (a 32-bit word, element 2i in the low nibble of byte i)
// times the scale pair s2, as four FP16 pairs (element 2i low), exact.
__device__ __forceinline__ uint4 e2m1x8_scaled_f16(uint32_t w, uint32_t s2) {
  uint32_t h[4];
  e2m1x8_to_half2x4(w, h);
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h[i]) : "r"(h[i]), "r"(s2));
  return make_uint4(h[0], h[1], h[2], h[3]);
}

struct HwTile {
  int m_tile, n_tile;   // tile coordinates (units of 128 A rows, BN weight rows)
  int a_row0;           // first A row (multiple of 128)
  int b_row0;           // first weight row (multiple of 128)
  const uint8_t* b_sf0; // scale chunks of the first 128 weight rows (K-group 0)
  const uint8_t* b_sf1; // ... of the second 128 (BN = 256)
  bool valid;
};

// Persistent tile loop over [0, n_tiles) (valid tiles form a prefix), one
// global stage counter across tiles; K a multiple of 64.  map_a: FP16 rows
// as bytes, box 128 rows x 128 B, SWIZZLE_128B; map_w: weight bytes [rows][K
// / 2], box BN rows x 32 B, no swizzle.  Epilogue functor `epi(tmem_row,
// row_in_tile, tile)` as for gemm_fp4_persistent.  Launch with kHwThreads
// threads and HwCfg<BN>::kSmem bytes of dynamic shared memory.
template <int BN, class TileOf, class Epi>
__device__ __forceinline__ void gemm_f16w4_persistent(const CUtensorMap* map_a, const CUtensorMap* map_w, int K,
                                                      uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                      const Epi& epi) {
  using Cfg = HwCfg<BN>;
  constexpr int S = Cfg::kStages, SB = Cfg::kBStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* bring = smem + S * Cfg::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bring + SB * Cfg::kStageB);
  uint64_t* empty = full + S;
  uint64_t* bready = empty + S;  // [SB]
  uint64_t* bfree = bready + SB; // [SB]
  uint64_t* done = bfree + SB;   // [2]
  uint64_t* accfree = done + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfree + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= n_tiles || !tile_of((int)blockIdx.x).valid) return;
  const int nk = K / kHwBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&bready[s], kHwDecWarps);
      mbar_init(&bfree[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&done[b], 1);
      mbar_init(&accfree[b], 4);
    }
    fence_mbar_init();
    tma_prefetch_desc(map_a);
    tma_prefetch_desc(map_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::kTmemCols);
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * Cfg::kStageBytes; };
  auto stage_raw = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA; };
  auto stage_sf = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageRaw; };
  auto stage_b = [&](int s) { return bring + s * Cfg::kStageB; };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        const HwTile t = tile_of(idx);
        if (!t.valid) break;
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % S, round = g / S;
          if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], Cfg::kStageA + Cfg::kStageRaw + Cfg::kStageSF);
          tma_load_2d(stage_a(slot), map_a, s * kHwBK * 2, t.a_row0, &full[slot]);
          tma_load_2d(stage_raw(slot), map_w, s * kHwBK / 2, t.b_row0, &full[slot]);
          bulk_load(stage_sf(slot), t.b_sf0 + (size_t)s * kChunkBytes, kChunkBytes, &full[slot]);
          if (BN == 256) bulk_load(stage_sf(slot) + kChunkBytes, t.b_sf1 + (size_t)s * kChunkBytes, kChunkBytes,
                                   &full[slot]);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    const uint32_t idesc = idesc_f16(kHwBM, BN);
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!tile_of(idx).valid) break;
      const int ab = it & 1, use = it >> 1;
      if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&accfree[ab], (use - 1) & 1, err, 16u))) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(ab * BN);
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % S, round = g / S, bs = g % SB, bround = g / SB;
        // the decode warps arrive on bready only after they saw the stage's
        // TMA complete (full), so bready alone orders the MMAs after both
        (void)round;
        const bool w = mbar_wait(&bready[bs], bround & 1, err, 2u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc(smem_u32(stage_a(slot)), 16, 1024, kLayoutSW128);
        const uint64_t db = smem_desc(smem_u32(stage_b(bs)), 16, 1024, kLayoutSW128);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K step of 16 = 32 bytes = 2 descriptor units
          mma_f16_warp(acc, da + 2 * k, db + 2 * k, idesc, s > 0 || k > 0);
        mma_commit_warp(&empty[slot]);
        mma_commit_warp(&bfree[bs]);
      }
      if (ok) mma_commit_warp(&done[ab]);
    }
  } else if (warp < 2 + kHwDecWarps) {
    // weight decode: work unit u = half a row (n = u / 2, K chunks 4 (u % 2)
    // .. + 3); thread t takes units t, t + 32 kHwDecWarps, ...
    const int t = threadIdx.x - 64;
    int g = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
      if (!tile_of(idx).valid) break;
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % S, round = g / S, bs = g % SB, bround = g / SB;
        bool w = mbar_wait(&full[slot], round & 1, err, 8u);
        if (bround > 0) w = w && mbar_wait(&bfree[bs], (bround - 1) & 1, err, 8u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint8_t* raw = stage_raw(slot);
        const uint8_t* sf = stage_sf(slot);
        uint8_t* dst = stage_b(bs);
#pragma unroll 1
        for (int u = t; u < 2 * BN; u += 32 * kHwDecWarps) {
          const int n = u >> 1, hh = u & 1, q = n >> 7, r = n & 127;
          const uint4 w = *reinterpret_cast<const uint4*>(raw + n * 32 + hh * 16);
          const uint32_t sb = *reinterpret_cast<const uint16_t*>(sf + q * kChunkBytes + (r & 31) * 16 + (r >> 5) * 4 +
                                                                 2 * hh);
          const uint32_t s0 = e4m3_scale_f16x2(sb & 0xFFu), s1 = e4m3_scale_f16x2(sb >> 8);
          uint8_t* row = dst + n * 128;
          const int sw = n & 7, c0 = 4 * hh;
          *reinterpret_cast<uint4*>(row + (((c0 + 0) ^ sw) << 4)) = e2m1x8_scaled_f16(w.x, s0);
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ sw) << 4)) = e2m1x8_scaled_f16(w.y, s0);
          *reinterpret_cast<uint4*>(row + (((c0 + 2) ^ sw) << 4)) = e2m1x8_scaled_f16(w.z, s1);
          *reinterpret_cast<uint4*>(row + (((c0 + 3) ^ sw) << 4)) = e2m1x8_scaled_f16(w.w, s1);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bready[bs]);
      }
    }
  } else {
    // epilogue: every warp reads its 32 lanes (rows) of the tile's accumulator
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;
    int it = 0;
    for (int idx = blockIdx.x; idx < n_tiles; idx += gridDim.x, ++it) {
      const HwTile t = tile_of(idx);
      if (!t.valid) break;
      const int ab = it & 1, use = it >> 1;
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
  if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

}  // namespace moe_fp4
