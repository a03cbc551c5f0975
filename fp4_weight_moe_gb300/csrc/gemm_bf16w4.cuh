// FP4 weights against BF16 activations on the BF16 tensor cores (sm_103a):
// D[m][n] = sum_k A[m][k] * W[n][k], A BF16 (K-major rows), W packed E2M1
// (K-major rows, low nibble = even k) with one E4M3 scale per 16 K-elements
// in the resident 512-byte chunk layout, FP32 accumulation in tensor memory.
// The weights are decoded to BF16 in shared memory on the CUDA cores; every
// product e2m1 x e4m3 has at most six significant bits, so the decoded
// weights are exact in BF16 and the only rounding before the FP32 sums is
// the activations' own (none: they are BF16 already).  This is the exact-
// numerics prefill: no activation quantisation at all.
//
// A persistent CTA (one per SM) computes 128 x BN tiles in turn with ten
// warps:
//   warp 0 lane 0  TMA producer: per 64-K stage the A box (128 rows x 128 B,
//                  SWIZZLE_128B), the raw weight box (BN rows x 32 B) and the
//                  stage's scale chunks (BN / 128 of 512 B) into a ring;
//   warp 1         allocates 2 x BN tensor-memory columns (two accumulators)
//                  and, converged, issues four tcgen05.mma kind::f16 (K = 16
//                  each) per stage and a commit that frees the stage;
//   warps 2-5      decode the stage's weights: E2M1 pairs to f16 (exact), times
//                  the E4M3 block scale in f16 (exact: at most 2 + 4
//                  significant bits, |v| <= 6 * 448), to BF16 (exact), written
//                  in the 128-byte-swizzled K-major layout the MMA reads;
//   warps 6-9      the epilogue: each reads its 32 accumulator lanes and hands
//                  them to the epilogue functor; the two accumulators
//                  alternate between tiles, so a tile's epilogue runs beside
//                  the next tile's MMAs.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

constexpr int kBwBM = 128;
constexpr int kBwBK = 64;  // K elements per stage (128 bytes of BF16 per A row)
constexpr int kBwThreads = 320;

template <int BN>
struct BwCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr uint32_t kStageA = kBwBM * kBwBK * 2;       // 16 KB
  static constexpr uint32_t kStageB = BN * kBwBK * 2;          // decoded BF16 weights
  static constexpr uint32_t kStageRaw = BN * kBwBK / 2;        // E2M1 bytes as loaded
  static constexpr uint32_t kStageSF = (BN / 128) * kChunkBytes;
  // (each stage starts 1024-byte aligned: the swizzled tiles need it)
  static constexpr uint32_t kStageBytes = (kStageA + kStageB + kStageRaw + kStageSF + 1023) / 1024 * 1024;
  static constexpr int kStages = BN == 256 ? 3 : 4;
  static constexpr uint32_t kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Instruction descriptor of tcgen05.mma kind::f16: BF16 A and B, both
// K-major, FP32 accumulator, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.u32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Eight E2M1 values (a 32-bit word, element 2i in the low nibble of byte i)
// times the E4M3 scale `s` (as f16x2, both halves), as eight BF16 values.
__device__ __forceinline__ uint4 e2m1x8_scaled_bf16(uint32_t w, uint32_t s2) {
  uint32_t h[4];
  e2m1x8_to_half2x4(w, h);
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t p;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h[i]), "r"(s2));  // exact (<= 6 significant bits)
    const float2 f = half2_bits_to_float2(p);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);  // exact
    r[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

struct BwTile {
  int m_tile, n_tile;   // tile coordinates (units of 128 A rows, BN weight rows)
  int a_row0;           // first A row (multiple of 128)
  int b_row0;           // first weight row (multiple of 128)
  const uint8_t* b_sf0; // scale chunks of the first 128 weight rows (K-group 0)
  const uint8_t* b_sf1; // ... of the second 128 (BN = 256)
  bool valid;
};

// Persistent tile loop over [0, n_tiles) (valid tiles form a prefix), one
// global stage counter across tiles; K a multiple of 64.  map_a: BF16 rows
// as bytes, box 128 rows x 128 B, SWIZZLE_128B; map_w: weight bytes [rows][K
// / 2], box BN rows x 32 B, no swizzle.  Epilogue functor `epi(tmem_row,
// row_in_tile, tile)` as for gemm_fp4_persistent.  Launch with kBwThreads
// threads and BwCfg<BN>::kSmem bytes of dynamic shared memory.
template <int BN, class TileOf, class Epi>
__device__ __forceinline__ void gemm_bf16w4_persistent(const CUtensorMap* map_a, const CUtensorMap* map_w, int K,
                                                       uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                       const Epi& epi) {
  using Cfg = BwCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* bready = empty + S;
  uint64_t* done = bready + S;  // [2]
  uint64_t* accfree = done + 2; // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfree + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= n_tiles || !tile_of((int)blockIdx.x).valid) return;
  const int nk = K / kBwBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&bready[s], 4);
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
  auto stage_b = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA; };
  auto stage_raw = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB; };
  auto stage_sf = [&](int s) { return smem + s * Cfg::kStageBytes + Cfg::kStageA + Cfg::kStageB + Cfg::kStageRaw; };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        const BwTile t = tile_of(idx);
        if (!t.valid) break;
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % S, round = g / S;
          if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], Cfg::kStageA + Cfg::kStageRaw + Cfg::kStageSF);
          tma_load_2d(stage_a(slot), map_a, s * kBwBK * 2, t.a_row0, &full[slot]);
          tma_load_2d(stage_raw(slot), map_w, s * kBwBK / 2, t.b_row0, &full[slot]);
          bulk_load(stage_sf(slot), t.b_sf0 + (size_t)s * kChunkBytes, kChunkBytes, &full[slot]);
          if (BN == 256) bulk_load(stage_sf(slot) + kChunkBytes, t.b_sf1 + (size_t)s * kChunkBytes, kChunkBytes,
                                   &full[slot]);
        }
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    const uint32_t idesc = idesc_bf16(kBwBM, BN);
    int g = 0, it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!tile_of(idx).valid) break;
      const int ab = it & 1, use = it >> 1;
      if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&accfree[ab], (use - 1) & 1, err, 16u))) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(ab * BN);
      for (int s = 0; s < nk; ++s, ++g) {
        const int slot = g % S, round = g / S;
        bool w = mbar_wait(&full[slot], round & 1, err, 2u);
        w = w && mbar_wait(&bready[slot], round & 1, err, 2u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = smem_desc(smem_u32(stage_a(slot)), 16, 1024, kLayoutSW128);
        const uint64_t db = smem_desc(smem_u32(stage_b(slot)), 16, 1024, kLayoutSW128);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K step of 16 = 32 bytes = 2 descriptor units
          mma_bf16_warp(acc, da + 2 * k, db + 2 * k, idesc, s > 0 || k > 0);
        mma_commit_warp(&empty[slot]);
      }
      if (ok) mma_commit_warp(&done[ab]);
    }
  } else if (warp < 6) {
    // weight decode: thread t handles 16-byte BF16 chunks t, t + 128, ...:
    // row n = chunk / 8, K chunk c = chunk % 8 (8 elements, half an E4M3
    // block), written at the 128-byte-swizzled position of (n, c)
    const int t = threadIdx.x - 64;
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
        const uint8_t* raw = stage_raw(slot);
        const uint8_t* sf = stage_sf(slot);
        uint8_t* dst = stage_b(slot);
#pragma unroll 4
        for (int ch = t; ch < BN * 8; ch += 128) {
          const int n = ch >> 3, c = ch & 7, q = n >> 7, r = n & 127;
          const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + n * 32 + c * 4);
          const uint32_t sb = sf[q * kChunkBytes + (r & 31) * 16 + (r >> 5) * 4 + (c >> 1)];
          uint32_t s2;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"((uint16_t)(sb | (sb << 8))));
          *reinterpret_cast<uint4*>(dst + n * 128 + ((c ^ (n & 7)) << 4)) = e2m1x8_scaled_bf16(w, s2);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bready[slot]);
      }
    }
  } else {
    // epilogue: every warp reads its 32 lanes (rows) of the tile's accumulator
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;
    int it = 0;
    for (int idx = blockIdx.x; idx < n_tiles; idx += gridDim.x, ++it) {
      const BwTile t = tile_of(idx);
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
