// Block-scaled FP4 x FP4 GEMM engine of the mid band (sm_103a): the expert
// weights on the MMA's 128-row side (A), an expert's routed rows on its N
// side (B: 16 or 32 rows), one E4M3 scale per 16 K-elements on both sides,
// FP32 accumulation in tensor memory.
//
// Batches of 9 to a few hundred tokens route a handful of rows to each
// expert.  With the routed rows on the 128-row side (the prefill engine,
// gemm_fp4.cuh) every weight stage travels beside 16 KB of mostly padding
// activation rows; here a 256-K slice of a weight tile (16 KB) travels with 2
// or 4 KB of activations.  Short expert dimensions (FC2's K = I = 320 is one
// 512-K stage) would leave a work item with too little to stream per
// accumulator hand-off, so a work item ("tile") multiplies one B tile (the
// <= 32 routed rows of a 32-row routing tile) with `subs` (<= kSwapSubs)
// consecutive 128-row weight tiles: weight tile j accumulates into columns
// [j N, j N + N) of one 128-column accumulator, and the epilogue runs once for
// all of them.
//
// Persistent CTA (one per SM), ten warps as in the prefill engine:
//   warp 0 lane 0  TMA producer: per (weight tile j, 512-K stage) two
//                  128 x 128 B weight boxes, two N x 128 B activation boxes
//                  (SWIZZLE_128B; the second pair only where the stage
//                  reaches past 256 K) and the two operands' scale chunks
//                  (512 B per 64-K group), into a 4-slot ring;
//   warp 1         tensor-memory allocation and, converged, the MMAs (eight
//                  K = 64 per full stage, four from one elected lane at a
//                  time) and the commits;
//   warps 2-5      scale chunks -> tensor memory (tcgen05.st, each warp its
//                  lane quarter); B's 32 rows sit in one 4-byte word of each
//                  lane's 16 bytes of a 128-row chunk (word b_word), which
//                  goes to the first column of its K group;
//   warps 6-9      the epilogue functor, per tile, after its accumulator is
//                  complete; two accumulators alternate between tiles.
// Every wait is bounded (mbar_wait) and reports into *err.
#pragma once

#include "common.cuh"
#include "gemm_fp4.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

constexpr int kSwapMaxN = 32;                    // B rows per tile at most
constexpr int kSwapSubs = 128 / kSwapMaxN;       // weight tiles per tile at most
constexpr int kSwapThreads = 320;

// A stage is 512 K: two 128-byte-wide boxes per operand (each 256 K, 128-byte
// swizzle) and eight 64-K scale groups, so that the MMA warp's per-stage cost
// (barrier wait, fence, commit) is paid once per eight MMAs.
struct SwapCfg {
  static constexpr int kStageK = 512;
  static constexpr uint32_t kBoxA = 128 * 128;                       // 16 KB: 128 rows x 256 K
  static constexpr uint32_t kBoxB = kSwapMaxN * 128;                 // 4 KB: up to 32 rows x 256 K
  static constexpr uint32_t kStageA = 2 * kBoxA;
  static constexpr uint32_t kStageB = 2 * kBoxB;
  static constexpr uint32_t kStageSF = 8 * kChunkBytes;              // 4 KB (A), 4 KB (B)
  static constexpr uint32_t kStageBytes = kStageA + kStageB + 2 * kStageSF;
  static constexpr int kStages = 4;
  static constexpr uint32_t kTmemSF = 2 * 128;                       // after two accumulators
  static constexpr uint32_t kSFPerSlot = 64;                         // 32 A + 32 B columns
  static constexpr uint32_t kExtra = 18 * 1024;                      // epilogue exchange area
  static constexpr uint32_t kSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/ + kExtra;
  static_assert(kStageBytes % 1024 == 0, "swizzled stages stay 1024-byte aligned");
  static_assert(kTmemSF + kStages * kSFPerSlot <= 512, "tensor memory");
  static_assert((3 * kStages + 4) * 8 + 4 <= 256, "barrier block");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct SwapTile {
  int m_tile;            // 32-row routing tile
  int group;             // weight-tile group (of the kernel's group size) within the expert
  int subs;              // weight tiles in this item (1..kSwapSubs), consecutive
  int a_row0;            // first A (weight) row of weight tile 0 of the group
  int b_row0;            // first B (routed) row, a multiple of 32
  int n_rows;            // 16 or 32: B box rows and the MMA's N
  int b_word;            // (b_row0 / 32) % 4: B's word in each lane's 16 chunk bytes
  const uint8_t* a_sf;   // scale chunks of weight tile 0 (K group 0); tile j at + j * a_sf_step
  size_t a_sf_step;
  const uint8_t* b_sf;   // the 128-row scale chunk set holding B's rows (K group 0)
  bool valid;
};

// 32 consecutive FP32 columns of this warp's 32 tensor-memory lanes, without
// waiting: several loads then one swap_tmem_ld_wait().
__device__ __forceinline__ void swap_tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void swap_tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The epilogue's exchange area (SwapCfg::kExtra bytes) behind the ring and
// the engine's barriers.
__device__ __forceinline__ uint8_t* swap_extra_smem() {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  return smem + SwapCfg::kStages * SwapCfg::kStageBytes + 256;
}

// Persistent tile loop: CTA b takes tiles b, b + gridDim.x, ... of [0,
// n_tiles) until tile_of(idx) reports an invalid tile (valid tiles form a
// prefix).  maps_b: two tensor maps of B with boxes of 16 and 32 rows.
// epi(tmem_row, row, tile): once per epilogue thread and tile; weight tile j
// of the group is at column j * n_rows of tmem_row.  K % 64 == 0; a ragged
// last stage multiplies only its valid 64-K groups.  Launch with
// kSwapThreads threads and SwapCfg::kSmem bytes of dynamic shared memory.
template <class TileOf, class Epi>
__device__ __forceinline__ void gemm_fp4_swap_persistent(const CUtensorMap* map_a, const CUtensorMap* maps_b, int K,
                                                         uint32_t* err, int n_tiles, const TileOf& tile_of,
                                                         const Epi& epi) {
  using Cfg = SwapCfg;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* sfready = empty + S;
  uint64_t* done = sfready + S;  // [2]
  uint64_t* accfree = done + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfree + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first tile's fields, read before the ring's TMA traffic starts: read
  // behind it, they held the first MMA back by 1.5 us (stage timestamps)
  const SwapTile t0 = tile_of((int)blockIdx.x);
  if ((int)blockIdx.x >= n_tiles || !t0.valid) return;
  const int nk = (K + Cfg::kStageK - 1) / Cfg::kStageK;
  auto groups = [&](int s) { return s + 1 < nk ? 8 : K / 64 - 8 * (nk - 1); };  // 64-K groups of stage s
  // the tile after idx for this CTA (invalid past the end); its loads are in
  // flight while the current tile is processed
  auto next_of = [&](int idx) {
    SwapTile t;
    t.valid = false;
    if (idx + (int)gridDim.x < n_tiles) t = tile_of(idx + (int)gridDim.x);
    return t;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&done[b], 1);
      mbar_init(&accfree[b], 4);
    }
    fence_mbar_init();
    tma_prefetch_desc(map_a);
    tma_prefetch_desc(maps_b);
    tma_prefetch_desc(maps_b + 1);
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
  auto stage_sfb = [&](int s) { return stage_sfa(s) + Cfg::kStageSF; };

  if (warp == 0) {
    // producer
    if (lane == 0) {
      // the weights stream through L2 once per routing tile
      const uint64_t wpol = l2_evict_first_policy();
      int g = 0;
      bool ok = true;
      SwapTile t = t0;
      for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
        if (!t.valid) break;
        const SwapTile tn = next_of(idx);
        const CUtensorMap* mb = maps_b + (t.n_rows == 32 ? 1 : 0);
        for (int j = 0; ok && j < t.subs; ++j) {
          for (int s = 0; s < nk; ++s, ++g) {
            const int slot = g % S, round = g / S;
            if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1, err, 1u)) {
              ok = false;
              break;
            }
            const int ng = groups(s);
            const uint32_t sfb = (uint32_t)ng * kChunkBytes, boxes = ng > 4 ? 2u : 1u;
            mbar_arrive_expect_tx(&full[slot], boxes * (Cfg::kBoxA + (uint32_t)t.n_rows * 128) + 2 * sfb);
            for (uint32_t h = 0; h < boxes; ++h) {
              tma_load_2d_hint(stage_a(slot) + h * Cfg::kBoxA, map_a, s * 256 + (int)h * 128, t.a_row0 + 128 * j,
                               &full[slot], wpol);
              tma_load_2d(stage_b(slot) + h * Cfg::kBoxB, mb, s * 256 + (int)h * 128, t.b_row0, &full[slot]);
            }
            bulk_load_hint(stage_sfa(slot), t.a_sf + j * t.a_sf_step + (size_t)(8 * s) * kChunkBytes, sfb, &full[slot],
                           wpol);
            bulk_load(stage_sfb(slot), t.b_sf + (size_t)(8 * s) * kChunkBytes, sfb, &full[slot]);
          }
        }
        t = tn;
      }
    }
  } else if (warp == 1) {
    // MMA issuer, converged
    int g = 0, it = 0;
    bool ok = true;
    SwapTile t = t0;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x, ++it) {
      if (!t.valid) break;
      const SwapTile tn = next_of(idx);
      const uint32_t idesc = idesc_mxf4nvf4(128, t.n_rows, false);
      const int ab = it & 1, use = it >> 1;
      // this accumulator's previous tile has been read out
      if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&accfree[ab], (use - 1) & 1, err, 16u))) break;
      tc_fence_after();
      for (int j = 0; ok && j < t.subs; ++j) {
        const uint32_t acc = tmem + (uint32_t)(ab * 128 + j * t.n_rows);
        for (int s = 0; s < nk; ++s, ++g) {
          const int slot = g % S, round = g / S;
          // the scale warps arrive on sfready only after they saw the
          // stage's TMA complete (full), so sfready alone orders the MMAs
          // after both (one wait per stage: measured 4% faster)
          const bool w = mbar_wait(&sfready[slot], round & 1, err, 2u);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // scale columns: A's group k at 4k, B's at 32 + 4k; boxes h = 0, 1
          // hold groups 0-3 and 4-7 (K step of 64 = 32 bytes = 2 descriptor
          // units within a box)
          const uint32_t sf_a = tmem + Cfg::kTmemSF + slot * Cfg::kSFPerSlot, sf_b = sf_a + 32;
          const int ng = groups(s);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k0 = 4 * h;
            if (ng <= k0) break;
            const uint64_t da = smem_desc(smem_u32(stage_a(slot) + h * Cfg::kBoxA), 16, 1024, kLayoutSW128);
            const uint64_t db = smem_desc(smem_u32(stage_b(slot) + h * Cfg::kBoxB), 16, 1024, kLayoutSW128);
            if (ng >= k0 + 4) {
              mma_nvf4_warp_x4(acc, da, db, idesc, sf_a + 4 * k0, sf_b + 4 * k0, 4, s > 0 || h > 0);
            } else {
              for (int k = k0; k < ng; ++k)
                mma_nvf4_warp(acc, da + 2 * (k - k0), db + 2 * (k - k0), idesc, sf_a + 4 * k, sf_b + 4 * k,
                              s > 0 || k > 0);
            }
          }
          mma_commit_warp(&empty[slot]);
        }
      }
      if (ok) mma_commit_warp(&done[ab]);
      t = tn;
    }
  } else if (warp < 6) {
    // scale chunks -> tensor memory (this warp's lane quarter), stage by stage
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int g = 0;
    bool ok = true;
    SwapTile t = t0;
    for (int idx = blockIdx.x; ok && idx < n_tiles; idx += gridDim.x) {
      if (!t.valid) break;
      const SwapTile tn = next_of(idx);
      const int stages = t.subs * nk;
      for (int q = 0; q < stages; ++q, ++g) {
        const int slot = g % S, round = g / S;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], round & 1, err, 8u))) {
          ok = false;
          break;
        }
        const uint32_t col = tmem + lane_base + Cfg::kTmemSF + slot * Cfg::kSFPerSlot;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // K groups 4h .. 4h + 3
          uint32_t r[16], rb[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint8_t* ca = stage_sfa(slot) + (4 * h + k) * kChunkBytes;
            const uint4 u = *reinterpret_cast<const uint4*>(ca + lane * 16);
            r[4 * k] = u.x;
            r[4 * k + 1] = u.y;
            r[4 * k + 2] = u.z;
            r[4 * k + 3] = u.w;
            // B row l of the tile is row 32 b_word + l of the chunk: lane l's
            // word b_word, into the first column of the K group
            const uint8_t* cb = stage_sfb(slot) + (4 * h + k) * kChunkBytes;
            rb[4 * k] = *reinterpret_cast<const uint32_t*>(cb + lane * 16 + 4 * t.b_word);
            rb[4 * k + 1] = 0u;
            rb[4 * k + 2] = 0u;
            rb[4 * k + 3] = 0u;
          }
          tmem_st16(col + 16 * h, r);
          tmem_st16(col + 32 + 16 * h, rb);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[slot]);
      }
      t = tn;
    }
  } else {
    // epilogue: every warp reads its 32 lanes (rows) of the tile's accumulator
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;
    int it = 0;
    for (int idx = blockIdx.x; idx < n_tiles; idx += gridDim.x, ++it) {
      const SwapTile t = it == 0 ? t0 : tile_of(idx);
      if (!t.valid) break;
      const int ab = it & 1, use = it >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&done[ab], use & 1, err, 4u))) break;
      tc_fence_after();
      epi(tmem + lane_base + (uint32_t)(ab * 128), row, t);
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
