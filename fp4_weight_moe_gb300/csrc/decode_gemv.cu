// Decode band (M <= 8 tokens), streaming-GEMV form of the layer: the routed
// experts' FP4 weights reach shared memory by TMA and are multiplied on the
// CUDA cores, with no reshaping into a tensor-core GEMM.
//
// What it computes is the layer of the tiny-decode PR ("What"): per routed
// token and valid expert, gate/up = x . W13 rows (FP32), h = SiLU(gate) * up,
// y = W2 . h, out = sum over slots of router weight * y (BF16); invalid ids
// contribute exactly zero (W4A16 route PR, invalid-route contract).  Like the
// pages' tiny decode it is two launches, FC1 and FC2, and streams each routed
// weight byte once; unlike it, the weights move by TMA into a shared-memory
// ring (no per-thread global loads), the K reduction of every output row
// stays inside one half-warp (no zero-fill, no atomics), and the output is
// written once per element in a fixed summation order (bitwise
// deterministic).
//
// Work split.  A row quad is the four rows r, r+32, r+64, r+96 of a 128-row
// resident tile: the rows whose scales share one 16-byte line of the tile's
// scale chunk, and (in w13, whose tiles hold 64 gate rows then the 64
// matching up rows) the gate and up rows of the intermediate indices r and
// r+32.  A CTA owns Q = 4 quads (16 rows).  One TMA box of 128 K-bytes x Q
// rows x 4 row blocks brings a stage (256 K) of those rows, a second one
// their 256 scale bytes.  Consumer warp w owns the four rows of quarter
// w % 4 and the stages (items) of parity w / 4; its lane owns two of those
// rows and one 16-element block of each stage (one activation block serves
// both rows), so a row's 16 blocks sit in one half-warp and its K sum is a
// shuffle reduction, then the sum of the two parity warps in fixed order.
//
//   FC1: one CTA per (route slot, w13 tile, quad set); slots naming an
//        expert that an earlier slot names leave at once, so every expert is
//        streamed once for all the tokens routed to it.  The CTA writes h =
//        SiLU(gate*g_gate) * (up*g_up) * (router weight * g_down) for its 8
//        intermediate indices and each routed token.
//   FC2: one CTA per (w2 tile, quad set) over all routed experts; items are
//        (expert, 256-K stage) pairs, h comes in by bulk copies once FC1 is
//        complete, and the CTA writes its 16 output rows of every token.
//
// Inner products: each weight byte becomes a half2 of its two E2M1 values
// (hardware cvt, exact).  FC1 scales x per (token, 256-K stage) by a power of
// two into FP16 (exact for every value above 2^-24 of the stage maximum) and
// accumulates the exact FP16 products in FP32; FC2 takes h in FP32 and the
// weights as FP32 pairs.  Block sums are scaled by the block's E4M3 scale.
#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

CUresult make_u8_map(CUtensorMap* m, const void* base, int rank, const uint64_t* d, const uint64_t* stride,
                     const uint32_t* box, bool swizzle128);

namespace {

constexpr int kGvQ = 4;                    // row quads per CTA
constexpr int kGvRows = 4 * kGvQ;          // rows per CTA
constexpr int kGvNQ = 32 / kGvQ;           // quad sets per 128-row tile
constexpr int kGvWarps = 8;                // consumer warps (warp 0 produces)
constexpr int kGvThreads = 32 * (kGvWarps + 1);
constexpr int kGvRingMax = 16;             // stages in flight
constexpr int kGvStageW = kGvRows * 128;   // weight bytes of one stage (16 rows x 256 K)
constexpr int kGvStageS = 4 * kGvQ * 16;   // their scale bytes
constexpr int kGvMaxSlots = 128;           // M * top_k <= 8 * 16
constexpr int kGvGroup = 68;               // floats per 64-K group of FP32 h in shared memory (64 + pad)
constexpr int kGvGroupH = 72;              // halves per 64-K group of FP16 x in shared memory (64 + pad)
constexpr int kGvSmemLimit = 227 * 1024;
static_assert(kGvWarps == 8 && kGvQ == 4, "warp w: row quarter w % 4, stage parity w / 4; lane: 2 rows x 1 block");

// status bits of the waits that can give up
constexpr uint32_t kErrGvFull = 256u, kErrGvEmpty = 512u, kErrGvH = 1024u;

struct GvArgs {
  const __nv_bfloat16* x;  // [M][H]
  const int32_t* ids;      // [M][top_k], int32 or (ids64) int64
  int ids64;
  const float* tw;         // [M][top_k]
  const uint8_t* s13;      // resident scales + multipliers (for the multipliers)
  const uint8_t* s2;
  float* h;                // [n_slots][M][I/64][kGvGroup]: FC1's output per (owner slot, token)
  __nv_bfloat16* out;      // [M][H]
  uint32_t* status;
  int M, E, H, I, top_k, n_slots, ring;
  ActParams act;           // FC1's gated activation
};

struct GvCtl {
  uint64_t full[kGvRingMax];
  uint64_t empty[kGvRingMax];
  uint64_t hbar;
  int ids[kGvMaxSlots];
  float tw[kGvMaxSlots];
  uint32_t tmask[kGvMaxSlots];  // FC2: tokens routed to the expert first named by slot j
  int own_slot[kGvMaxSlots];    // FC2: owner slots in slot order
  int own_e[kGvMaxSlots];
  uint32_t own_mask[kGvMaxSlots];
  int own_pbase[kGvMaxSlots];   // first (owner, token) pair of each owner
  int pair_src[kGvMaxSlots];    // float offset of each pair's h row
  int n_own, n_pairs;
  int expert, ntok;             // FC1
  int tok[8];
  float wtok[8];
  float g3[3];
};

struct GvLayout {
  int ring_s, ctl, act, red, total;
};

// Shared-memory layout: weight ring (stages at multiples of 2 KB from a
// 1024-byte aligned base, as the 128-byte swizzle wants), scale ring,
// control block, activations [act_bytes], row sums [2 parities][kGvRows][8].
__host__ __device__ inline GvLayout gv_layout(int ring, int act_bytes) {
  GvLayout L;
  L.ring_s = ring * kGvStageW;
  L.ctl = L.ring_s + ring * kGvStageS;
  L.act = (L.ctl + (int)sizeof(GvCtl) + 15) & ~15;
  L.red = (L.act + act_bytes + 15) & ~15;
  L.total = L.red + 2 * kGvRows * 8 * 4 + 1024;  // + alignment slack of the dynamic base
  return L;
}

__device__ __forceinline__ uint8_t* gv_smem_base() {
  extern __shared__ uint8_t gv_smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gv_smem_raw) + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ float gv_ld_f32(const void* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 gv_ld_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// named barrier of the consumer warps only
__device__ __forceinline__ void gv_consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kGvWarps) : "memory"); }

// One row's 16-element block l of a stage: its 8 weight bytes in the
// swizzled box (smem row z*Q + q holds tile row q + 32 z of the quad set) as
// 8 half2, and its E4M3 block scale.
__device__ __forceinline__ float unit_weights(const uint8_t* wst, const uint8_t* sst, int row, int l,
                                              uint32_t (&wh)[8]) {
  const int z = row / kGvQ, q = row % kGvQ, g = l >> 2, b = l & 3;
  const uint2 wv = *reinterpret_cast<const uint2*>(wst + row * 128 + (((l >> 1) ^ (row & 7)) << 4) + ((l & 1) << 3));
  uint32_t t4[4];
  e2m1x8_to_half2x4(wv.x, t4);
  wh[0] = t4[0], wh[1] = t4[1], wh[2] = t4[2], wh[3] = t4[3];
  e2m1x8_to_half2x4(wv.y, t4);
  wh[4] = t4[0], wh[5] = t4[1], wh[6] = t4[2], wh[7] = t4[3];
  return e4m3_to_float(sst[(g * kGvQ + q) * 16 + z * 4 + b]);
}

// sum over 16 elements of w (8 half2) * x (16 FP16 in shared memory):
// exact products accumulated in FP32, two chains.
__device__ __forceinline__ float block_dot_h(const uint32_t (&w)[8], const uint32_t* x) {
  const uint4 a = *reinterpret_cast<const uint4*>(x);
  const uint4 b = *reinterpret_cast<const uint4*>(x + 4);
  const uint32_t xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm("{\n\t.reg .f16 w0, w1, x0, x1;\n\tmov.b32 {w0, w1}, %2;\n\tmov.b32 {x0, x1}, %3;\n\t"
        "fma.rn.f32.f16 %0, w0, x0, %0;\n\tfma.rn.f32.f16 %1, w1, x1, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(w[i]), "r"(xv[i]));
  return s0 + s1;
}

// sum over 16 elements of w (8 half2) * x (16 FP32 in shared memory).
__device__ __forceinline__ float block_dot_f(const uint32_t (&w)[8], const float* x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  const float4 c = *reinterpret_cast<const float4*>(x + 8);
  const float4 d = *reinterpret_cast<const float4*>(x + 12);
  const float xv[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
  float2 p = make_float2(0.f, 0.f), r = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    p = ffma2(half2_bits_to_float2(w[i]), make_float2(xv[2 * i], xv[2 * i + 1]), p);
    r = ffma2(half2_bits_to_float2(w[i + 1]), make_float2(xv[2 * i + 2], xv[2 * i + 3]), r);
  }
  return (p.x + r.x) + (p.y + r.y);
}

// Sum of the 16 lanes of a half-warp (the blocks of one row).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

template <int MT>
__global__ void __launch_bounds__(kGvThreads, 4)
    gemv_fc1_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s, GvArgs a) {
  uint8_t* sm = gv_smem_base();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, M = a.M, n = a.n_slots, ring = a.ring;
  const int tiles1 = I / 64, G = H / 64, S = H / 256;
  const int qs = blockIdx.x % kGvNQ, t = (blockIdx.x / kGvNQ) % tiles1, slot = blockIdx.x / (kGvNQ * tiles1);
  const GvLayout L = gv_layout(ring, M * G * kGvGroupH * 2 + M * S * 4);
  GvCtl& C = *reinterpret_cast<GvCtl*>(sm + L.ctl);
  __half* acth = reinterpret_cast<__half*>(sm + L.act);
  float* xfac = reinterpret_cast<float*>(sm + L.act + M * G * kGvGroupH * 2);
  float* red = reinterpret_cast<float*>(sm + L.red);

  // x and the routing of this call may come from the kernel just before it
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    for (int j = lane; j < n; j += 32) {
      C.ids[j] = route_id(a.ids, j, a.ids64, a.E);
      C.tw[j] = gv_ld_f32(a.tw + j);
    }
    __syncwarp();
    const int e = C.ids[slot];
    const bool valid = e >= 0 && e < a.E;
    bool dup = false;
    for (int j = lane; j < slot; j += 32) dup = dup || C.ids[j] == e;
    const bool own = valid && !__any_sync(0xffffffffu, dup);
    // tokens of the expert in token order; duplicate slots of a token sum
    float w = 0.f;
    bool hit = false;
    if (own && lane < M)
      for (int k = 0; k < a.top_k; ++k) {
        const int j = lane * a.top_k + k;
        if (C.ids[j] == e) {
          w += C.tw[j];
          hit = true;
        }
      }
    const uint32_t hm = __ballot_sync(0xffffffffu, hit);
    if (hit) {
      const int i = __popc(hm & ((1u << lane) - 1u));
      C.tok[i] = lane;
      C.wtok[i] = w;
    }
    if (lane == 0) {
      C.expert = own ? e : -1;
      C.ntok = __popc(hm);
    }
    if (own && lane < 3) {
      const float* gl13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * tiles1 * (H / 64) * kChunkBytes);
      const float* gl2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * (H / 128) * (I / 64) * kChunkBytes);
      C.g3[lane] = gv_ld_f32(lane < 2 ? gl13 + 2 * e + lane : gl2 + e);
    }
    if (own && lane == 0) {
      for (int b = 0; b < ring; ++b) {
        mbar_init(&C.full[b], 1);
        mbar_init(&C.empty[b], kGvWarps / 2);  // the four warps of the stage's parity
      }
      fence_mbar_init();
      const int zw = e * (2 * I / 32) + 4 * t;
      const int zs = (e * tiles1 + t) * G;
      for (int s = 0; s < S && s < ring; ++s) {
        mbar_arrive_expect_tx(&C.full[s], kGvStageW + kGvStageS);
        tma_load_3d(sm + s * kGvStageW, &map_w, 128 * s, qs * kGvQ, zw, &C.full[s]);
        tma_load_3d(sm + L.ring_s + s * kGvStageS, &map_s, 0, qs * kGvQ, zs + 4 * s, &C.full[s]);
      }
    }
  }
  __syncthreads();
  if (C.expert < 0) return;
  const int e = C.expert, ntok = C.ntok;

  if (warp == 0) {
    if (lane == 0) {
      const int zw = e * (2 * I / 32) + 4 * t;
      const int zs = (e * tiles1 + t) * G;
      for (int s = ring; s < S; ++s) {
        const int b = s % ring;
        if (!mbar_wait(&C.empty[b], ((s / ring) - 1) & 1, a.status, kErrGvEmpty)) break;
        mbar_arrive_expect_tx(&C.full[b], kGvStageW + kGvStageS);
        tma_load_3d(sm + b * kGvStageW, &map_w, 128 * s, qs * kGvQ, zw, &C.full[b]);
        tma_load_3d(sm + L.ring_s + b * kGvStageS, &map_s, 0, qs * kGvQ, zs + 4 * s, &C.full[b]);
      }
    }
    return;
  }

  // consumers: x of the expert's tokens as FP16 scaled by a power of two per
  // (token, 256-K stage) so that the stage's largest value lies in [1, 2):
  // [token][64-K group][kGvGroupH] halves, and the factors [token][stage]
  const int ct = threadIdx.x - 32;
  const int n8 = H / 8;
  for (int v = ct; v < ntok * n8; v += 32 * kGvWarps) {  // a warp covers one stage of one token
    const int i = v / n8, k = (v % n8) * 8;
    const uint4 u = gv_ld_v4(a.x + (size_t)C.tok[i] * H + k);
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
    float f[8];
    float mx = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      f[2 * c] = __uint_as_float(wv[c] << 16);
      f[2 * c + 1] = __uint_as_float(wv[c] & 0xffff0000u);
      mx = fmaxf(mx, fmaxf(fabsf(f[2 * c]), fabsf(f[2 * c + 1])));
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    // 2^-e with e = floor(log2(amax)) (0 for a zero stage): exact scaling
    const int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xff) - 127 : 0;
    const float down = __uint_as_float((uint32_t)(127 - ex) << 23);
    uint32_t hv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __half2 h2 = __floats2half2_rn(f[2 * c] * down, f[2 * c + 1] * down);
      hv[c] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(acth + (i * G + k / 64) * kGvGroupH + k % 64) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    if (lane == 0) xfac[i * S + k / 256] = __uint_as_float((uint32_t)(127 + ex) << 23);
  }
  gv_consumer_sync();

  // warp: row quarter rq (smem rows 4 rq .. 4 rq + 3) and stage parity sp;
  // lane: block l of each of its stages for rows row0 and row0 + 1
  const int cw = warp - 1, rq = cw & 3, sp = cw >> 2, l = lane & 15;
  const int row0 = 4 * rq + 2 * (lane >> 4), g = l >> 2, blk = l & 3;
  float acc[2][MT];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[j][m] = 0.f;
  for (int s = sp; s < S; s += 2) {
    const int b = s % ring;
    if (!mbar_wait(&C.full[b], (s / ring) & 1, a.status, kErrGvFull)) break;
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(acth + (4 * s + g) * kGvGroupH + 16 * blk);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t wh[8];
      const float sc = unit_weights(sm + b * kGvStageW, sm + L.ring_s + b * kGvStageS, row0 + j, l, wh);
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < ntok)
          acc[j][m] = fmaf(block_dot_h(wh, xs + m * G * (kGvGroupH / 2)), sc * xfac[m * S + s], acc[j][m]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.empty[b]);
  }
  // row sums over the half-warp's 16 blocks, per stage parity
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float v = half_warp_sum(acc[j][m]);
      if (l == 0 && m < ntok) red[(sp * kGvRows + row0 + j) * 8 + m] = v;
    }
  gv_consumer_sync();
  // h of the CTA's 2Q intermediate indices: row z*Q + q is tile row q' + 32 z
  // (q' = quad line), z = 0/1 gate of index q' / q' + 32, z = 2/3 their up
  if (ct < 2 * kGvQ * ntok) {
    const int i = ct % ntok, p = (ct / ntok) & 1, q = ct / (2 * ntok);
    const int rg = p * kGvQ + q, ru = (2 + p) * kGvQ + q;
    const float gate = red[rg * 8 + i] + red[(kGvRows + rg) * 8 + i];
    const float up = red[ru * 8 + i] + red[(kGvRows + ru) * 8 + i];
    const int ni = 64 * t + qs * kGvQ + q + 32 * p;
    const float hv = gated_act(gate * C.g3[0], up * C.g3[1], a.act) * (C.wtok[i] * C.g3[2]);
    a.h[(((size_t)slot * M + C.tok[i]) * (I / 64) + ni / 64) * kGvGroup + ni % 64] = hv;
  }
}

template <int MT>
__global__ void __launch_bounds__(kGvThreads, 4)
    gemv_fc2_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s, GvArgs a) {
  uint8_t* sm = gv_smem_base();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, M = a.M, n = a.n_slots, ring = a.ring;
  const int tiles2 = H / 128, G = I / 64, S2 = (I + 255) / 256;
  const int qs = blockIdx.x % kGvNQ, t = blockIdx.x / kGvNQ;
  const GvLayout L = gv_layout(ring, n * G * kGvGroup * 4);
  GvCtl& C = *reinterpret_cast<GvCtl*>(sm + L.ctl);
  float* act = reinterpret_cast<float*>(sm + L.act);
  float* red = reinterpret_cast<float*>(sm + L.red);

  // the next kernel waits for this grid before it reads or writes anything
  pdl_launch_dependents();

  if (warp == 0) {
    // The routing is stable for the whole call (FC1 waited for its
    // producer), so the weight stream starts before FC1 is done.
    for (int j = lane; j < kGvMaxSlots; j += 32) {
      C.ids[j] = j < n ? route_id(a.ids, j, a.ids64, a.E) : -1;
      C.tmask[j] = 0u;
    }
    __syncwarp();
    int base = 0;
    for (int c = 0; c < (n + 31) / 32; ++c) {
      const int j = 32 * c + lane;
      const int id = C.ids[j];
      const bool valid = j < n && id >= 0 && id < a.E;
      const uint32_t mm = __match_any_sync(0xffffffffu, valid ? id : -1 - lane);
      int first = 32 * c + __ffs(mm) - 1;
      for (int jj = 0; valid && jj < 32 * c; ++jj)
        if (C.ids[jj] == id) {
          first = jj;
          break;
        }
      if (valid) atomicOr(&C.tmask[first], 1u << (j / a.top_k));
      const bool own = valid && first == j;
      const uint32_t bal = __ballot_sync(0xffffffffu, own);
      if (own) {
        const int u = base + __popc(bal & ((1u << lane) - 1u));
        C.own_slot[u] = j;
        C.own_e[u] = id;
      }
      base += __popc(bal);
    }
    __syncwarp();
    // (owner, token) pairs in owner order, tokens ascending
    int pb = 0;
    for (int u0 = 0; u0 < base; u0 += 32) {
      const int u = u0 + lane;
      const uint32_t mk = u < base ? C.tmask[C.own_slot[u]] : 0u;
      const int cnt = __popc(mk);
      int incl = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      if (u < base) {
        const int p0 = pb + incl - cnt;
        C.own_mask[u] = mk;
        C.own_pbase[u] = p0;
        uint32_t r = mk;
        for (int i = 0; r; ++i) {
          const int m = __ffs(r) - 1;
          r &= r - 1u;
          C.pair_src[p0 + i] = ((C.own_slot[u] * M + m) * G) * kGvGroup;
        }
      }
      pb += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      C.n_own = base;
      C.n_pairs = pb;
      for (int b = 0; b < ring; ++b) {
        mbar_init(&C.full[b], 1);
        mbar_init(&C.empty[b], kGvWarps / 2);  // the four warps of the item's parity
      }
      mbar_init(&C.hbar, 1);
      fence_mbar_init();
      const int items = base * S2;
      for (int i = 0; i < items && i < ring; ++i) {
        const int e = C.own_e[i / S2], s = i % S2;
        mbar_arrive_expect_tx(&C.full[i], kGvStageW + kGvStageS);
        tma_load_3d(sm + i * kGvStageW, &map_w, 128 * s, qs * kGvQ, e * (H / 32) + 4 * t, &C.full[i]);
        tma_load_3d(sm + L.ring_s + i * kGvStageS, &map_s, 0, qs * kGvQ, (e * tiles2 + t) * G + 4 * s, &C.full[i]);
      }
    }
  }
  __syncthreads();
  const int n_own = C.n_own, n_items = n_own * S2;

  if (warp == 0) {
    // h of every (owner, token) pair, once FC1 is complete
    pdl_wait();
    if (lane == 0) mbar_arrive_expect_tx(&C.hbar, (uint32_t)(C.n_pairs * G * kGvGroup * 4));
    __syncwarp();
    for (int p = lane; p < C.n_pairs; p += 32)
      bulk_load(act + p * G * kGvGroup, a.h + C.pair_src[p], (uint32_t)(G * kGvGroup * 4), &C.hbar);
    if (lane == 0) {
      for (int i = ring; i < n_items; ++i) {
        const int b = i % ring, e = C.own_e[i / S2], s = i % S2;
        if (!mbar_wait(&C.empty[b], ((i / ring) - 1) & 1, a.status, kErrGvEmpty)) break;
        mbar_arrive_expect_tx(&C.full[b], kGvStageW + kGvStageS);
        tma_load_3d(sm + b * kGvStageW, &map_w, 128 * s, qs * kGvQ, e * (H / 32) + 4 * t, &C.full[b]);
        tma_load_3d(sm + L.ring_s + b * kGvStageS, &map_s, 0, qs * kGvQ, (e * tiles2 + t) * G + 4 * s, &C.full[b]);
      }
    }
    return;
  }

  const int ct = threadIdx.x - 32;
  const int cw = warp - 1, rq = cw & 3, ip = cw >> 2, l = lane & 15;
  const int row0 = 4 * rq + 2 * (lane >> 4), g = l >> 2, blk = l & 3;
  float acc[2][MT];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[j][m] = 0.f;
  const bool h_ok = mbar_wait(&C.hbar, 0, a.status, kErrGvH);
  for (int i = ip; h_ok && i < n_items; i += 2) {
    const int b = i % ring, u = i / S2, s = i % S2;
    if (!mbar_wait(&C.full[b], (i / ring) & 1, a.status, kErrGvFull)) break;
    if (4 * s + g < G) {  // the last stage of a ragged I holds fewer groups
      const uint32_t mk = C.own_mask[u];
      const float* hs = act + (C.own_pbase[u] * G + 4 * s + g) * kGvGroup + 16 * blk;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t wh[8];
        const float sc = unit_weights(sm + b * kGvStageW, sm + L.ring_s + b * kGvStageS, row0 + j, l, wh);
        int p = 0;
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if ((mk >> m) & 1u) {
            acc[j][m] = fmaf(block_dot_f(wh, hs + p * G * kGvGroup), sc, acc[j][m]);
            ++p;
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.empty[b]);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float v = half_warp_sum(acc[j][m]);
      if (l == 0 && m < M) red[(ip * kGvRows + row0 + j) * 8 + m] = v;
    }
  gv_consumer_sync();
  // output rows: row z*Q + q is w2 tile row q' + 32 z (q' = quad line)
  for (int v = ct; v < kGvRows * M; v += 32 * kGvWarps) {
    const int m = v % M, r = v / M, z = r / kGvQ, q = r % kGvQ;
    a.out[(size_t)m * H + 128 * t + 32 * z + qs * kGvQ + q] =
        __float2bfloat16_rn(red[r * 8 + m] + red[(kGvRows + r) * 8 + m]);
  }
}

int gv_mt(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

int gv_ring1(int H) { return H / 256 < kGvRingMax ? H / 256 : kGvRingMax; }
int gv_ring2(int n_slots, int I) {
  const int items = n_slots * ((I + 255) / 256);
  return items < kGvRingMax ? (items < 1 ? 1 : items) : kGvRingMax;
}
int gv_smem1(int M, int H) {
  return gv_layout(gv_ring1(H), M * (H / 64) * kGvGroupH * 2 + M * (H / 256) * 4).total;
}
int gv_smem2(int M, int I, int top_k) { return gv_layout(gv_ring2(M * top_k, I), M * top_k * (I / 64) * kGvGroup * 4).total; }

template <int MT>
cudaError_t gv_set_attrs() {
  cudaError_t e = cudaFuncSetAttribute(gemv_fc1_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGvSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_fc2_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGvSmemLimit);
  return e;
}

template <int MT>
cudaError_t gv_launch(const CUtensorMap& w13m, const CUtensorMap& s13m, const CUtensorMap& w2m,
                      const CUtensorMap& s2m, GvArgs a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.blockDim = dim3(kGvThreads);
  c.stream = st;
  c.attrs = at;
  c.numAttrs = 1;
  GvArgs a1 = a;
  a1.ring = gv_ring1(a.H);
  c.gridDim = dim3((unsigned)(a.n_slots * (a.I / 64) * kGvNQ));
  c.dynamicSmemBytes = (size_t)gv_smem1(a.M, a.H);
  cudaError_t e = cudaLaunchKernelEx(&c, gemv_fc1_kernel<MT>, w13m, s13m, a1);
  if (e != cudaSuccess) return e;
  GvArgs a2 = a;
  a2.ring = gv_ring2(a.n_slots, a.I);
  c.gridDim = dim3((unsigned)((a.H / 128) * kGvNQ));
  c.dynamicSmemBytes = (size_t)gv_smem2(a.M, a.I, a.top_k);
  return cudaLaunchKernelEx(&c, gemv_fc2_kernel<MT>, w2m, s2m, a2);
}

}  // namespace

// Shapes the streaming-GEMV kernels take: shared memory for the activations
// of all tokens (FC1) and h of every routed pair (FC2) within one CTA's
// limit, and TMA coordinates within int range.
bool decode_gemv_fits(int M, int E, int H, int I, int top_k) {
  if (M < 1 || M > 8 || M * top_k > kGvMaxSlots) return false;
  if (gv_smem1(M, H) > kGvSmemLimit || gv_smem2(M, I, top_k) > kGvSmemLimit) return false;
  const double rows13 = (double)E * 2 * I / 32, rows2 = (double)E * H / 32;
  const double ch13 = (double)E * (2 * I / 128) * (H / 64), ch2 = (double)E * (H / 128) * (I / 64);
  return rows13 < 2147483647.0 && rows2 < 2147483647.0 && ch13 < 2147483647.0 && ch2 < 2147483647.0;
}

// h [n_slots][M][I/64][68] FP32.
size_t decode_gemv_scratch_bytes(int M, int I, int top_k) {
  const size_t b = (size_t)M * top_k * M * (I / 64) * kGvGroup * sizeof(float);
  return (b + 255) & ~(size_t)255;
}

cudaError_t launch_decode_gemv(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                               const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H,
                               int I, int top_k, const ActParams& act, float* scratch, uint32_t* status, cudaStream_t st,
                               int* cu_err) {
  CUtensorMap w13m, s13m, w2m, s2m;
  {
    const uint64_t d[3] = {(uint64_t)H / 2, 32, (uint64_t)E * 2 * I / 32};
    const uint64_t sd[2] = {(uint64_t)H / 2, (uint64_t)H / 2 * 32};
    const uint32_t box[3] = {128, kGvQ, 4};
    CUresult r = make_u8_map(&w13m, w13, 3, d, sd, box, true);
    const uint64_t ds[3] = {16, 32, (uint64_t)E * (2 * I / 128) * (H / 64)};
    const uint64_t ss[2] = {16, kChunkBytes};
    const uint32_t bs[3] = {16, kGvQ, 4};
    if (r == CUDA_SUCCESS) r = make_u8_map(&s13m, s13, 3, ds, ss, bs, false);
    const uint64_t d2[3] = {(uint64_t)I / 2, 32, (uint64_t)E * H / 32};
    const uint64_t sd2[2] = {(uint64_t)I / 2, (uint64_t)I / 2 * 32};
    if (r == CUDA_SUCCESS) r = make_u8_map(&w2m, w2, 3, d2, sd2, box, true);
    const uint64_t ds2[3] = {16, 32, (uint64_t)E * (H / 128) * (I / 64)};
    if (r == CUDA_SUCCESS) r = make_u8_map(&s2m, s2, 3, ds2, ss, bs, false);
    if (r != CUDA_SUCCESS) {
      *cu_err = (int)r;
      return cudaErrorInvalidValue;
    }
  }
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    err = gv_set_attrs<1>();
    if (err == cudaSuccess) err = gv_set_attrs<2>();
    if (err == cudaSuccess) err = gv_set_attrs<4>();
    if (err == cudaSuccess) err = gv_set_attrs<8>();
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  GvArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ids = ids;
  a.ids64 = ids64;
  a.tw = tw;
  a.s13 = static_cast<const uint8_t*>(s13);
  a.s2 = static_cast<const uint8_t*>(s2);
  a.h = scratch;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.M = M;
  a.E = E;
  a.H = H;
  a.I = I;
  a.top_k = top_k;
  a.n_slots = M * top_k;
  a.ring = 1;
  a.act = act;
  switch (gv_mt(M)) {
    case 1: return gv_launch<1>(w13m, s13m, w2m, s2m, a, st);
    case 2: return gv_launch<2>(w13m, s13m, w2m, s2m, a, st);
    case 4: return gv_launch<4>(w13m, s13m, w2m, s2m, a, st);
    default: return gv_launch<8>(w13m, s13m, w2m, s2m, a, st);
  }
}

}  // namespace moe_fp4
