// Decode band (M <= 8 tokens) on the 5th-generation tensor cores: the expert
// weights (NVFP4, or MXFP4 re-expressed at prepare time with E4M3 block
// scales) are streamed by TMA straight into shared memory and consumed by
// tcgen05.mma kind::mxf4nvf4 with their own block scales, so no instruction
// is spent decoding a weight nibble.
//
// Prior art: the pages' tiny-decode kernel pair (b12x PR #22, "rp-native
// tiny-decode kernel for w4a8_mx (M=1)", section What): FC1 streams the
// routed experts' packed weights and writes an FP32 gate/up intermediate,
// FC2 applies the activation and performs the router-weighted sum; two plain
// launches rather than one cooperative launch (section Notes).  The routing is
// read directly by the GEMM kernels (the small-batch "direct" path of
// flashinfer PR #4285, "sync SM12x NVFP4 fused-MoE kernels"), ids outside
// [0, E) contribute exactly zero (b12x PR #311, conversation).
//
// The tensor-core MMA wants both operands in FP4.  The activations (BF16 x
// for FC1, FP32 h for FC2) enter as a sum of kTerms NVFP4 terms:
//   r_1 = a;  for t = 1..T:  term_t = NVFP4(r_t; G_t),  r_{t+1} = r_t - term_t
// where NVFP4(r; G) is the per-16-element quantisation with block scale
// s = e4m3_rn_satfinite(bmax / (6 G)) and codes e2m1_rn_satfinite(r / (s G)),
// and G_1 is the smallest power of two >= amax / (6 * 448) over the 256
// values of one (token, K stage), G_{t+1} = G_t / 4.  Every term is exact in
// FP32 and the dropped remainder r_{T+1} is about 10^-T of the block maximum
// (four terms: ~1e-4 relative error of the dot products, below the BF16
// rounding of the inputs).  Each (token, term) is one B row of the MMA
// (N = kTerms * M rounded up to 16), so for M <= 4 the terms ride in columns
// the N = 16 minimum would leave empty.  Each K stage ("item") accumulates
// into its own group of tensor-memory columns; the accumulator warps fold
// the group with its multipliers into FP32 registers, in item order, and
// release it for the item four stages later.
//
// FC1: a CTA owns one (route slot, 128-row w13 tile = 64 gate/up pairs, K
//      range); the K ranges of one tile form a thread-block cluster.  Each
//      CTA sends its partial rows to the CTA that owns them with asynchronous
//      distributed-shared-memory stores counted on the owner's mbarrier (no
//      cluster-wide barrier at the end); the owner sums them in rank order and
//      writes h = SiLU(gate) * up * (router weight) * (down multiplier) in
//      FP32 (FC2 is linear in h, so it only sums).
// FC2: a CTA owns one (128-row w2 tile, share of the (route slot, K stage)
//      items); the CTAs of one tile form a cluster and reduce the same way;
//      each output element is written once, in BF16.  Both kernels use
//      programmatic dependent launch: FC1's prologue overlaps the previous
//      kernel, and FC2's CTAs that find room beside FC1's (at most two CTAs
//      per SM) start streaming their weights before FC1 is done; only the
//      warps that read h wait for FC1.
//
// The tensor cores issue an MMA about every hundred cycles however small N
// is, so with N = 16 the issue, not the arithmetic, sets the pace: the MMAs
// are issued by two converged warps (alternate items), and the scale factors
// reach tensor memory through tcgen05.st from the warps that produce or
// receive them instead of through tcgen05.cp from the issuing thread.
//
// Roles in a 352-thread CTA: warp 0 lane 0 issues the TMA weight tiles and
// scale chunks into a 4-deep ring; warps 1-2 issue the MMAs (alternate
// items; warp 1 also owns the tensor-memory allocation); warps 3-6 build the
// activation terms (B operand, one warp per (stage, token)) and write their
// scales into tensor memory; warps 7-10 write the weight scales into tensor
// memory and drain the accumulator groups.  At most two CTAs share an SM
// (shared memory), so their 2 x 256 tensor-memory columns always fit and no
// allocation waits on another grid.
#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {

CUresult make_fp4_map(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows);

namespace {

constexpr int kTerms = 4;
constexpr int kRing = 4;                               // ring slots = accumulator groups
constexpr int kGSlots = 2 * kRing;                     // term-multiplier sets in flight
constexpr int kMmaWarp0 = 1, kMmaWarps = 2;            // warps 1..2 issue the MMAs
constexpr int kQuantWarp0 = 3, kQuantWarps = 4;        // warps 3..6 build B
constexpr int kEpiWarp0 = 7;                           // warps 7..10 drain the accumulator
constexpr int kTcThreads = 32 * (kEpiWarp0 + 4);
constexpr int kMaxN = 32;                              // kTerms * 8 tokens
constexpr uint32_t kSlotA = 128 * 128;                 // 128 rows x 256 K (FP4)
constexpr uint32_t kSlotB = kMaxN * 128;               // N rows x 256 K
constexpr uint32_t kSlotSF = 4 * kChunkBytes;          // 4 K-groups
constexpr uint32_t kSlotBytes = kSlotA + kSlotB + 2 * kSlotSF;  // 24 KB, 1024-aligned
constexpr int kMaxSlotsTc = 128;
constexpr uint32_t kTmemColsTc = 256;
constexpr uint32_t kTmemSFBase = 32 * kRing;           // accumulator groups in [0, 128)

// FC2: split * M * ceil(128 / split) floats; split <= 8 gives at most
// 7 * 19 = 133 per token (split 7), so 8 tokens fit in 8 * 136.
// FC1 (cluster of K ranges): split * M * 2 * ceil(64 / split) floats, at
// most 7 * 2 * 10 = 140 per token (split 7); FC2: split * M * ceil(128 /
// split), at most 133 per token.  8 tokens: 8 * 140.
constexpr int kPartFloats = 8 * 140;

struct SmemTc {
  float part[kPartFloats];         // partial sums received from the cluster
  float G[kGSlots][8][kTerms];     // term multipliers per (item, token)
  int ids[kMaxSlotsTc];
  float tw[kMaxSlotsTc];
  int own[kMaxSlotsTc];            // FC2: first slot naming each valid expert, in slot order
  int own_cnt[4];                  // FC2: owners per 32-slot chunk
  int expert;                      // FC1: this CTA's expert (-1: nothing to do)
  float wtok[8];                   // FC1: router weight of the expert per token
  float g3[3];                     // FC1: gate, up, down multipliers of the expert
  uint32_t routed;                 // FC1: tokens routed to the expert (bit mask)
  uint64_t fullA[kRing];           // weight tile + its scale chunks landed (TMA)
  uint64_t fullB[kRing];           // activation terms + their scales in place (builders)
  uint64_t sfa[kRing];             // weight scales copied to tensor memory
  uint64_t done[kRing];            // MMAs of the slot complete (slot and group reusable)
  uint64_t acce[kRing];            // accumulator group drained
  uint64_t gready[kGSlots];        // term multipliers written
  uint64_t bsf;                    // a wave's B scales are staged (all builder warps)
  uint64_t red;                    // every partial row this CTA reduces has landed
  uint32_t tmem;
};
constexpr uint32_t kTcSmem = kRing * kSlotBytes + sizeof(SmemTc) + 1024;

struct TcArgs {
  const __nv_bfloat16* x;
  const int32_t* ids;  // [M][top_k], int32 or (ids64) int64
  int ids64;
  const float* tw;
  const uint8_t* s13;
  const uint8_t* s2;
  float* h;      // [n_slots][M][I]: FC1's output, SiLU(gate)*up*(router weight)*(down multiplier)
  uint8_t* ximg;  // per K stage of x: B tile (N rows x 128 B, swizzled), 512 B of scales, G [M][kTerms]
  int ximg_stride;
  uint8_t* himg;  // per (route slot, K stage of h): the same images for FC2, or null (FC2 builds its own)
  __nv_bfloat16* out;
  uint32_t* status;
  int M, E, H, I, top_k, n_slots;
  int split;   // FC1: K ranges per w13 tile; FC2: CTAs (cluster size) per w2 tile
  int N;      // B rows per item (accumulator columns)
  ActParams act;  // FC1's gated activation
  // single-launch layer only: h-ready counters and reader counts, both
  // [owner][K stage of h], and the K ranges per w13 tile
  uint32_t* hflag;
  uint32_t* hused;
  int s1;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Asynchronous FP32 store to the same shared-memory offset in another CTA of
// the cluster; its completion is counted (4 bytes) on that CTA's mbarrier.
__device__ __forceinline__ void st_async_peer_f32(float* local, uint64_t* local_bar, uint32_t rank, float v) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(local_bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
               "r"(__float_as_uint(v)), "r"(rb)
               : "memory");
}


__device__ __forceinline__ uint32_t e4m3_rn_satf(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}
// Two E2M1 codes, `lo` in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn_satf(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xffu;
}

// Smallest power of two >= amax / 2688 (0 for amax == 0).
__device__ __forceinline__ float term_g1(float amax) {
  if (!(amax > 0.f)) return 0.f;
  const float q = amax * (1.0f / 2688.0f) * 1.0000002f;
  uint32_t b = __float_as_uint(q);
  uint32_t e = b >> 23;
  if (b & 0x7fffffu) ++e;
  if (e < 1u) e = 1u;
  if (e > 254u) e = 254u;
  return __uint_as_float(e << 23);
}

// Byte offset of 16-element block b of B row n in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t b_tile_offset(int n, int b) {
  return (uint32_t)(n * 128 + ((((b >> 1) ^ (n & 7)) & 7) << 4) + ((b & 1) << 3));
}
// Byte offset of the scale of (B row n < 32, block b of the 256-K stage) in
// the item's B scale staging: row n's 16 scale bytes, 64-K group g in bytes
// 4g .. 4g+3 (the 32-bit word tensor memory holds per row and group).
__device__ __forceinline__ uint32_t sf_offset(int n, int b) { return (uint32_t)((n & 31) * 16 + b); }

// 1/g for a power of two g in [2^-126, 2^126] (exact).
__device__ __forceinline__ float pow2_inv(float g) { return __uint_as_float((254u << 23) - __float_as_uint(g)); }

__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// The kTerms NVFP4 terms of one token's 256-value K stage, built by one warp:
// lane l holds values 8l .. 8l+7 (half l%2 of 16-element block l/2).  The
// term multipliers are G1 * 4^-t.  Lane l writes its 4 code bytes of each
// term's B row token*kTerms + t, the even lane of a block its scale byte.
// Any quotient rounding is corrected by the next term (the residual is
// formed from the exact term values), so the reciprocals are approximate.
__device__ __forceinline__ void emit_stage_terms(float (&v)[8], float G1, uint8_t* btile, uint8_t* sfb, int token,
                                                 int lane, bool store) {
  const int b = lane >> 1, half = lane & 1;
  float g = G1;
#pragma unroll
  for (int t = 0; t < kTerms; ++t, g *= 0.25f) {
    const int n = token * kTerms + t;
    float m01 = fmaxf(fabsf(v[0]), fabsf(v[1])), m23 = fmaxf(fabsf(v[2]), fabsf(v[3]));
    float m45 = fmaxf(fabsf(v[4]), fabsf(v[5])), m67 = fmaxf(fabsf(v[6]), fabsf(v[7]));
    float bm = fmaxf(fmaxf(m01, m23), fmaxf(m45, m67));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
    uint32_t sc = 0, w = 0;
    if (g > 0.f) {
      const float inv_g = pow2_inv(g);
      sc = e4m3_rn_satf(bm * (inv_g * (1.0f / 6.0f)));
      const float s = e4m3_to_float(sc);
      if (s > 0.f) {
        const float sg = s * g, inv = rcp_approx(s) * inv_g;
#pragma unroll
        for (int j = 0; j < 4; ++j) w |= e2m1x2_rn_satf(v[2 * j] * inv, v[2 * j + 1] * inv) << (8 * j);
        uint32_t hv[4];
        e2m1x8_to_half2x4(w, hv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = half2_bits_to_float2(hv[j]);
          v[2 * j] = fmaf(-d.x, sg, v[2 * j]);
          v[2 * j + 1] = fmaf(-d.y, sg, v[2 * j + 1]);
        }
      } else {
        sc = 0;
      }
    }
    if (store) {
      *reinterpret_cast<uint32_t*>(btile + b_tile_offset(n, b) + 4 * half) = w;
      if (!half) sfb[sf_offset(n, b)] = (uint8_t)sc;
    }
  }
}

// Loads issued where they stand (volatile): the activation prefetch must not
// be moved below the barriers that follow it.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ float ld_nc_f32(const void* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
// 8 consecutive BF16 / FP32 activations as FP32.
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = ld_nc_v4(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// FC2's activations for route slot j and `token`: h at pairs p0 .. p0+7.
__device__ __forceinline__ void fc2_activation(const TcArgs& a, int j, int token, int p0, float (&v)[8]) {
  const float* p = a.h + ((size_t)j * a.M + token) * a.I + p0;
  const uint4 u0 = ld_cg_v4(p), u1 = ld_cg_v4(p + 4);
  v[0] = __uint_as_float(u0.x);
  v[1] = __uint_as_float(u0.y);
  v[2] = __uint_as_float(u0.z);
  v[3] = __uint_as_float(u0.w);
  v[4] = __uint_as_float(u1.x);
  v[5] = __uint_as_float(u1.y);
  v[6] = __uint_as_float(u1.z);
  v[7] = __uint_as_float(u1.w);
}

// Activation pre-pass of FC1: the four NVFP4 terms of x for every (K stage,
// token), built once per layer call and stored as the images FC1 copies
// into its ring: the B tile (rows token*kTerms + t, 128-byte swizzle), the
// scales (row n's 16 bytes at 16n) and the term multipliers G [M][kTerms].
// One CTA per K stage, one warp per token.
__global__ void __launch_bounds__(256) decode_quant_x_kernel(TcArgs a) {
  pdl_wait();               // x comes from the previous kernel
  pdl_launch_dependents();  // FC1 may start: the routing is final as well
  const int st = blockIdx.x, token = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (token >= a.M) return;
  uint8_t* img = a.ximg + (size_t)st * a.ximg_stride;
  float v[8];
  load_bf16x8(a.x + (size_t)token * a.H + st * 256 + lane * 8, v);
  float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                  fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float G1 = term_g1(m);
  const uint32_t tb = (uint32_t)a.N * 128;
  if (lane < kTerms)
    reinterpret_cast<float*>(img + tb + kChunkBytes)[token * kTerms + lane] =
        G1 * __uint_as_float((127u - 2u * lane) << 23);
  emit_stage_terms(v, G1, img, img + tb, token, lane, true);
}

// Activation pre-pass of FC2 (larger M): the four NVFP4 terms of h for every
// (route slot that owns its expert, K stage of the intermediate, token),
// stored as FC2's images.  One CTA per (slot,
// stage), one warp per token.
__global__ void __launch_bounds__(256) decode_quant_h_kernel(TcArgs a) {
  __shared__ int s_ids[kMaxSlotsTc];
  pdl_launch_dependents();  // FC2 may start streaming its weights
  const int ns2 = (a.I + 255) / 256;
  const int j = blockIdx.x / ns2, st = blockIdx.x % ns2;
  const int token = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = threadIdx.x; k < a.n_slots; k += blockDim.x) s_ids[k] = route_id(a.ids, k, a.ids64, a.E);
  __syncthreads();
  const int e = s_ids[j];
  bool skip = e < 0 || e >= a.E;
  for (int k = 0; !skip && k < j; ++k) skip = s_ids[k] == e;  // an earlier slot owns this expert
  // every CTA waits, the ones with nothing to do too: FC2 takes this grid's
  // completion for FC1's
  pdl_wait();  // FC1's h is complete
  if (skip) return;
  if (token >= a.M) return;
  const int rem = a.I / 64 - 4 * st;
  const bool act = lane < 8 * (rem < 4 ? rem : 4);
  float v[8];
  if (act) {
    fc2_activation(a, j, token, st * 256 + lane * 8, v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                  fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float G1 = term_g1(m);
  uint8_t* img = a.himg + ((size_t)j * ns2 + st) * a.ximg_stride;
  const uint32_t tb = (uint32_t)a.N * 128;
  if (lane < kTerms)
    reinterpret_cast<float*>(img + tb + kChunkBytes)[token * kTerms + lane] =
        G1 * __uint_as_float((127u - 2u * lane) << 23);
  emit_stage_terms(v, G1, img, img + tb, token, lane, act);
}

// FC1 (kFc2 = false) and FC2 (kFc2 = true).
template <bool kFc2>
__global__ void __launch_bounds__(kTcThreads, 2) decode_tc_kernel(const __grid_constant__ CUtensorMap map_w, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  SmemTc& S = *reinterpret_cast<SmemTc*>(ring + kRing * kSlotBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.M, H = a.H, I = a.I, n = a.n_slots, N = a.N;
  const int split = a.split;
  // FC1: clusters of `split` K ranges per (slot, w13 tile); FC2: clusters of
  // `split` CTAs per w2 row tile
  const uint32_t rank = cluster_rank();
  const int unit = blockIdx.x / split;  // FC1: slot * tiles1 + tile; FC2: w2 row tile
  // FC1 of non-gated experts (squared ReLU): w1 tiles of 128 rows (h values),
  // the last one padded (its scale rows past I are zero)
  const bool relu2 = !kFc2 && a.act.kind == MOE_FP4_ACT_RELU2;
  const int tiles1 = relu2 ? (I + 127) / 128 : I / 64, ns2 = (I + 255) / 256;
  const bool is_quant = warp >= kQuantWarp0 && warp < kQuantWarp0 + kQuantWarps;
  // activation terms from a pre-pass image (FC1 always, FC2 for larger M)
  // or built in this CTA (FC2 for small M)
  const bool use_img = !kFc2 || a.himg != nullptr;
  const bool is_epi = warp >= kEpiWarp0;

  // the routing first: its latency overlaps the barrier setup below (the
  // kernels are launched only after whatever produced it is complete)
  int idr[4];
  float twr[4];
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      idr[k] = j < n ? route_id(a.ids, j, a.ids64, a.E) : -1;
      twr[k] = j < n ? ld_nc_f32(a.tw + j) : 0.f;
    }
  }

  // ---- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&S.fullA[s], 1);
      mbar_init(&S.fullB[s], use_img ? 1 : kQuantWarps);
      mbar_init(&S.sfa[s], 4);
      mbar_init(&S.done[s], 1);
      mbar_init(&S.acce[s], 4);
    }
    for (int s = 0; s < kGSlots; ++s) mbar_init(&S.gready[s], kQuantWarps);
    mbar_init(&S.bsf, kQuantWarps);
    // the partial rows this CTA reduces, one from every CTA of the cluster:
    // FC1 the gate and up rows of pairs p = rank mod split, FC2 the rows
    // r = rank mod split
    mbar_init(&S.red, 1);
    const int own = kFc2 || relu2 ? (128 - (int)rank + split - 1) / split : 2 * ((64 - (int)rank + split - 1) / split);
    mbar_arrive_expect_tx(&S.red, (uint32_t)(split * own * M * 4));
    fence_mbar_init();
    tma_prefetch_desc(&map_w);
  }
  // cluster phase 1: this CTA runs and its barriers are initialised
  // (awaited before any remote store)
  cluster_arrive_release();
  if (warp == kMmaWarp0) tmem_alloc(&S.tmem, kTmemColsTc);
  // Both kernels are launched only after the activation pre-pass has passed
  // its wait on whatever produced x and the routing, so they may read the
  // routing right away; FC1 waits (griddepcontrol.wait) before it reads the
  // pre-pass's activation terms, FC2 before it reads FC1's partial sums.
  pdl_launch_dependents();

  int slot1 = 0, tile = 0, k0 = 0, n_items = 0, n_own = 0;
  auto item_slot = [&](int i) { return kFc2 ? S.own[((int)rank + split * i) % n_own] : slot1; };
  auto item_stage = [&](int i) { return kFc2 ? ((int)rank + split * i) / n_own : k0 + i; };
  auto item_groups = [&](int i) {
    if (!kFc2) return 4;
    const int rem = I / 64 - 4 * item_stage(i);
    return rem < 4 ? rem : 4;
  };
  const uint64_t KG = kFc2 ? (uint64_t)(I / 64) : (uint64_t)(H / 64);
  auto issue = [&](int i, int e) {  // TMA of item i's weight tile and scale chunks
    const int sl = i % kRing, st = item_stage(i), ng = item_groups(i);
    uint8_t* slotp = ring + sl * kSlotBytes;
    mbar_arrive_expect_tx(&S.fullA[sl], kSlotA + (uint32_t)ng * kChunkBytes);
    int row0;
    const uint8_t* sfa;
    if (!kFc2) {
      row0 = (relu2 ? e * I : e * 2 * I) + tile * 128;
      sfa = a.s13 + (((uint64_t)e * tiles1 + tile) * KG + 4 * (uint64_t)st) * kChunkBytes;
    } else {
      row0 = e * H + unit * 128;
      sfa = a.s2 + (((uint64_t)e * (H / 128) + unit) * KG + 4 * (uint64_t)st) * kChunkBytes;
    }
    // the weights stream through L2 once per layer: evict-first
    const uint64_t wpol = l2_evict_first_policy();
    tma_load_2d_hint(slotp, &map_w, st * 128, row0, &S.fullA[sl], wpol);
    bulk_load_hint(slotp + kSlotA + kSlotB, sfa, (uint32_t)ng * kChunkBytes, &S.fullA[sl], wpol);
  };
  // FC1: bulk copy of item i's activation terms (B tile, scales, G) from the
  // pre-pass's image into the ring slot
  auto issue_b = [&](int i) {
    const int sl = i % kRing;
    uint8_t* slotp = ring + sl * kSlotBytes;
    const uint8_t* img = kFc2 ? a.himg + ((size_t)item_slot(i) * ns2 + item_stage(i)) * a.ximg_stride
                              : a.ximg + (size_t)item_stage(i) * a.ximg_stride;
    const uint32_t tb = (uint32_t)N * 128, sb = kChunkBytes + 16u * (uint32_t)M;
    mbar_arrive_expect_tx(&S.fullB[sl], tb + sb);
    bulk_load(slotp + kSlotA, img, tb, &S.fullB[sl]);
    bulk_load(slotp + kSlotA + kSlotB + kSlotSF, img + tb, sb, &S.fullB[sl]);
  };

  const int qw = warp - kQuantWarp0;  // FC2 quantiser warp: one (item, token) per round
  if (!kFc2) {
    slot1 = unit / tiles1;
    tile = unit % tiles1;
    const int nk = H / 256;
    k0 = (int)rank * nk / split;
    n_items = ((int)rank + 1) * nk / split - k0;
  }
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (lane + 32 * k < n) {
        S.ids[lane + 32 * k] = idr[k];
        S.tw[lane + 32 * k] = twr[k];
      }
    __syncwarp();
    if (!kFc2) {
      // does an earlier slot name the same expert?  If not, stream the first
      // ring wave of weight tiles right away.
      const int e = S.ids[slot1];
      bool ok = e >= 0 && e < a.E;
      for (int base = 0; ok && base < slot1; base += 32) {
        const int j = base + lane;
        ok = !__any_sync(0xffffffffu, j < slot1 && S.ids[j] == e);
      }
      if (lane == 0) {
        S.expert = ok ? e : -1;
        if (ok)
          for (int i = 0; i < n_items && i < kRing; ++i) issue(i, e);
      }
      // router weight of this expert per token
      float wt = 0.f;
      bool rt = false;
      if (lane < M)
        for (int k = 0; k < a.top_k; ++k)
          if (S.ids[lane * a.top_k + k] == e) {
            wt += S.tw[lane * a.top_k + k];
            rt = true;
          }
      const uint32_t rm = __ballot_sync(0xffffffffu, rt);
      if (lane < M) S.wtok[lane] = wt;
      if (lane == 0) S.routed = rm;
    }
  }
  tc_fence_before();
  __syncwarp();  // converge every warp before the CTA barrier (it counts whole warps)
  __syncthreads();
  tc_fence_after();

  int e1 = -1;
  if (!kFc2) {
    e1 = S.expert;
    if (e1 < 0) {  // an earlier slot names this expert: the whole cluster leaves
      // (not before the x pre-pass is complete: FC2 and the next layer take
      // FC1's completion for the pre-pass's, and a layer whose slots all
      // leave here would otherwise let them run beside a pre-pass still
      // writing its images)
      pdl_wait();
      if (warp == kMmaWarp0) tmem_dealloc(S.tmem, kTmemColsTc);
      return;
    }
    if (warp == kQuantWarp0 && lane < 3) {  // (FC1's builder warps are free)
      const float* gl13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * tiles1 * (H / 64) * kChunkBytes);
      const float* gl2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * (H / 128) * (I / 64) * kChunkBytes);
      // gated: gate, up, down multipliers; non-gated: w1's ([E]) twice, down
      S.g3[lane] = ld_nc_f32(lane < 2 ? (relu2 ? gl13 + e1 : gl13 + 2 * e1 + lane) : gl2 + e1);
    }
  } else {
    // owners: the first slot naming each valid expert, in slot order
    bool own_j = false;
    uint32_t bal = 0;
    const int j = 32 * warp + lane;
    if (warp < 4) {
      const int id = j < n ? S.ids[j] : -1;
      const bool valid = j < n && id >= 0 && id < a.E;
      const uint32_t mm = __match_any_sync(0xffffffffu, valid ? id : -1 - lane);
      bool dup = (mm & ((1u << lane) - 1u)) != 0;
      for (int c = 0; valid && !dup && c < warp; ++c)
        for (int k = 0; k < 32; ++k) dup = dup || S.ids[32 * c + k] == id;
      own_j = valid && !dup;
      bal = __ballot_sync(0xffffffffu, own_j);
      if (lane == 0) S.own_cnt[warp] = __popc(bal);
    }
    __syncwarp();
    __syncthreads();
    if (own_j) {
      int base = 0;
      for (int c = 0; c < warp; ++c) base += S.own_cnt[c];
      S.own[base + __popc(bal & ((1u << lane) - 1u))] = j;
    }
    n_own = S.own_cnt[0] + S.own_cnt[1] + S.own_cnt[2] + S.own_cnt[3];
    __syncwarp();
    __syncthreads();
    // items (owner, K stage) stage-major, dealt round-robin to the cluster
    const int total = n_own * ns2;
    n_items = total > (int)rank ? (total - (int)rank + split - 1) / split : 0;
  }

  float vout[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) vout[t] = 0.f;

  // An item's weight scales (and, with pre-pass images, its activation scales
  // and term multipliers) into tensor memory, this warp's lane quarter
  // (replicated), as soon as the item's TMA lands; returns false if a wait
  // gave up.
  auto store_sfa = [&](int i, uint32_t tq) -> bool {
      const int sl = i % kRing;
      bool ok = mbar_wait(&S.fullA[sl], (i / kRing) & 1, a.status, 32u);
      if (use_img) ok = ok && mbar_wait(&S.fullB[sl], (i / kRing) & 1, a.status, 32u);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      const uint8_t* src = ring + sl * kSlotBytes + kSlotA + kSlotB;
      uint32_t r[16];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 u = *reinterpret_cast<const uint4*>(src + g * kChunkBytes + lane * 16);
        r[4 * g] = u.x;
        r[4 * g + 1] = u.y;
        r[4 * g + 2] = u.z;
        r[4 * g + 3] = u.w;
      }
      tmem_st16(tq + kTmemSFBase + sl * 32, r);
      if (use_img) {
        // the item's activation scales (B rows 0..31, 64-K group g in column
        // 4g) and its term multipliers, copied from the pre-pass image
        const uint8_t* bsf = src + kSlotSF;
        const uint4 u = *reinterpret_cast<const uint4*>(bsf + lane * 16);
        const uint32_t rb[16] = {u.x, 0u, 0u, 0u, u.y, 0u, 0u, 0u, u.z, 0u, 0u, 0u, u.w, 0u, 0u, 0u};
        tmem_st16(tq + kTmemSFBase + sl * 32 + 16, rb);
        const float* gi = reinterpret_cast<const float*>(bsf + kChunkBytes);
        if (lane < M * kTerms) S.G[i % kGSlots][lane / kTerms][lane % kTerms] = gi[lane];
        __syncwarp();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sfa[sl]);
      return true;
  };

  if (warp == 0) {
    // ---------------- TMA producer (the weights need nothing from FC1)
    if (lane == 0) {
      const int wave0 = n_items < kRing ? n_items : kRing;
      if (kFc2)  // (FC1 issued its first wave of weight tiles already)
        for (int i = 0; i < wave0; ++i) issue(i, S.ids[item_slot(i)]);
      if (use_img) {
        pdl_wait();  // the pre-pass images are complete
        for (int i = 0; i < wave0; ++i) issue_b(i);
      }
      for (int i = wave0; i < n_items; ++i) {
        const int sl = i % kRing, round = i / kRing;
        if (!mbar_wait(&S.done[sl], (round - 1) & 1, a.status, 1u)) break;
        issue(i, kFc2 ? S.ids[item_slot(i)] : e1);
        if (use_img) issue_b(i);
      }
    }
  } else if (warp < kMmaWarp0 + kMmaWarps) {
    // ---------------- MMA issuers: items alternate between two warps (the
    // issue cost of an MMA, not its execution, bounds these tiny-N tiles);
    // each warp runs converged and one elected lane issues
    const int mw = warp - kMmaWarp0;
    const uint32_t tmem = S.tmem;
    const uint32_t idesc = idesc_mxf4nvf4(128, N, false);
    for (int i = mw; i < n_items; i += kMmaWarps) {
      const int sl = i % kRing, round = i / kRing;
      // the scale writers arrive on sfa only after they saw the item's
      // weight tile (and, from a pre-pass image, its activation terms) land
      bool ok = mbar_wait(&S.sfa[sl], round & 1, a.status, 2u);
      if (!use_img) ok = ok && mbar_wait(&S.fullB[sl], round & 1, a.status, 2u);
      ok = ok && (round == 0 || mbar_wait(&S.acce[sl], (round - 1) & 1, a.status, 2u));
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int ng = item_groups(i);
      uint8_t* slotp = ring + sl * kSlotBytes;
      const uint32_t sfa_t = tmem + kTmemSFBase + sl * 32, sfb_t = sfa_t + 16;
      const uint64_t da = smem_desc(smem_u32(slotp), 16, 1024, kLayoutSW128);
      const uint64_t db = smem_desc(smem_u32(slotp + kSlotA), 16, 1024, kLayoutSW128);
      for (int k = 0; k < ng; ++k)  // K step of 64 = 32 bytes = 2 descriptor units
        mma_nvf4_warp(tmem + 32 * sl, da + 2 * k, db + 2 * k, idesc, sfa_t + 4 * k, sfb_t + 4 * k, k > 0);
      mma_commit_warp(&S.done[sl]);
    }
  } else if (is_quant) {
    // ---------------- FC2: activation terms (B operand), one wave of ring slots at a time
    if (use_img) {
      // the terms come from a pre-pass image: these warps put every item's
      // scales into tensor memory instead, running ahead of the drain
      const uint32_t tq = S.tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      for (int i = 0; i < n_items; ++i)
        if (!store_sfa(i, tq)) break;
    }
    if (!use_img) {  // (otherwise the terms come from a pre-pass)
    pdl_wait();  // FC1's h is complete and visible
    const int waves = (n_items + kRing - 1) / kRing;
    for (int w = 0; w < waves; ++w) {
      const int i0 = w * kRing, wi = n_items - i0 < kRing ? n_items - i0 : kRing;
      if (w > 0) {
        bool ok = true;
        for (int k = 0; k < wi; ++k) ok = ok && mbar_wait(&S.done[(i0 + k) % kRing], (w - 1) & 1, a.status, 8u);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int pairs = wi * M;
      for (int r = 0; r * kQuantWarps < pairs; ++r) {
        const int p = r * kQuantWarps + qw;
        if (p >= pairs) break;  // warp-uniform
        const int item = i0 + p / M, token = p % M;
        const bool act = lane < 8 * item_groups(item);  // lanes beyond the stage's valid K
        float v[8];
        if (act) {
          fc2_activation(a, item_slot(item), token, item_stage(item) * 256 + lane * 8, v);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        // G1 of this (item, token): the maximum over the whole stage
        float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                        fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float G1 = term_g1(m);
        if (lane < kTerms) S.G[item % kGSlots][token][lane] = G1 * __uint_as_float((127u - 2u * lane) << 23);
        uint8_t* slotp = ring + (item % kRing) * kSlotBytes;
        emit_stage_terms(v, G1, slotp + kSlotA, slotp + kSlotA + kSlotB + kSlotSF, token, lane, act);
      }
      fence_proxy_async_smem();
      // the wave's B scales -> tensor memory: each warp fills its lane quarter
      // (the scales of B rows 0..31 are replicated in all four)
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.bsf);
      if (!__all_sync(0xffffffffu, mbar_wait(&S.bsf, w & 1, a.status, 64u))) break;
      for (int k = 0; k < wi; ++k) {
        const int sl = (i0 + k) % kRing;
        const uint4 u = *reinterpret_cast<const uint4*>(ring + sl * kSlotBytes + kSlotA + kSlotB + kSlotSF + lane * 16);
        const uint32_t r[16] = {u.x, 0u, 0u, 0u, u.y, 0u, 0u, 0u, u.z, 0u, 0u, 0u, u.w, 0u, 0u, 0u};
        tmem_st16(S.tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kTmemSFBase + sl * 32 + 16, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < wi; ++k) {
          mbar_arrive(&S.gready[(i0 + k) % kGSlots]);
          mbar_arrive(&S.fullB[(i0 + k) % kRing]);
        }
    }
    }
  } else {
    // ---------------- accumulator drain (and, when this CTA builds its own
    // activation terms, the weight scales -> tensor memory).  Warps 7..10
    // own lanes 32*(warp%4) ...
    const int q = warp & 3;
    const uint32_t tq = S.tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;
    if (!use_img)
      for (int i = 0; ok && i < n_items && i < kRing; ++i) ok = store_sfa(i, tq);
    for (int i = 0; ok && i < n_items; ++i) {
      const int sl = i % kRing, gs = i % kGSlots;
      ok = use_img || mbar_wait(&S.gready[gs], (i / kGSlots) & 1, a.status, 16u);
      ok = ok && mbar_wait(&S.done[sl], (i / kRing) & 1, a.status, 4u);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float acc[kMaxN];
      uint32_t r[16];
      tmem_ld16(tq + 32 * sl, r);
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(r[c]);
      if (N > 16) {
        tmem_ld16(tq + 32 * sl + 16, r);
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[16 + c] = __uint_as_float(r[c]);
      } else {
#pragma unroll
        for (int c = 16; c < kMaxN; ++c) acc[c] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (t < M) {
#pragma unroll
          for (int u = 0; u < kTerms; ++u) vout[t] = fmaf(acc[t * kTerms + u], S.G[gs][t][u], vout[t]);
        }
      // (the multipliers are read before the slot is released: with images,
      // the scale warps refill S.G for later items as soon as they may)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acce[sl]);
      if (!use_img && i + kRing < n_items) ok = ok && store_sfa(i + kRing, tq);
    }
  }

  // ---- cluster reduction: partial rows go to their owner CTA (asynchronous
  // stores counted on its barrier), summed there in rank order
  tc_fence_before();
  __syncwarp();
  cluster_wait();  // phase 1: every CTA of the cluster runs
  // FC1: pair p is owned by rank p % split (cpo pairs each, gate and up rows);
  // FC2 and non-gated FC1: row r by rank r % split
  const int cpo = (64 + split - 1) / split;
  const int rpo = kFc2 || relu2 ? (128 + split - 1) / split : 2 * cpo;
  if (is_epi) {
    const int row = 32 * (warp & 3) + lane;
    int owner, j;
    if (!kFc2 && !relu2) {
      const int pr = row & 63;
      owner = pr % split;
      j = (row >> 6) * cpo + pr / split;
    } else {
      owner = row % split;
      j = row / split;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < M) st_async_peer_f32(&S.part[((int)rank * M + t) * rpo + j], &S.red, (uint32_t)owner, vout[t]);
  }
  __syncwarp();
  __syncthreads();  // tensor memory is no longer read
  if (warp == kMmaWarp0) tmem_dealloc(S.tmem, kTmemColsTc);
  if (!__all_sync(0xffffffffu, mbar_wait(&S.red, 0, a.status, 128u))) return;
  if (relu2) {
    // h_n = max(u_n, 0)^2 x (router weight) x (down multiplier), rows of the
    // tile below I
    for (int idx = threadIdx.x; idx < M * rpo; idx += kTcThreads) {
      const int token = idx / rpo, j = idx % rpo, row = (int)rank + split * j;
      if (row >= 128 || tile * 128 + row >= I) continue;
      float u = 0.f;
      for (int src = 0; src < split; ++src) u += S.part[(src * M + token) * rpo + j];
      const float r = fmaxf(u * S.g3[0], 0.f);
      const float hv = (S.routed >> token) & 1u ? r * r * (S.wtok[token] * S.g3[2]) : 0.f;
      a.h[((size_t)slot1 * M + token) * I + tile * 128 + row] = hv;
    }
  } else if (!kFc2) {
    for (int idx = threadIdx.x; idx < M * cpo; idx += kTcThreads) {
      const int token = idx / cpo, jj = idx % cpo, pair = (int)rank + split * jj;
      if (pair >= 64) continue;
      float gate = 0.f, up = 0.f;
      for (int src = 0; src < split; ++src) {
        gate += S.part[(src * M + token) * rpo + jj];
        up += S.part[(src * M + token) * rpo + cpo + jj];
      }
      const float hv =
          (S.routed >> token) & 1u ? gated_act(gate * S.g3[0], up * S.g3[1], a.act) * (S.wtok[token] * S.g3[2]) : 0.f;
      a.h[((size_t)slot1 * M + token) * I + tile * 64 + pair] = hv;
    }
  } else {
    for (int idx = threadIdx.x; idx < M * rpo; idx += kTcThreads) {
      const int token = idx / rpo, j = idx % rpo, row = (int)rank + split * j;
      if (row >= 128) continue;
      float v = 0.f;
      for (int src = 0; src < split; ++src) v += S.part[(src * M + token) * rpo + j];
      a.out[(size_t)token * H + unit * 128 + row] = __float2bfloat16_rn(v);
    }
  }
}

// ---------------------------------------------------------------- single launch
// The whole decode layer in one launch, for shapes whose work fits one
// resident grid with every CTA's weight tiles in flight at once (see
// launch_decode_fused).  A CTA owns one FC1 share (a K range of one 128-row
// w13 tile of one routed expert) and one FC2 share (some of the (expert, K
// stage) items of one 128-row w2 tile); its shared-memory ring has a slot for
// every item, so the producer issues all of its weight tiles as the CTA
// starts and FC2's weights are in shared memory before h exists.  The
// tiny-decode PR keeps FC1 and FC2 as two launches and found one cooperative
// launch slower because of its grid synchronisation (b12x PR #22, section
// Notes); here nothing waits for the whole grid: an FC2 item waits only for
// the h values it reads, published per (expert, w13 tile, K range) by a flag
// in global memory, and both reductions stay inside thread-block clusters.
//
// Cluster of C CTAs (rank r): FC1 sub-clusters of s1 CTAs (the K ranges of one
// w13 tile; C / s1 tiles per cluster), FC2 the whole cluster (the items of
// one w2 tile dealt round-robin).  Unit index of an FC1 share: cluster * (C /
// s1) + r / s1 over the (owner, w13 tile) pairs; w2 tile: the cluster index.
//
// Roles (352 threads): warp 0 lane 0 issues every weight TMA at the start;
// warps 1-2 issue the MMAs (alternate items, each into its own accumulator
// group); warps 3-6 build the activation terms (x for FC1's items, h for
// FC2's, items or (item, token) pairs spread over the four warps) and write
// both scale sets of every item into tensor memory (each warp its lane
// quarter); warps 7-10 drain the accumulators, then run the FC1 and FC2
// reductions.
//
// h-ready protocol: the CTA that reduces pairs p = r1 mod s1 of an FC1 unit
// writes their h and adds 1 (release, GPU scope) to the counter of the
// (expert, 256-wide K stage of h) the unit belongs to; the stage is complete
// when its counter reaches (its w13 tiles) x s1.  One lane of each FC2
// builder polls that counter (acquire) before the warp loads h.  Every
// (expert, K stage) item is read by exactly one CTA of each w2 tile; after
// its items are published each reader counts itself in a second counter, and
// the last reader sets both back to zero, so every call ends with them all at
// zero (the workspace starts with them zero).

// Ring geometry of the single launch for N activation-term rows (16 up to 4
// tokens, 32 up to 8): slot = weight tile (128 rows x 256 K), the B tile (N
// rows, 128-byte swizzle), the weight scale chunks (4 K-groups) and the B
// scales (row n's 16 bytes at 16n), rounded to 1 KB; as many slots as fit
// one CTA per SM, and tensor memory for one accumulator group of N columns
// plus 32 scale columns per slot.
template <int kN>
struct FzCfg {
  static constexpr uint32_t kB = kN * 128;
  static constexpr uint32_t kSFA = kSlotA + kB;
  static constexpr uint32_t kSFB = kSFA + 4 * kChunkBytes;
  static constexpr uint32_t kSlot = (kSFB + 512 + 1023) / 1024 * 1024;
  static constexpr int kRing = kN == 16 ? 10 : 8;
  static constexpr uint32_t kTmemSF = kRing * kN;  // scale columns after the accumulator groups
  static_assert(kTmemSF + 32 * kRing <= 512, "tensor memory");
};

struct SmemFz {
  float part1[8 * 144];            // FC1 partials received from the sub-cluster
  float part2[8 * 144];            // FC2 partials received from the cluster
  float G[10][8][kTerms];          // term multipliers per (item, token)
  int ids[kMaxSlotsTc];
  float tw[kMaxSlotsTc];
  int own[kMaxSlotsTc];            // first slot naming each valid expert, in slot order
  int own_cnt[4];
  float wtok[8];                   // FC1: router weight of the unit's expert per token
  float g3[3];                     // FC1: gate, up, down multipliers of the expert
  uint32_t routed;                 // FC1: tokens routed to the expert (bit mask)
  uint64_t fullA[10];              // weight tile + its scale chunks landed (TMA)
  uint64_t ready[10];              // activation terms, both scale sets and G in place (builders)
  uint64_t done[10];               // MMAs of the item complete
  uint64_t red1, red2;             // FC1 / FC2 partial rows this CTA reduces have landed
  uint32_t tmem;
};
template <int kN>
constexpr uint32_t fz_smem() {
  return FzCfg<kN>::kRing * FzCfg<kN>::kSlot + sizeof(SmemFz) + 1024;
}
static_assert(fz_smem<16>() <= 227 * 1024 && fz_smem<32>() <= 227 * 1024, "shared memory");

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Polls of an h-ready counter before the builder gives up (each poll is an
// L2 round trip of a few hundred nanoseconds: about two seconds in all).
constexpr uint32_t kFlagPollLimit = 1u << 22;
constexpr uint32_t kErrHFlag = 2048u, kErrFzRed = 4096u;

// One (item, token) activation row: the kTerms NVFP4 terms of 256 values
// (v, zero past `act` lanes) into the item's slot, its multipliers into G.
__device__ __forceinline__ void fz_build_row(float (&v)[8], uint8_t* slotp, uint32_t sfa_off, float* G, int token,
                                             int lane, bool act) {
  float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                  fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float G1 = term_g1(m);
  if (lane < kTerms) G[lane] = G1 * __uint_as_float((127u - 2u * lane) << 23);
  emit_stage_terms(v, G1, slotp + kSlotA, slotp + sfa_off + 4 * kChunkBytes, token, lane, act);
}

template <int kN>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap map13, const __grid_constant__ CUtensorMap map2, TcArgs a) {
  using Cfg = FzCfg<kN>;
  constexpr int R = Cfg::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  SmemFz& S = *reinterpret_cast<SmemFz*>(ring + R * Cfg::kSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = a.M, H = a.H, I = a.I, n = a.n_slots;
  const int C = a.split, s1 = a.s1;
  const int rank = (int)cluster_rank();
  const int q = blockIdx.x / C, sub = rank / s1, r1 = rank % s1;
  const int tiles1 = I / 64, ns2 = (I + 255) / 256, tiles2 = H / 128, nk = H / 256;
  const int cpo = (64 + s1 - 1) / s1, rpo1 = 2 * cpo;  // FC1 pairs per owner, partial rows per sender
  const int rpo2 = (128 + C - 1) / C;                   // FC2 rows per owner
  const bool is_epi = warp >= kEpiWarp0;
  const bool is_quant = warp >= kQuantWarp0 && warp < kQuantWarp0 + kQuantWarps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(&S.fullA[s], 1);
      mbar_init(&S.ready[s], kQuantWarps);
      mbar_init(&S.done[s], 1);
    }
    mbar_init(&S.red1, 1);
    mbar_init(&S.red2, 1);
    fence_mbar_init();
    tma_prefetch_desc(&map13);
    tma_prefetch_desc(&map2);
  }
  // cluster phase 1: this CTA runs and its barriers are initialised (awaited
  // before any remote store)
  cluster_arrive_release();
  if (warp == kMmaWarp0) tmem_alloc(&S.tmem, 512);
  // The next kernel may start its prologue; it waits (griddepcontrol.wait)
  // for this whole grid before it reads anything this launch writes.
  pdl_launch_dependents();
  pdl_wait();  // x and the routing come from the previous kernel

  // ---- routing: owners (the first slot naming each valid expert, in slot order)
  bool own_j = false;
  uint32_t bal = 0;
  if (warp < 4) {
    const int j = 32 * warp + lane;
    const int id = j < n ? route_id(a.ids, j, a.ids64, a.E) : -1;
    S.ids[j] = id;
    S.tw[j] = j < n ? ld_nc_f32(a.tw + j) : 0.f;
    const bool valid = j < n && id >= 0 && id < a.E;
    const uint32_t mm = __match_any_sync(0xffffffffu, valid ? id : -1 - lane);
    own_j = valid && (mm & ((1u << lane) - 1u)) == 0;  // earlier 32-slot chunks are checked below
  }
  __syncthreads();
  if (warp < 4) {
    const int j = 32 * warp + lane;
    for (int c = 0; own_j && c < warp; ++c)
      for (int k = 0; k < 32; ++k) own_j = own_j && S.ids[32 * c + k] != S.ids[j];
    bal = __ballot_sync(0xffffffffu, own_j);
    if (lane == 0) S.own_cnt[warp] = __popc(bal);
  }
  __syncthreads();
  if (own_j) {
    const int j = 32 * warp + lane;
    int base = 0;
    for (int c = 0; c < warp; ++c) base += S.own_cnt[c];
    S.own[base + __popc(bal & ((1u << lane) - 1u))] = j;
  }
  const int n_own = S.own_cnt[0] + S.own_cnt[1] + S.own_cnt[2] + S.own_cnt[3];
  __syncthreads();

  // ---- this CTA's work: an FC1 share, then an FC2 share (at most R items)
  const int u1 = q * (C / s1) + sub;
  const bool valid1 = u1 < n_own * tiles1;
  const int o1 = valid1 ? u1 / tiles1 : 0, tile1 = valid1 ? u1 % tiles1 : 0;
  const int e1 = valid1 ? S.ids[S.own[o1]] : -1;
  const int k0 = r1 * nk / s1;
  const int n1 = valid1 ? (r1 + 1) * nk / s1 - k0 : 0;
  const int t2 = q;
  const bool valid2 = t2 < tiles2;
  const int T2 = n_own * ns2;
  const int n2 = valid2 && T2 > rank ? (T2 - rank + C - 1) / C : 0;
  const int n_items = n1 + n2 < R ? n1 + n2 : R;  // (the plan keeps n1 + n2 <= R)
  auto item_o = [&](int i) { return (rank + C * (i - n1)) % n_own; };
  auto item_s2 = [&](int i) { return (rank + C * (i - n1)) / n_own; };
  auto item_groups = [&](int i) {
    if (i < n1) return 4;
    const int rem = tiles1 - 4 * item_s2(i);
    return rem < 4 ? rem : 4;
  };
  const uint64_t KG1 = (uint64_t)(H / 64), KG2 = (uint64_t)(I / 64);
  if (threadIdx.x == 0) {
    // every weight tile of the CTA, FC1's first (streaming once per layer:
    // evict-first in L2)
    const uint64_t wpol = l2_evict_first_policy();
    for (int i = 0; i < n_items; ++i) {
      uint8_t* slotp = ring + i * Cfg::kSlot;
      const int ng = item_groups(i);
      mbar_arrive_expect_tx(&S.fullA[i], kSlotA + (uint32_t)ng * kChunkBytes);
      if (i < n1) {
        const int st = k0 + i;
        const uint8_t* sfa = a.s13 + (((uint64_t)e1 * tiles1 + tile1) * KG1 + 4 * (uint64_t)st) * kChunkBytes;
        tma_load_2d_hint(slotp, &map13, st * 128, e1 * 2 * I + tile1 * 128, &S.fullA[i], wpol);
        bulk_load_hint(slotp + Cfg::kSFA, sfa, (uint32_t)ng * kChunkBytes, &S.fullA[i], wpol);
      } else {
        const int st = item_s2(i), e = S.ids[S.own[item_o(i)]];
        const uint8_t* sfa = a.s2 + (((uint64_t)e * tiles2 + t2) * KG2 + 4 * (uint64_t)st) * kChunkBytes;
        tma_load_2d_hint(slotp, &map2, st * 128, e * H + t2 * 128, &S.fullA[i], wpol);
        bulk_load_hint(slotp + Cfg::kSFA, sfa, (uint32_t)ng * kChunkBytes, &S.fullA[i], wpol);
      }
    }
    // the partial rows this CTA reduces: FC1 from the s1 CTAs of its
    // sub-cluster (gate and up rows of its pairs), FC2 from the C CTAs of
    // the cluster (its rows)
    if (valid1)
      mbar_arrive_expect_tx(&S.red1, (uint32_t)(s1 * 2 * ((64 - r1 + s1 - 1) / s1) * M * 4));
    else
      mbar_arrive(&S.red1);
    if (valid2)
      mbar_arrive_expect_tx(&S.red2, (uint32_t)(C * ((128 - rank + C - 1) / C) * M * 4));
    else
      mbar_arrive(&S.red2);
  }
  if (warp == 0 && valid1) {
    // router weight of the unit's expert per token
    float wt = 0.f;
    bool rt = false;
    if (lane < M)
      for (int k = 0; k < a.top_k; ++k)
        if (S.ids[lane * a.top_k + k] == e1) {
          wt += S.tw[lane * a.top_k + k];
          rt = true;
        }
    const uint32_t rm = __ballot_sync(0xffffffffu, rt);
    if (lane < M) S.wtok[lane] = wt;
    if (lane == 0) S.routed = rm;
  }
  if (warp == kQuantWarp0 && valid1 && lane < 3) {
    const float* gl13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * tiles1 * (H / 64) * kChunkBytes);
    const float* gl2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * tiles2 * (I / 64) * kChunkBytes);
    S.g3[lane] = ld_nc_f32(lane < 2 ? gl13 + 2 * e1 + lane : gl2 + e1);
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();

  if (warp < kMmaWarp0) {
    // (the producer issued everything above)
  } else if (warp < kMmaWarp0 + kMmaWarps) {
    // ---------------- MMA issuers (alternate items, one elected lane each)
    const int mw = warp - kMmaWarp0;
    const uint32_t tmem = S.tmem;
    const uint32_t idesc = idesc_mxf4nvf4(128, kN, false);
    for (int i = mw; i < n_items; i += kMmaWarps) {
      bool ok = mbar_wait(&S.fullA[i], 0, a.status, 2u);
      ok = ok && mbar_wait(&S.ready[i], 0, a.status, 2u);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int ng = item_groups(i);
      uint8_t* slotp = ring + i * Cfg::kSlot;
      const uint32_t sfa_t = tmem + Cfg::kTmemSF + i * 32, sfb_t = sfa_t + 16;
      const uint64_t da = smem_desc(smem_u32(slotp), 16, 1024, kLayoutSW128);
      const uint64_t db = smem_desc(smem_u32(slotp + kSlotA), 16, 1024, kLayoutSW128);
      for (int k = 0; k < ng; ++k)
        mma_nvf4_warp(tmem + kN * i, da + 2 * k, db + 2 * k, idesc, sfa_t + 4 * k, sfb_t + 4 * k, k > 0);
      mma_commit_warp(&S.done[i]);
    }
  } else if (is_quant) {
    // ---------------- activation terms and scales.  (No early exit: the four
    // warps meet at named barriers; after a wait that gave up they go on
    // without waiting.)
    const int qw = warp - kQuantWarp0;
    const uint32_t tq = S.tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    bool live = true;
    // both scale sets of item i into this warp's lane quarter, then its
    // arrival (the weight scales once the item's TMA has landed)
    auto publish = [&](int i) {
      uint8_t* slotp = ring + i * Cfg::kSlot;
      {
        const uint4 u = *reinterpret_cast<const uint4*>(slotp + Cfg::kSFB + lane * 16);
        const uint32_t r[16] = {u.x, 0u, 0u, 0u, u.y, 0u, 0u, 0u, u.z, 0u, 0u, 0u, u.w, 0u, 0u, 0u};
        tmem_st16(tq + Cfg::kTmemSF + i * 32 + 16, r);
      }
      if (live) live = __all_sync(0xffffffffu, mbar_wait(&S.fullA[i], 0, a.status, 32u));
      uint32_t r[16];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 u = *reinterpret_cast<const uint4*>(slotp + Cfg::kSFA + g * kChunkBytes + lane * 16);
        r[4 * g] = u.x;
        r[4 * g + 1] = u.y;
        r[4 * g + 2] = u.z;
        r[4 * g + 3] = u.w;
      }
      tmem_st16(tq + Cfg::kTmemSF + i * 32, r);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.ready[i]);
    };
    // FC1: the (item, token) rows of x, dealt over the four warps
    for (int p = qw; p < n1 * M; p += kQuantWarps) {
      const int i = p / M, t = p % M;
      float v[8];
      load_bf16x8(a.x + (size_t)t * H + (k0 + i) * 256 + lane * 8, v);
      fz_build_row(v, ring + i * Cfg::kSlot, Cfg::kSFA, S.G[i][t], t, lane, true);
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 32 * kQuantWarps);  // FC1's terms and scales are staged
    for (int i = 0; i < n1; ++i) publish(i);
    // FC2: warp qw takes items n1 + qw, n1 + qw + 4, ...: waits for the flags
    // of the w13 tiles its K stage of h comes from, loads h, builds the terms
    for (int i = n1 + qw; i < n_items; i += kQuantWarps) {
      const int o = item_o(i), s2 = item_s2(i);
      const int ntl = tiles1 - 4 * s2 < 4 ? tiles1 - 4 * s2 : 4;
      if (lane == 0) {
        const uint32_t* f = a.hflag + (size_t)o * ns2 + s2;
        const uint32_t want = (uint32_t)(ntl * s1);
        for (uint32_t pl = 0; ld_acquire_gpu(f) != want;)
          if (++pl > kFlagPollLimit) {
            atomicOr(a.status, kErrHFlag);
            break;
          }
      }
      __syncwarp();  // (lane 0's acquire orders the warp's loads of h below)
      const bool act = lane < 8 * ntl;  // lanes past the stage's valid K
      for (int t = 0; t < M; ++t) {
        float v[8];
        if (act) {
          fc2_activation(a, o, t, s2 * 256 + lane * 8, v);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        fz_build_row(v, ring + i * Cfg::kSlot, Cfg::kSFA, S.G[i][t], t, lane, act);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 32 * kQuantWarps);  // FC2's terms and scales are staged
    for (int i = n1; i < n_items; ++i) publish(i);
    // this CTA has read its share of each of its items' h; the last reader
    // of an item in the layer puts its two counters back to zero
    for (int i = n1 + qw; lane == 0 && i < n_items; i += kQuantWarps) {
      const size_t c = (size_t)item_o(i) * ns2 + item_s2(i);
      if (atomicAdd(a.hused + c, 1u) == (uint32_t)(tiles2 - 1)) {
        a.hflag[c] = 0u;
        a.hused[c] = 0u;
      }
    }
  } else {
    // ---------------- accumulator drain; after FC1's last item the FC1
    // reduction and h, after FC2's the FC2 partial rows.  Warps 7..10 own
    // lanes 32*(warp%4) ...
    const int qd = warp & 3;
    const int row = 32 * qd + lane;
    const uint32_t tq = S.tmem + ((uint32_t)(32 * qd) << 16);
    cluster_wait();  // phase 1: every CTA of the cluster runs (before remote stores)
    bool ok = true;
    float vout[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) vout[t] = 0.f;
    for (int i = 0; i < n_items; ++i) {
      if (ok) {
        // (ready: the builders' multipliers of the item are visible here)
        ok = mbar_wait(&S.ready[i], 0, a.status, 4u) && mbar_wait(&S.done[i], 0, a.status, 4u);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        uint32_t r[16];
        float acc[kN];
        tmem_ld16(tq + kN * i, r);
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(r[c]);
        if (kN > 16) {
          tmem_ld16(tq + kN * i + 16, r);
#pragma unroll
          for (int c = 0; c < 16; ++c) acc[(16 + c) % kN] = __uint_as_float(r[c]);
        }
#pragma unroll
        for (int t = 0; t < kN / kTerms; ++t)
          if (t < M) {
#pragma unroll
            for (int u = 0; u < kTerms; ++u) vout[t] = fmaf(acc[t * kTerms + u], S.G[i][t][u], vout[t]);
          }
      }
      if (i == n1 - 1) {
        // ---- FC1 reduction: pair p of the unit is owned by rank
        // sub*s1 + p % s1 of the sub-cluster; partial gate/up rows go there
        // by asynchronous stores counted on its barrier and are summed in
        // rank order; the owner writes h and publishes it
        const int pr = row & 63, owner = sub * s1 + pr % s1, j = (row >> 6) * cpo + pr / s1;
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (t < M) st_async_peer_f32(&S.part1[(r1 * M + t) * rpo1 + j], &S.red1, (uint32_t)owner, vout[t]);
#pragma unroll
        for (int t = 0; t < 8; ++t) vout[t] = 0.f;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&S.red1, 0, a.status, kErrFzRed));
        if (got)
          for (int idx = row; idx < M * cpo; idx += 128) {
            const int t = idx / cpo, jj = idx % cpo, pair = r1 + s1 * jj;
            if (pair >= 64) continue;
            float gate = 0.f, up = 0.f;
            for (int src = 0; src < s1; ++src) {
              gate += S.part1[(src * M + t) * rpo1 + jj];
              up += S.part1[(src * M + t) * rpo1 + cpo + jj];
            }
            const float hv =
                (S.routed >> t) & 1u ? gated_act(gate * S.g3[0], up * S.g3[1], a.act) * (S.wtok[t] * S.g3[2]) : 0.f;
            a.h[((size_t)o1 * M + t) * I + tile1 * 64 + pair] = hv;
          }
        named_bar_sync(2, 128);  // every h store of this CTA is made
        if (row == 0 && got) {
          fence_acq_rel_gpu();  // (cumulative: the drain warps' stores, ordered by the barrier)
          red_release_gpu_add(a.hflag + (size_t)o1 * ns2 + tile1 / 4, 1u);
        }
      }
    }
    if (valid2) {
      // ---- FC2 reduction: row r of the tile is owned by rank r % C
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (t < M)
          st_async_peer_f32(&S.part2[(rank * M + t) * rpo2 + row / C], &S.red2, (uint32_t)(row % C), vout[t]);
    }
  }

  tc_fence_before();
  __syncwarp();
  __syncthreads();  // tensor memory is no longer read or written
  if (warp == kMmaWarp0) tmem_dealloc(S.tmem, 512);
  if (!is_epi) cluster_wait();  // (the drain warps completed phase 1 already)
  if (is_epi && valid2 && __all_sync(0xffffffffu, mbar_wait(&S.red2, 0, a.status, kErrFzRed))) {
    const int row = 32 * (warp & 3) + lane;
    for (int idx = row; idx < M * rpo2; idx += 128) {
      const int t = idx / rpo2, j = idx % rpo2, orow = rank + C * j;
      if (orow >= 128) continue;
      float v = 0.f;
      for (int src = 0; src < C; ++src) v += S.part2[(src * M + t) * rpo2 + j];
      a.out[(size_t)t * H + t2 * 128 + orow] = __float2bfloat16_rn(v);
    }
  }
}

// K ranges per w13 tile: about 1.5 CTAs per SM in total (measured best on
// GB300 for 1..8 tokens: more ranges shorten each CTA's weight stream, fewer
// leave room for FC2's CTAs beside them), at most 8.
int fc1_split(int units, int H, int sms) {
  const int nk = H / 256;
  int s = 3 * sms / (2 * units);
  s = s > 8 ? 8 : s;
  s = s > nk ? nk : s;
  return s < 1 ? 1 : s;
}

// CTAs per w2 row tile (the cluster): 8, or the number of (slot, K stage)
// items if smaller (the items of a tile spread over more SMs), but never
// more than about 1.5 CTAs per SM, so that FC2 runs in one wave once FC1
// leaves the SMs instead of a wave and a tail.  Measured on GB300: H = 4096
// at 4 tokens 33.7-34.1 us with 6-8 CTAs per tile against 35.7 with 4;
// H = 2560, 4 and 8 tokens, 8 beats 7 by 2-4%; H = 7168 (56 tiles), 4 CTAs
// (224) beat 8 (448) by 9% at one token and 5 (280) by 15% at two.
int fc2_split(int n_slots, int H, int I, int sms) {
  const int tiles = H / 128, items = n_slots * ((I + 255) / 256);
  int q = items < 8 ? (items < 1 ? 1 : items) : 8;
  if (2 * q * tiles > 3 * sms) q = 3 * sms / (2 * tiles);
  return q < 1 ? 1 : q;
}

}  // namespace

// Bytes of one K stage's activation image: B tile, scales, multipliers.
static int ximg_stride(int M) {
  const int N = (kTerms * M + 15) / 16 * 16;
  return (N * 128 + kChunkBytes + 16 * M + 127) / 128 * 128;
}
static size_t h_bytes(int M, int I, int top_k) {
  const size_t b = (size_t)M * top_k * M * (size_t)I * sizeof(float);
  return (b + 255) & ~(size_t)255;
}

// From this batch size on, FC2's activation terms come from a pre-pass (built
// once per slot instead of once per CTA of the slot's row tiles); below it
// FC2 builds them itself and the layer saves a launch on its critical path.
constexpr int kHPrepassMinM = 2;

// h [M*top_k slots][M][I] FP32, the activation images of x's H/256 K
// stages, and (M >= kHPrepassMinM) those of h's (slot, K stage) pairs.
size_t decode_tc_scratch_bytes(int M, int H, int I, int top_k, int num_sms) {
  (void)num_sms;
  size_t b = h_bytes(M, I, top_k) + (size_t)(H / 256) * ximg_stride(M);
  if (M >= kHPrepassMinM) b += (size_t)M * top_k * ((I + 255) / 256) * ximg_stride(M);
  return b;
}

cudaError_t launch_decode_tc(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                             const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                             int top_k, const ActParams& act, float* scratch, uint32_t* status, int num_sms, cudaStream_t st,
                             int* cu_err) {
  CUtensorMap m13, m2;
  // (w13: 2I rows per expert; the w1 of non-gated experts: I)
  const uint64_t rows13 = (uint64_t)E * (act.kind == MOE_FP4_ACT_RELU2 ? I : 2 * I);
  CUresult r = make_fp4_map(&m13, w13, (uint64_t)H / 2, rows13, 128);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&m2, w2, (uint64_t)I / 2, (uint64_t)E * H, 128);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    err = cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    // all of the unified L1/shared array as shared memory: two CTAs per SM
    // (FC2's beside FC1's)
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  TcArgs a = {};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ids = ids;
  a.ids64 = ids64;
  a.tw = tw;
  a.s13 = static_cast<const uint8_t*>(s13);
  a.s2 = static_cast<const uint8_t*>(s2);
  a.h = scratch;
  a.ximg = reinterpret_cast<uint8_t*>(scratch) + h_bytes(M, I, top_k);
  a.ximg_stride = ximg_stride(M);
  a.himg = M >= kHPrepassMinM ? a.ximg + (size_t)(H / 256) * a.ximg_stride : nullptr;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.status = status;
  a.M = M;
  a.E = E;
  a.H = H;
  a.I = I;
  a.top_k = top_k;
  a.n_slots = M * top_k;
  a.N = (kTerms * M + 15) / 16 * 16;
  a.act = act;
  const int sms = num_sms > 0 ? num_sms : 152;

  // activation pre-pass: one CTA per K stage, one warp per token
  cudaLaunchAttribute at0[1];
  at0[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at0[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c0 = {};
  c0.gridDim = dim3((unsigned)(H / 256));
  c0.blockDim = dim3((unsigned)(32 * M));
  c0.stream = st;
  c0.attrs = at0;
  c0.numAttrs = 1;
  err = cudaLaunchKernelEx(&c0, decode_quant_x_kernel, a);
  if (err != cudaSuccess) return err;

  // FC1: K ranges per w13 tile (independent CTAs); programmatic dependent
  // launch so that its prologue overlaps the pre-pass
  const int tiles1 = act.kind == MOE_FP4_ACT_RELU2 ? (I + 127) / 128 : I / 64;
  const int units1 = a.n_slots * tiles1;
  const int s1 = fc1_split(units1, H, sms);
  a.split = s1;
  cudaLaunchAttribute at1[2];
  at1[0].id = cudaLaunchAttributeClusterDimension;
  at1[0].val.clusterDim.x = (unsigned)s1;
  at1[0].val.clusterDim.y = 1;
  at1[0].val.clusterDim.z = 1;
  at1[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at1[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c1 = {};
  c1.gridDim = dim3((unsigned)(units1 * s1));
  c1.blockDim = dim3(kTcThreads);
  c1.dynamicSmemBytes = kTcSmem;
  c1.stream = st;
  c1.attrs = at1;
  c1.numAttrs = 2;
  err = cudaLaunchKernelEx(&c1, decode_tc_kernel<false>, m13, a);
  if (err != cudaSuccess) return err;

  if (a.himg) {
    // h's activation pre-pass: one CTA per (route slot, K stage), a warp per token
    cudaLaunchConfig_t ch = {};
    ch.gridDim = dim3((unsigned)(a.n_slots * ((I + 255) / 256)));
    ch.blockDim = dim3((unsigned)(32 * M));
    ch.stream = st;
    ch.attrs = at0;
    ch.numAttrs = 1;
    err = cudaLaunchKernelEx(&ch, decode_quant_h_kernel, a);
    if (err != cudaSuccess) return err;
  }

  // FC2: clusters of CTAs per w2 row tile, dependent launch on the kernel before
  const int tiles2 = H / 128;
  const int q = fc2_split(a.n_slots, H, I, sms);
  a.split = q;
  cudaLaunchAttribute at2[2];
  at2[0].id = cudaLaunchAttributeClusterDimension;
  at2[0].val.clusterDim.x = (unsigned)q;
  at2[0].val.clusterDim.y = 1;
  at2[0].val.clusterDim.z = 1;
  at2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at2[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c2 = {};
  c2.gridDim = dim3((unsigned)(tiles2 * q));
  c2.blockDim = dim3(kTcThreads);
  c2.dynamicSmemBytes = kTcSmem;
  c2.stream = st;
  c2.attrs = at2;
  c2.numAttrs = 2;
  return cudaLaunchKernelEx(&c2, decode_tc_kernel<true>, m2, a);
}


// ---------------------------------------------------------------- single launch, host side

// Words of the single-launch kernel's synchronisation area: an h-ready
// counter and a reader count per (owner, K stage of h), for up to
// MOE_FP4_DECODE_MAX_M tokens (so that its place in the workspace does not
// depend on the batch).  Zero between calls.
size_t decode_sync_bytes(int H, int I, int top_k) {
  (void)H;
  const size_t slots = (size_t)MOE_FP4_DECODE_MAX_M * top_k;
  const size_t words = 2 * slots * ((I + 255) / 256);
  return (words * 4 + 255) & ~(size_t)255;
}

namespace {
// Clusters of `C` single-launch CTAs for kN activation rows that can be
// resident at once on the current device (cached per device, cluster size
// and kN); 0 if the query fails.
template <int kN>
int fused_max_clusters(int C) {
  static int cache[64][9] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || C < 1 || C > 8) return 0;
  if (cache[dev][C] != 0) return cache[dev][C] > 0 ? cache[dev][C] : 0;
  int n = 0;
  cudaError_t e =
      cudaFuncSetAttribute(decode_fused_kernel<kN>, cudaFuncAttributeMaxDynamicSharedMemorySize, fz_smem<kN>());
  if (e == cudaSuccess) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3((unsigned)(C * 16));
    c.blockDim = dim3(kTcThreads);
    c.dynamicSmemBytes = fz_smem<kN>();
    c.attrs = at;
    c.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, decode_fused_kernel<kN>, &c);
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[dev][C] = n > 0 ? n : -1;
  return n;
}
}  // namespace

// The single-launch geometry for a shape, or false if none fits: clusters of
// C = 8 CTAs, else 4 (the w2 tile's items dealt over C), FC1 K ranges s1 per
// w13 tile (C, C/2, ... 1, at most H/256; the largest that fits), as many
// clusters Q as the larger of the (slot, w13 tile) units / (C / s1) and the
// w2 tiles; all Q clusters resident at once on the current device (the CTAs
// wait for each other's h), and every CTA's items (its FC1 K stages and its
// share of the w2 tile's (slot, K stage) items) within the ring, so that all
// weight tiles are in flight from the start.  Up to 8 tokens (4 with the
// larger ring).  *cap_out (if non-null) receives the resident-cluster limit
// of the chosen C.
bool decode_fused_plan(int M, int H, int I, int top_k, int* C_out, int* s1_out, int* Q_out, int* cap_out) {
  if (M < 1 || M > 8) return false;
  const int n_slots = M * top_k;
  const int units = n_slots * (I / 64), tiles2 = H / 128, nk = H / 256, ns2 = (I + 255) / 256;
  const int ring = M <= 4 ? FzCfg<16>::kRing : FzCfg<32>::kRing;
  for (int C = 8; C >= 4; C /= 2) {
    const int cap = M <= 4 ? fused_max_clusters<16>(C) : fused_max_clusters<32>(C);
    if (cap <= 0) continue;
    for (int s1 = C; s1 >= 1; s1 /= 2) {
      if (s1 > nk) continue;
      const int per = C / s1;
      int Q = (units + per - 1) / per;
      if (Q < tiles2) Q = tiles2;
      const int items = (nk + s1 - 1) / s1 + (n_slots * ns2 + C - 1) / C;
      if (Q <= cap && items <= ring) {
        *C_out = C;
        *s1_out = s1;
        *Q_out = Q;
        if (cap_out) *cap_out = cap;
        return true;
      }
    }
  }
  return false;
}

cudaError_t launch_decode_fused(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                                const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                                int top_k, const ActParams& act, float* scratch, uint32_t* sync, uint32_t* status,
                                cudaStream_t st, int* cu_err) {
  int C = 0, s1 = 0, Q = 0;
  if (!decode_fused_plan(M, H, I, top_k, &C, &s1, &Q, nullptr)) return cudaErrorInvalidConfiguration;
  CUtensorMap m13, m2;
  CUresult r = make_fp4_map(&m13, w13, (uint64_t)H / 2, (uint64_t)E * 2 * I, 128);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&m2, w2, (uint64_t)I / 2, (uint64_t)E * H, 128);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  TcArgs a = {};
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
  a.N = (kTerms * M + 15) / 16 * 16;
  a.act = act;
  a.split = C;
  a.s1 = s1;
  a.hflag = sync;
  a.hused = sync + (size_t)MOE_FP4_DECODE_MAX_M * top_k * ((I + 255) / 256);
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3((unsigned)(Q * C));
  c.blockDim = dim3(kTcThreads);
  c.stream = st;
  c.attrs = at;
  c.numAttrs = 2;
  if (M <= 4) {
    c.dynamicSmemBytes = fz_smem<16>();
    return cudaLaunchKernelEx(&c, decode_fused_kernel<16>, m13, m2, a);
  }
  c.dynamicSmemBytes = fz_smem<32>();
  return cudaLaunchKernelEx(&c, decode_fused_kernel<32>, m13, m2, a);
}

}  // namespace moe_fp4
