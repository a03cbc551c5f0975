// Decode band (M <= 8 tokens) for MXFP4 weights: the layer as the HBM-bound
// GEMV it is, on the warp-level tensor-core MMA.  (NVFP4 weights take the
// tcgen05 path in decode_tc.cu; launch_decode below dispatches.)
//
// Prior art: the pages' tiny-decode kernel pair (b12x PR #22, "rp-native
// tiny-decode kernel for w4a8_mx (M=1)", section What) -- FC1 streams the
// routed experts' packed nibbles with one 16 B ld.global.nc per 32
// K-elements, decodes them in registers and writes an FP32 gate/up
// intermediate; FC2 applies SiLU inline, decodes the down weights and does
// the router-weighted sum into the BF16 output.  The section's Notes record
// why two plain launches beat a single cooperative launch (a grid barrier
// deadlocked when CTAs were not co-resident) and list folding the wrapper's
// zero-fills into the kernels as a follow-up.
//
// This implementation, for sm_103a:
//   * Routing lives inside the kernels (the small-batch "direct" idea of
//     flashinfer PR #4285, "sync SM12x NVFP4 fused-MoE kernels": read the
//     top-k ids directly instead of a separate routing pass).  An expert's
//     work is owned by the first slot that names it, so every routed expert's
//     weights are streamed exactly once; ids < 0 or >= E are never
//     dereferenced and contribute exactly zero (b12x PR #311, conversation).
//   * The multiply-adds run on the warp-level tensor-core MMA
//     (mma.sync m16n8k16, f16 inputs, FP32 accumulate) so that the FP32 pipe
//     is left to the decode: each streamed 16 B of nibbles is decoded in
//     registers by the hardware E2M1 -> f16 convert (exact) and multiplied by
//     its block scale in f16 (exact: an E4M3 scale, or an MXFP4 scale divided
//     by the projection's power-of-two multiplier), and the up-to-8 tokens
//     are the MMA's N = 8 columns, so the cost per weight byte does not grow
//     with M.  A lane (g, c) of a warp holds rows g and g+8 of a 16-row tile
//     and bytes 16c..16c+15 of each 64-byte K segment (128 elements); the
//     activations of token g are the B fragments, scaled per (segment, token)
//     by a power of two so they convert to f16 exactly (BF16 inputs) or to
//     f16 rounding (the FP32 intermediate), and the scale is undone on the
//     FP32 result of the segment.
//   * FC1: a CTA owns 16 (gate, up) pairs of one expert over the whole K; its
//     8 warps split the K segments and meet in shared memory, so
//     h = SiLU(gate) * up is final inside the CTA.  The router weight (summed
//     over the token's slots naming this expert) and the down projection's
//     multiplier are folded into h (FC2 is linear in h), so FC2 only sums.
//     Each CTA also bulk-prefetches its share of the expert's down projection
//     into L2 for FC2.
//   * FC2: a CTA owns 16 output rows for every routed expert; its warps take
//     (expert, K segment) units round-robin and meet in shared memory in a
//     fixed order, so each output element is written once, deterministically
//     (no zero-fill, no atomics, no cross-CTA synchronisation).  It is
//     launched with programmatic dependent launch and waits for FC1 with
//     griddepcontrol.wait (a hardware dependency, not a spin).
#include "common.cuh"

namespace moe_fp4 {

constexpr int kThreads = 256;  // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 128;       // K elements per warp segment (4 lanes x 32)
constexpr int kMaxSlots = 128;  // M <= 8, top_k <= 16

struct DecodeParams {
  const __nv_bfloat16* x;
  const uint8_t* w13;
  const uint8_t* s13;
  const uint8_t* w2;
  const uint8_t* s2;
  const int32_t* ids;
  const float* tw;
  __nv_bfloat16* out;
  int M, E, H, I, top_k, fmt;
  int n_slots;
  float* h;  // [n_slots][M][I]: router-weighted SiLU(gate)*up of the slot's expert
};

// ---------------------------------------------------------------- helpers
// Warp-cooperative over the staged ids: does a slot before `slot` name e, and
// which tokens route to e.
__device__ __forceinline__ void warp_route(const int* s_ids, int n, int top_k, int e, int slot, bool* dup,
                                           uint32_t* mask) {
  const int lane = threadIdx.x & 31;
  bool d = false;
  uint32_t m = 0;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const bool hit = j < n && s_ids[j] == e;
    d |= __any_sync(0xffffffffu, hit && j < slot);
    m |= __reduce_or_sync(0xffffffffu, hit ? (1u << (j / top_k)) : 0u);
  }
  *dup = d;
  *mask = m;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 {s, s} for one block scale byte: E4M3 as is; UE8M0 divided by the
// projection's multiplier 2^bias (flushed to zero below 2^-24, NaN kept).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t b, int fmt, int bias) {
  if (fmt == MOE_FP4_NVFP4) {
    uint32_t h2;
    const uint16_t in = (uint16_t)(b | (b << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return h2;
  }
  const int k = (int)b - 127 - bias;
  uint32_t h;
  if (b == 255u)
    h = 0x7e00u;
  else if (k >= -14)
    h = (uint32_t)(k + 15) << 10;
  else if (k >= -24)
    h = 1u << (k + 24);
  else
    h = 0u;
  return h | (h << 16);
}

// Power-of-two exponent s so that amax * 2^s lies in [2^14, 2^15).
__device__ __forceinline__ int act_scale_exp(float amax) {
  const int E = (int)((__float_as_uint(amax) >> 23) & 0xffu);
  int s = 141 - E;
  return s > 126 ? 126 : s;
}
__device__ __forceinline__ float exp2i(int s) { return __int_as_float((127 + s) << 23); }

// Pack two FP32 values (lo, hi) times f into f16x2.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi, float f) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi * f), "f"(lo * f));
  return r;
}

// B fragments of one segment for this lane's token: 32 BF16 activations ->
// 16 f16x2 registers scaled by 2^s (s shared by the 4 lanes of the token).
// Returns 2^-s.
__device__ __forceinline__ float act_from_bf16(const uint4 (&u)[4], uint32_t (&b)[16]) {
  uint32_t m = 0;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t ws[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t a = ws[j] & 0x7fff7fffu;
      m = max(m, max(a & 0xffffu, a >> 16));
    }
  }
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const int s = act_scale_exp(__uint_as_float(m << 16));
  const float f = exp2i(s);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t ws[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      b[4 * v + j] = pack_f16x2(__uint_as_float(ws[j] << 16), __uint_as_float(ws[j] & 0xffff0000u), f);
  }
  return exp2i(-s);
}

__device__ __forceinline__ float act_from_f32(const float4 (&u)[8], uint32_t (&b)[16]) {
  float m = 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) m = fmaxf(m, fmaxf(fmaxf(fabsf(u[v].x), fabsf(u[v].y)), fmaxf(fabsf(u[v].z), fabsf(u[v].w))));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const int s = act_scale_exp(m);
  const float f = exp2i(s);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    b[2 * v] = pack_f16x2(u[v].x, u[v].y, f);
    b[2 * v + 1] = pack_f16x2(u[v].z, u[v].w, f);
  }
  return exp2i(-s);
}

// One 16-row x 128-K tile segment: rows g (wg) and g+8 (wh), block scales
// (f16x2) of the two 16-element halves of each row's 32-element chunk.
__device__ __forceinline__ void tile_segment(float (&d)[4], const uint4& wg, const uint4& wh, uint32_t sg0,
                                             uint32_t sg1, uint32_t sh0, uint32_t sh1, const uint32_t (&b)[16]) {
  const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w};
  const uint32_t hw[4] = {wh.x, wh.y, wh.z, wh.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t hg[4], hh[4];
    e2m1x8_to_half2x4(gw[j], hg);
    e2m1x8_to_half2x4(hw[j], hh);
    const uint32_t sg = j < 2 ? sg0 : sg1, sh = j < 2 ? sh0 : sh1;
    mma16816(d, hmul2(hg[0], sg), hmul2(hh[0], sh), hmul2(hg[1], sg), hmul2(hh[1], sh), b[4 * j], b[4 * j + 1]);
    mma16816(d, hmul2(hg[2], sg), hmul2(hh[2], sh), hmul2(hg[3], sg), hmul2(hh[3], sh), b[4 * j + 2],
             b[4 * j + 3]);
  }
}

// Scale bytes for a lane's 32-element chunk of a row: (half 0, half 1).
__device__ __forceinline__ void chunk_scale_pair(uint32_t word, int kb, int fmt, int bias, uint32_t* s0,
                                                 uint32_t* s1) {
  if (fmt == MOE_FP4_MXFP4) {
    *s0 = *s1 = scale_f16x2((word >> (8 * (kb & 3))) & 0xffu, fmt, bias);
  } else {
    *s0 = scale_f16x2((word >> (8 * (kb & 3))) & 0xffu, fmt, bias);
    *s1 = scale_f16x2((word >> (8 * ((kb & 3) + 1))) & 0xffu, fmt, bias);
  }
}

// Exponent of a power-of-two FP32 multiplier (the MXFP4 per-projection one).
__device__ __forceinline__ int pow2_exp(float g) { return (int)((__float_as_uint(g) >> 23) & 0xffu) - 127; }

// ---------------------------------------------------------------- FC1
// grid.x = I/16 pair tiles, grid.y = route slot.
__global__ void __launch_bounds__(kThreads, 2) decode_fc1_kernel(DecodeParams p) {
  pdl_launch_dependents();
  const int slot = blockIdx.y;
  const int e = __ldg(p.ids + slot);
  if (e < 0 || e >= p.E) return;

  __shared__ int s_ids[kMaxSlots];
  __shared__ float s_tw[kMaxSlots];
  __shared__ float s_red[kWarps][2][32][4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int H = p.H, I = p.I, fmt = p.fmt, n = p.n_slots, M = p.M;
  const int KG = k_groups(H, fmt);
  const int nseg = H / kSeg;
  const int nmy = warp < nseg ? (nseg - warp + kWarps - 1) / kWarps : 0;
  const size_t row_bytes = (size_t)H / 2;
  const uint8_t* wexp = p.w13 + (size_t)e * 2 * I * row_bytes;
  const uint8_t* sexp = p.s13 + (size_t)e * scale_chunk_bytes(2 * I, H, fmt);
  const float* gl13 = reinterpret_cast<const float*>(p.s13 + (size_t)p.E * scale_chunk_bytes(2 * I, H, fmt));
  const float* gl2 = reinterpret_cast<const float*>(p.s2 + (size_t)p.E * scale_chunk_bytes(H, I, fmt));
  const float g_gate = __ldg(gl13 + 2 * e), g_up = __ldg(gl13 + 2 * e + 1);
  const int bias_g = fmt == MOE_FP4_MXFP4 ? pow2_exp(g_gate) : 0;
  const int bias_u = fmt == MOE_FP4_MXFP4 ? pow2_exp(g_up) : 0;
  const uint64_t pol = l2_evict_first_policy();

  const int n0 = 16 * blockIdx.x;  // first pair of this CTA
  const int rg = (n0 / 64) * kRowTile + (n0 % 64) + g;  // gate row of pair n0 + g
  const int rows[4] = {rg, rg + 8, rg + 64, rg + 72};  // gate g, gate g+8, up g, up g+8
  const bool has_tok = g < M;

  struct Seg {
    uint4 w[4];
    uint32_t s[4];
    uint4 x[4];
  };
  auto load_seg = [&](int jj, Seg& sg) {
    const int seg = warp + kWarps * jj;
    const int kb = fmt == MOE_FP4_MXFP4 ? 4 * seg + c : 8 * seg + 2 * c;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sg.w[i] = ld_stream_16_ef(wexp + (size_t)rows[i] * row_bytes + seg * (kSeg / 2) + 16 * c, pol);
      sg.s[i] = ld_nc_u32(sexp + (scale_offset(rows[i], kb, KG) & ~(size_t)3));
    }
    if (has_tok) {
      const uint4* xp = reinterpret_cast<const uint4*>(p.x + (size_t)g * H + seg * kSeg + 32 * c);
#pragma unroll
      for (int v = 0; v < 4; ++v) sg.x[v] = __ldg(xp + v);
    } else {
#pragma unroll
      for (int v = 0; v < 4; ++v) sg.x[v] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  Seg sa, sb;
  if (nmy > 0) load_seg(0, sa);
  if (nmy > 1) load_seg(1, sb);

  // stage routes; prefetch this CTA's share of the expert's FC2 rows into L2
  for (int j = threadIdx.x; j < n; j += kThreads) {
    s_ids[j] = __ldg(p.ids + j);
    s_tw[j] = __ldg(p.tw + j);
  }
  if (threadIdx.x == 32) {
    const size_t w2_bytes = (size_t)H * (I / 2);
    const size_t share = ((w2_bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t off = share * blockIdx.x;
    if (off < w2_bytes) {
      const size_t len = off + share <= w2_bytes ? share : w2_bytes - off;
      prefetch_l2_bulk(p.w2 + (size_t)e * w2_bytes + off, (uint32_t)len);
    }
    if (blockIdx.x == 0) {
      const size_t sb2 = scale_chunk_bytes(H, I, fmt);
      prefetch_l2_bulk(p.s2 + (size_t)e * sb2, (uint32_t)sb2);
    }
  }
  __syncthreads();
  bool dup;
  uint32_t mask;
  warp_route(s_ids, n, p.top_k, e, slot, &dup, &mask);
  if (dup) return;  // another slot names the same expert and does the work

  float acc_g[4] = {0.f, 0.f, 0.f, 0.f}, acc_u[4] = {0.f, 0.f, 0.f, 0.f};
  auto compute_seg = [&](int jj, const Seg& sg) {
    const int seg = warp + kWarps * jj;
    const int kb = fmt == MOE_FP4_MXFP4 ? 4 * seg + c : 8 * seg + 2 * c;
    uint32_t b[16];
    const float inv = act_from_bf16(sg.x, b);
    const float inv0 = __shfl_sync(0xffffffffu, inv, (2 * c) << 2);
    const float inv1 = __shfl_sync(0xffffffffu, inv, (2 * c + 1) << 2);
    uint32_t sc[4][2];
    chunk_scale_pair(sg.s[0], kb, fmt, bias_g, &sc[0][0], &sc[0][1]);
    chunk_scale_pair(sg.s[1], kb, fmt, bias_g, &sc[1][0], &sc[1][1]);
    chunk_scale_pair(sg.s[2], kb, fmt, bias_u, &sc[2][0], &sc[2][1]);
    chunk_scale_pair(sg.s[3], kb, fmt, bias_u, &sc[3][0], &sc[3][1]);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_segment(d, sg.w[0], sg.w[1], sc[0][0], sc[0][1], sc[1][0], sc[1][1], b);
    acc_g[0] = fmaf(d[0], inv0, acc_g[0]);
    acc_g[1] = fmaf(d[1], inv1, acc_g[1]);
    acc_g[2] = fmaf(d[2], inv0, acc_g[2]);
    acc_g[3] = fmaf(d[3], inv1, acc_g[3]);
    float du[4] = {0.f, 0.f, 0.f, 0.f};
    tile_segment(du, sg.w[2], sg.w[3], sc[2][0], sc[2][1], sc[3][0], sc[3][1], b);
    acc_u[0] = fmaf(du[0], inv0, acc_u[0]);
    acc_u[1] = fmaf(du[1], inv1, acc_u[1]);
    acc_u[2] = fmaf(du[2], inv0, acc_u[2]);
    acc_u[3] = fmaf(du[3], inv1, acc_u[3]);
  };
  for (int jj = 0; jj < nmy; jj += 2) {
    compute_seg(jj, sa);
    if (jj + 2 < nmy) load_seg(jj + 2, sa);
    if (jj + 1 < nmy) {
      compute_seg(jj + 1, sb);
      if (jj + 3 < nmy) load_seg(jj + 3, sb);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s_red[warp][0][lane][i] = acc_g[i];
    s_red[warp][1][lane][i] = acc_u[i];
  }
  __syncthreads();

  // one thread per (row, token) of the 16x8 tile
  if (threadIdx.x < 128) {
    const int ln = threadIdx.x >> 2, i = threadIdx.x & 3;
    const int row = (ln >> 2) + 8 * (i >> 1);
    const int t = 2 * (ln & 3) + (i & 1);
    if (t < M && ((mask >> t) & 1u)) {
      float gsum = 0.f, usum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        gsum += s_red[w][0][ln][i];
        usum += s_red[w][1][ln][i];
      }
      float wsum = 0.f;
      for (int j = 0; j < p.top_k; ++j)
        if (s_ids[t * p.top_k + j] == e) wsum += s_tw[t * p.top_k + j];
      const float gate = gsum * g_gate, up = usum * g_up;
      p.h[((size_t)slot * M + t) * I + n0 + row] = silu(gate) * up * (wsum * __ldg(gl2 + e));
    }
  }
}

// ---------------------------------------------------------------- FC2
// grid.x = H/16 output row tiles.
__global__ void __launch_bounds__(kThreads, 2) decode_fc2_kernel(DecodeParams p) {
  const int H = p.H, I = p.I, fmt = p.fmt, n = p.n_slots, M = p.M;
  __shared__ int s_ids[kMaxSlots];
  __shared__ int s_list[kMaxSlots];
  __shared__ int s_nact;
  __shared__ float s_red[kWarps][32][4];

  for (int j = threadIdx.x; j < n; j += kThreads) s_ids[j] = __ldg(p.ids + j);
  __syncthreads();
  // active slots (first slot naming each valid expert), in slot order
  if (threadIdx.x < 32) {
    int cnt = 0;
    for (int base = 0; base < n; base += 32) {
      const int j = base + threadIdx.x;
      const int ej = j < n ? s_ids[j] : -1;
      bool act = ej >= 0 && ej < p.E;
      for (int i = 0; act && i < j; ++i)
        if (s_ids[i] == ej) act = false;
      const uint32_t bal = __ballot_sync(0xffffffffu, act);
      if (act) s_list[cnt + __popc(bal & ((1u << threadIdx.x) - 1u))] = j;
      cnt += __popc(bal);
    }
    if (threadIdx.x == 0) s_nact = cnt;
  }
  __syncthreads();
  const int nact = s_nact;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const size_t row_bytes = (size_t)I / 2;
  const int KG = k_groups(I, fmt);
  const size_t s_bytes = scale_chunk_bytes(H, I, fmt);
  const float* gl2 = reinterpret_cast<const float*>(p.s2 + (size_t)p.E * s_bytes);
  const int r0 = 16 * blockIdx.x;
  const int nseg = (I + kSeg - 1) / kSeg;
  const int nunits = nact * nseg;

  pdl_wait();  // FC1's h is complete and visible

  struct Unit {
    uint4 w[2];
    uint32_t s[2];
    float4 h[8];
    uint32_t mask;
    int bias;
  };
  auto load_unit = [&](int u, Unit& un) {
    const int a = u / nseg, seg = u % nseg;
    const int slot = s_list[a];
    const int e = s_ids[slot];
    bool dup;
    warp_route(s_ids, n, p.top_k, e, slot, &dup, &un.mask);
    un.bias = fmt == MOE_FP4_MXFP4 ? pow2_exp(__ldg(gl2 + e)) : 0;
    const bool in_k = seg * kSeg + 32 * c < I;
    const int kb = fmt == MOE_FP4_MXFP4 ? 4 * seg + c : 8 * seg + 2 * c;
    const uint8_t* wexp = p.w2 + (size_t)e * H * row_bytes;
    const uint8_t* sexp = p.s2 + (size_t)e * s_bytes;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + g + 8 * i;
      if (in_k) {
        un.w[i] = ld_stream_16(wexp + (size_t)r * row_bytes + seg * (kSeg / 2) + 16 * c);
        un.s[i] = ld_nc_u32(sexp + (scale_offset(r, kb, KG) & ~(size_t)3));
      } else {
        un.w[i] = make_uint4(0u, 0u, 0u, 0u);
        un.s[i] = 0u;
      }
    }
    const bool tok = g < M && ((un.mask >> g) & 1u) && in_k;
    const float4* hp = reinterpret_cast<const float4*>(p.h + ((size_t)slot * M + (g < M ? g : 0)) * I + seg * kSeg + 32 * c);
#pragma unroll
    for (int v = 0; v < 8; ++v) un.h[v] = tok ? __ldcg(hp + v) : make_float4(0.f, 0.f, 0.f, 0.f);
  };

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  auto compute_unit = [&](int u, const Unit& un) {
    const int seg = u % nseg;
    const int kb = fmt == MOE_FP4_MXFP4 ? 4 * seg + c : 8 * seg + 2 * c;
    uint32_t b[16];
    const float inv = act_from_f32(un.h, b);
    const float inv0 = __shfl_sync(0xffffffffu, inv, (2 * c) << 2);
    const float inv1 = __shfl_sync(0xffffffffu, inv, (2 * c + 1) << 2);
    uint32_t sg0, sg1, sh0, sh1;
    chunk_scale_pair(un.s[0], kb, fmt, un.bias, &sg0, &sg1);
    chunk_scale_pair(un.s[1], kb, fmt, un.bias, &sh0, &sh1);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    tile_segment(d, un.w[0], un.w[1], sg0, sg1, sh0, sh1, b);
    acc[0] = fmaf(d[0], inv0, acc[0]);
    acc[1] = fmaf(d[1], inv1, acc[1]);
    acc[2] = fmaf(d[2], inv0, acc[2]);
    acc[3] = fmaf(d[3], inv1, acc[3]);
  };
  Unit ua, ub;
  const int u0 = warp;
  if (u0 < nunits) load_unit(u0, ua);
  if (u0 + kWarps < nunits) load_unit(u0 + kWarps, ub);
  for (int u = u0; u < nunits; u += 2 * kWarps) {
    compute_unit(u, ua);
    if (u + 2 * kWarps < nunits) load_unit(u + 2 * kWarps, ua);
    if (u + kWarps < nunits) {
      compute_unit(u + kWarps, ub);
      if (u + 3 * kWarps < nunits) load_unit(u + 3 * kWarps, ub);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s_red[warp][lane][i] = acc[i];
  __syncthreads();
  // sum the warps in a fixed order, apply nothing else (weights and
  // multipliers are in h), cast once, write every output element
  if (threadIdx.x < 128) {
    const int ln = threadIdx.x >> 2, i = threadIdx.x & 3;
    const int row = (ln >> 2) + 8 * (i >> 1);
    const int t = 2 * (ln & 3) + (i & 1);
    if (t < M) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += s_red[w][ln][i];
      p.out[(size_t)t * H + r0 + row] = __float2bfloat16_rn(v);
    }
  }
}

// ---------------------------------------------------------------- host side
bool decode_tc_supported(int fmt);
size_t decode_tc_scratch_bytes(int M, int H, int I, int top_k, int num_sms);
cudaError_t launch_decode_tc(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                             const int32_t* ids, const float* tw, void* out, int M, int E, int H, int I, int top_k,
                             float* part1, uint32_t* status, int num_sms, cudaStream_t st, int* cu_err);

// Scratch before the 256-byte status block: MXFP4, h [M*top_k][M][I] FP32;
// NVFP4, FC1's partial sums (decode_tc_scratch_bytes).
static size_t decode_scratch_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms) {
  const size_t b = decode_tc_supported(fmt) ? decode_tc_scratch_bytes(M_max, H, I, top_k, num_sms)
                                            : sizeof(float) * (size_t)M_max * top_k * M_max * I;
  return (b + 255) & ~(size_t)255;
}

// Scratch, then a 256-byte status block (bit flags of bounded waits that
// gave up; sticky).
size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms) {
  return decode_scratch_bytes(M_max, H, I, top_k, fmt, num_sms) + 256;
}

cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, const float* tw, void* out, int M, int E, int H, int I, int top_k,
                          int fmt, void* ws, int num_sms, cudaStream_t st) {
  if (decode_tc_supported(fmt)) {
    int cu = 0;
    uint32_t* status =
        reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + decode_scratch_bytes(M, H, I, top_k, fmt, num_sms));
    return launch_decode_tc(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, static_cast<float*>(ws), status,
                            num_sms, st, &cu);
  }
  DecodeParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w13 = static_cast<const uint8_t*>(w13);
  p.s13 = static_cast<const uint8_t*>(s13);
  p.w2 = static_cast<const uint8_t*>(w2);
  p.s2 = static_cast<const uint8_t*>(s2);
  p.ids = ids;
  p.tw = tw;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.M = M;
  p.E = E;
  p.H = H;
  p.I = I;
  p.top_k = top_k;
  p.fmt = fmt;
  p.n_slots = M * top_k;
  p.h = static_cast<float*>(ws);
  cudaLaunchConfig_t c1 = {};
  c1.gridDim = dim3((unsigned)(I / 16), (unsigned)p.n_slots);
  c1.blockDim = dim3(kThreads);
  c1.stream = st;
  cudaError_t err = cudaLaunchKernelEx(&c1, decode_fc1_kernel, p);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t c2 = {};
  c2.gridDim = dim3((unsigned)(H / 16));
  c2.blockDim = dim3(kThreads);
  c2.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  c2.attrs = attr;
  c2.numAttrs = 1;
  return cudaLaunchKernelEx(&c2, decode_fc2_kernel, p);
}

}  // namespace moe_fp4
