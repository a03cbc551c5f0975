// Decode band (M <= 8 tokens): the layer as the HBM-bound GEMV it is.
//
// Prior art: the pages' tiny-decode kernel pair (b12x PR #22, "rp-native
// tiny-decode kernel for w4a8_mx (M=1)", section What) -- FC1 streams the
// routed experts' packed nibbles with one 16 B ld.global.nc per 32
// K-elements, folds K with a lane butterfly and writes an FP32 gate/up
// intermediate; FC2 applies SiLU inline, decodes the down weights and does
// the router-weighted sum into the BF16 output.  The section's Notes also
// record why two plain launches beat a single cooperative launch (a grid
// barrier deadlocked when CTAs were not co-resident), and its follow-ups ask
// to fold the wrapper's zero-fills into the kernels.
//
// This implementation, for sm_103a:
//   * Routing lives inside the kernels (the small-batch "direct" idea of
//     flashinfer PR #4285, "sync SM12x NVFP4 fused-MoE kernels": read the
//     top-k ids directly instead of a separate routing pass).  CTA row y is a
//     route slot; it is active only for the first slot naming a valid expert,
//     so every routed expert's weights are streamed exactly once, and invalid
//     ids (< 0 or >= E) are never dereferenced (b12x PR #311, conversation:
//     exact-zero contribution, route tensors untouched).
//   * A warp owns rows r0, r0+32, r0+64, r0+96 of a 128-row resident tile
//     (lane group q = lane/8) and splits K over the 8 lanes of a group (16 B =
//     32 elements per lane per 256-element K-slab).  Each warp load is four
//     fully used 128 B lines; the four rows' scale bytes share one 16 B run.
//     In w13 the lanes 16 apart hold gate n and up n, so SiLU(gate)*up needs
//     one shuffle.
//   * E2M1 -> f16 pairs by the hardware cvt (exact), widened to FP32; FP32
//     accumulation per scale block, scale applied once per block; NVFP4
//     multipliers applied after the K sum.
//   * K may be split across CTAs; partial sums go to the workspace and the
//     last CTA to arrive (atomic counter, no waiting) reduces them in a fixed
//     order, so results are bitwise deterministic.  FC2 reduces the routed
//     experts of each 128-row output tile the same way and writes every
//     output element exactly once (no zero-fill launch, no output atomics).
//   * FC2 is launched with programmatic dependent launch: its CTAs bulk-
//     prefetch their down-projection weights into L2 while FC1 still runs,
//     then wait for FC1's results (griddepcontrol.wait, a hardware
//     dependency, not a spin).
#include "common.cuh"

namespace moe_fp4 {

constexpr int kThreads = 256;  // 8 warps x 16 rows = one 128-row tile
constexpr int kSlab = 256;     // K elements per lane-group pass (8 lanes x 32)

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
  int s1;           // FC1 K splits
  int slabs_per_s1; // FC1 K-slabs per split
  uint32_t* cnt1;   // [n_slots][2I/128]
  uint32_t* cnt2;   // [H/128]
  float* part1;     // [n_slots][2I/128][s1][128][M]
  float* h;         // [n_slots][M][I]
  float* part2;     // [n_slots][H/128][128][M]
};

struct RouteInfo {
  int e;         // expert of this slot
  int active;    // first valid slot naming e
  uint32_t mask; // tokens routed to e (bit t)
};

// Warp 0 of the CTA: expert, activity and token mask of slot `slot`.
__device__ __forceinline__ RouteInfo route_slot(const int32_t* ids, int n_slots, int top_k, int E, int slot) {
  const int lane = threadIdx.x & 31;
  RouteInfo ri;
  ri.e = ids[slot];
  const bool valid = ri.e >= 0 && ri.e < E;
  bool earlier = false;
  uint32_t mask = 0;
  for (int base = 0; base < n_slots; base += 32) {
    int j = base + lane;
    int ej = j < n_slots ? ids[j] : -1;
    bool match = valid && j < n_slots && ej == ri.e;
    if (match && j < slot) earlier = true;
    uint32_t m = match ? (1u << (j / top_k)) : 0u;
    mask |= __reduce_or_sync(0xffffffffu, m);
  }
  earlier = __any_sync(0xffffffffu, earlier);
  ri.active = valid && !earlier;
  ri.mask = mask;
  return ri;
}

// Router weight of token t summed over its slots that name expert e.
__device__ __forceinline__ float slot_weight_sum(const int32_t* ids, const float* tw, int top_k, int t, int e) {
  float s = 0.f;
  for (int j = 0; j < top_k; ++j)
    if (ids[t * top_k + j] == e) s += tw[t * top_k + j];
  return s;
}

// Dot product of one 16 B chunk (32 E2M1 elements) with 32 FP32 activations,
// returned as the two 16-element halves (separate NVFP4 scale blocks).
__device__ __forceinline__ float2 chunk_dot(const uint4& w, const float (&a)[32]) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t hb[4];
    e2m1x8_to_half2x4(words[j], hb);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float2 f = half2_bits_to_float2(hb[p]);
      const int k = 8 * j + 2 * p;
      if (j < 2) {
        s0 = fmaf(f.x, a[k], s0);
        s1 = fmaf(f.y, a[k + 1], s1);
      } else {
        s2 = fmaf(f.x, a[k], s2);
        s3 = fmaf(f.y, a[k + 1], s3);
      }
    }
  }
  return make_float2(s0 + s1, s2 + s3);
}

__device__ __forceinline__ void load_x_chunk(const __nv_bfloat16* xrow, int k0, float (&a)[32]) {
  const uint4* p = reinterpret_cast<const uint4*>(xrow + k0);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 u = __ldg(p + v);
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a[8 * v + 2 * j] = __uint_as_float(ws[j] << 16);
      a[8 * v + 2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ void load_h_chunk(const float* hrow, int k0, float (&a)[32]) {
  const float4* p = reinterpret_cast<const float4*>(hrow + k0);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    float4 u = __ldcg(p + v);
    a[4 * v] = u.x;
    a[4 * v + 1] = u.y;
    a[4 * v + 2] = u.z;
    a[4 * v + 3] = u.w;
  }
}

// Block-scale contribution of one chunk for lane kpart l.
// MX: one UE8M0 block of 32; NV: two E4M3 blocks of 16.
__device__ __forceinline__ float apply_scales(float2 d, uint32_t sword, int fmt, int byte0) {
  if (fmt == MOE_FP4_MXFP4) {
    return (d.x + d.y) * ue8m0_to_float((sword >> (8 * byte0)) & 0xffu);
  }
  float a = e4m3_to_float((sword >> (8 * byte0)) & 0xffu);
  float b = e4m3_to_float((sword >> (8 * (byte0 + 1))) & 0xffu);
  return fmaf(d.x, a, d.y * b);
}

// Signal the next kernel in the stream and return whether this CTA is the
// last of `target` CTAs to arrive at *cnt (after publishing its writes).
__device__ __forceinline__ bool arrive_last(uint32_t* cnt, uint32_t target) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t prev = atomicAdd(cnt, 1u);
    s_last = (prev == target - 1) ? 1 : 0;
    if (s_last) *cnt = 0u;  // leave the counter zeroed for the next call
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

// ---------------------------------------------------------------- FC1
template <int TM>
__global__ void __launch_bounds__(kThreads, TM == 1 ? 3 : 2) decode_fc1_kernel(DecodeParams p) {
  pdl_launch_dependents();
  const int slot = blockIdx.y;
  const int rt = blockIdx.x / p.s1, split = blockIdx.x % p.s1;
  __shared__ RouteInfo s_ri;
  if (threadIdx.x < 32) {
    RouteInfo ri = route_slot(p.ids, p.n_slots, p.top_k, p.E, slot);
    if (threadIdx.x == 0) s_ri = ri;
  }
  __syncthreads();
  const RouteInfo ri = s_ri;
  if (!ri.active) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = lane >> 3, l = lane & 7;
  const int H = p.H, I = p.I, fmt = p.fmt;
  const int KG = k_groups(H, fmt);
  const int nslab = H / kSlab;
  const int s_begin = split * p.slabs_per_s1;
  const int s_end = min(nslab, s_begin + p.slabs_per_s1);

  int tok[TM];
  int Mu = 0;
#pragma unroll
  for (int t = 0; t < TM; ++t) tok[t] = 0;
  {
    uint32_t m = ri.mask;
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      if (m) {
        tok[t] = __ffs(m) - 1;
        m &= m - 1;
        Mu = t + 1;
      }
    }
  }

  const size_t row_bytes = (size_t)H / 2;
  const uint8_t* wexp = p.w13 + (size_t)ri.e * 2 * I * row_bytes;
  const uint8_t* sexp = p.s13 + (size_t)ri.e * scale_chunk_bytes(2 * I, H, fmt);
  int rows[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) rows[i] = rt * kRowTile + 4 * warp + i + 32 * q;

  float acc[4][TM];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[i][t] = 0.f;

  for (int s = s_begin; s < s_end; ++s) {
    uint4 wv[4];
    uint32_t sw[4];
    const int byte_off = s * (kSlab / 2) + l * 16;
    // scale word: MX K-block = 8s+l, NV K-blocks = 16s+2l, +1
    const int kb = fmt == MOE_FP4_MXFP4 ? 8 * s + l : 16 * s + 2 * l;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wv[i] = ld_stream_16(wexp + (size_t)rows[i] * row_bytes + byte_off);
      sw[i] = ld_nc_u32(sexp + (scale_offset(rows[i], kb, KG) & ~(size_t)3));
    }
    const int byte0 = kb & 3;
#pragma unroll 1
    for (int t = 0; t < Mu; ++t) {
      float a[32];
      load_x_chunk(p.x + (size_t)tok[t] * H, s * kSlab + l * 32, a);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 d = chunk_dot(wv[i], a);
        float c = apply_scales(d, sw[i], fmt, byte0);
#pragma unroll
        for (int tt = 0; tt < TM; ++tt)
          if (tt == t) acc[i][tt] += c;
      }
    }
  }
  // fold K across the 8 lanes of each group
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      float v = acc[i][t];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      acc[i][t] = v;
    }

  float gmul_gate = 1.f, gmul_up = 1.f;
  if (fmt == MOE_FP4_NVFP4) {
    const float* gl = reinterpret_cast<const float*>(p.s13 + (size_t)p.E * scale_chunk_bytes(2 * I, H, fmt));
    gmul_gate = gl[2 * ri.e];
    gmul_up = gl[2 * ri.e + 1];
  }
  const int rows_total_tiles = 2 * I / kRowTile;
  float* hslot = p.h + (size_t)slot * p.M * I;

  if (p.s1 == 1) {
    // lanes (q, l=0) and (q+2, l=0) hold gate n and up n of the same n
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        float other = __shfl_xor_sync(0xffffffffu, acc[i][t], 16);
        if (l == 0 && q < 2 && t < Mu) {
          const int n = rt * (kRowTile / 2) + 4 * warp + i + 32 * q;
          float g = acc[i][t] * gmul_gate, u = other * gmul_up;
          hslot[(size_t)tok[t] * I + n] = silu(g) * u;
        }
      }
    return;
  }

  // split K: publish partials, the last CTA of this (slot, tile) reduces
  float* part = p.part1 + (((size_t)slot * rows_total_tiles + rt) * p.s1 + split) * kRowTile * p.M;
  if (l == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < TM; ++t)
        if (t < Mu) part[(size_t)(4 * warp + i + 32 * q) * p.M + tok[t]] = acc[i][t];
  }
  if (!arrive_last(p.cnt1 + (size_t)slot * rows_total_tiles + rt, (uint32_t)p.s1)) return;
  const float* part0 = p.part1 + ((size_t)slot * rows_total_tiles + rt) * p.s1 * kRowTile * p.M;
  for (int idx = threadIdx.x; idx < (kRowTile / 2) * Mu; idx += kThreads) {
    const int r = idx % (kRowTile / 2), tt = idx / (kRowTile / 2);
    int tk = tok[0];
#pragma unroll
    for (int z = 0; z < TM; ++z)
      if (z == tt) tk = tok[z];
    float g = 0.f, u = 0.f;
    for (int sp = 0; sp < p.s1; ++sp) {
      const float* ps = part0 + (size_t)sp * kRowTile * p.M;
      g += __ldcg(ps + (size_t)r * p.M + tk);
      u += __ldcg(ps + (size_t)(r + kRowTile / 2) * p.M + tk);
    }
    const int n = rt * (kRowTile / 2) + r;
    hslot[(size_t)tk * I + n] = silu(g * gmul_gate) * (u * gmul_up);
  }
}

// ---------------------------------------------------------------- FC2
template <int TM>
__global__ void __launch_bounds__(kThreads, TM == 1 ? 3 : 2) decode_fc2_kernel(DecodeParams p) {
  const int slot = blockIdx.y;
  const int rt = blockIdx.x;
  const int H = p.H, I = p.I, fmt = p.fmt;
  const int n_tiles = H / kRowTile;
  __shared__ RouteInfo s_ri;
  if (threadIdx.x < 32) {
    RouteInfo ri = route_slot(p.ids, p.n_slots, p.top_k, p.E, slot);
    if (threadIdx.x == 0) s_ri = ri;
  }
  __syncthreads();
  const RouteInfo ri = s_ri;
  const size_t row_bytes = (size_t)I / 2;
  const int KG = k_groups(I, fmt);

  if (ri.active) {
    const uint8_t* wexp = p.w2 + (size_t)ri.e * H * row_bytes;
    const uint8_t* sexp = p.s2 + (size_t)ri.e * scale_chunk_bytes(H, I, fmt);
    if (threadIdx.x == 0) {
      // stream this CTA's down-projection tile into L2 while FC1 finishes
      const uint8_t* wt = wexp + (size_t)rt * kRowTile * row_bytes;
      const uint32_t wbytes = (uint32_t)(kRowTile * row_bytes);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(wt), "r"(wbytes) : "memory");
      const uint8_t* st = sexp + (size_t)rt * KG * kChunkBytes;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(st), "r"((uint32_t)(KG * kChunkBytes))
                   : "memory");
    }
    pdl_wait();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane >> 3, l = lane & 7;
    int tok[TM];
    int Mu = 0;
#pragma unroll
    for (int t = 0; t < TM; ++t) tok[t] = 0;
    {
      uint32_t m = ri.mask;
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (m) {
          tok[t] = __ffs(m) - 1;
          m &= m - 1;
          Mu = t + 1;
        }
      }
    }
    int rows[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rows[i] = rt * kRowTile + 4 * warp + i + 32 * q;
    float acc[4][TM];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < TM; ++t) acc[i][t] = 0.f;

    const float* hslot = p.h + (size_t)slot * p.M * I;
    const int nchunk = I / 32;
    for (int c = l; c < nchunk; c += 8) {
      uint4 wv[4];
      uint32_t sw[4];
      const int kb = fmt == MOE_FP4_MXFP4 ? c : 2 * c;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wv[i] = ld_stream_16(wexp + (size_t)rows[i] * row_bytes + c * 16);
        sw[i] = ld_nc_u32(sexp + (scale_offset(rows[i], kb, KG) & ~(size_t)3));
      }
      const int byte0 = kb & 3;
#pragma unroll 1
      for (int t = 0; t < Mu; ++t) {
        float a[32];
        load_h_chunk(hslot + (size_t)tok[t] * I, c * 32, a);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 d = chunk_dot(wv[i], a);
          float cc = apply_scales(d, sw[i], fmt, byte0);
#pragma unroll
          for (int tt = 0; tt < TM; ++tt)
            if (tt == t) acc[i][tt] += cc;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        float v = acc[i][t];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        acc[i][t] = v;
      }
    float gmul = 1.f;
    if (fmt == MOE_FP4_NVFP4) {
      const float* gl = reinterpret_cast<const float*>(p.s2 + (size_t)p.E * scale_chunk_bytes(H, I, fmt));
      gmul = gl[ri.e];
    }
    float* part = p.part2 + ((size_t)slot * n_tiles + rt) * kRowTile * p.M;
    if (l == 0) {
      for (int t = 0; t < p.M; ++t) {
        float wsum = 0.f;
        int ti = -1;
#pragma unroll
        for (int z = 0; z < TM; ++z)
          if (z < Mu && tok[z] == t) ti = z;
        if (ti >= 0) wsum = slot_weight_sum(p.ids, p.tw, p.top_k, t, ri.e) * gmul;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v = 0.f;
#pragma unroll
          for (int z = 0; z < TM; ++z)
            if (z == ti) v = acc[i][z] * wsum;
          part[(size_t)(4 * warp + i + 32 * q) * p.M + t] = v;
        }
      }
    }
  }

  if (!arrive_last(p.cnt2 + rt, (uint32_t)p.n_slots)) return;

  // last CTA of this output tile: sum the active slots in slot order, cast once
  __shared__ int s_active[128];
  for (int sl = threadIdx.x; sl < p.n_slots; sl += kThreads) {
    int e = p.ids[sl];
    int act = e >= 0 && e < p.E;
    for (int j = 0; act && j < sl; ++j)
      if (p.ids[j] == e) act = 0;
    s_active[sl] = act;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRowTile * p.M; idx += kThreads) {
    const int r = idx % kRowTile, t = idx / kRowTile;
    float v = 0.f;
    for (int sl = 0; sl < p.n_slots; ++sl)
      if (s_active[sl]) v += __ldcg(p.part2 + (((size_t)sl * n_tiles + rt) * kRowTile + r) * p.M + t);
    p.out[(size_t)t * H + rt * kRowTile + r] = __float2bfloat16_rn(v);
  }
}

// ---------------------------------------------------------------- host side
static void choose_split(int n_slots, int I, int H, int num_sms, int* s1, int* per);

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace carve-up for M tokens: counters | FC1 partials | h | FC2 partials.
struct DecodeCarve {
  size_t cnt, part1, h, part2, total;
};
static DecodeCarve decode_carve(int M, int H, int I, int top_k, int num_sms) {
  const size_t n = (size_t)M * top_k;
  const size_t t13 = 2 * I / kRowTile, t2 = H / kRowTile;
  int s1, per;
  choose_split((int)n, I, H, num_sms, &s1, &per);
  DecodeCarve c;
  c.cnt = 0;
  c.part1 = align256(sizeof(uint32_t) * (n * t13 + t2));
  c.h = c.part1 + align256(sizeof(float) * n * t13 * (size_t)s1 * kRowTile * M);
  c.part2 = c.h + align256(sizeof(float) * n * M * I);
  c.total = c.part2 + align256(sizeof(float) * n * t2 * kRowTile * M);
  return c;
}

// Largest carve over every M <= M_max (a workspace sized for M_max serves any
// smaller M; the counters always sit at offset 0).
size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int num_sms) {
  size_t b = 0;
  for (int m = 1; m <= M_max; ++m) {
    size_t t = decode_carve(m, H, I, top_k, num_sms).total;
    if (t > b) b = t;
  }
  return b;
}

static void choose_split(int n_slots, int I, int H, int num_sms, int* s1, int* per) {
  const int t13 = 2 * I / kRowTile;
  const int nslab = H / kSlab;
  const int target = 2 * num_sms;
  int want = (target + n_slots * t13 - 1) / (n_slots * t13);
  if (want < 1) want = 1;
  if (want > nslab) want = nslab;
  int p_ = (nslab + want - 1) / want;
  *per = p_;
  *s1 = (nslab + p_ - 1) / p_;
}

cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, const float* tw, void* out, int M, int E, int H, int I, int top_k,
                          int fmt, void* ws, int num_sms, cudaStream_t st) {
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
  choose_split(p.n_slots, I, H, num_sms, &p.s1, &p.slabs_per_s1);
  const size_t n = p.n_slots;
  const size_t t13 = 2 * I / kRowTile, t2 = H / kRowTile;
  const DecodeCarve cv = decode_carve(M, H, I, top_k, num_sms);
  char* b = static_cast<char*>(ws);
  p.cnt1 = reinterpret_cast<uint32_t*>(b);
  p.cnt2 = p.cnt1 + n * t13;
  p.part1 = reinterpret_cast<float*>(b + cv.part1);
  p.h = reinterpret_cast<float*>(b + cv.h);
  p.part2 = reinterpret_cast<float*>(b + cv.part2);

  dim3 g1((unsigned)(t13 * p.s1), (unsigned)n);
  dim3 g2((unsigned)t2, (unsigned)n);
  cudaLaunchConfig_t c1 = {};
  c1.gridDim = g1;
  c1.blockDim = dim3(kThreads);
  c1.stream = st;
  cudaLaunchConfig_t c2 = {};
  c2.gridDim = g2;
  c2.blockDim = dim3(kThreads);
  c2.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  c2.attrs = attr;
  c2.numAttrs = 1;
  cudaError_t err;
#define MOE_FP4_DECODE_CASE(TMV)                                  \
  err = cudaLaunchKernelEx(&c1, decode_fc1_kernel<TMV>, p);       \
  if (err != cudaSuccess) return err;                             \
  err = cudaLaunchKernelEx(&c2, decode_fc2_kernel<TMV>, p);       \
  return err;
  if (M <= 1) {
    MOE_FP4_DECODE_CASE(1)
  } else if (M <= 2) {
    MOE_FP4_DECODE_CASE(2)
  } else if (M <= 4) {
    MOE_FP4_DECODE_CASE(4)
  } else {
    MOE_FP4_DECODE_CASE(8)
  }
#undef MOE_FP4_DECODE_CASE
}

}  // namespace moe_fp4
