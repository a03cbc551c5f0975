// The prefill bands (batches past the decode band): routing compaction
// (count, scan, stable scatter into routing tiles per expert; one kernel for
// up to 8192 routing entries), then one of four launch chains over the same
// routed rows and FP32 token accumulator:
//   NVFP4 activations  x and h quantised to NVFP4, both GEMMs on the FP4
//                      tensor cores (gemm_fp4.cuh, kind::mxf4nvf4), routed
//                      rows on the MMA's 128-row side;
//   mid band           the same layer with the operands swapped for experts
//                      with few routed rows (gemm_fp4_swap.cuh: weights on the
//                      128-row side, 32-row routing tiles on N);
//   exact BF16         x and h carried exactly in row-scaled FP16, the FP4
//                      weights decoded to FP16 in shared memory (gemm_f16w4.cuh);
//   W4A8-MX            x and h quantised to MXFP8, both GEMMs on the FP8 tensor
//                      cores with the MXFP4 weights as stored (gemm_mxf8.cuh,
//                      kind::mxf8f6f4) where I % 128 == 0, else the 16-bit chain;
// and the test-support entry points (GEMM, routing, quantisers).  Every
// kernel of a chain is launched with programmatic dependent launch and waits
// for its predecessor before it touches global memory.
#include <mutex>

#include "gemm_f16w4.cuh"
#include "gemm_fp4.cuh"
#include "gemm_fp4_swap.cuh"
#include "gemm_mxf8.cuh"

namespace moe_fp4 {

// The driver's tensor-map encoder, resolved through the runtime so that the
// library does not link against libcuda (it stays loadable without a GPU).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map over a byte array of up to three dimensions (d[0] innermost,
// stride[i] the byte distance between consecutive indices of dimension i+1),
// boxes of box[0..rank) bytes x rows, optional 128-byte swizzle.  Encoded
// maps are kept in a small cache keyed by every argument (a map depends on
// nothing else), so repeated layer calls skip the encoding.
static CUresult make_typed_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* d,
                               const uint64_t* stride, const uint32_t* box, bool swizzle128);
CUresult make_u8_map(CUtensorMap* m, const void* base, int rank, const uint64_t* d, const uint64_t* stride,
                     const uint32_t* box, bool swizzle128) {
  return make_typed_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, d, stride, box, swizzle128);
}

// 2-D tensor map over packed E2M1 rows [rows][K / 2 bytes] that unpacks them
// into shared memory as 16-byte groups (8 bytes of 16 packed values, then 8
// bytes of gap: the layout tcgen05.mma kind::mxf8f6f4 reads 4-bit operands
// in), box of box_rows x 128 elements (128 bytes in shared memory), 128-byte
// swizzle.  K % 128 == 0, base 32-byte aligned (the driver checks both).
CUresult make_e2m1_unpacked_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  const uint64_t d[2] = {K, rows};
  const uint64_t stride[1] = {K / 2};
  const uint32_t box[2] = {128, box_rows};
  return make_typed_map(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, base, 2, d, stride, box, true);
}

static CUresult make_typed_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, int rank, const uint64_t* d,
                               const uint64_t* stride, const uint32_t* box, bool swizzle128) {
  struct Entry {
    const void* base;
    CUtensorMapDataType dtype;
    int rank;
    uint64_t d[3], stride[2];
    uint32_t box[3];
    bool sw;
    CUtensorMap map;
  };
  static Entry cache[64];
  static int n_used = 0, next = 0;
  static std::mutex mu;
  if (rank < 1 || rank > 3) return CUDA_ERROR_INVALID_VALUE;
  auto same = [&](const Entry& e) {
    if (e.base != base || e.dtype != dtype || e.rank != rank || e.sw != swizzle128) return false;
    for (int i = 0; i < rank; ++i)
      if (e.d[i] != d[i] || e.box[i] != box[i] || (i + 1 < rank && e.stride[i] != stride[i])) return false;
    return true;
  };
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_used; ++i)
      if (same(cache[i])) {
        *m = cache[i].map;
        return CUDA_SUCCESS;
      }
  }
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3], strides[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    dims[i] = d[i];
    bx[i] = box[i];
    if (i + 1 < rank) strides[i] = stride[i];
  }
  const CUresult r = enc(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides,
                         bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lk(mu);
    Entry& e = cache[next];
    e = Entry{};
    e.base = base;
    e.dtype = dtype;
    e.rank = rank;
    e.sw = swizzle128;
    for (int i = 0; i < rank; ++i) {
      e.d[i] = d[i];
      e.box[i] = box[i];
      if (i + 1 < rank) e.stride[i] = stride[i];
    }
    e.map = *m;
    next = (next + 1) % 64;
    if (n_used < 64) ++n_used;
  }
  return r;
}

// 2-D tensor map over a row-major byte matrix [rows][inner_bytes], box of
// box_rows x 128 bytes, 128-byte swizzle (the K-major SW128 operand layout).
CUresult make_fp4_map(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows) {
  const uint64_t d[2] = {inner_bytes, rows};
  const uint64_t stride[1] = {inner_bytes};
  const uint32_t box[2] = {128, box_rows};
  return make_u8_map(m, base, 2, d, stride, box, true);
}

// SM count of the current device (cached): the persistent GEMMs launch one
// CTA per SM.
// Launch with programmatic dependent launch: the kernel may become resident
// while its predecessor on the stream finishes; every prefill kernel waits
// for the predecessor's completion (griddepcontrol.wait) before it touches
// global memory, so only the launch latency overlaps.
template <class Kern, class... Args>
static cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned threads, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(grid);
  c.blockDim = dim3(threads);
  c.dynamicSmemBytes = smem;
  c.stream = st;
  c.attrs = at;
  c.numAttrs = 1;
  return cudaLaunchKernelEx(&c, kern, args...);
}

static cudaError_t gemm_sms(int* sms) {
  static int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *sms = cache[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev] = *sms;
  return e;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    debug_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                      const uint8_t* a_sf, const uint8_t* b_sf, float* d, int K, int N, int n_tiles, uint32_t* err) {
  const int KG = K / 64;
  const int NT = N / kGemmBN;
  auto tile_of = [&](int idx) {
    GemmTile t;
    t.m_tile = idx / NT;
    t.n_tile = idx % NT;
    t.a_row0 = t.m_tile * kGemmBM;
    t.b_row0 = t.n_tile * kGemmBN;
    t.a_sf = a_sf + (size_t)t.m_tile * KG * kChunkBytes;
    t.b_sf0 = b_sf + (size_t)(2 * t.n_tile) * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    t.valid = true;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const GemmTile& t) {
#pragma unroll 1
    for (int c = 0; c < kGemmBN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem_row + 32 * c, r);
      float4* dst = reinterpret_cast<float4*>(d + (size_t)(t.a_row0 + row) * N + t.b_row0 + 32 * c);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                             __uint_as_float(r[4 * i + 3]));
    }
  };
  gemm_fp4_persistent<kGemmBN>(&map_a, &map_b, K, err, n_tiles, tile_of, epi);
}

cudaError_t launch_debug_gemm(const void* a_q, const void* a_sf, const void* b_q, const void* b_sf, float* d,
                              int M_rows, int N_rows, int K, uint32_t* status, cudaStream_t st, int* cu_err) {
  CUtensorMap ma, mb;
  CUresult r = make_fp4_map(&ma, a_q, (uint64_t)K / 2, (uint64_t)M_rows, kGemmBM);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mb, b_q, (uint64_t)K / 2, (uint64_t)N_rows, kGemmBN);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(debug_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  const int n_tiles = (M_rows / kGemmBM) * (N_rows / kGemmBN);
  int sms = 0;
  e = gemm_sms(&sms);
  if (e != cudaSuccess) return e;
  debug_gemm_kernel<<<n_tiles < sms ? n_tiles : sms, kGemmThreads, kGemmSmem, st>>>(
      ma, mb, static_cast<const uint8_t*>(a_sf), static_cast<const uint8_t*>(b_sf), d, K, N_rows, n_tiles, status);
  return cudaGetLastError();
}


// ============================================================================
// Prefill band (M > 8): route -> quantise x -> FC1 GEMM (SiLU*up) ->
// quantise h -> FC2 GEMM (router-weighted FP32 accumulation) -> cast.
//
// Prior art: the SM12x sync PR's dynamic prefill backend (flashinfer PR
// #4285): routed rows grouped per expert and processed as MMA tiles, W4A4
// NVFP4 with a fast FP4 activation quantiser for gated activations; and the
// W4A16 route PR's prefill epilogue (b12x PR #311, conversation): routed
// outputs reduced with relaxed FP32 global reductions into a caller-owned
// FP32 token accumulator and cast to BF16 once.
//
// Activations: x per token and h per routed row are quantised to NVFP4 (E2M1,
// one E4M3 scale per 16 elements, one FP32 multiplier per row):
//   G = amax/(6*448) (1 if the row is zero), s = e4m3_rn_satfinite(bmax/(6G)),
//   q = e2m1_rn_satfinite(a/(s*G)) (0 where s*G == 0),
// every step an IEEE FP32 operation; h is staged in BF16 between FC1 and its
// quantiser.  Each expert's routed rows are padded to a multiple of the
// routing-tile height (128; 32 in the mid band) so a tile never straddles two
// experts.
// ============================================================================

size_t decode_sync_bytes(int H, int I, int top_k);

namespace {

constexpr int kRouteBlock = 256;  // routing entries per count/scatter block
// W4A8-MX engine choice (test support): 1 = FP8 tensor cores where the shape
// allows, 0 = always the 16-bit engine
int g_w4a8_fp8 = 1;
// W4A8-MX FC1 tile width (I % 128 == 0 makes either fit).  Measured on GB300
// at E=128 H=4096 I=1536 M=4096: 1022 us per layer with 128-wide tiles (two
// accumulators, the epilogue beside the next tile's MMAs) against 1046 with
// 256-wide ones (one accumulator).
constexpr int kMxFc1BN = 128;
// FC2 tile widths of the 16-bit and FP8 bands.  Measured on GB300 at
// prefill_e128 (us per layer, 256 / 128): exact 1699 / 1970 (the 16-bit
// engine decodes the weights once per tile: twice as often per FLOP at 128);
// W4A8-MX 997 / 983 (two accumulators, the reductions beside the MMAs).
constexpr int kFc2ExactBN = 256;
constexpr int kMxFc2BN = 128;
constexpr int kMaxPrefillE = 4096;

struct PrefillArgs {
  const __nv_bfloat16* x;
  const int32_t* ids;  // [M][top_k], int32 or (ids64) int64
  int ids64;
  const float* tw;
  const uint8_t* s13;  // resident scale chunks (+ multipliers)
  const uint8_t* s2;
  __nv_bfloat16* out;
  int M, E, H, I, top_k, n_entries, n_route_blocks, max_tiles;
  ActParams act;  // FC1's gated activation
  int* counts;      // [n_route_blocks][E]
  int* block_base;  // [n_route_blocks][E]
  int* expert_off;  // [E+1]
  int* expert_poff; // [E+1]
  int* tile_expert; // [max_tiles]
  int* tile_rows;   // [max_tiles] routed rows of each 128-row routing tile (1..128)
  int* num_tiles;   // [1]
  int* pos;         // [n_entries]
  int* row_src;     // [128 * max_tiles]
  uint8_t* xq;      // [rows][H/2]
  uint8_t* xsf;     // chunks [rows/128][H/64][512]
  float* xG;        // [rows]
  __nv_bfloat16* hbuf;  // [rows][I]
  __half* xb;           // 16-bit bands: x (or its MXFP8 image) in FP16, row-scaled, per routed row [rows][H]
  int amode;            // 16-bit bands: 0 exact BF16 activations, 1 MXFP8 (W4A8-MX)
  uint8_t* hq;      // [rows][I/2]
  uint8_t* hsf;     // chunks [rows/128][I/64][512]
  float* hG;        // [rows]
  float* acc;       // [M][H]
  // W4A8-MX band on the FP8 tensor cores (inside the 16-bit bands' x and h areas)
  uint8_t* xq8;     // [rows][H] E4M3
  uint8_t* xsf8;    // UE8M0 chunks [rows/128][H/128][512]
  uint8_t* hq8;     // [rows][I] E4M3
  uint8_t* hsf8;    // UE8M0 chunks [rows/128][I/128][512]
  uint32_t* status;
};

// Byte offset of (row, 16-element block kb) in a chunk array of K = 64*KG.
__device__ __forceinline__ size_t sf_chunk_offset(int row, int kb, int KG) {
  return ((size_t)(row >> 7) * KG + (kb >> 2)) * kChunkBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kb & 3);
}

__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}
// Two E2M1 codes, element `lo` in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xffu;
}

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp quantises a row of K elements given by load16(block, float[16]).
// For each 16-element block calls emit(block, scale_byte, code words w0, w1
// (8 bytes of codes)).  Returns G.
template <class Load16, class Emit>
__device__ __forceinline__ float quant_row_nvfp4(int K, const Load16& load16, const Emit& emit) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 16;
  float amax = 0.f;
  for (int b = lane; b < nb; b += 32) {
    float v[16];
    load16(b, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  const float G = amax == 0.f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  const float six_g = __fmul_rn(6.0f, G);
  for (int b = lane; b < nb; b += 32) {
    float v[16];
    load16(b, v);
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
    const uint32_t sb = e4m3_rn_sat(__fdiv_rn(bmax, six_g));
    const float sdec = e4m3_to_float(sb);
    const float sg = __fmul_rn(sdec, G);
    uint32_t w0 = 0, w1 = 0;
    if (sg != 0.f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) w0 |= e2m1x2_rn_sat(__fdiv_rn(v[2 * i], sg), __fdiv_rn(v[2 * i + 1], sg)) << (8 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w1 |= e2m1x2_rn_sat(__fdiv_rn(v[8 + 2 * i], sg), __fdiv_rn(v[8 + 2 * i + 1], sg)) << (8 * i);
    }
    emit(b, sb, w0, w1);
  }
  return G;
}

__device__ __forceinline__ void bf16x16_to_f32(const __nv_bfloat16* p, float (&v)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const uint4 u0 = __ldg(q), u1 = __ldg(q + 1);
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// ---------------------------------------------------------------- routing
__global__ void route_count_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  extern __shared__ int s_hist[];
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int i = blockIdx.x * kRouteBlock + threadIdx.x;
  if (i < a.n_entries) {
    const int e = route_id(a.ids, i, a.ids64, a.E);
    if (e >= 0 && e < a.E) atomicAdd(&s_hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.counts[(size_t)blockIdx.x * a.E + e] = s_hist[e];
}

// One CTA: per-expert totals, unpadded and P-padded exclusive offsets, the
// per-block bases of the stable scatter, the list of P-row routing tiles and
// the padding rows (P = 128: the prefill band; 32: the mid band).
template <int P>
__global__ void route_scan_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  __shared__ int s_tot[kMaxPrefillE];
  __shared__ int s_part[2][1024];
  __shared__ int s_poff[kMaxPrefillE];
  const int E = a.E, nb = a.n_route_blocks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // lanes per expert column (a power of two <= 32 that divides the warp):
  // the column's count blocks are split in contiguous segments
  int tpe = 1;
  while (tpe < 32 && tpe * 2 * E <= (int)blockDim.x) tpe *= 2;
  const int seg = (nb + tpe - 1) / tpe;
  for (int base = 0; base < E * tpe; base += blockDim.x) {
    const int v = base + threadIdx.x, e = v / tpe, part = v % tpe;
    int t = 0;
    if (e < E) {
      const int b1 = min(nb, part * seg + seg);
#pragma unroll 8  // independent loads in flight together (the sum is the only chain)
      for (int b = part * seg; b < b1; ++b) t += __ldg(a.counts + (size_t)b * E + e);
    }
    for (int d = 1; d < tpe; d <<= 1) t += __shfl_xor_sync(0xffffffffu, t, d);
    if (e < E && part == 0) s_tot[e] = t;
  }
  __syncthreads();
  // exclusive scans over experts: each thread owns a contiguous run
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
  int su = 0, sp = 0;
  for (int e = e0; e < e1; ++e) {
    su += s_tot[e];
    sp += (s_tot[e] + P - 1) & ~(P - 1);
  }
  // exclusive block scan of (su, sp): within warps by shuffles, then over
  // the warp totals
  int iu = su, ip = sp;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int ou = __shfl_up_sync(0xffffffffu, iu, d), op = __shfl_up_sync(0xffffffffu, ip, d);
    if (lane >= d) {
      iu += ou;
      ip += op;
    }
  }
  if (lane == 31) {
    s_part[0][warp] = iu;
    s_part[1][warp] = ip;
  }
  __syncthreads();
  if (warp == 0) {
    int wu = lane < nw ? s_part[0][lane] : 0, wp = lane < nw ? s_part[1][lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int ou = __shfl_up_sync(0xffffffffu, wu, d), op = __shfl_up_sync(0xffffffffu, wp, d);
      if (lane >= d) {
        wu += ou;
        wp += op;
      }
    }
    if (lane < nw) {
      s_part[0][32 + lane] = wu;  // inclusive warp prefixes
      s_part[1][32 + lane] = wp;
    }
    if (lane == nw - 1) {
      a.expert_off[E] = wu;
      a.expert_poff[E] = wp;
      *a.num_tiles = wp / P;
    }
  }
  __syncthreads();
  int ru = iu - su + (warp > 0 ? s_part[0][32 + warp - 1] : 0);
  int rp = ip - sp + (warp > 0 ? s_part[1][32 + warp - 1] : 0);
  for (int e = e0; e < e1; ++e) {
    const int tot = s_tot[e], padded = (tot + P - 1) & ~(P - 1);
    a.expert_off[e] = ru;
    a.expert_poff[e] = rp;
    s_poff[e] = rp;
    for (int t = 0; t < padded / P; ++t) {
      a.tile_expert[rp / P + t] = e;
      a.tile_rows[rp / P + t] = min(P, tot - P * t);
    }
    ru += tot;
    rp += padded;
  }
  __syncthreads();
  // padding rows (past the routed rows of each expert's last tile) -> -1,
  // all threads over all tiles, coalesced
  const int n_rows = s_part[1][32 + nw - 1];
  for (int v = threadIdx.x; v < n_rows; v += blockDim.x)
    if (v % P >= a.tile_rows[v / P]) a.row_src[v] = -1;
  // per-block bases of the stable scatter: the expert's padded offset plus
  // the counts of the earlier blocks (segment sums, then a scan in order)
  for (int base = 0; base < E * tpe; base += blockDim.x) {
    const int v = base + threadIdx.x, e = v / tpe, part = v % tpe;
    const int b0 = part * seg, b1 = e < E ? min(nb, b0 + seg) : b0;
    int t = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) t += __ldg(a.counts + (size_t)b * E + e);
    int incl = t;  // inclusive scan over the parts of this expert
    for (int d = 1; d < tpe; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (part >= d) incl += o;
    }
    if (e < E) {
      int run = s_poff[e] + incl - t;
#pragma unroll 8
      for (int b = b0; b < b1; ++b) {
        const int cnt = __ldg(a.counts + (size_t)b * E + e);
        a.block_base[(size_t)b * E + e] = run;
        run += cnt;
      }
    }
  }
}

// Small batches (n_entries <= kRouteSmallMax): the whole routing in one CTA
// of 1024 threads -- per-expert counts and each entry's rank among its
// expert's entries by shared-memory atomics, the exclusive scans (unpadded
// and P-padded), the tile list, the rows, the padding rows.  The rank order
// within an expert is the atomics' order, not the entries' (every routed
// row computes the same products wherever it sits).
constexpr int kRouteSmallMax = 8192;
template <int P>
__global__ void __launch_bounds__(1024, 1) route_small_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  __shared__ int s_cnt[kMaxPrefillE];
  __shared__ int s_off[kMaxPrefillE];
  __shared__ int s_wsum[2][32];
  const int E = a.E, n = a.n_entries;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += 1024) s_cnt[e] = 0;
  __syncthreads();
  constexpr int R = kRouteSmallMax / 1024;
  int ex[R], rk[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = tid + 1024 * r;
    ex[r] = i < n ? route_id(a.ids, i, a.ids64, E) : -1;
    rk[r] = ex[r] >= 0 && ex[r] < E ? atomicAdd(&s_cnt[ex[r]], 1) : -1;
  }
  __syncthreads();
  // exclusive scans over experts (counts, P-padded counts): each thread a
  // contiguous run of experts, then the runs' totals across the block
  const int per = (E + 1023) / 1024;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int su = 0, sp = 0;
  for (int e = e0; e < e1; ++e) {
    su += s_cnt[e];
    sp += (s_cnt[e] + P - 1) & ~(P - 1);
  }
  int iu = su, ip = sp;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int ou = __shfl_up_sync(0xffffffffu, iu, d), op = __shfl_up_sync(0xffffffffu, ip, d);
    if (lane >= d) {
      iu += ou;
      ip += op;
    }
  }
  if (lane == 31) {
    s_wsum[0][warp] = iu;
    s_wsum[1][warp] = ip;
  }
  __syncthreads();
  if (warp == 0) {
    int wu = s_wsum[0][lane], wp = s_wsum[1][lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int ou = __shfl_up_sync(0xffffffffu, wu, d), op = __shfl_up_sync(0xffffffffu, wp, d);
      if (lane >= d) {
        wu += ou;
        wp += op;
      }
    }
    s_wsum[0][lane] = wu;  // inclusive over warps
    s_wsum[1][lane] = wp;
    if (lane == 31) {
      a.expert_off[E] = wu;
      a.expert_poff[E] = wp;
      *a.num_tiles = wp / P;
    }
  }
  __syncthreads();
  int ru = iu - su + (warp > 0 ? s_wsum[0][warp - 1] : 0);
  int rp = ip - sp + (warp > 0 ? s_wsum[1][warp - 1] : 0);
  for (int e = e0; e < e1; ++e) {
    const int tot = s_cnt[e], padded = (tot + P - 1) & ~(P - 1);
    a.expert_off[e] = ru;
    a.expert_poff[e] = rp;
    s_off[e] = rp;
    for (int t = 0; t < padded / P; ++t) {
      a.tile_expert[rp / P + t] = e;
      a.tile_rows[rp / P + t] = min(P, tot - P * t);
    }
    ru += tot;
    rp += padded;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = tid + 1024 * r;
    if (i >= n) break;
    if (rk[r] >= 0) {
      const int row = s_off[ex[r]] + rk[r];
      a.pos[i] = row;
      a.row_src[row] = i;
    } else {
      a.pos[i] = -1;
    }
  }
  // padding rows (past the routed rows of each expert's last tile) -> -1
  const int n_rows = s_wsum[1][31];
  for (int v = tid; v < n_rows; v += 1024)
    if (v % P >= a.tile_rows[v / P]) a.row_src[v] = -1;
}

// One warp per block of entries: stable ranks by expert in index order.
__global__ void route_scatter_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  extern __shared__ int s_base[];
  const int lane = threadIdx.x;
  for (int e = lane; e < a.E; e += 32) s_base[e] = a.block_base[(size_t)blockIdx.x * a.E + e];
  __syncwarp();
  for (int r0 = 0; r0 < kRouteBlock; r0 += 32) {
    const int i = blockIdx.x * kRouteBlock + r0 + lane;
    const int e = i < a.n_entries ? route_id(a.ids, i, a.ids64, a.E) : -1;
    const bool valid = e >= 0 && e < a.E;
    const int key = valid ? e : -1 - lane;  // invalid entries stay alone
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const uint32_t below = peers & ((1u << lane) - 1u);
    if (valid) {
      const int row = s_base[e] + __popc(below);
      a.pos[i] = row;
      a.row_src[row] = i;
    } else if (i < a.n_entries) {
      a.pos[i] = -1;
    }
    __syncwarp();
    if (valid && below == 0) s_base[e] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------- quantisers
// Largest magnitude over the 128 threads of a block (every thread gets it).
__device__ __forceinline__ float block128_max(float v, float* red4) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red4[threadIdx.x >> 5] = v;
  __syncthreads();
  return fmaxf(fmaxf(red4[0], red4[1]), fmaxf(red4[2], red4[3]));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One warp per token: NVFP4 row of x into every routed row of the token;
// also zeroes the token's FP32 accumulator row.
__global__ void quant_x_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t >= a.M) return;
  const int lane = threadIdx.x & 31;
  const int H = a.H, KG = H / 64, k = a.top_k;
  const __nv_bfloat16* xr = a.x + (size_t)t * H;
  const int* prow = a.pos + (size_t)t * k;
  const float G = quant_row_nvfp4(
      H, [&](int b, float (&v)[16]) { bf16x16_to_f32(xr + 16 * b, v); },
      [&](int b, uint32_t sb, uint32_t w0, uint32_t w1) {
        for (int j = 0; j < k; ++j) {
          const int r = prow[j];
          if (r < 0) continue;
          *reinterpret_cast<uint2*>(a.xq + (size_t)r * (H / 2) + 8 * b) = make_uint2(w0, w1);
          a.xsf[sf_chunk_offset(r, b, KG)] = (uint8_t)sb;
        }
      });
  if (lane == 0)
    for (int j = 0; j < k; ++j)
      if (prow[j] >= 0) a.xG[prow[j]] = G;
  float4* accr = reinterpret_cast<float4*>(a.acc + (size_t)t * H);
  for (int v = lane; v < H / 4; v += 32) accr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Small batches: one warp per routing entry quantises its token's row into
// the entry's routed row (the same codes as quant_x_kernel, k times the
// arithmetic for k times the warps); the token's first entry zeroes its FP32
// accumulator row.
__global__ void quant_x_entry_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int i = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (i >= a.n_entries) return;
  const int lane = threadIdx.x & 31;
  const int H = a.H, KG = H / 64, t = i / a.top_k;
  const int r = a.pos[i];
  if (r >= 0) {
    const __nv_bfloat16* xr = a.x + (size_t)t * H;
    const float G = quant_row_nvfp4(
        H, [&](int b, float (&v)[16]) { bf16x16_to_f32(xr + 16 * b, v); },
        [&](int b, uint32_t sb, uint32_t w0, uint32_t w1) {
          *reinterpret_cast<uint2*>(a.xq + (size_t)r * (H / 2) + 8 * b) = make_uint2(w0, w1);
          a.xsf[sf_chunk_offset(r, b, KG)] = (uint8_t)sb;
        });
    if (lane == 0) a.xG[r] = G;
  }
  if (i % a.top_k == 0) {
    float4* accr = reinterpret_cast<float4*>(a.acc + (size_t)t * H);
    for (int v = lane; v < H / 4; v += 32) accr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
// Batches up to this many tokens quantise x per routing entry.
constexpr int kQuantXEntryMaxM = 256;

// NVFP4 row r of h (BF16) for FC2, by one warp; returns the row's G.
__device__ __forceinline__ float quant_h_row(const PrefillArgs& a, int r) {
  const int I = a.I, KG = I / 64;
  const __nv_bfloat16* hr = a.hbuf + (size_t)r * I;
  return quant_row_nvfp4(
      I, [&](int b, float (&v)[16]) { bf16x16_to_f32(hr + 16 * b, v); },
      [&](int b, uint32_t sb, uint32_t w0, uint32_t w1) {
        *reinterpret_cast<uint2*>(a.hq + (size_t)r * (I / 2) + 8 * b) = make_uint2(w0, w1);
        a.hsf[sf_chunk_offset(r, b, KG)] = (uint8_t)sb;
      });
}

// One warp per routed row: NVFP4 row of h (BF16) for FC2; padding rows get
// zero codes, zero scales and G = 0.
__global__ void quant_h_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= 128 * *a.num_tiles) return;
  const int lane = threadIdx.x & 31;
  const int I = a.I, KG = I / 64;
  if (a.row_src[r] < 0) {
    for (int b = lane; b < I / 16; b += 32) {
      *reinterpret_cast<uint2*>(a.hq + (size_t)r * (I / 2) + 8 * b) = make_uint2(0u, 0u);
      a.hsf[sf_chunk_offset(r, b, KG)] = 0;
    }
    if (lane == 0) a.hG[r] = 0.f;
    return;
  }
  const float G = quant_h_row(a, r);
  if (lane == 0) a.hG[r] = G;
}

// Mid band: one warp per routing entry, the routed rows only (the swapped
// GEMMs never use a padding row's products, so its bytes stay as they are).
// The row's FC2 factor G * (down multiplier) * (router weight) -- the
// product the prefill band's FC2 epilogue forms, in the same order -- takes
// G's place.
__global__ void quant_h_routed_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int i = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (i >= a.n_entries) return;
  const int r = a.pos[i];
  if (r < 0) return;
  const float G = quant_h_row(a, r);
  if ((threadIdx.x & 31) == 0) {
    const float* g2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * scale_chunk_bytes(a.H, a.I));
    a.hG[r] = G * g2[route_id(a.ids, i, a.ids64, a.E)] * a.tw[i];
  }
}

// ---------------------------------------------------------------- GEMMs
// 16 lanes x 256 bits of tensor memory, eight times along the columns (64
// FP32 columns): thread t holds, per 8-column block q, columns 2 (t % 4) and
// 2 (t % 4) + 1 of lanes t / 4 (registers 4q, 4q + 1) and t / 4 + 8 (4q + 2,
// 4q + 3) of the 16 lanes at the address's lane field.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// FC2 epilogue of a BN-column accumulator tile, one routed row per lane of
// this warp's 32 tensor-memory lanes (tmem_row: their lane field):
// out[tok][col] += f * D[row][col] for the rows with tok >= 0 (tok and f are
// this lane's row's).  The accumulator is read in the 16-lane x 256-bit shape
// (a thread holds two consecutive columns of rows g and g + 8 of a 16-row
// half), so that a warp's FP32 reductions cover 8 rows x 32 contiguous bytes
// (whole sectors) instead of 32 rows x 16 bytes: measured on prefill_e128,
// NVFP4 layer 731 -> 689 us.
template <int BN>
__device__ __forceinline__ void reduce_rows_to_tokens(uint32_t tmem_row, float f, int tok, float* out, int H) {
  const int lane = threadIdx.x & 31;
  out += 2 * (lane & 3);
#pragma unroll 1
  for (int hf = 0; hf < 2; ++hf) {  // 16-lane halves of the warp's 32 rows
    const int ra = 16 * hf + (lane >> 2), rb = ra + 8;  // this thread's two rows
    const int ta = __shfl_sync(0xffffffffu, tok, ra), tb = __shfl_sync(0xffffffffu, tok, rb);
    const float fa = __shfl_sync(0xffffffffu, f, ra), fb = __shfl_sync(0xffffffffu, f, rb);
    if (!__any_sync(0xffffffffu, ta >= 0 || tb >= 0)) continue;  // a half of padding rows (small batches)
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {  // 64 columns per load
      uint32_t v[32];
      tmem_ld_16x256b_x8(tmem_row + ((uint32_t)(16 * hf) << 16) + 64 * c, v);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int col = 64 * c + 8 * q;
        if (ta >= 0)
          asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(out + (size_t)ta * H + col),
                       "f"(__uint_as_float(v[4 * q]) * fa), "f"(__uint_as_float(v[4 * q + 1]) * fa)
                       : "memory");
        if (tb >= 0)
          asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(out + (size_t)tb * H + col),
                       "f"(__uint_as_float(v[4 * q + 2]) * fb), "f"(__uint_as_float(v[4 * q + 3]) * fb)
                       : "memory");
      }
    }
  }
}
// FC2's tile width: 128, two accumulators, so that a tile's reduction
// epilogue runs beside the next tile's MMAs.  Measured on GB300 at
// prefill_e128 (us per layer, 128 / 256): 672 / 685 with the reductions in
// whole sectors; with the earlier row-wise reductions 256 was ahead (737 /
// 756): the narrower tiles stage a third more bytes per FLOP.
constexpr int kFc2BN = 128;
// Tile (m, n) with n fastest, dealt round-robin to one persistent CTA per
// SM: CTAs sharing an activation tile run together, and the M-tiles of one
// expert (sharing weight tiles) follow each other.
// FC1 N tiles span BN / 128 resident w13 tiles (64 gate/up pairs each);
// launched with BN = 128 (one resident tile per N tile).
template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    fc1_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  // non-gated experts (squared ReLU): N tiles of 128 w1 rows, the expert's
  // last one padded (its scale rows past I are zero); gated: 2I rows
  const bool relu2 = a.act.kind == MOE_FP4_ACT_RELU2;
  const int NT = relu2 ? (a.I + 127) / 128 : 2 * a.I / BN;
  const int KG = a.H / 64;
  const size_t scb = scale_chunk_bytes(relu2 ? NT * 128 : 2 * a.I, a.H);
  const float* g13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    GemmTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kGemmBM * mt;
    t.b_row0 = (relu2 ? e * a.I : e * 2 * a.I) + BN * nt;
    t.a_sf = a.xsf + (size_t)mt * KG * kChunkBytes;
    t.b_sf0 = a.s13 + (size_t)e * scb + (size_t)(BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const GemmTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const bool live = a.row_src[r] >= 0;
    const float xg = live ? a.xG[r] : 0.f;
    if (relu2) {
      // h = max(u, 0)^2 in BF16 for the tile's rows of w1 below I (BN = 128)
      const float s1 = xg * g13[e];
      __nv_bfloat16* hrow = a.hbuf + (size_t)r * a.I;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // 32-column chunks (I % 64 == 0: whole chunks)
        uint32_t u[32];
        tmem_ld32(tmem_row + 32 * c, u);
        const int n0 = 128 * t.n_tile + 32 * c;
        if (!live || n0 >= a.I) continue;
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float r0 = fmaxf(__uint_as_float(u[2 * j]) * s1, 0.f);
          const float r1 = fmaxf(__uint_as_float(u[2 * j + 1]) * s1, 0.f);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(r0 * r0, r1 * r1);
          packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        uint4* dst = reinterpret_cast<uint4*>(hrow + n0);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
      }
      return;
    }
    const float sgate = xg * g13[2 * e], sup = xg * g13[2 * e + 1];
    __nv_bfloat16* hrow = a.hbuf + (size_t)r * a.I;
#pragma unroll 1
    for (int q = 0; q < BN / 128; ++q) {  // the 128-row resident tiles of this N tile
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 32-pair chunks of the tile's 64 pairs
        uint32_t g[32], u[32];
        tmem_ld32(tmem_row + 128 * q + 32 * c, g);
        tmem_ld32(tmem_row + 128 * q + 64 + 32 * c, u);
        if (live) {
          const int n0 = 64 * ((BN / 128) * t.n_tile + q) + 32 * c;
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = gated_act(__uint_as_float(g[2 * j]) * sgate, __uint_as_float(u[2 * j]) * sup, a.act);
            const float h1 =
                gated_act(__uint_as_float(g[2 * j + 1]) * sgate, __uint_as_float(u[2 * j + 1]) * sup, a.act);
            const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
            packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          uint4* dst = reinterpret_cast<uint4*>(hrow + n0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
    }
  };
  gemm_fp4_persistent<BN>(&map_x, &map_w, a.H, a.status, n_mt * NT, tile_of, epi);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    fc2_gemm_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                    PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int NT = a.H / kFc2BN;
  const int KG = a.I / 64;
  const size_t scb = scale_chunk_bytes(a.H, a.I);
  const float* g2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    GemmTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kGemmBM * mt;
    t.b_row0 = e * a.H + kFc2BN * nt;
    t.a_sf = a.hsf + (size_t)mt * KG * kChunkBytes;
    t.b_sf0 = a.s2 + (size_t)e * scb + (size_t)(kFc2BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const GemmTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const int src = a.row_src[r];
    const float f = src >= 0 ? a.hG[r] * g2[e] * a.tw[src] : 0.f;
    reduce_rows_to_tokens<kFc2BN>(tmem_row, f, src >= 0 ? src / a.top_k : -1, a.acc + kFc2BN * t.n_tile, a.H);
  };
  gemm_fp4_persistent<kFc2BN>(&map_h, &map_w, a.I, a.status, n_mt * NT, tile_of, epi);
}

// ---------------------------------------------------------------- mid band
// Batches with few routed rows per expert: the same layer (same activation
// quantisation, same products) with the GEMM operands swapped
// (gemm_fp4_swap.cuh): the weights fill the MMA's 128-row side, and the
// routed rows of a 32-row routing tile (each expert's rows padded to a
// multiple of 32) are its N side, 16 or 32 of them.  A tile is (routing
// tile, group of up to four 128-row weight tiles), the group fastest.
struct BMaps {
  CUtensorMap m[2];  // B boxes of 16 and 32 rows
};
constexpr int kMidPad = 32;  // the mid band's routing-tile height
constexpr int kFc1SwapSubs = 2;  // FC1's weight tiles per item at most (the gate/up exchange area)
static_assert(kFc1SwapSubs * 32 * 64 * 4 + 16 <= SwapCfg::kExtra, "epilogue exchange area");

// Per-routing-tile values of the epilogues, fetched by each epilogue thread
// for its next tile while it finishes the current one (lane j: column j).
struct MidCols {
  int mt = -1, nv = 0, src = 0;
  float v = 0.f, m0 = 0.f, m1 = 0.f;
};

// FC1: D[w13 row][routed row].  A 128-row w13 tile holds 64 gate rows then
// the 64 matching up rows, so the up lanes hand their values to the gate
// lanes through shared memory (mbarriers: up values written / read).
__global__ void __launch_bounds__(kSwapThreads, 1)
    fc1_swap_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ BMaps maps_x, PrefillArgs a,
                    int subs) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const bool relu2 = a.act.kind == MOE_FP4_ACT_RELU2;
  const int NT = relu2 ? (a.I + 127) / 128 : 2 * a.I / 128;  // weight tiles per expert
  const int NG = (NT + subs - 1) / subs;  // weight-tile groups per routing tile
  const int KG = a.H / 64;
  const size_t scb = scale_chunk_bytes(relu2 ? NT * 128 : 2 * a.I, a.H);
  const float* g13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  const int lane = threadIdx.x & 31;
  // [weight tile][column][64] up values of at most kFc1SwapSubs weight tiles
  float* xch = reinterpret_cast<float*>(swap_extra_smem());
  uint64_t* xbar = reinterpret_cast<uint64_t*>(xch + kFc1SwapSubs * 32 * 64);  // [0] written, [1] read
  if (threadIdx.x == 0) {
    mbar_init(&xbar[0], 64);
    mbar_init(&xbar[1], 64);
  }
  auto tile_of = [&](int idx) {
    SwapTile t;
    const int mt = idx / NG, g = idx % NG;
    t.m_tile = mt;
    t.group = g;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.subs = NT - subs * g < subs ? NT - subs * g : subs;
    t.n_rows = a.tile_rows[mt] <= 16 ? 16 : 32;
    t.a_row0 = (relu2 ? e * a.I : e * 2 * a.I) + 128 * subs * g;
    t.b_row0 = kMidPad * mt;
    t.b_word = mt & 3;
    t.a_sf = a.s13 + (size_t)e * scb + (size_t)subs * g * KG * kChunkBytes;
    t.a_sf_step = (size_t)KG * kChunkBytes;
    t.b_sf = a.xsf + (size_t)(mt >> 2) * KG * kChunkBytes;
    return t;
  };
  auto fetch = [&](int mt) {
    MidCols c;
    c.mt = mt;
    const int e = a.tile_expert[mt];
    c.nv = a.tile_rows[mt];
    c.v = a.xG[kMidPad * mt + lane];
    c.m0 = relu2 ? g13[e] : g13[2 * e];  // gate (w1) multiplier
    c.m1 = relu2 ? 0.f : g13[2 * e + 1];  // up multiplier
    return c;
  };
  // the epilogue warps fetch their first tile's values while its stages stream
  MidCols cur, pf;
  if (threadIdx.x >= 192 && (int)blockIdx.x < n_mt * NG) pf = fetch((int)blockIdx.x / NG);
  int xi = 0;  // tiles this epilogue thread has finished
  auto epi = [&](uint32_t tmem_row, int row, const SwapTile& t) {
    cur = pf.mt == t.m_tile ? pf : fetch(t.m_tile);
    const int next = t.m_tile * NG + t.group + (int)gridDim.x;
    if (next < n_mt * NG && next / NG != t.m_tile) pf = fetch(next / NG);
    const int nv = cur.nv, N = t.n_rows;
    const float xg = cur.v;  // lane c: column c's x multiplier
    if (relu2) {
      // h = max(u, 0)^2 for w1 rows below I
      const float m0 = cur.m0;
#pragma unroll 1
      for (int j = 0; j < t.subs; ++j) {
        const int n = 128 * (subs * t.group + j) + row;
        uint32_t v[32];
        tmem_ld32(tmem_row + j * N, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= nv) break;  // (warp-uniform)
          const float xc = __shfl_sync(0xffffffffu, xg, c);
          if (n < a.I) {
            const float u = fmaxf(__uint_as_float(v[c]) * (xc * m0), 0.f);
            a.hbuf[(size_t)(t.b_row0 + c) * a.I + n] = __float2bfloat16_rn(u * u);
          }
        }
      }
      return;
    }
    const int l = row & 63;
    if (row >= 64) {
      // up lanes: this tile's up values into the exchange area once the gate
      // lanes have read the previous tile's
      if (xi > 0) mbar_wait(&xbar[1], (xi - 1) & 1, a.status, 16u);
#pragma unroll 1
      for (int j = 0; j < t.subs; ++j) {
        uint32_t v[32];
        tmem_ld32(tmem_row + j * N, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) xch[(j * 32 + c) * 64 + l] = __uint_as_float(v[c]);
      }
      mbar_arrive(&xbar[0]);
    } else {
      const float mg = cur.m0, mu = cur.m1;
      mbar_wait(&xbar[0], xi & 1, a.status, 16u);
#pragma unroll 1
      for (int j = 0; j < t.subs; ++j) {
        const int n = 64 * (subs * t.group + j) + l;
        uint32_t v[32];
        tmem_ld32(tmem_row + j * N, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          // (warp-uniform) leaving at the first padding column keeps the
          // unrolled loop's later iterations out of the instruction stream:
          // skipping them one by one fetched each from memory, and the first
          // tile's epilogue took 12 us against 2 (decode_e512 M=64 126 ->
          // 118 us per layer)
          if (c >= nv) break;
          const float xc = __shfl_sync(0xffffffffu, xg, c);
          const float h =
              gated_act(__uint_as_float(v[c]) * (xc * mg), xch[(j * 32 + c) * 64 + l] * (xc * mu), a.act);
          a.hbuf[(size_t)(t.b_row0 + c) * a.I + n] = __float2bfloat16_rn(h);
        }
      }
      mbar_arrive(&xbar[1]);
    }
    ++xi;
  };
  gemm_fp4_swap_persistent(&map_w, &maps_x.m[0], a.H, a.status, n_mt * NG, tile_of, epi);
}

// FC2: D[w2 row][routed row]; each lane owns an output column and reduces its
// routed rows' products, times the rows' factors (hG, with the down
// multiplier and router weight folded in), into the FP32 token accumulator.
__global__ void __launch_bounds__(kSwapThreads, 1)
    fc2_swap_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ BMaps maps_h, PrefillArgs a,
                    int subs) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int NT = a.H / 128;
  const int NG = (NT + subs - 1) / subs;  // weight-tile groups per routing tile
  const int KG = a.I / 64;
  const size_t scb = scale_chunk_bytes(a.H, a.I);
  const int n_mt = *a.num_tiles;
  const int lane = threadIdx.x & 31;
  auto tile_of = [&](int idx) {
    SwapTile t;
    const int mt = idx / NG, g = idx % NG;
    t.m_tile = mt;
    t.group = g;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.subs = NT - subs * g < subs ? NT - subs * g : subs;
    t.n_rows = a.tile_rows[mt] <= 16 ? 16 : 32;
    t.a_row0 = e * a.H + 128 * subs * g;
    t.b_row0 = kMidPad * mt;
    t.b_word = mt & 3;
    t.a_sf = a.s2 + (size_t)e * scb + (size_t)subs * g * KG * kChunkBytes;
    t.a_sf_step = (size_t)KG * kChunkBytes;
    t.b_sf = a.hsf + (size_t)(mt >> 2) * KG * kChunkBytes;
    return t;
  };
  auto fetch = [&](int mt) {
    MidCols c;
    c.mt = mt;
    c.nv = a.tile_rows[mt];
    c.src = a.row_src[kMidPad * mt + lane];  // (-1 on padding rows, never used)
    c.v = a.hG[kMidPad * mt + lane];
    return c;
  };
  // the epilogue warps fetch their first tile's values while its stages stream
  MidCols cur, pf;
  if (threadIdx.x >= 192 && (int)blockIdx.x < n_mt * NG) pf = fetch((int)blockIdx.x / NG);
  // one red.add per (output row, routed row): a warp's 32 lanes reduce 32
  // consecutive outputs of one token; the tile's accumulator columns come
  // out of tensor memory 64 at a time under one wait
  auto epi = [&](uint32_t tmem_row, int row, const SwapTile& t) {
    cur = pf.mt == t.m_tile ? pf : fetch(t.m_tile);
    const int next = t.m_tile * NG + t.group + (int)gridDim.x;
    if (next < n_mt * NG && next / NG != t.m_tile) pf = fetch(next / NG);
    const int nv = cur.nv, N = t.n_rows, tok = cur.src / a.top_k;
    float* out0 = a.acc + 128 * (subs * t.group) + row;
    // sub-tile j's column c: value v, token and factor of routed row c
    auto put = [&](int j, int c, uint32_t v) {
      const int tc = __shfl_sync(0xffffffffu, tok, c);
      const float fc = __shfl_sync(0xffffffffu, cur.v, c);
      asm volatile("red.global.add.f32 [%0], %1;" ::"l"(out0 + (size_t)tc * a.H + 128 * j), "f"(__uint_as_float(v) * fc)
                   : "memory");
    };
#pragma unroll 1
    for (int j0 = 0; j0 < t.subs; j0 += 64 / N) {  // 64 accumulator columns per round
      uint32_t v0[32], v1[32];
      swap_tmem_ld32(tmem_row + j0 * N, v0);
      swap_tmem_ld32(tmem_row + j0 * N + 32, v1);
      swap_tmem_ld_wait();
      if (N == 16) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c >= nv) break;  // (warp-uniform)
          put(j0, c, v0[c]);
          if (j0 + 1 < t.subs) put(j0 + 1, c, v0[16 + c]);
          if (j0 + 2 < t.subs) put(j0 + 2, c, v1[c]);
          if (j0 + 3 < t.subs) put(j0 + 3, c, v1[16 + c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= nv) break;  // (warp-uniform)
          put(j0, c, v0[c]);
          if (j0 + 1 < t.subs) put(j0 + 1, c, v1[c]);
        }
      }
    }
  };
  gemm_fp4_swap_persistent(&map_w, &maps_h.m[0], a.I, a.status, n_mt * NG, tile_of, epi);
}

// MXFP8 (W4A8-MX activations): E4M3 elements with one UE8M0 scale per 32
// K-elements; block scale 2^e with e = ceil(log2(amax_blk / 448)) (0 for an
// all-zero block), clamped to [-127, 127]; elements e4m3_rn(a / 2^e), never
// above 448 by construction.  ceil(log2(amax / 448)) from amax's bits:
// amax = m 2^E with m in [1, 2) and 448 = 1.75 2^8, so it is E - 8, plus one
// when m > 1.75 (mantissa field above 0x600000); amaxes below the normal
// range give less than -127.
__device__ __forceinline__ int mxfp8_scale_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0u) return 0;
  const int E = (int)(b >> 23) - 127;
  if (E == -127) return -127;
  const int e = E - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// One warp quantises a row of K elements (K % 32 == 0): lane l takes the
// 32-element blocks l, l + 32, ...; load32(block, float[32]) supplies a
// block, emit(block, scale_byte, 32 code bytes as 8 words) takes the result.
template <class Load32, class Emit>
__device__ __forceinline__ void quant_row_mxfp8(int K, const Load32& load32, const Emit& emit) {
  const int lane = threadIdx.x & 31;
  for (int b = lane; b < K / 32; b += 32) {
    float v[32];
    load32(b, v);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mxfp8_scale_exponent(amax);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, exact (e <= 120 for finite FP32)
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // (the second source lands in the low byte)
      uint16_t lo, hi;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[4 * j + 1] * inv), "f"(v[4 * j] * inv));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[4 * j + 3] * inv), "f"(v[4 * j + 2] * inv));
      w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    emit(b, (uint32_t)(e + 127), w);
  }
}

// One MXFP8 block of 32 values quantised and dequantised in place: the
// scale exponent and E4M3 rounding of quant_row_mxfp8, then each code times
// 2^e, exact in FP32 (at most four significant bits, magnitudes >= 2^-136).
__device__ __forceinline__ void mxfp8_qdq32(float (&v)[32]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mxfp8_scale_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e (e <= 120 for finite FP32)
  const float sc = e > -127 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);  // 2^e
#pragma unroll
  for (int j = 0; j < 16; ++j) {  // (the second source lands in the low byte, which widens to the low half)
    uint16_t c;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(v[2 * j + 1] * inv), "f"(v[2 * j] * inv));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    const float2 f = half2_bits_to_float2(h2);
    v[2 * j] = f.x * sc;
    v[2 * j + 1] = f.y * sc;
  }
}

// Eight values of an MXFP8 block whose largest magnitude is amax, quantised
// and dequantised in place (the same exponent and per-element rounding as
// mxfp8_qdq32, for a block spread over four threads).
__device__ __forceinline__ void mxfp8_qdq8(float (&v)[8], float amax) {
  const int e = mxfp8_scale_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
  const float sc = e > -127 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint16_t c;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(v[2 * j + 1] * inv), "f"(v[2 * j] * inv));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    const float2 f = half2_bits_to_float2(h2);
    v[2 * j] = f.x * sc;
    v[2 * j + 1] = f.y * sc;
  }
}

// ---------------------------------------------------------------- exact numerics
// The prefill band without NVFP4 activations, on the FP16 tensor cores: x in
// BF16 (or its MXFP8 image, W4A8-MX) against the FP4 weights decoded to FP16
// (exact), FP32 sums; h = act(gate, up) staged in BF16 (then, W4A8-MX,
// through MXFP8), FC2 into the same FP32 token accumulator, one cast.  Every
// 16-bit operand row is scaled by a power of two so that its largest
// magnitude lies in [2^14, 2^15): BF16 and MXFP8 values are then exact in
// FP16 unless they lie more than 2^31 below their row's largest, and the
// epilogues multiply the power back out (exact).

// FP16 row scale: 2^s with max |v| 2^s in [2^14, 2^15), s in [-126, 126];
// 0 for a zero or non-finite maximum.
__device__ __forceinline__ int f16_row_shift(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0u || b >= 0x7F800000u) return 0;
  const int E = b >= 0x00800000u ? (int)(b >> 23) - 127 : -127;  // floor(log2 amax) (subnormals: below -126)
  const int sft = 14 - E;
  return sft < -126 ? -126 : (sft > 126 ? 126 : sft);
}
__device__ __forceinline__ float pow2f(int e) {  // e in [-126, 127]
  return __uint_as_float((uint32_t)(e + 127) << 23);
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One block of 128 threads per token: x's BF16 row (amode 0), or its MXFP8
// image (amode 1: quantised per 32-element block, then dequantised), scaled
// by the row's power of two and stored in FP16 into every routed row of the
// token (the GEMM's A tiles are rows of routed rows), with 2^-s in xG; also
// zeroes the token's FP32 accumulator row.  Thread t takes the 8-element
// chunks t, t + 128, ...; the four threads of a 32-element block are
// neighbouring lanes.  The MXFP8 image never exceeds max |x| by more than
// 2^-4 of it (E4M3 rounds to nearest), so the FP16 range holds.
__global__ void __launch_bounds__(128) stage_x_f16_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  __shared__ float red4[4];
  const int t = blockIdx.x;
  const int H = a.H, k = a.top_k, nc = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * H);
  const int* prow = a.pos + (size_t)t * k;
  float amax = 0.f;
  for (int c = threadIdx.x; c < nc; c += 128) {
    float v[8];
    bf16x8_to_f32(__ldg(xr + c), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = block128_max(amax, red4);
  const int sft = f16_row_shift(amax);
  const float up = pow2f(sft);
  if (threadIdx.x < k) {
    const int r = prow[threadIdx.x];
    if (r >= 0) a.xG[r] = pow2f(-sft);
  }
  int rows[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) rows[j] = j < k ? prow[j] : -1;
  for (int c = threadIdx.x; c < nc; c += 128) {  // (nc % 32 == 0: a warp's lanes stay converged)
    float v[8];
    bf16x8_to_f32(__ldg(xr + c), v);
    if (a.amode) {
      float bm = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) bm = fmaxf(bm, fabsf(v[i]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      mxfp8_qdq8(v, bm);
    }
    const uint4 o = make_uint4(f16x2_of(v[0] * up, v[1] * up), f16x2_of(v[2] * up, v[3] * up),
                               f16x2_of(v[4] * up, v[5] * up), f16x2_of(v[6] * up, v[7] * up));
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (rows[j] >= 0) reinterpret_cast<uint4*>(a.xb + (size_t)rows[j] * H)[c] = o;
  }
  float4* accr = reinterpret_cast<float4*>(a.acc + (size_t)t * H);
  for (int v = threadIdx.x; v < H / 4; v += 128) accr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// One warp per live routed row: h (BF16, written by FC1) rescaled by the
// row's power of two and converted to FP16 in place, 2^-s in hG.
__global__ void stage_h_f16_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= 128 * *a.num_tiles || a.row_src[r] < 0) return;
  const int lane = threadIdx.x & 31;
  uint4* hr = reinterpret_cast<uint4*>(a.hbuf + (size_t)r * a.I);
  float amax = 0.f;
  for (int v = lane; v < a.I / 8; v += 32) {
    const uint4 u = hr[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int sft = f16_row_shift(amax);
  const float up = pow2f(sft);
  if (lane == 0) a.hG[r] = pow2f(-sft);
  for (int v = lane; v < a.I / 8; v += 32) {
    const uint4 u = hr[v];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = f16x2_of(__uint_as_float(w[i] << 16) * up, __uint_as_float(w[i] & 0xFFFF0000u) * up);
    hr[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// FC1, exact, on BN-wide N tiles: BN / 128 resident 128-row tiles of 64
// gate/up pairs each, or (BN = 128) 128 rows of a non-gated expert's w1.
template <int BN>
__global__ void __launch_bounds__(kHwThreads, 1)
    fc1_exact_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                     PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const bool relu2 = a.act.kind == MOE_FP4_ACT_RELU2;
  const int NT = relu2 ? (a.I + 127) / 128 : 2 * a.I / BN;
  const int KG = a.H / 64;
  const size_t scb = scale_chunk_bytes(relu2 ? (a.I + 127) / 128 * 128 : 2 * a.I, a.H);
  const float* g13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    HwTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kHwBM * mt;
    t.b_row0 = (relu2 ? e * a.I : e * 2 * a.I) + BN * nt;
    t.b_sf0 = a.s13 + (size_t)e * scb + (size_t)(BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const HwTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const bool live = a.row_src[r] >= 0;
    const float xs = live ? a.xG[r] : 0.f;  // the row's 2^-s
    __nv_bfloat16* hrow = a.hbuf + (size_t)r * a.I;
    if (relu2) {
      const float g1 = g13[e] * xs;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem_row + 32 * c, u);
        const int n0 = 128 * t.n_tile + 32 * c;
        if (!live || n0 >= a.I) continue;
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float r0 = fmaxf(__uint_as_float(u[2 * j]) * g1, 0.f);
          const float r1 = fmaxf(__uint_as_float(u[2 * j + 1]) * g1, 0.f);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(r0 * r0, r1 * r1);
          packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        uint4* dst = reinterpret_cast<uint4*>(hrow + n0);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
      }
      return;
    }
    const float sgate = g13[2 * e] * xs, sup = g13[2 * e + 1] * xs;
#pragma unroll 1
    for (int q = 0; q < BN / 128; ++q) {  // the 128-row resident tiles of this N tile
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 32-pair chunks of the tile's 64 pairs
        uint32_t g[32], u[32];
        tmem_ld32(tmem_row + 128 * q + 32 * c, g);
        tmem_ld32(tmem_row + 128 * q + 64 + 32 * c, u);
        if (live) {
          const int n0 = 64 * ((BN / 128) * t.n_tile + q) + 32 * c;
          float hf[32];  // h staged in BF16 (one 32-element block of the row)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            hf[j] = __bfloat162float(__float2bfloat16_rn(
                gated_act(__uint_as_float(g[j]) * sgate, __uint_as_float(u[j]) * sup, a.act)));
          if (a.amode) mxfp8_qdq32(hf);  // W4A8-MX: h quantised per routed row, block of 32
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 hv = __floats2bfloat162_rn(hf[2 * j], hf[2 * j + 1]);  // exact
            packed[j] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          uint4* dst = reinterpret_cast<uint4*>(hrow + n0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
    }
  };
  gemm_f16w4_persistent<BN>(&map_x, &map_w, a.H, a.status, n_mt * NT, tile_of, epi);
}

// FC2, exact: h (BF16) against w2 decoded to BF16, router-weighted FP32
// reductions into the token accumulator.
__global__ void __launch_bounds__(kHwThreads, 1)
    fc2_exact_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                     PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  constexpr int BN = kFc2ExactBN;
  const int NT = a.H / BN;
  const int KG = a.I / 64;
  const size_t scb = scale_chunk_bytes(a.H, a.I);
  const float* g2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    HwTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kHwBM * mt;
    t.b_row0 = e * a.H + BN * nt;
    t.b_sf0 = a.s2 + (size_t)e * scb + (size_t)(BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const HwTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const int src = a.row_src[r];
    const float f = src >= 0 ? g2[e] * a.tw[src] * a.hG[r] : 0.f;
    reduce_rows_to_tokens<BN>(tmem_row, f, src >= 0 ? src / a.top_k : -1, a.acc + BN * t.n_tile, a.H);
  };
  gemm_f16w4_persistent<BN>(&map_h, &map_w, a.I, a.status, n_mt * NT, tile_of, epi);
}

// ---------------------------------------------------------------- W4A8-MX, FP8 tensor cores
// MXFP8 x (per token) and h (per routed row) against the MXFP4 weights on
// tcgen05.mma kind::mxf8f6f4 (gemm_mxf8.cuh): the products are those of the
// W4A8-MX definition exactly, summed in FP32.  Needs I % 128 == 0 (the
// unpacking tensor map's row length); gated activations.

// Byte offset of (row, 32-element block b) in a UE8M0 chunk array of K =
// 128 * nst: chunk (row / 128, b / 4), byte (row % 32) * 16 + (row / 32 % 4) * 4
// + b % 4.
__device__ __forceinline__ size_t mx_sf_offset(int row, int b, int nst) {
  return ((size_t)(row >> 7) * nst + (b >> 2)) * kChunkBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (b & 3);
}

// One block of 128 threads per token: x quantised to MXFP8 into every
// routed row of the token, thread t taking the 8-element chunks t, t + 128,
// ... (the four threads of a 32-element block are neighbouring lanes and
// share its largest magnitude by shuffles; the first writes the scale byte);
// zeroes the token's accumulator.  The rule is quant_row_mxfp8's.
__global__ void __launch_bounds__(128) quant_x_mx_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int t = blockIdx.x;
  const int H = a.H, k = a.top_k, nst = H / 128, nc = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * H);
  const int* prow = a.pos + (size_t)t * k;
  int rows[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) rows[j] = j < k ? prow[j] : -1;
  for (int c = threadIdx.x; c < nc; c += 128) {  // (nc % 32 == 0: a warp's lanes stay converged)
    float v[8];
    bf16x8_to_f32(__ldg(xr + c), v);
    float bm = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) bm = fmaxf(bm, fabsf(v[i]));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
    const int e = mxfp8_scale_exponent(bm);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e (e <= 120 for finite FP32)
    uint32_t w[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // (the second source lands in the low byte)
      uint16_t lo, hi;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[4 * j + 1] * inv), "f"(v[4 * j] * inv));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[4 * j + 3] * inv), "f"(v[4 * j + 2] * inv));
      w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      reinterpret_cast<uint2*>(a.xq8 + (size_t)r * H)[c] = make_uint2(w[0], w[1]);
      if ((c & 3) == 0) a.xsf8[mx_sf_offset(r, c >> 2, nst)] = (uint8_t)(e + 127);
    }
  }
  float4* accr = reinterpret_cast<float4*>(a.acc + (size_t)t * H);
  for (int v = threadIdx.x; v < H / 4; v += 128) accr[v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// One MXFP8 block of 32 values (this thread's): E4M3 codes as 8 words
// (element 4j + i in byte i of word j) and the UE8M0 scale byte, by the rule
// of quant_row_mxfp8.
__device__ __forceinline__ uint32_t mxfp8_block32(const float (&v)[32], uint32_t (&w)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mxfp8_scale_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e (e <= 120 for finite FP32)
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // (the second source lands in the low byte)
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[4 * j + 1] * inv), "f"(v[4 * j] * inv));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[4 * j + 3] * inv), "f"(v[4 * j + 2] * inv));
    w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return (uint32_t)(e + 127);
}

// FC1, W4A8-MX: BN-wide N tiles (BN / 128 resident 128-row tiles of 64
// gate/up pairs; two accumulators at BN = 128, one at 256); the epilogue
// applies the activation, stages h in BF16 and quantises it per 32-block of
// the routed row (the thread owns the row) for FC2.
template <int BN>
__global__ void __launch_bounds__(kMxThreads, 1)
    fc1_mx_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                  PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const int NT = 2 * a.I / BN;
  const int KG = a.H / 64, nst = a.H / 128, nsth = a.I / 128;
  const size_t scb = scale_chunk_bytes(2 * a.I, a.H);
  const float* g13 = reinterpret_cast<const float*>(a.s13 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    MxTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kMxBM * mt;
    t.a_sf = a.xsf8 + (size_t)mt * nst * kChunkBytes;
    t.b_row0 = e * 2 * a.I + BN * nt;
    t.b_sf0 = a.s13 + (size_t)e * scb + (size_t)(BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const MxTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const bool live = a.row_src[r] >= 0;
    const float sgate = g13[2 * e], sup = g13[2 * e + 1];
#pragma unroll 1
    for (int q = 0; q < BN / 128; ++q) {  // the 128-row resident tiles of this N tile
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // 32-pair chunks of the tile's 64 pairs
        uint32_t g[32], u[32];
        tmem_ld32(tmem_row + 128 * q + 32 * c, g);
        tmem_ld32(tmem_row + 128 * q + 64 + 32 * c, u);
        const int n0 = 64 * ((BN / 128) * t.n_tile + q) + 32 * c;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t sb = 0u;
        if (live) {
          float hf[32];  // h staged in BF16
#pragma unroll
          for (int j = 0; j < 32; ++j)
            hf[j] = __bfloat162float(__float2bfloat16_rn(
                gated_act(__uint_as_float(g[j]) * sgate, __uint_as_float(u[j]) * sup, a.act)));
          sb = mxfp8_block32(hf, w);
        }
        uint4* dst = reinterpret_cast<uint4*>(a.hq8 + (size_t)r * a.I + n0);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        a.hsf8[mx_sf_offset(r, n0 / 32, nsth)] = (uint8_t)sb;
      }
    }
  };
  gemm_mxf8_persistent<BN>(&map_x, &map_w, a.H, a.status, n_mt * NT, tile_of, epi);
}

// FC2, W4A8-MX: MXFP8 h against w2, router-weighted FP32 reductions into the
// token accumulator.
__global__ void __launch_bounds__(kMxThreads, 1)
    fc2_mx_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                  PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  constexpr int BN = kMxFc2BN;
  const int NT = a.H / BN;
  const int KG = a.I / 64, nst = a.I / 128;
  const size_t scb = scale_chunk_bytes(a.H, a.I);
  const float* g2 = reinterpret_cast<const float*>(a.s2 + (size_t)a.E * scb);
  const int n_mt = *a.num_tiles;
  auto tile_of = [&](int idx) {
    MxTile t;
    const int mt = idx / NT, nt = idx % NT;
    t.m_tile = mt;
    t.n_tile = nt;
    t.valid = mt < n_mt;
    if (!t.valid) return t;
    const int e = a.tile_expert[mt];
    t.a_row0 = kMxBM * mt;
    t.a_sf = a.hsf8 + (size_t)mt * nst * kChunkBytes;
    t.b_row0 = e * a.H + BN * nt;
    t.b_sf0 = a.s2 + (size_t)e * scb + (size_t)(BN / 128) * nt * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    return t;
  };
  auto epi = [&](uint32_t tmem_row, int row, const MxTile& t) {
    const int r = t.a_row0 + row;
    const int e = a.tile_expert[t.m_tile];
    const int src = a.row_src[r];
    const float f = src >= 0 ? g2[e] * a.tw[src] : 0.f;
    reduce_rows_to_tokens<BN>(tmem_row, f, src >= 0 ? src / a.top_k : -1, a.acc + BN * t.n_tile, a.H);
  };
  gemm_mxf8_persistent<BN>(&map_h, &map_w, a.I, a.status, n_mt * NT, tile_of, epi);
}

__global__ void cast_out_kernel(PrefillArgs a) {
  pdl_wait();               // the previous kernel on the stream is complete and visible
  pdl_launch_dependents();  // the next may start its prologue (it waits the same way)
  const size_t n8 = (size_t)a.M * a.H / 8;
  for (size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x; v < n8; v += (size_t)gridDim.x * blockDim.x) {
    const float4 p = reinterpret_cast<const float4*>(a.acc)[2 * v];
    const float4 q = reinterpret_cast<const float4*>(a.acc)[2 * v + 1];
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(p.x, p.y), b1 = __floats2bfloat162_rn(p.z, p.w);
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(q.x, q.y), b3 = __floats2bfloat162_rn(q.z, q.w);
    reinterpret_cast<uint4*>(a.out)[v] =
        make_uint4(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1),
                   *reinterpret_cast<const uint32_t*>(&b2), *reinterpret_cast<const uint32_t*>(&b3));
  }
}

// Grouped routed rows -> unpadded permutation (test support).
__global__ void route_perm_kernel(PrefillArgs a, int32_t* perm) {
  const int e = blockIdx.x;
  const int n = a.expert_off[e + 1] - a.expert_off[e];
  for (int i = threadIdx.x; i < n; i += blockDim.x) perm[a.expert_off[e] + i] = a.row_src[a.expert_poff[e] + i];
}
__global__ void fill_i32_kernel(int32_t* p, int n, int v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

// One warp per row: the MXFP8 quantiser alone (test support).
__global__ void debug_quant_mxfp8_kernel(const float* in, int rows, int K, uint8_t* q, uint8_t* s) {
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* row = in + (size_t)r * K;
  quant_row_mxfp8(
      K, [&](int b, float (&v)[32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = row[32 * b + i];
      },
      [&](int b, uint32_t sb, const uint32_t (&w)[8]) {
        uint4* dst = reinterpret_cast<uint4*>(q + (size_t)r * K + 32 * b);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        s[(size_t)r * (K / 32) + b] = (uint8_t)sb;
      });
}

// One warp per row: the quantiser alone (test support), logical outputs.
__global__ void debug_quant_kernel(const float* in, int rows, int K, uint8_t* q, uint8_t* s, float* G) {
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* row = in + (size_t)r * K;
  const float g = quant_row_nvfp4(
      K, [&](int b, float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = row[16 * b + i];
      },
      [&](int b, uint32_t sb, uint32_t w0, uint32_t w1) {
        *reinterpret_cast<uint2*>(q + (size_t)r * (K / 2) + 8 * b) = make_uint2(w0, w1);
        s[(size_t)r * (K / 16) + b] = (uint8_t)sb;
      });
  if ((threadIdx.x & 31) == 0) G[r] = g;
}

size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

struct PrefillCarve {
  size_t counts, block_base, expert_off, expert_poff, tile_expert, tile_rows, num_tiles, pos, row_src, xq, xsf, xG,
      hbuf, hq,
      hsf, hG, acc, xb, status, total;
  int n_route_blocks, max_tiles;
};

// Workspace carve of the band; the exact-numerics band appends x's BF16 copy
// per routed row after the common part (a workspace sized for it serves both).
PrefillCarve prefill_carve(int M, int E, int H, int I, int top_k, bool exact = false) {
  PrefillCarve c;
  const size_t n = (size_t)M * top_k;
  c.n_route_blocks = (int)((n + kRouteBlock - 1) / kRouteBlock);
  c.max_tiles = (int)((n + 127) / 128) + E;
  const int max_tiles_mid = (int)((n + kMidPad - 1) / kMidPad) + E;  // the mid band's 32-row tiles
  const size_t rows = (size_t)128 * c.max_tiles;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes);
    return at;
  };
  c.status = take(256);
  // the decode band's synchronisation words of the same shape sit right
  // after the status block in every workspace: this band leaves them alone
  // (they must stay zero for a decode call sharing the workspace)
  (void)take(decode_sync_bytes(H, I, top_k));
  c.counts = take(sizeof(int) * c.n_route_blocks * E);
  c.block_base = take(sizeof(int) * c.n_route_blocks * E);
  c.expert_off = take(sizeof(int) * (E + 1));
  c.expert_poff = take(sizeof(int) * (E + 1));
  c.tile_expert = take(sizeof(int) * max_tiles_mid);
  c.tile_rows = take(sizeof(int) * max_tiles_mid);
  c.num_tiles = take(sizeof(int));
  c.pos = take(sizeof(int) * n);
  c.row_src = take(sizeof(int) * rows);
  c.xq = take(rows * H / 2);
  c.xsf = take(rows * H / 16);
  c.xG = take(sizeof(float) * rows);
  c.hbuf = take(rows * I * 2);
  c.hq = take(rows * I / 2);
  c.hsf = take(rows * I / 16);
  c.hG = take(sizeof(float) * rows);
  c.acc = take(sizeof(float) * M * H);
  c.xb = exact ? take(rows * H * 2) : 0;
  c.total = o;
  return c;
}

PrefillArgs prefill_args(const PrefillCarve& c, void* ws, int M, int E, int H, int I, int top_k) {
  char* b = static_cast<char*>(ws);
  PrefillArgs a;
  a.x = nullptr;
  a.ids = nullptr;
  a.ids64 = 0;
  a.tw = nullptr;
  a.s13 = a.s2 = nullptr;
  a.out = nullptr;
  a.amode = 0;
  a.xq8 = a.xsf8 = a.hq8 = a.hsf8 = nullptr;
  a.M = M;
  a.E = E;
  a.H = H;
  a.I = I;
  a.top_k = top_k;
  a.n_entries = M * top_k;
  a.n_route_blocks = c.n_route_blocks;
  a.max_tiles = c.max_tiles;
  a.status = reinterpret_cast<uint32_t*>(b + c.status);
  a.counts = reinterpret_cast<int*>(b + c.counts);
  a.block_base = reinterpret_cast<int*>(b + c.block_base);
  a.expert_off = reinterpret_cast<int*>(b + c.expert_off);
  a.expert_poff = reinterpret_cast<int*>(b + c.expert_poff);
  a.tile_expert = reinterpret_cast<int*>(b + c.tile_expert);
  a.tile_rows = reinterpret_cast<int*>(b + c.tile_rows);
  a.num_tiles = reinterpret_cast<int*>(b + c.num_tiles);
  a.pos = reinterpret_cast<int*>(b + c.pos);
  a.row_src = reinterpret_cast<int*>(b + c.row_src);
  a.xq = reinterpret_cast<uint8_t*>(b + c.xq);
  a.xsf = reinterpret_cast<uint8_t*>(b + c.xsf);
  a.xG = reinterpret_cast<float*>(b + c.xG);
  a.hbuf = reinterpret_cast<__nv_bfloat16*>(b + c.hbuf);
  a.hq = reinterpret_cast<uint8_t*>(b + c.hq);
  a.hsf = reinterpret_cast<uint8_t*>(b + c.hsf);
  a.hG = reinterpret_cast<float*>(b + c.hG);
  a.acc = reinterpret_cast<float*>(b + c.acc);
  a.xb = c.xb ? reinterpret_cast<__half*>(b + c.xb) : nullptr;
  return a;
}

cudaError_t launch_route(PrefillArgs& a, cudaStream_t st, int pad = 128, bool stable = false) {
  if (!stable && a.n_entries <= kRouteSmallMax)
    return pad == 128 ? launch_pdl(route_small_kernel<128>, 1u, 1024u, 0, st, a)
                      : launch_pdl(route_small_kernel<kMidPad>, 1u, 1024u, 0, st, a);
  cudaError_t e = launch_pdl(route_count_kernel, (unsigned)a.n_route_blocks, kRouteBlock, sizeof(int) * a.E, st, a);
  if (e == cudaSuccess)
    e = pad == 128 ? launch_pdl(route_scan_kernel<128>, 1u, 1024u, 0, st, a)
                   : launch_pdl(route_scan_kernel<kMidPad>, 1u, 1024u, 0, st, a);
  if (e == cudaSuccess) e = launch_pdl(route_scatter_kernel, (unsigned)a.n_route_blocks, 32u, sizeof(int) * a.E, st, a);
  return e;
}

}  // namespace

// ---------------------------------------------------------------- host side
// Test support: the W4A8-MX engine (1 FP8 tensor cores where the shape
// allows, 0 the 16-bit engine); returns the previous choice.
int set_w4a8_fp8_engine(int on) {
  const int prev = g_w4a8_fp8;
  g_w4a8_fp8 = on ? 1 : 0;
  return prev;
}

size_t prefill_workspace_bytes(int M, int E, int H, int I, int top_k, bool exact) {
  return prefill_carve(M, E, H, I, top_k, exact).total;
}

// The exact-numerics band: route, x copied per routed row, FC1 and FC2 on the
// BF16 tensor cores with the weights decoded to BF16, the cast.
static cudaError_t launch_prefill_exact(PrefillArgs& a, const PrefillCarve& c, const void* w13, const void* w2,
                                        cudaStream_t st, int* cu_err) {
  const int E = a.E, H = a.H, I = a.I;
  const bool relu2 = a.act.kind == MOE_FP4_ACT_RELU2;
  const size_t rows = (size_t)128 * c.max_tiles;
  CUtensorMap mx, mw13, mh, mw2;
  auto raw_map = [](CUtensorMap* m, const void* base, uint64_t inner, uint64_t nrows, uint32_t box_rows) {
    const uint64_t d[2] = {inner, nrows};
    const uint64_t stride[1] = {inner};
    const uint32_t box[2] = {32, box_rows};  // 64 E2M1 elements per row and stage
    return make_u8_map(m, base, 2, d, stride, box, false);
  };
  // FC1 tile width: 256 (two resident 128-row tiles of gate/up pairs) for
  // gated experts when I % 128 == 0, else 128.  Measured on GB300 at E=128
  // H=4096 I=1536 M=4096 (exact BF16): 1791 us per layer against 2087 with
  // 128-wide tiles (A, the activations, staged half as often per FLOP).
  constexpr int kFc1Wide = 256;
  const int bn1 = (!relu2 && kFc1Wide == 256 && I % 128 == 0) ? 256 : 128;
  const int nt1 = relu2 ? (I + 127) / 128 : 2 * I / bn1, nt2 = H / kFc2ExactBN;
  CUresult r = make_fp4_map(&mx, a.xb, (uint64_t)H * 2, rows, kHwBM);
  if (r == CUDA_SUCCESS) r = raw_map(&mw13, w13, (uint64_t)H / 2, (uint64_t)E * (relu2 ? I : 2 * I), (uint32_t)bn1);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mh, a.hbuf, (uint64_t)I * 2, rows, kHwBM);
  if (r == CUDA_SUCCESS) r = raw_map(&mw2, w2, (uint64_t)I / 2, (uint64_t)E * H, kFc2ExactBN);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  static bool attrs = false;
  if (!attrs) {
    cudaError_t e = cudaSuccess;
    auto smem_attr = [&](const void* f, uint32_t bytes) {
      if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    };
    smem_attr((const void*)fc1_exact_kernel<128>, HwCfg<128>::kSmem);
    smem_attr((const void*)fc1_exact_kernel<256>, HwCfg<256>::kSmem);
    smem_attr((const void*)fc2_exact_kernel, HwCfg<kFc2ExactBN>::kSmem);
    if (e != cudaSuccess) return e;
    attrs = true;
  }
  cudaError_t e = launch_route(a, st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(stage_x_f16_kernel, (unsigned)a.M, 128u, 0, st, a);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = gemm_sms(&sms);
  if (e != cudaSuccess) return e;
  const int g1 = c.max_tiles * nt1, g2 = c.max_tiles * nt2;
  const int p1 = g1 < sms ? g1 : sms, p2 = g2 < sms ? g2 : sms;
  if (bn1 == 256)
    e = launch_pdl(fc1_exact_kernel<256>, (unsigned)p1, kHwThreads, HwCfg<256>::kSmem, st, mx, mw13, a);
  else
    e = launch_pdl(fc1_exact_kernel<128>, (unsigned)p1, kHwThreads, HwCfg<128>::kSmem, st, mx, mw13, a);
  if (e == cudaSuccess) e = launch_pdl(stage_h_f16_kernel, (unsigned)(rows / 8), 256u, 0, st, a);
  if (e == cudaSuccess)
    e = launch_pdl(fc2_exact_kernel, (unsigned)p2, kHwThreads, HwCfg<kFc2ExactBN>::kSmem, st, mh, mw2, a);
  if (e == cudaSuccess) e = launch_pdl(cast_out_kernel, 4u * 152u, 256u, 0, st, a);
  return e;
}

// The W4A8-MX band on the FP8 tensor cores: route, x to MXFP8 per routed row,
// FC1 (h quantised to MXFP8 in its epilogue), FC2, the cast.  The MXFP8 x and
// h with their scale chunks live in the 16-bit bands' x and h areas.
static cudaError_t launch_prefill_mx(PrefillArgs& a, const PrefillCarve& c, const void* w13, const void* w2,
                                     cudaStream_t st, int* cu_err) {
  const int E = a.E, H = a.H, I = a.I;
  const size_t rows = (size_t)128 * c.max_tiles;
  a.xq8 = reinterpret_cast<uint8_t*>(a.xb);
  a.xsf8 = a.xq8 + rows * H;
  a.hq8 = reinterpret_cast<uint8_t*>(a.hbuf);
  a.hsf8 = a.hq8 + rows * I;
  // FC1 tile width (128: two accumulators, the epilogue beside the next
  // tile's MMAs; 256: A staged half as often per FLOP, one accumulator)
  constexpr int bn1 = kMxFc1BN;
  CUtensorMap mx, mw13, mh, mw2;
  CUresult r = make_fp4_map(&mx, a.xq8, (uint64_t)H, rows, kMxBM);
  if (r == CUDA_SUCCESS) r = make_e2m1_unpacked_map(&mw13, w13, (uint64_t)H, (uint64_t)E * 2 * I, bn1);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mh, a.hq8, (uint64_t)I, rows, kMxBM);
  if (r == CUDA_SUCCESS) r = make_e2m1_unpacked_map(&mw2, w2, (uint64_t)I, (uint64_t)E * H, kMxFc2BN);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  static bool attrs = false;
  if (!attrs) {
    cudaError_t e =
        cudaFuncSetAttribute(fc1_mx_kernel<bn1>, cudaFuncAttributeMaxDynamicSharedMemorySize, MxCfg<bn1>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fc2_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MxCfg<kMxFc2BN>::kSmem);
    if (e != cudaSuccess) return e;
    attrs = true;
  }
  cudaError_t e = launch_route(a, st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(quant_x_mx_kernel, (unsigned)a.M, 128u, 0, st, a);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = gemm_sms(&sms);
  if (e != cudaSuccess) return e;
  const int g1 = c.max_tiles * (2 * I / bn1), g2 = c.max_tiles * (H / kMxFc2BN);
  e = launch_pdl(fc1_mx_kernel<bn1>, (unsigned)(g1 < sms ? g1 : sms), kMxThreads, MxCfg<bn1>::kSmem, st, mx, mw13, a);
  if (e == cudaSuccess)
    e = launch_pdl(fc2_mx_kernel, (unsigned)(g2 < sms ? g2 : sms), kMxThreads, MxCfg<kMxFc2BN>::kSmem, st, mh, mw2,
                   a);
  if (e == cudaSuccess) e = launch_pdl(cast_out_kernel, 4u * 152u, 256u, 0, st, a);
  return e;
}

// The mid band: route, x quantised per routed row, the swapped FC1, h
// quantised per routed row, the swapped FC2, the cast (same numerics as the
// prefill band).
static cudaError_t launch_prefill_mid(PrefillArgs& a, const PrefillCarve& c, const void* w13, const void* w2,
                                      cudaStream_t st, int* cu_err) {
  const int E = a.E, H = a.H, I = a.I;
  const bool relu2 = a.act.kind == MOE_FP4_ACT_RELU2;
  const size_t rows = (size_t)128 * c.max_tiles;
  CUtensorMap mw13, mw2;
  BMaps mx, mh;
  CUresult r = make_fp4_map(&mw13, w13, (uint64_t)H / 2, (uint64_t)E * (relu2 ? I : 2 * I), 128u);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mw2, w2, (uint64_t)I / 2, (uint64_t)E * H, 128u);
  for (int i = 0; i < 2 && r == CUDA_SUCCESS; ++i) {
    r = make_fp4_map(&mx.m[i], a.xq, (uint64_t)H / 2, rows, 16u << i);
    if (r == CUDA_SUCCESS) r = make_fp4_map(&mh.m[i], a.hq, (uint64_t)I / 2, rows, 16u << i);
  }
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  static bool attrs = false;
  if (!attrs) {
    cudaError_t e = cudaFuncSetAttribute(fc1_swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SwapCfg::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fc2_swap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SwapCfg::kSmem);
    if (e != cudaSuccess) return e;
    attrs = true;
  }
  cudaError_t e = launch_route(a, st, kMidPad);
  if (e == cudaSuccess)
    e = a.M <= kQuantXEntryMaxM ? launch_pdl(quant_x_entry_kernel, (unsigned)((a.n_entries + 7) / 8), 256u, 0, st, a)
                                : launch_pdl(quant_x_kernel, (unsigned)((a.M + 7) / 8), 256u, 0, st, a);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = gemm_sms(&sms);
  if (e != cudaSuccess) return e;
  // persistent, one CTA per SM; tiles: (32-row routing tile, group of up to
  // four weight tiles)
  // weight tiles per item: enough for about four 512-K stages between
  // accumulator hand-offs (FC2's K = I is often one stage)
  auto subs_for = [](int K) {
    const int nk = (K + SwapCfg::kStageK - 1) / SwapCfg::kStageK, sb = (4 + nk - 1) / nk;
    return sb < kSwapSubs ? sb : kSwapSubs;
  };
  const int s1 = subs_for(H) < kFc1SwapSubs ? subs_for(H) : kFc1SwapSubs, s2 = subs_for(I);
  const int n = a.n_entries, max_mid = (n + kMidPad - 1) / kMidPad + E;
  const int nt1 = relu2 ? (I + 127) / 128 : 2 * I / 128, nt2 = H / 128;
  const int g1 = max_mid * ((nt1 + s1 - 1) / s1), g2 = max_mid * ((nt2 + s2 - 1) / s2);
  e = launch_pdl(fc1_swap_kernel, (unsigned)(g1 < sms ? g1 : sms), kSwapThreads, SwapCfg::kSmem, st, mw13, mx, a,
                 s1);
  if (e == cudaSuccess)
    e = launch_pdl(quant_h_routed_kernel, (unsigned)((a.n_entries + 7) / 8), 256u, 0, st, a);
  if (e == cudaSuccess)
    e = launch_pdl(fc2_swap_kernel, (unsigned)(g2 < sms ? g2 : sms), kSwapThreads, SwapCfg::kSmem, st, mw2, mh, a,
                   s2);
  if (e == cudaSuccess) e = launch_pdl(cast_out_kernel, 4u * 152u, 256u, 0, st, a);
  return e;
}

cudaError_t launch_prefill(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                           const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                           int top_k, const ActParams& act, int band, bool mid, void* ws, cudaStream_t st,
                           int* cu_err) {
  const bool exact = band != MOE_FP4_PREFILL_NVFP4;  // the BF16-engine bands
  const PrefillCarve c = prefill_carve(M, E, H, I, top_k, exact);
  PrefillArgs a = prefill_args(c, ws, M, E, H, I, top_k);
  a.act = act;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ids = ids;
  a.ids64 = ids64;
  a.tw = tw;
  a.s13 = static_cast<const uint8_t*>(s13);
  a.s2 = static_cast<const uint8_t*>(s2);
  a.out = static_cast<__nv_bfloat16*>(out);
  if (exact) {
    // W4A8-MX on the FP8 tensor cores where w2's rows suit the unpacking
    // tensor map (I % 128 == 0), else on the 16-bit engine (same products)
    if (band == MOE_FP4_PREFILL_W4A8_MX && I % 128 == 0 && g_w4a8_fp8) return launch_prefill_mx(a, c, w13, w2, st, cu_err);
    a.amode = band == MOE_FP4_PREFILL_W4A8_MX ? 1 : 0;
    return launch_prefill_exact(a, c, w13, w2, st, cu_err);
  }
  const size_t rows = (size_t)128 * c.max_tiles;
  CUtensorMap mx, mw13, mh, mw2;
  CUresult r = make_fp4_map(&mx, a.xq, (uint64_t)H / 2, rows, kGemmBM);
  // FC1 tile width 128: two accumulators, so that a tile's epilogue (the
  // activation and the h store) overlaps the next tile's MMAs.  Measured on
  // GB300 at E=128 H=4096 I=1536 M=4096: 790.8 us per layer against 842.5
  // with 256-wide tiles (one accumulator: tensor memory also holds the ring's
  // scale factors).
  constexpr int bn1 = 128;
  const bool relu2 = act.kind == MOE_FP4_ACT_RELU2;  // non-gated experts: w1 of I rows
  if (r == CUDA_SUCCESS)
    r = make_fp4_map(&mw13, w13, (uint64_t)H / 2, (uint64_t)E * (relu2 ? I : 2 * I), (uint32_t)bn1);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mh, a.hq, (uint64_t)I / 2, rows, kGemmBM);
  if (r == CUDA_SUCCESS) r = make_fp4_map(&mw2, w2, (uint64_t)I / 2, (uint64_t)E * H, kFc2BN);
  if (r != CUDA_SUCCESS) {
    *cu_err = (int)r;
    return cudaErrorInvalidValue;
  }
  if (mid) return launch_prefill_mid(a, c, w13, w2, st, cu_err);
  static bool attrs = false;
  if (!attrs) {
    cudaError_t e =
        cudaFuncSetAttribute(fc1_gemm_kernel<bn1>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg<bn1>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fc2_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               GemmCfg<kFc2BN>::kSmem);
    if (e != cudaSuccess) return e;
    attrs = true;
  }
  cudaError_t e = launch_route(a, st);
  if (e != cudaSuccess) return e;
  e = M <= kQuantXEntryMaxM ? launch_pdl(quant_x_entry_kernel, (unsigned)((a.n_entries + 7) / 8), 256u, 0, st, a)
                            : launch_pdl(quant_x_kernel, (unsigned)((M + 7) / 8), 256u, 0, st, a);
  if (e != cudaSuccess) return e;
  int sms = 0;
  cudaError_t es = gemm_sms(&sms);
  if (es != cudaSuccess) return es;
  // persistent: one CTA per SM (the valid tile count is known on the device)
  const int g1 = c.max_tiles * (relu2 ? (I + 127) / 128 : 2 * I / bn1), g2 = c.max_tiles * (H / kFc2BN);
  e = launch_pdl(fc1_gemm_kernel<bn1>, (unsigned)(g1 < sms ? g1 : sms), kGemmThreads, GemmCfg<bn1>::kSmem, st, mx,
                 mw13, a);
  if (e == cudaSuccess) e = launch_pdl(quant_h_kernel, (unsigned)((rows + 7) / 8), 256u, 0, st, a);
  if (e == cudaSuccess)
    e = launch_pdl(fc2_gemm_kernel, (unsigned)(g2 < sms ? g2 : sms), kGemmThreads, GemmCfg<kFc2BN>::kSmem,
                   st, mh,
                   mw2, a);
  if (e == cudaSuccess) e = launch_pdl(cast_out_kernel, 4u * 152u, 256u, 0, st, a);
  return e;
}

size_t debug_route_workspace_bytes(int M, int E, int top_k) { return prefill_carve(M, E, 256, 256, top_k).total; }

cudaError_t launch_debug_route(const int32_t* ids, int M, int E, int top_k, int32_t* perm, int32_t* expert_offset,
                               void* ws, cudaStream_t st, bool small) {
  const PrefillCarve c = prefill_carve(M, E, 256, 256, top_k);
  PrefillArgs a = prefill_args(c, ws, M, E, 256, 256, top_k);
  a.ids = ids;
  if (small && a.n_entries > kRouteSmallMax) return cudaErrorInvalidValue;
  cudaError_t e = launch_route(a, st, 128, !small);
  if (e != cudaSuccess) return e;
  fill_i32_kernel<<<64, 256, 0, st>>>(perm, M * top_k, -1);
  route_perm_kernel<<<E, 256, 0, st>>>(a, perm);
  return cudaMemcpyAsync(expert_offset, a.expert_off, sizeof(int) * (E + 1), cudaMemcpyDeviceToDevice, st);
}

cudaError_t launch_debug_quant(const float* in, int rows, int K, uint8_t* q, uint8_t* s, float* G, cudaStream_t st) {
  debug_quant_kernel<<<(rows + 7) / 8, 256, 0, st>>>(in, rows, K, q, s, G);
  return cudaGetLastError();
}

cudaError_t launch_debug_quant_mxfp8(const float* in, int rows, int K, uint8_t* q, uint8_t* s, cudaStream_t st) {
  debug_quant_mxfp8_kernel<<<(rows + 7) / 8, 256, 0, st>>>(in, rows, K, q, s);
  return cudaGetLastError();
}

}  // namespace moe_fp4
