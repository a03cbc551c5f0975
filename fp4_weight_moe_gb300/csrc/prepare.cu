// One-time weight repack into the resident layout, its inverse, and the
// test-support dequantiser.
//
// The pages repack FP4 weights once at load time into an in-place layout that
// the decode kernel streams with fully coalesced 512 B warp runs (b12x PR
// #22, "rp-native tiny-decode kernel for w4a8_mx (M=1)", section What:
// "N256/K128 in-place-repacked storage", built by a logical->rp transform with
// a tested inverse mapping).  Our resident layout serves both bands on
// sm_103a:
//   - w13 rows interleave gate and up in groups of 64, so a 128-row tile
//     holds 64 matching (gate n, up n) pairs: the decode warp that owns rows
//     r, r+32, r+64, r+96 of a tile gets gate n and up n in lanes 16 apart,
//     and a prefill MMA tile of 128/256 rows carries whole pairs;
//   - rows stay K-contiguous (what a TMA box of the prefill GEMM reads);
//   - scale bytes are grouped in 512 B chunks (128 rows x 4 K-blocks), byte
//     (r%32)*16 + (r/32)*4 + b, the order of a 128-row scale tile in tensor
//     memory (lane r%32, column r/32, byte b);
//   - one E4M3 scale byte per 16 elements for BOTH formats.  An MXFP4 block
//     scale 2^(e-127) becomes, for each of its two 16-element halves, the
//     E4M3 power of two 2^(e-127-b) and the projection's FP32 multiplier
//     2^b, with b chosen so that the projection's largest block scale maps
//     to 2^8; E4M3 holds the powers of two 2^-9 .. 2^8 exactly, so every
//     block scale within 2^17 of the projection's largest is carried
//     exactly (smaller ones are stored as 0).  MXFP4 weights then run on the
//     same block-scaled kernels as NVFP4.
#include "common.cuh"

namespace moe_fp4 {

// w13: copy 16 B units, permuting rows (gate/up interleave).
__global__ void repack_w13_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int E, int I, int H,
                                  bool inverse) {
  const int units_per_row = H / 32;  // 16 B = 32 elements
  const size_t total = (size_t)E * 2 * I * units_per_row;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    size_t row_all = idx / units_per_row;
    int c = (int)(idx % units_per_row);
    int e = (int)(row_all / (2 * I)), R = (int)(row_all % (2 * I));
    int L = w13_logical_row(R, I);
    size_t res = ((size_t)e * 2 * I + R) * units_per_row + c;
    size_t log = ((size_t)e * 2 * I + L) * units_per_row + c;
    if (!inverse)
      out[res] = in[log];
    else
      out[log] = in[res];
  }
}

// E4M3 byte of 2^p for p in [-9, 8] (exact); 0 below.
__device__ __forceinline__ uint32_t e4m3_pow2(int p) {
  if (p >= -6) return (uint32_t)(p + 7) << 3;
  if (p >= -9) return 1u << (p + 9);
  return 0u;
}
// Exponent p of an E4M3 power of two written by e4m3_pow2 (byte != 0).
__device__ __forceinline__ int e4m3_pow2_exp(uint32_t b) {
  if (b >= 8u) return (int)(b >> 3) - 7;
  return b == 4u ? -7 : (b == 2u ? -8 : -9);
}

// Scales: logical [E][lrows][K/B] <-> resident chunks of E4M3 bytes per 16,
// `rows` (lrows rounded up to a multiple of 128) per expert; the resident
// bytes of rows past lrows are zero.  g [E][nproj]: the projection
// multipliers (MXFP4: 2^b, written before this kernel runs); nproj = 2 for
// w13 (rows < I gate, >= I up), 1 for w2 and w1.
__global__ void repack_scales_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, int E, int rows,
                                     int lrows, int K, int fmt, int I_for_w13, const float* __restrict__ g,
                                     bool inverse) {
  const int KB = K / block_size(fmt);    // logical blocks per row
  const int KBr = K / kResBlock;         // resident blocks per row
  const int KG = k_groups(K);
  const size_t per_expert = scale_chunk_bytes(rows, K);
  const size_t total = (size_t)E * per_expert;
  const bool mx = fmt == MOE_FP4_MXFP4;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(idx / per_expert);
    const size_t o = idx % per_expert;
    const int chunk = (int)(o / kChunkBytes), pos = (int)(o % kChunkBytes);
    const int rt = chunk / KG, kg = chunk % KG;
    const int r = (pos / 16) + 32 * ((pos % 16) / 4);
    const int kb = kg * 4 + pos % 4;  // resident 16-element block
    const int row = rt * kRowTile + r;
    const int lrow = I_for_w13 > 0 ? w13_logical_row(row, I_for_w13) : row;
    const int proj = I_for_w13 > 0 && lrow >= I_for_w13 ? 1 : 0;
    const int lkb = mx ? kb / 2 : kb;  // logical block
    const size_t li = ((size_t)e * lrows + lrow) * KB + lkb;
    if (kb >= KBr || row >= lrows) {
      if (!inverse) out[idx] = 0;
      continue;
    }
    if (!mx) {
      if (!inverse)
        out[idx] = in[li];
      else
        out[li] = in[idx];
      continue;
    }
    const int bias = (int)((__float_as_uint(g[e * (I_for_w13 > 0 ? 2 : 1) + proj]) >> 23) & 0xffu) - 127;
    if (!inverse) {
      const uint32_t eb = in[li];
      out[idx] = eb == 255u ? (uint8_t)0x7f : (uint8_t)e4m3_pow2((int)eb - 127 - bias);
    } else if ((kb & 1) == 0) {
      const uint32_t b = in[idx];
      // a block stored as 0 (more than 2^17 below the projection's largest)
      // comes back as the smallest scale, 2^-127
      out[li] = b == 0x7fu ? (uint8_t)255 : (b == 0u ? (uint8_t)0 : (uint8_t)(e4m3_pow2_exp(b) + 127 + bias));
    }
  }
}

// MXFP4: per (expert, projection) multiplier 2^b with b = (largest block
// scale exponent) - 8, clamped to the FP32 normal range, so that the largest
// block scale of the projection becomes the E4M3 power of two 2^8.  One CTA
// per (expert, projection); scale byte 255 (NaN) is ignored.
__global__ void mx_multiplier_kernel(const uint8_t* __restrict__ s_logical, int rows_per_proj, int KB, int nproj,
                                     float* __restrict__ g_out) {
  const int e = blockIdx.x / nproj, proj = blockIdx.x % nproj;
  const uint8_t* base = s_logical + ((size_t)e * nproj + proj) * rows_per_proj * KB;
  const size_t n = (size_t)rows_per_proj * KB;
  uint32_t mx = 0;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t b = base[i];
    if (b != 255u && b > mx) mx = b;
  }
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __shared__ uint32_t s_mx[32];
  if ((threadIdx.x & 31) == 0) s_mx[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) m = max(m, s_mx[w]);
    int k = (int)m - 127 - 8;
    if (k < -126) k = -126;
    g_out[blockIdx.x] = __int_as_float((k + 127) << 23);
  }
}

// Dequantise one expert's projection (logical row order) for tests:
// e2m1 * scale * g, as the kernels use them.  which: 0 w13, 1 w2, 2 w1
// (non-gated experts: I rows, scale rows padded to a multiple of 128).
__global__ void debug_dequant_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ s, int which, int e,
                                     int E, int H, int I, float* __restrict__ out) {
  const int rows = which == 0 ? 2 * I : (which == 1 ? H : I);
  const int K = which == 1 ? I : H;
  const int srows = which == 2 ? (I + kRowTile - 1) / kRowTile * kRowTile : rows;
  const int KG = k_groups(K);
  const uint8_t* wexp = w + (size_t)e * rows * (K / 2);
  const uint8_t* sexp = s + (size_t)e * scale_chunk_bytes(srows, K);
  const float* gl = reinterpret_cast<const float*>(s + (size_t)E * scale_chunk_bytes(srows, K));
  const size_t total = (size_t)rows * K;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    int L = (int)(idx / K), k = (int)(idx % K);
    int R = which == 0 ? w13_resident_row(L, I) : L;
    uint32_t byte = wexp[(size_t)R * (K / 2) + k / 2];
    uint32_t h[4];
    e2m1x8_to_half2x4(byte, h);
    float2 v = half2_bits_to_float2(h[0]);
    float q = (k & 1) ? v.y : v.x;
    float sc = e4m3_to_float(sexp[scale_offset(R, k / kResBlock, KG)]);
    float g = which == 0 ? gl[2 * e + (L >= I ? 1 : 0)] : gl[e];
    out[idx] = (q * sc) * g;  // q * sc exact (<= 2 + 4 significant bits); one rounding
  }
}

static int grid_for(size_t n, int threads) {
  size_t b = (n + threads - 1) / threads;
  if (b > 152 * 32) b = 152 * 32;
  if (b < 1) b = 1;
  return (int)b;
}

// w2 and its scales (shared by the gated and the non-gated layouts): the
// multipliers first (the MXFP4 scale conversion reads them), then the scale
// chunks and the nibbles (the logical layout).
static cudaError_t prepare_w2(const void* w2_l, const void* s2_l, const float* g2, int E, int H, int I, int fmt,
                              void* w2, void* s2, cudaStream_t st, bool inverse) {
  const size_t s2_bytes = (size_t)E * scale_chunk_bytes(H, I);
  float* s2g = reinterpret_cast<float*>(static_cast<uint8_t*>(s2) + s2_bytes);
  cudaError_t err = cudaSuccess;
  if (fmt == MOE_FP4_MXFP4 && !inverse) {
    mx_multiplier_kernel<<<E, 256, 0, st>>>(static_cast<const uint8_t*>(s2_l), H, I / 32, 1, s2g);
    err = cudaGetLastError();
  }
  if (fmt == MOE_FP4_NVFP4)
    err = inverse ? cudaMemcpyAsync(const_cast<float*>(g2), s2g, sizeof(float) * E, cudaMemcpyDeviceToDevice, st)
                  : cudaMemcpyAsync(s2g, g2, sizeof(float) * E, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return err;
  repack_scales_kernel<<<grid_for(s2_bytes, 256), 256, 0, st>>>(
      static_cast<const uint8_t*>(inverse ? s2 : s2_l), static_cast<uint8_t*>(inverse ? const_cast<void*>(s2_l) : s2),
      E, H, H, I, fmt, 0, s2g, inverse);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t w2_bytes = (size_t)E * H * (I / 2);
  return inverse ? cudaMemcpyAsync(const_cast<void*>(w2_l), w2, w2_bytes, cudaMemcpyDeviceToDevice, st)
                 : cudaMemcpyAsync(w2, w2_l, w2_bytes, cudaMemcpyDeviceToDevice, st);
}

cudaError_t launch_prepare(const void* w13_l, const void* s13_l, const float* g13, const void* w2_l,
                           const void* s2_l, const float* g2, int E, int H, int I, int fmt, void* w13, void* s13,
                           void* w2, void* s2, cudaStream_t st, bool inverse) {
  const size_t w13_units = (size_t)E * 2 * I * (H / 32);
  repack_w13_kernel<<<grid_for(w13_units, 256), 256, 0, st>>>(
      static_cast<const uint4*>(inverse ? w13 : w13_l), static_cast<uint4*>(inverse ? const_cast<void*>(w13_l) : w13),
      E, I, H, inverse);
  const size_t s13_bytes = (size_t)E * scale_chunk_bytes(2 * I, H);
  float* s13g = reinterpret_cast<float*>(static_cast<uint8_t*>(s13) + s13_bytes);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // the multipliers first: the MXFP4 scale conversion reads them
  if (fmt == MOE_FP4_MXFP4 && !inverse) {
    mx_multiplier_kernel<<<E * 2, 256, 0, st>>>(static_cast<const uint8_t*>(s13_l), I, H / 32, 2, s13g);
    err = cudaGetLastError();
  }
  if (fmt == MOE_FP4_NVFP4)
    err = inverse ? cudaMemcpyAsync(const_cast<float*>(g13), s13g, sizeof(float) * 2 * E, cudaMemcpyDeviceToDevice, st)
                  : cudaMemcpyAsync(s13g, g13, sizeof(float) * 2 * E, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return err;
  repack_scales_kernel<<<grid_for(s13_bytes, 256), 256, 0, st>>>(
      static_cast<const uint8_t*>(inverse ? s13 : s13_l),
      static_cast<uint8_t*>(inverse ? const_cast<void*>(s13_l) : s13), E, 2 * I, 2 * I, H, fmt, I, s13g, inverse);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return prepare_w2(w2_l, s2_l, g2, E, H, I, fmt, w2, s2, st, inverse);
}

// Non-gated experts (squared ReLU): w1 [E][I][H/2] kept in logical row order,
// its scales in chunks with each expert's rows padded to a multiple of 128,
// then the multipliers [E]; w2 as for the gated layout.
cudaError_t launch_prepare_relu2(const void* w1_l, const void* s1_l, const float* g1, const void* w2_l,
                                 const void* s2_l, const float* g2, int E, int H, int I, int fmt, void* w1, void* s1,
                                 void* w2, void* s2, cudaStream_t st, bool inverse) {
  const int rows = (I + kRowTile - 1) / kRowTile * kRowTile;
  const size_t s1_bytes = (size_t)E * scale_chunk_bytes(rows, H);
  float* s1g = reinterpret_cast<float*>(static_cast<uint8_t*>(s1) + s1_bytes);
  const size_t w1_bytes = (size_t)E * I * (H / 2);
  cudaError_t err = inverse ? cudaMemcpyAsync(const_cast<void*>(w1_l), w1, w1_bytes, cudaMemcpyDeviceToDevice, st)
                            : cudaMemcpyAsync(w1, w1_l, w1_bytes, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return err;
  if (fmt == MOE_FP4_MXFP4 && !inverse) {
    mx_multiplier_kernel<<<E, 256, 0, st>>>(static_cast<const uint8_t*>(s1_l), I, H / 32, 1, s1g);
    err = cudaGetLastError();
  }
  if (fmt == MOE_FP4_NVFP4)
    err = inverse ? cudaMemcpyAsync(const_cast<float*>(g1), s1g, sizeof(float) * E, cudaMemcpyDeviceToDevice, st)
                  : cudaMemcpyAsync(s1g, g1, sizeof(float) * E, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return err;
  repack_scales_kernel<<<grid_for(s1_bytes, 256), 256, 0, st>>>(
      static_cast<const uint8_t*>(inverse ? s1 : s1_l), static_cast<uint8_t*>(inverse ? const_cast<void*>(s1_l) : s1),
      E, rows, I, H, fmt, 0, s1g, inverse);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return prepare_w2(w2_l, s2_l, g2, E, H, I, fmt, w2, s2, st, inverse);
}

cudaError_t launch_debug_dequant(const void* w, const void* s, int which, int e, int E, int H, int I, int fmt,
                                 float* out, cudaStream_t st) {
  const size_t n = (size_t)(which == 0 ? 2 * I : (which == 1 ? H : I)) * (which == 1 ? I : H);
  (void)fmt;
  debug_dequant_kernel<<<grid_for(n, 256), 256, 0, st>>>(static_cast<const uint8_t*>(w),
                                                          static_cast<const uint8_t*>(s), which, e, E, H, I, out);
  return cudaGetLastError();
}

}  // namespace moe_fp4
