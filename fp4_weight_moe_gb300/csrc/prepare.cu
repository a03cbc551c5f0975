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
//     (r%32)*16 + (r/32)*4 + b, the order in which tcgen05.cp copies 32x128b
//     scale-factor tiles into tensor memory; the decode warp's four rows r0,
//     r0+32, r0+64, r0+96 share one 16 B run of a chunk.
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

// Scales: logical [E][rows][K/B] <-> resident chunks.
__global__ void repack_scales_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ out, int E, int rows,
                                     int K, int fmt, int I_for_w13, bool inverse) {
  const int KB = K / block_size(fmt);
  const int KG = k_groups(K, fmt);
  const size_t per_expert = scale_chunk_bytes(rows, K, fmt);
  const size_t total = (size_t)E * per_expert;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    int e = (int)(idx / per_expert);
    size_t o = idx % per_expert;
    int chunk = (int)(o / kChunkBytes), pos = (int)(o % kChunkBytes);
    int rt = chunk / KG, kg = chunk % KG;
    int r = (pos / 16) + 32 * ((pos % 16) / 4);
    int kb = kg * 4 + pos % 4;
    int row = rt * kRowTile + r;
    int lrow = I_for_w13 > 0 ? w13_logical_row(row, I_for_w13) : row;
    size_t li = ((size_t)e * rows + lrow) * KB + kb;
    if (!inverse) {
      out[idx] = kb < KB ? in[li] : (uint8_t)0;
    } else if (kb < KB) {
      out[li] = in[idx];
    }
  }
}

// MXFP4: per (expert, projection) multiplier g = 2^(max scale exponent - 12),
// so the decode band can carry each block scale divided by g as an exact f16
// (2^-24 .. 2^12) and apply g after the K sum, like the NVFP4 multiplier.
// One CTA per (expert, projection); scale byte 255 (NaN) is ignored.
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
    int k = (int)m - 127 - 12;
    if (k < -126) k = -126;
    g_out[blockIdx.x] = __int_as_float((k + 127) << 23);
  }
}

// Dequantise one expert's projection (logical row order) for tests.
__global__ void debug_dequant_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ s, int which, int e,
                                     int E, int H, int I, int fmt, float* __restrict__ out) {
  const int rows = which == 0 ? 2 * I : H;
  const int K = which == 0 ? H : I;
  const int KG = k_groups(K, fmt);
  const int B = block_size(fmt);
  const uint8_t* wexp = w + (size_t)e * rows * (K / 2);
  const uint8_t* sexp = s + (size_t)e * scale_chunk_bytes(rows, K, fmt);
  const float* gl = reinterpret_cast<const float*>(s + (size_t)E * scale_chunk_bytes(rows, K, fmt));
  const size_t total = (size_t)rows * K;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    int L = (int)(idx / K), k = (int)(idx % K);
    int R = which == 0 ? w13_resident_row(L, I) : L;
    uint32_t byte = wexp[(size_t)R * (K / 2) + k / 2];
    uint32_t h[4];
    e2m1x8_to_half2x4(byte, h);
    float2 v = half2_bits_to_float2(h[0]);
    float q = (k & 1) ? v.y : v.x;
    float sc = scale_to_float(sexp[scale_offset(R, k / B, KG)], fmt);
    float val = q * sc;  // exact: <= 2 + 4 significant bits, in range
    if (fmt == MOE_FP4_NVFP4) {
      float g = which == 0 ? gl[2 * e + (L >= I ? 1 : 0)] : gl[e];
      val = val * g;
    }
    out[idx] = val;
  }
}

static int grid_for(size_t n, int threads) {
  size_t b = (n + threads - 1) / threads;
  if (b > 152 * 32) b = 152 * 32;
  if (b < 1) b = 1;
  return (int)b;
}

cudaError_t launch_prepare(const void* w13_l, const void* s13_l, const float* g13, const void* w2_l,
                           const void* s2_l, const float* g2, int E, int H, int I, int fmt, void* w13, void* s13,
                           void* w2, void* s2, cudaStream_t st, bool inverse) {
  const size_t w13_units = (size_t)E * 2 * I * (H / 32);
  repack_w13_kernel<<<grid_for(w13_units, 256), 256, 0, st>>>(
      static_cast<const uint4*>(inverse ? w13 : w13_l), static_cast<uint4*>(inverse ? const_cast<void*>(w13_l) : w13),
      E, I, H, inverse);
  const size_t s13_bytes = (size_t)E * scale_chunk_bytes(2 * I, H, fmt);
  const size_t s2_bytes = (size_t)E * scale_chunk_bytes(H, I, fmt);
  repack_scales_kernel<<<grid_for(s13_bytes, 256), 256, 0, st>>>(
      static_cast<const uint8_t*>(inverse ? s13 : s13_l),
      static_cast<uint8_t*>(inverse ? const_cast<void*>(s13_l) : s13), E, 2 * I, H, fmt, I, inverse);
  repack_scales_kernel<<<grid_for(s2_bytes, 256), 256, 0, st>>>(
      static_cast<const uint8_t*>(inverse ? s2 : s2_l), static_cast<uint8_t*>(inverse ? const_cast<void*>(s2_l) : s2),
      E, H, I, fmt, 0, inverse);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t w2_bytes = (size_t)E * H * (I / 2);
  if (!inverse)
    err = cudaMemcpyAsync(w2, w2_l, w2_bytes, cudaMemcpyDeviceToDevice, st);
  else
    err = cudaMemcpyAsync(const_cast<void*>(w2_l), w2, w2_bytes, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return err;
  if (fmt == MOE_FP4_MXFP4 && !inverse) {
    float* s13g = reinterpret_cast<float*>(static_cast<uint8_t*>(s13) + s13_bytes);
    float* s2g = reinterpret_cast<float*>(static_cast<uint8_t*>(s2) + s2_bytes);
    mx_multiplier_kernel<<<E * 2, 256, 0, st>>>(static_cast<const uint8_t*>(s13_l), I, H / 32, 2, s13g);
    mx_multiplier_kernel<<<E, 256, 0, st>>>(static_cast<const uint8_t*>(s2_l), H, I / 32, 1, s2g);
    err = cudaGetLastError();
  }
  if (fmt == MOE_FP4_NVFP4) {
    uint8_t* s13g = static_cast<uint8_t*>(s13) + s13_bytes;
    uint8_t* s2g = static_cast<uint8_t*>(s2) + s2_bytes;
    if (!inverse) {
      err = cudaMemcpyAsync(s13g, g13, sizeof(float) * 2 * E, cudaMemcpyDeviceToDevice, st);
      if (err == cudaSuccess) err = cudaMemcpyAsync(s2g, g2, sizeof(float) * E, cudaMemcpyDeviceToDevice, st);
    } else {
      err = cudaMemcpyAsync(const_cast<float*>(g13), s13g, sizeof(float) * 2 * E, cudaMemcpyDeviceToDevice, st);
      if (err == cudaSuccess)
        err = cudaMemcpyAsync(const_cast<float*>(g2), s2g, sizeof(float) * E, cudaMemcpyDeviceToDevice, st);
    }
  }
  return err;
}

cudaError_t launch_debug_dequant(const void* w, const void* s, int which, int e, int E, int H, int I, int fmt,
                                 float* out, cudaStream_t st) {
  const size_t n = (size_t)(which == 0 ? 2 * I : H) * (which == 0 ? H : I);
  debug_dequant_kernel<<<grid_for(n, 256), 256, 0, st>>>(static_cast<const uint8_t*>(w),
                                                          static_cast<const uint8_t*>(s), which, e, E, H, I, fmt, out);
  return cudaGetLastError();
}

}  // namespace moe_fp4
