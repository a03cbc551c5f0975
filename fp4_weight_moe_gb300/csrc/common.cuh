// Shared device helpers of libmoe_fp4: resident-layout index math, E2M1 /
// scale decode, and the inline PTX the kernels use (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_fp4.h"

namespace moe_fp4 {

constexpr int kRowTile = 128;     // rows per resident tile (scale chunk height)
constexpr int kChunkBytes = 512;  // one scale chunk: 128 rows x 4 K-blocks
constexpr int kInterleave = 64;   // gate/up interleave granularity in w13

// Scale block of the LOGICAL (checkpoint) layout: 32 elements for MXFP4
// (UE8M0 bytes), 16 for NVFP4 (E4M3 bytes).
__host__ __device__ constexpr int block_size(int fmt) { return fmt == MOE_FP4_MXFP4 ? 32 : 16; }
__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// The RESIDENT layout has one E4M3 scale byte per 16 elements for both
// formats (MXFP4 block scales are re-expressed at prepare time, see
// prepare.cu), so both run on the same block-scaled MMA.
constexpr int kResBlock = 16;

// Number of 4-block groups along K (resident).
__host__ __device__ inline int k_groups(int K) { return ceil_div(K / kResBlock, 4); }

// Bytes of one expert-projection's scale chunks (rows x K), resident.
__host__ __device__ inline size_t scale_chunk_bytes(int rows, int K) {
  return (size_t)(rows / kRowTile) * k_groups(K) * kChunkBytes;
}

// Offset of (row, kblock) inside one expert-projection's chunk array.
__host__ __device__ inline size_t scale_offset(int row, int kb, int KG) {
  int rt = row / kRowTile, r = row % kRowTile;
  return ((size_t)rt * KG + kb / 4) * kChunkBytes + (r % 32) * 16 + (r / 32) * 4 + (kb % 4);
}

// Resident w13 row -> logical row (gate rows 0..I-1, up rows I..2I-1).
__host__ __device__ inline int w13_logical_row(int R, int I) {
  int j = R / (2 * kInterleave), r = R % (2 * kInterleave);
  return r < kInterleave ? j * kInterleave + r : I + j * kInterleave + (r - kInterleave);
}
// Logical w13 row -> resident row.
__host__ __device__ inline int w13_resident_row(int L, int I) {
  bool up = L >= I;
  int n = up ? L - I : L;
  return (n / kInterleave) * (2 * kInterleave) + (up ? kInterleave : 0) + n % kInterleave;
}

// ---------------------------------------------------------------- decode helpers
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// Eight E2M1 values (a 32-bit word, element 2i in the low nibble of byte i)
// -> four half2 {element 2i, element 2i+1}; exact (hardware cvt).
__device__ __forceinline__ void e2m1x8_to_half2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Streaming 16-byte load that bypasses L1 (weights are read exactly once).
__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Routing id j of the caller's top-k ids: int32 as stored, or int64 (wide)
// narrowed to int32 with every value outside [0, E) mapped to -1, so that the
// narrowing never turns an invalid id into a valid one.  The ids are inputs
// of the call and stay unchanged during it (non-coherent loads).
__device__ __forceinline__ int route_id(const int32_t* ids, int j, int wide, int E) {
  if (wide) {
    long long v;
    asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(v) : "l"(reinterpret_cast<const long long*>(ids) + j));
    return v >= 0 && v < (long long)E ? (int)v : -1;
  }
  int r;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(r) : "l"(ids + j));
  return r;
}

// L2 policy: lines loaded with it are the first candidates for eviction.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Streaming 16-byte load, no L1 allocation, L2 evict-first.
__device__ __forceinline__ uint4 ld_stream_16_ef(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Bring [p, p + bytes) into L2 without a destination (bytes % 16 == 0).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// d = a * b + c on two FP32 lanes at once.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\t"
      "mov.b64 rc, {%6,%7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0,%1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and (in that kernel) wait until this grid's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float silu(float v) { return v / (1.0f + __expf(-v)); }

// The gated activation of FC1's (gate, up) pair (MOE_FP4_ACT_*): SiLU(gate) *
// up; GELU in its tanh form; SwiGLU-OAI with gate' = min(gate, limit), up' =
// clamp(up, -limit, limit), (up' + beta) * gate' * sigmoid(alpha * gate').
struct ActParams {
  int kind;
  float alpha, beta, limit;
};

__device__ __forceinline__ float gated_act(float gate, float up, const ActParams& p) {
  if (p.kind == MOE_FP4_ACT_GELU_TANH) {
    const float c = 0.7978845608028654f;  // sqrt(2 / pi)
    return 0.5f * gate * (1.0f + tanhf(c * fmaf(0.044715f * gate, gate * gate, gate))) * up;
  }
  if (p.kind == MOE_FP4_ACT_SWIGLUOAI) {
    const float g = fminf(gate, p.limit);
    const float u = fminf(fmaxf(up, -p.limit), p.limit);
    return (u + p.beta) * g / (1.0f + __expf(-p.alpha * g));
  }
  return silu(gate) * up;
}

}  // namespace moe_fp4
