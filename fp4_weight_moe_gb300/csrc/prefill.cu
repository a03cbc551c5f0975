// Prefill band building blocks: the tcgen05 block-scaled FP4 GEMM and its
// test-support entry point.
#include "gemm_fp4.cuh"

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

// 2-D tensor map over a row-major byte matrix [rows][inner_bytes], box of
// box_rows x 128 bytes, 128-byte swizzle (the K-major SW128 operand layout).
CUresult make_fp4_map(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    debug_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                      const uint8_t* a_sf, const uint8_t* b_sf, float* d, int K, int N, uint32_t* err) {
  const int KG = K / 64;
  auto tile_of = [&]() {
    GemmTile t;
    t.a_row0 = blockIdx.x * kGemmBM;
    t.b_row0 = blockIdx.y * kGemmBN;
    t.a_sf = a_sf + (size_t)blockIdx.x * KG * kChunkBytes;
    t.b_sf0 = b_sf + (size_t)(2 * blockIdx.y) * KG * kChunkBytes;
    t.b_sf1 = t.b_sf0 + (size_t)KG * kChunkBytes;
    t.valid = true;
    return t;
  };
  auto epi = [&](int row, int col0, const float* v, const GemmTile& t) {
    float4* dst = reinterpret_cast<float4*>(d + (size_t)(t.a_row0 + row) * N + t.b_row0 + col0);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  };
  gemm_fp4_tile(&map_a, &map_b, K, err, tile_of, epi);
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
  dim3 grid(M_rows / kGemmBM, N_rows / kGemmBN);
  debug_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, st>>>(ma, mb, static_cast<const uint8_t*>(a_sf),
                                                           static_cast<const uint8_t*>(b_sf), d, K, N_rows, status);
  return cudaGetLastError();
}

}  // namespace moe_fp4
