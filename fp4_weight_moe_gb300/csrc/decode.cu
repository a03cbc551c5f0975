// Decode band (M <= 8 tokens): host-side entry of the layer for both weight
// formats.  MXFP4 and NVFP4 weights share the resident layout (E4M3 scale
// bytes per 16 elements and FP32 projection multipliers, see prepare.cu), so
// both run the tcgen05 kernels of decode_tc.cu.
#include "common.cuh"

namespace moe_fp4 {

size_t decode_tc_scratch_bytes(int M, int H, int I, int top_k, int num_sms);
cudaError_t launch_decode_tc(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                             const int32_t* ids, const float* tw, void* out, int M, int E, int H, int I, int top_k,
                             float* scratch, uint32_t* status, int num_sms, cudaStream_t st, int* cu_err);

static size_t decode_scratch_bytes(int M_max, int H, int I, int top_k, int num_sms) {
  return (decode_tc_scratch_bytes(M_max, H, I, top_k, num_sms) + 255) & ~(size_t)255;
}

// Scratch (h, activation-term images), then a 256-byte status
// block (bit flags of bounded waits that gave up; sticky).
size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms) {
  (void)fmt;
  return decode_scratch_bytes(M_max, H, I, top_k, num_sms) + 256;
}

cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, const float* tw, void* out, int M, int E, int H, int I, int top_k,
                          int fmt, void* ws, int num_sms, cudaStream_t st) {
  (void)fmt;
  int cu = 0;
  uint32_t* status =
      reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + decode_scratch_bytes(M, H, I, top_k, num_sms));
  return launch_decode_tc(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, static_cast<float*>(ws), status,
                          num_sms, st, &cu);
}

}  // namespace moe_fp4
