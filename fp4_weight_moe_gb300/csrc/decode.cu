// Decode band (M <= 8 tokens): host-side entry of the layer for both weight
// formats.  MXFP4 and NVFP4 weights share the resident layout (E4M3 scale
// bytes per 16 elements and FP32 projection multipliers, see prepare.cu), so
// both run the same kernels.  Three kernel plans serve the band:
//   decode_gemv.cu  TMA-staged streaming GEMV on the CUDA cores, one pass
//                   over each routed expert's weights for all of its tokens
//                   (two launches);
//   decode_tc.cu    tcgen05 block-scaled MMA with the activations split into
//                   four NVFP4 terms, either as one launch whose CTAs hand h
//                   over through flags in global memory (shapes whose whole
//                   grid is resident at once) or as a chain of three or four
//                   launches.
// By default the shape decides (decode_family_of below).
#include <atomic>

#include "common.cuh"

namespace moe_fp4 {

// Which plan serves the band: 0 chooses by shape, 1 the streaming GEMV where
// it fits, 2 the tcgen05 launch chain, 3 the tcgen05 single launch where it
// fits.  Set only by moe_fp4_debug_set_decode_family (test support).
std::atomic<int> g_decode_family{0};

size_t decode_tc_scratch_bytes(int M, int H, int I, int top_k, int num_sms);
cudaError_t launch_decode_tc(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                             const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                             int top_k, const ActParams& act, float* scratch, uint32_t* status, int num_sms,
                             cudaStream_t st, int* cu_err);
size_t decode_sync_bytes(int H, int I, int top_k);
bool decode_fused_plan(int M, int H, int I, int top_k, int* C, int* s1, int* Q, int* cap);
cudaError_t launch_decode_fused(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                                const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                                int top_k, const ActParams& act, float* scratch, uint32_t* sync, uint32_t* status,
                                cudaStream_t st, int* cu_err);
bool decode_gemv_fits(int M, int E, int H, int I, int top_k);
size_t decode_gemv_scratch_bytes(int M, int I, int top_k);
cudaError_t launch_decode_gemv(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                               const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H,
                               int I, int top_k, const ActParams& act, float* scratch, uint32_t* status,
                               cudaStream_t st, int* cu_err);

static size_t decode_scratch_bytes(int M_max, int H, int I, int top_k, int num_sms) {
  const size_t tc = decode_tc_scratch_bytes(M_max, H, I, top_k, num_sms);
  const size_t gv = decode_gemv_scratch_bytes(M_max, I, top_k);
  return ((tc > gv ? tc : gv) + 255) & ~(size_t)255;
}

// The streaming GEMV wins where the layer is mostly fixed latency: one token
// and at most 4 MB of routed weights (measured on GB300: 5.2 vs 9.4 us at
// 0.1 MB, 7.4 vs 9.2 us at 1.8 MB, even at 7 MB, and the tcgen05 kernels
// ahead at every M >= 2).  Past that the CUDA cores' FP4 decode rate, not
// HBM, bounds it, while the tensor cores take FP4 operands directly.
static bool gemv_preferred(int M, int H, int I, int top_k) {
  const double expert = 3.0 * I * H / 2 + 3.0 * I * H / 16 + 12;
  return M == 1 && (double)M * top_k * expert <= 4.0 * (1 << 20);
}

// Workspace of the band: a 256-byte status block first (bit flags of bounded
// waits that gave up; sticky until cleared), then the single-launch kernel's
// synchronisation area (its size does not depend on the batch, so workspaces
// shared by batches of different sizes keep it in one place), then the
// scratch (the larger of the kernel families' intermediates).
constexpr size_t kStatusBytes = 256;

size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms) {
  (void)fmt;
  return kStatusBytes + decode_sync_bytes(H, I, top_k) + decode_scratch_bytes(M_max, H, I, top_k, num_sms);
}

// The plan the current setting picks for a decode-band shape: 1 streaming
// GEMV, 2 tcgen05 launch chain, 3 tcgen05 single launch.
int decode_family_of(int M, int E, int H, int I, int top_k) {
  const int family = g_decode_family.load(std::memory_order_relaxed);
  const bool fits = decode_gemv_fits(M, E, H, I, top_k);
  if (family == 1 ? fits : family == 0 && fits && gemv_preferred(M, H, I, top_k)) return 1;
  if (family != 3) return 2;
  int C, s1, Q;
  return decode_fused_plan(M, H, I, top_k, &C, &s1, &Q, nullptr) ? 3 : 2;
}

// Kernel launches of one decode-band layer under the current family setting.
int decode_launches(int M, int E, int H, int I, int top_k) {
  switch (decode_family_of(M, E, H, I, top_k)) {
    case 1: return 2;
    case 3: return 1;
    default: return M >= 2 ? 4 : 3;  // x pre-pass, FC1, (h pre-pass,) FC2
  }
}

cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                          int top_k, int fmt, const ActParams& act, void* ws, int num_sms, cudaStream_t st) {
  (void)fmt;
  int cu = 0;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  uint32_t* sync = reinterpret_cast<uint32_t*>(base + kStatusBytes);
  float* scratch = reinterpret_cast<float*>(base + kStatusBytes + decode_sync_bytes(H, I, top_k));
  // non-gated experts (squared ReLU) run on the tcgen05 launch chain only
  const int plan = act.kind == MOE_FP4_ACT_RELU2 ? 2 : decode_family_of(M, E, H, I, top_k);
  switch (plan) {
    case 1:
      return launch_decode_gemv(x, w13, s13, w2, s2, ids, ids64, tw, out, M, E, H, I, top_k, act, scratch, status, st,
                                &cu);
    case 3:
      return launch_decode_fused(x, w13, s13, w2, s2, ids, ids64, tw, out, M, E, H, I, top_k, act, scratch, sync,
                                 status, st, &cu);
    default:
      return launch_decode_tc(x, w13, s13, w2, s2, ids, ids64, tw, out, M, E, H, I, top_k, act, scratch, status,
                              num_sms, st, &cu);
  }
}

}  // namespace moe_fp4
