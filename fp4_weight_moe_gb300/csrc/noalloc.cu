// moe_fp4_forward_noalloc: the decode-band layer for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at the point where they run the layer:
// code inside a stream capture (allocation is not a capturable operation),
// runtimes that hand out all device memory from their own fixed pool and
// forbid other allocations, or latency-critical paths where an allocation's
// implicit device synchronisation is not acceptable.  This entry point takes
// the same inputs and outputs as moe_fp4_forward, but its scratch memory is a
// fixed array of this library's device image instead of a workspace the
// caller allocates.
//
// The array lives in device memory on every GPU where the library's device
// code is loaded, from the first use until the process exits.  Host code may
// not use the array's name as a device address (in host code it names a
// host-side stand-in), so the first call on each device looks up the array's
// device address with cudaGetSymbolAddress while that device is current and
// caches it; make that first call before any stream capture.
//
// The array is laid out as the decode band's workspace: the 256-byte status
// block, the single-launch kernel's synchronisation words, then the
// intermediate.  The synchronisation words must be zero when a call starts:
// the array is zero when the library's device code is loaded, and every call
// that completes leaves them at zero again.
#include <mutex>

#include "common.cuh"

namespace moe_fp4 {
size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms);
cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                          int top_k, int fmt, const ActParams& act, void* ws, int num_sms, cudaStream_t st);
int check_layer_shape(int E, int H, int I, int top_k, int fmt);
}  // namespace moe_fp4

namespace {

// Scratch of moe_fp4_forward_noalloc, shared by all its calls on a device:
// the decode band's 256-byte status block and synchronisation words, and the
// intermediate (MOE_FP4_NOALLOC_SCRATCH_BYTES in all with the 256 bytes).
constexpr size_t kNoallocStatusBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_FP4_NOALLOC_SCRATCH_BYTES + kNoallocStatusBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device address of the scratch array and the SM count on the current
// device, looked up on the first call per device.
int scratch_for_current_device(void** ptr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return MOE_FP4_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_FP4_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_FP4_ECUDA;
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return MOE_FP4_ECUDA;
    g_scratch_ptr[dev] = p;
    g_sms[dev] = v;
  }
  *ptr = g_scratch_ptr[dev];
  *sms = g_sms[dev];
  return MOE_FP4_OK;
}

}  // namespace

extern "C" int moe_fp4_forward_noalloc(const void* x_bf16, const void* w13, const void* s13, const void* w2,
                                       const void* s2, const int32_t* topk_ids, const float* topk_weights,
                                       void* out_bf16, int M, int E, int H, int I, int top_k, int fmt,
                                       void* stream) {
  using namespace moe_fp4;
  const int shape = check_layer_shape(E, H, I, top_k, fmt);
  if (shape != MOE_FP4_OK) return shape;
  if (M < 0) return MOE_FP4_EINVAL;
  if (M == 0) return MOE_FP4_OK;
  if (M > MOE_FP4_DECODE_MAX_M) return MOE_FP4_EUNSUPPORTED;  // decode band only
  if (!x_bf16 || !w13 || !s13 || !w2 || !s2 || !topk_ids || !topk_weights || !out_bf16) return MOE_FP4_EINVAL;
  if (!aligned16(x_bf16) || !aligned16(w13) || !aligned16(w2) || !aligned16(s13) || !aligned16(s2))
    return MOE_FP4_EINVAL;
  void* scratch = nullptr;
  int sms = 0;
  int st = scratch_for_current_device(&scratch, &sms);
  if (st != MOE_FP4_OK) return st;
  if (decode_workspace_bytes(M, H, I, top_k, fmt, sms) > (size_t)MOE_FP4_NOALLOC_SCRATCH_BYTES + kNoallocStatusBytes)
    return MOE_FP4_EWORKSPACE;
  // The intermediate needs no clearing (each call writes every element it
  // reads); the synchronisation words are zero between calls (see above).
  const ActParams silu_act = {MOE_FP4_ACT_SILU, 0.f, 0.f, 0.f};
  cudaError_t e = launch_decode(x_bf16, w13, s13, w2, s2, topk_ids, 0, topk_weights, out_bf16, M, E, H, I, top_k, fmt,
                                silu_act, scratch, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_FP4_OK : MOE_FP4_ECUDA;
}

extern "C" int moe_fp4_noalloc_status(uint32_t* flags, int clear, void* stream) {
  if (!flags) return MOE_FP4_EINVAL;
  void* scratch = nullptr;
  int sms = 0;
  int st = scratch_for_current_device(&scratch, &sms);
  if (st != MOE_FP4_OK) return st;
  uint32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess && clear) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOE_FP4_ECUDA;
  *flags = v;
  return MOE_FP4_OK;
}
