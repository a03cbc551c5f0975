// extern "C" entry points of libmoe_fp4.so: argument validation, workspace
// management and band dispatch.  The declarations and the contract of each
// function are in include/moe_fp4.h.
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace moe_fp4 {
cudaError_t launch_prepare(const void* w13_l, const void* s13_l, const float* g13, const void* w2_l,
                           const void* s2_l, const float* g2, int E, int H, int I, int fmt, void* w13, void* s13,
                           void* w2, void* s2, cudaStream_t st, bool inverse);
cudaError_t launch_debug_dequant(const void* w, const void* s, int which, int e, int E, int H, int I, int fmt,
                                 float* out, cudaStream_t st);
cudaError_t launch_prepare_relu2(const void* w1_l, const void* s1_l, const float* g1, const void* w2_l,
                                 const void* s2_l, const float* g2, int E, int H, int I, int fmt, void* w1, void* s1,
                                 void* w2, void* s2, cudaStream_t st, bool inverse);
size_t decode_workspace_bytes(int M_max, int H, int I, int top_k, int fmt, int num_sms);
size_t decode_sync_bytes(int H, int I, int top_k);
cudaError_t launch_debug_gemm(const void* a_q, const void* a_sf, const void* b_q, const void* b_sf, float* d,
                              int M_rows, int N_rows, int K, uint32_t* status, cudaStream_t st, int* cu_err);
size_t prefill_workspace_bytes(int M, int E, int H, int I, int top_k, bool exact);
int set_w4a8_fp8_engine(int on);
size_t debug_route_workspace_bytes(int M, int E, int top_k);
cudaError_t launch_prefill(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                           const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                           int top_k, const ActParams& act, int band, bool mid, void* ws, cudaStream_t st,
                           int* cu_err);
cudaError_t launch_debug_route(const int32_t* ids, int M, int E, int top_k, int32_t* perm, int32_t* expert_offset,
                               void* ws, cudaStream_t st, bool small);
cudaError_t launch_debug_quant(const float* in, int rows, int K, uint8_t* q, uint8_t* s, float* G, cudaStream_t st);
cudaError_t launch_debug_quant_mxfp8(const float* in, int rows, int K, uint8_t* q, uint8_t* s, cudaStream_t st);
extern std::atomic<int> g_decode_family;
bool decode_gemv_fits(int M, int E, int H, int I, int top_k);
int decode_launches(int M, int E, int H, int I, int top_k);
int decode_family_of(int M, int E, int H, int I, int top_k);
bool decode_fused_plan(int M, int H, int I, int top_k, int* C, int* s1, int* Q, int* cap);
cudaError_t launch_decode(const void* x, const void* w13, const void* s13, const void* w2, const void* s2,
                          const int32_t* ids, int ids64, const float* tw, void* out, int M, int E, int H, int I,
                          int top_k, int fmt, const ActParams& act, void* ws, int num_sms, cudaStream_t st);
}  // namespace moe_fp4

using namespace moe_fp4;

namespace {
// Test support: one thread waits on an mbarrier that nothing arrives on,
// polling it `polls` times, so that the bounded wait gives up and records
// MOE_FP4_STATUS_TEST_WAIT in the status word.
__global__ void wait_timeout_kernel(uint32_t* status, uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  (void)mbar_wait_for(&bar, 0, status, MOE_FP4_STATUS_TEST_WAIT, polls);
}

// Copy the status word at `word` (device) to *flags and, if asked, clear it;
// the stream is synchronised.
int read_status_word(void* word, uint32_t* flags, int clear, cudaStream_t st);
}  // namespace

namespace moe_fp4 {
// Shape limits shared by every entry point that runs the layer: a known
// format, positive sizes, E <= 65536, top_k <= 16, H % 256 == 0, I % 64 == 0,
// and one expert projection's elements (2I x H) within 2^31, so that the
// kernels' 32-bit element offsets cannot overflow.
int check_layer_shape(int E, int H, int I, int top_k, int fmt) {
  if (fmt != MOE_FP4_MXFP4 && fmt != MOE_FP4_NVFP4) return MOE_FP4_EINVAL;
  if (E <= 0 || H <= 0 || I <= 0 || top_k <= 0) return MOE_FP4_EINVAL;
  if (E > 65536 || top_k > 16) return MOE_FP4_EUNSUPPORTED;
  if (H % 256 != 0 || I % 64 != 0) return MOE_FP4_EUNSUPPORTED;
  if ((long long)H * 2 * I > (1LL << 31)) return MOE_FP4_EUNSUPPORTED;
  return MOE_FP4_OK;
}
}  // namespace moe_fp4

namespace {

thread_local int g_last_cuda_error = 0;
constexpr size_t kMaxWorkspace = (size_t)1 << 31;  // workspaces past 2^31 bytes are rejected

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return MOE_FP4_ECUDA;
}

int device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *sms = cache[dev];
    return MOE_FP4_OK;
  }
  int v = 0;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev >= 0 && dev < 64) cache[dev] = v;
  *sms = v;
  return MOE_FP4_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int read_status_word(void* word, uint32_t* flags, int clear, cudaStream_t st) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(word, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess && clear) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e);
  *flags = v;
  return MOE_FP4_OK;
}

int check_shape(int E, int H, int I, int top_k, int fmt) { return check_layer_shape(E, H, I, top_k, fmt); }

// Extra limits of the prefill band (M > MOE_FP4_DECODE_MAX_M).
int check_prefill(int M, int E, int I, int top_k, int fmt) {
  (void)fmt;  // both formats share the resident layout and the kernels
  if (E > 4096) return MOE_FP4_EUNSUPPORTED;
  if ((long long)M * top_k >= (1LL << 30)) return MOE_FP4_EUNSUPPORTED;
  return MOE_FP4_OK;
}

// Scratch for every batch size up to M (a workspace reserved for M_max serves
// all smaller batches).
size_t workspace_need(int M, int E, int H, int I, int top_k, int fmt, int sms, bool exact = false) {
  size_t d = 0;
  for (int m = 1; m <= M && m <= MOE_FP4_DECODE_MAX_M; ++m) {
    const size_t b = decode_workspace_bytes(m, H, I, top_k, fmt, sms);
    if (b > d) d = b;
  }
  if (M > MOE_FP4_DECODE_MAX_M) {
    const size_t p = prefill_workspace_bytes(M, E, H, I, top_k, exact);
    if (p > d) d = p;
  }
  return d;
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Host-buffer staging area of moe_fp4_forward_host: x, ids, router weights and
// the output, each 256-byte aligned, placed right after the layer's own
// workspace for M tokens.
struct HostStage {
  size_t x, ids, tw, out, total;
};
HostStage host_stage(int M, int H, int top_k) {
  HostStage h;
  h.x = 0;
  h.ids = h.x + align256((size_t)M * H * 2);
  h.tw = h.ids + align256((size_t)M * top_k * 4);
  h.out = h.tw + align256((size_t)M * top_k * 4);
  h.total = h.out + align256((size_t)M * H * 2);
  return h;
}

// The address under which the current device reaches `p`, or null if it
// cannot (pageable host memory, another device's memory) or `p` is not
// 16-byte aligned.  Page-locked host memory is mapped for every device on a
// unified-address system, so its device view is usable by the kernels.
void* device_view(const void* p) {
  if (!aligned16(p)) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  if (a.type == cudaMemoryTypeDevice && a.device == dev) return a.devicePointer;
  return nullptr;
}

struct LibWorkspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::mutex g_ws_mutex;
LibWorkspace g_ws[64];

}  // namespace

extern "C" {

const char* moe_fp4_status_string(int status) {
  switch (status) {
    case MOE_FP4_OK: return "ok";
    case MOE_FP4_EINVAL: return "invalid argument";
    case MOE_FP4_EUNSUPPORTED: return "unsupported shape";
    case MOE_FP4_ECUDA: return "CUDA error";
    case MOE_FP4_EWORKSPACE: return "workspace missing, too small or too large";
    default: return "unknown status";
  }
}

int moe_fp4_last_cuda_error(void) { return g_last_cuda_error; }

int moe_fp4_version(void) { return 100; }

int moe_fp4_prepared_sizes(int E, int H, int I, int fmt, size_t* w13_bytes, size_t* s13_bytes, size_t* w2_bytes,
                           size_t* s2_bytes) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  const size_t g13 = sizeof(float) * 2 * (size_t)E;
  const size_t g2 = sizeof(float) * (size_t)E;
  auto pad16 = [](size_t v) { return (v + 15) & ~(size_t)15; };
  if (w13_bytes) *w13_bytes = (size_t)E * 2 * I * (H / 2);
  if (s13_bytes) *s13_bytes = pad16((size_t)E * scale_chunk_bytes(2 * I, H) + g13);
  if (w2_bytes) *w2_bytes = (size_t)E * H * (I / 2);
  if (s2_bytes) *s2_bytes = pad16((size_t)E * scale_chunk_bytes(H, I) + g2);
  return MOE_FP4_OK;
}

int moe_fp4_prepared_sizes_relu2(int E, int H, int I, int fmt, size_t* w1_bytes, size_t* s1_bytes, size_t* w2_bytes,
                                 size_t* s2_bytes) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  auto pad16 = [](size_t v) { return (v + 15) & ~(size_t)15; };
  const int rows1 = (I + kRowTile - 1) / kRowTile * kRowTile;
  if (w1_bytes) *w1_bytes = (size_t)E * I * (H / 2);
  if (s1_bytes) *s1_bytes = pad16((size_t)E * scale_chunk_bytes(rows1, H) + sizeof(float) * (size_t)E);
  if (w2_bytes) *w2_bytes = (size_t)E * H * (I / 2);
  if (s2_bytes) *s2_bytes = pad16((size_t)E * scale_chunk_bytes(H, I) + sizeof(float) * (size_t)E);
  return MOE_FP4_OK;
}

int moe_fp4_prepare_weights_relu2(const void* w1_logical, const void* s1_logical, const float* g1,
                                  const void* w2_logical, const void* s2_logical, const float* g2, int E, int H, int I,
                                  int fmt, void* w1, void* s1, void* w2, void* s2, void* stream) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  if (!w1_logical || !s1_logical || !w2_logical || !s2_logical || !w1 || !s1 || !w2 || !s2) return MOE_FP4_EINVAL;
  if (fmt == MOE_FP4_NVFP4 && (!g1 || !g2)) return MOE_FP4_EINVAL;
  if (!aligned16(w1) || !aligned16(s1) || !aligned16(w2) || !aligned16(s2)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_prepare_relu2(w1_logical, s1_logical, g1, w2_logical, s2_logical, g2, E, H, I, fmt, w1, s1,
                                       w2, s2, static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_unprepare_weights_relu2(const void* w1, const void* s1, const void* w2, const void* s2, int E, int H,
                                    int I, int fmt, void* w1_logical, void* s1_logical, float* g1, void* w2_logical,
                                    void* s2_logical, float* g2, void* stream) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  if (!w1_logical || !s1_logical || !w2_logical || !s2_logical || !w1 || !s1 || !w2 || !s2) return MOE_FP4_EINVAL;
  if (fmt == MOE_FP4_NVFP4 && (!g1 || !g2)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_prepare_relu2(w1_logical, s1_logical, g1, w2_logical, s2_logical, g2, E, H, I, fmt,
                                       const_cast<void*>(w1), const_cast<void*>(s1), const_cast<void*>(w2),
                                       const_cast<void*>(s2), static_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_prepare_weights(const void* w13_logical, const void* s13_logical, const float* g13,
                            const void* w2_logical, const void* s2_logical, const float* g2, int E, int H, int I,
                            int fmt, void* w13, void* s13, void* w2, void* s2, void* stream) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  if (!w13_logical || !s13_logical || !w2_logical || !s2_logical || !w13 || !s13 || !w2 || !s2)
    return MOE_FP4_EINVAL;
  if (fmt == MOE_FP4_NVFP4 && (!g13 || !g2)) return MOE_FP4_EINVAL;
  if (!aligned16(w13_logical) || !aligned16(w13) || !aligned16(s13) || !aligned16(s2)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_prepare(w13_logical, s13_logical, g13, w2_logical, s2_logical, g2, E, H, I, fmt, w13, s13,
                                 w2, s2, static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_unprepare_weights(const void* w13, const void* s13, const void* w2, const void* s2, int E, int H, int I,
                              int fmt, void* w13_logical, void* s13_logical, float* g13, void* w2_logical,
                              void* s2_logical, float* g2, void* stream) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  if (!w13_logical || !s13_logical || !w2_logical || !s2_logical || !w13 || !s13 || !w2 || !s2)
    return MOE_FP4_EINVAL;
  if (fmt == MOE_FP4_NVFP4 && (!g13 || !g2)) return MOE_FP4_EINVAL;
  if (!aligned16(w13_logical) || !aligned16(w13)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_prepare(w13_logical, s13_logical, g13, w2_logical, s2_logical, g2, E, H, I, fmt,
                                 const_cast<void*>(w13), const_cast<void*>(s13), const_cast<void*>(w2),
                                 const_cast<void*>(s2), static_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

size_t moe_fp4_workspace_zero_bytes(int E, int H, int I, int top_k, int fmt) {
  if (check_shape(E, H, I, top_k, fmt) != MOE_FP4_OK) return 0;
  return 256 + decode_sync_bytes(H, I, top_k);
}

size_t moe_fp4_workspace_bytes(int M_max, int E, int H, int I, int top_k, int fmt) {
  if (M_max < 0 || check_shape(E, H, I, top_k, fmt) != MOE_FP4_OK) return 0;
  if (M_max > MOE_FP4_DECODE_MAX_M && check_prefill(M_max, E, I, top_k, fmt) != MOE_FP4_OK) return 0;
  int sms = 0;
  if (device_sms(&sms) != MOE_FP4_OK) return 0;
  return workspace_need(M_max < 1 ? 1 : M_max, E, H, I, top_k, fmt, sms);
}

int moe_fp4_reserve_workspace(int M_max, int E, int H, int I, int top_k, int fmt, void* stream) {
  size_t need = moe_fp4_workspace_bytes(M_max, E, H, I, top_k, fmt);
  if (need == 0) return check_shape(E, H, I, top_k, fmt) != MOE_FP4_OK ? check_shape(E, H, I, top_k, fmt)
                                                                        : MOE_FP4_EUNSUPPORTED;
  if (need >= kMaxWorkspace) return MOE_FP4_EWORKSPACE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= 64) return MOE_FP4_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_ws_mutex);
  LibWorkspace& w = g_ws[dev];
  if (w.bytes >= need) return MOE_FP4_OK;
  if (w.ptr) {
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e);
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
  }
  void* p = nullptr;
  e = cudaMalloc(&p, need);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaMemsetAsync(p, 0, need, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaFree(p);
    return fail_cuda(e);
  }
  w.ptr = p;
  w.bytes = need;
  return MOE_FP4_OK;
}

int moe_fp4_release_workspace(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= 64) return MOE_FP4_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_ws_mutex);
  LibWorkspace& w = g_ws[dev];
  if (w.ptr) {
    e = cudaDeviceSynchronize();
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return MOE_FP4_OK;
}

namespace {
// Batches past the decode band: 0 by shape, 1 the prefill band's GEMMs, 2 the
// decode kernels in chunks, 3 the mid band's swapped GEMMs (test support:
// moe_fp4_debug_set_mid_band).
std::atomic<int> g_mid_band{0};
constexpr int kMidBandMaxM = 3 * MOE_FP4_DECODE_MAX_M;

// Does a batch of M > MOE_FP4_DECODE_MAX_M tokens run as decode-band chunks?
// Only when forced (mode 2), for up to kMidBandMaxM tokens.  Chunks stream an
// expert once per chunk that routes to it instead of once per layer, but skip
// the routing, quantisation and cast launches, and keep the decode band's
// BF16-activation numerics.  They led the mid band for up to 12 tokens with
// small experts until the mid band's first-tile latency came down; measured
// on GB300 since (us per layer, chunks / mid band): E=512 H=2560 I=320 k=10:
// M=9 47.7 / 43.6, 12 55.3 / 50.8; E=288 H=4096 I=512 k=10: M=9 80.6 / 69.7,
// 12 99.8 / 80.2; E=8 H=256 I=128 k=2: M=9 21.3 / 20.1, 12 22.5 / 20.3.
bool mid_band_chunks(int M) {
  return M <= kMidBandMaxM && g_mid_band.load(std::memory_order_relaxed) == 2;
}

// Does a batch past the decode band (and not in chunks) run on the mid band's
// swapped GEMMs rather than the prefill band's?  By shape: while the experts
// average at most kMidBandMaxRows routed rows, where the prefill tiles would
// stage mostly padding rows of activations.  Measured on GB300 (us per layer,
// prefill / mid band, routed rows per expert in brackets): E=512 H=2560 I=320
// k=10: M=64 (1.25) 196.9 / 107.7, 1024 (20) 334.1 / 210.8, 1536 (30) 352.9 /
// 290.3, 1792 (35) 351.8 / 338.9, 2048 (40) 357.0 / 377.5; E=288 H=4096 I=512
// k=10: M=768 (26.7) 344.8 / 264.0, 1024 (35.6) 347.3 / 357.0; E=256 H=7168
// I=2048 k=8: M=832 (26) 1091.1 / 1065.7, 1024 (32) 1108.9 / 1241.5; E=128
// H=4096 I=1536 k=8: M=416 (26) 283.1 / 261.5, 512 (32) 287.1 / 301.2.
// With I <= 384 the prefill band's FC2 has one or two K stages per tile and
// the mid band stays ahead further (the E=512 rows above): up to
// kMidBandMaxRowsShortI rows there.
constexpr int kMidBandMaxRows = 28;
constexpr int kMidBandMaxRowsShortI = 36;
bool mid_band_swap(int M, int E, int I, int top_k) {
  const int mode = g_mid_band.load(std::memory_order_relaxed);
  if (mode == 1 || mode == 3) return mode == 3;
  const int rows = I <= 384 ? kMidBandMaxRowsShortI : kMidBandMaxRows;
  return (int64_t)M * top_k <= (int64_t)rows * E;  // (mode 2: past the chunks' reach)
}

// moe_fp4_forward_ex and moe_fp4_forward_ex_i64: topk_ids int32 (ids64 = 0)
// or int64 (ids64 = 1)
int forward_any_ids(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                    const void* topk_ids, int ids64, const float* topk_weights, void* out_bf16, int M, int E, int H,
                    int I, int top_k, int fmt, const moe_fp4_activation* act, void* workspace, size_t workspace_bytes,
                    void* stream, int prefill_mode = MOE_FP4_PREFILL_NVFP4) {
  if (prefill_mode != MOE_FP4_PREFILL_NVFP4 && prefill_mode != MOE_FP4_PREFILL_BF16 &&
      prefill_mode != MOE_FP4_PREFILL_W4A8_MX)
    return MOE_FP4_EINVAL;
  const bool exact = prefill_mode != MOE_FP4_PREFILL_NVFP4;  // the BF16-engine bands
  const int32_t* ids = static_cast<const int32_t*>(topk_ids);
  ActParams ap = {MOE_FP4_ACT_SILU, 0.f, 0.f, 0.f};
  if (act) {
    if (act->kind != MOE_FP4_ACT_SILU && act->kind != MOE_FP4_ACT_GELU_TANH && act->kind != MOE_FP4_ACT_SWIGLUOAI &&
        act->kind != MOE_FP4_ACT_RELU2)
      return MOE_FP4_EINVAL;
    if (act->kind == MOE_FP4_ACT_SWIGLUOAI &&
        (!std::isfinite(act->alpha) || !std::isfinite(act->beta) || !(act->limit > 0.f)))
      return MOE_FP4_EINVAL;
    ap = {act->kind, act->alpha, act->beta, act->limit};
  }
  int st = check_shape(E, H, I, top_k, fmt);
  if (st != MOE_FP4_OK) return st;
  // W4A8-MX: MXFP4 weights, gated activations (the mirror the band follows)
  if (prefill_mode == MOE_FP4_PREFILL_W4A8_MX && (fmt != MOE_FP4_MXFP4 || ap.kind == MOE_FP4_ACT_RELU2))
    return MOE_FP4_EUNSUPPORTED;
  if (M < 0) return MOE_FP4_EINVAL;
  if (M == 0) return MOE_FP4_OK;
  if (!x_bf16 || !w13 || !s13 || !w2 || !s2 || !topk_ids || !topk_weights || !out_bf16) return MOE_FP4_EINVAL;
  if (!aligned16(x_bf16) || !aligned16(w13) || !aligned16(w2) || !aligned16(s13) || !aligned16(s2))
    return MOE_FP4_EINVAL;
  if (M > MOE_FP4_DECODE_MAX_M) {
    st = check_prefill(M, E, I, top_k, fmt);
    if (st != MOE_FP4_OK) return st;
  }
  if (!workspace || ((uintptr_t)workspace & 255u)) return MOE_FP4_EWORKSPACE;
  int sms = 0;
  st = device_sms(&sms);
  if (st != MOE_FP4_OK) return st;
  if (M > MOE_FP4_DECODE_MAX_M && !exact && mid_band_chunks(M)) {
    // balanced chunks of at most MOE_FP4_DECODE_MAX_M tokens, one after
    // another on the stream (each overwrites only its own rows of out; a
    // chunk's first kernel waits for the previous chunk before it touches
    // the shared workspace)
    const int n = (M + MOE_FP4_DECODE_MAX_M - 1) / MOE_FP4_DECODE_MAX_M;
    size_t need = 0;
    for (int c = 0, m0 = 0; c < n; ++c) {
      const int mc = (M - m0) / (n - c);
      const size_t b = decode_workspace_bytes(mc, H, I, top_k, fmt, sms);
      need = b > need ? b : need;
      m0 += mc;
    }
    if (need >= kMaxWorkspace || workspace_bytes < need) return MOE_FP4_EWORKSPACE;
    const size_t id_bytes = ids64 ? 8 : 4;
    for (int c = 0, m0 = 0; c < n; ++c) {
      const int mc = (M - m0) / (n - c);
      const size_t r0 = (size_t)m0 * top_k;
      cudaError_t e = launch_decode(
          static_cast<const uint16_t*>(x_bf16) + (size_t)m0 * H, w13, s13, w2, s2,
          reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(topk_ids) + r0 * id_bytes), ids64,
          topk_weights + r0, static_cast<uint16_t*>(out_bf16) + (size_t)m0 * H, mc, E, H, I, top_k, fmt, ap,
          workspace, sms, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return fail_cuda(e);
      m0 += mc;
    }
    return MOE_FP4_OK;
  }
  if (M <= MOE_FP4_DECODE_MAX_M) {
    const size_t need = decode_workspace_bytes(M, H, I, top_k, fmt, sms);
    if (need >= kMaxWorkspace || workspace_bytes < need) return MOE_FP4_EWORKSPACE;
    cudaError_t e = launch_decode(x_bf16, w13, s13, w2, s2, ids, ids64, topk_weights, out_bf16, M, E, H, I, top_k,
                                  fmt, ap, workspace, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
  }
  const size_t need = prefill_workspace_bytes(M, E, H, I, top_k, exact);
  if (need >= kMaxWorkspace || workspace_bytes < need) return MOE_FP4_EWORKSPACE;
  int cu = 0;
  cudaError_t e = launch_prefill(x_bf16, w13, s13, w2, s2, ids, ids64, topk_weights, out_bf16, M, E, H, I, top_k,
                                 ap, prefill_mode, !exact && mid_band_swap(M, E, I, top_k), workspace,
                                 static_cast<cudaStream_t>(stream), &cu);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}
}  // namespace

int moe_fp4_forward_ex(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                       const int32_t* topk_ids, const float* topk_weights, void* out_bf16, int M, int E, int H,
                       int I, int top_k, int fmt, const moe_fp4_activation* act, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return forward_any_ids(x_bf16, w13, s13, w2, s2, topk_ids, 0, topk_weights, out_bf16, M, E, H, I, top_k, fmt, act,
                         workspace, workspace_bytes, stream);
}

int moe_fp4_forward_ex_i64(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                           const int64_t* topk_ids, const float* topk_weights, void* out_bf16, int M, int E, int H,
                           int I, int top_k, int fmt, const moe_fp4_activation* act, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (((uintptr_t)topk_ids & 7u) != 0) return MOE_FP4_EINVAL;
  return forward_any_ids(x_bf16, w13, s13, w2, s2, topk_ids, 1, topk_weights, out_bf16, M, E, H, I, top_k, fmt, act,
                         workspace, workspace_bytes, stream);
}

int moe_fp4_forward_mode(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                         const void* topk_ids, int ids_int64, const float* topk_weights, void* out_bf16, int M, int E,
                         int H, int I, int top_k, int fmt, const moe_fp4_activation* act, int prefill_mode,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (ids_int64 != 0 && ids_int64 != 1) return MOE_FP4_EINVAL;
  if (ids_int64 && ((uintptr_t)topk_ids & 7u) != 0) return MOE_FP4_EINVAL;
  return forward_any_ids(x_bf16, w13, s13, w2, s2, topk_ids, ids_int64, topk_weights, out_bf16, M, E, H, I, top_k,
                         fmt, act, workspace, workspace_bytes, stream, prefill_mode);
}

int moe_fp4_debug_set_w4a8_engine(int fp8) { return moe_fp4::set_w4a8_fp8_engine(fp8); }

size_t moe_fp4_workspace_bytes_mode(int M_max, int E, int H, int I, int top_k, int fmt, int prefill_mode) {
  if (prefill_mode != MOE_FP4_PREFILL_NVFP4 && prefill_mode != MOE_FP4_PREFILL_BF16 &&
      prefill_mode != MOE_FP4_PREFILL_W4A8_MX)
    return 0;
  if (M_max < 0 || check_shape(E, H, I, top_k, fmt) != MOE_FP4_OK) return 0;
  if (prefill_mode == MOE_FP4_PREFILL_W4A8_MX && fmt != MOE_FP4_MXFP4) return 0;
  if (M_max > MOE_FP4_DECODE_MAX_M && check_prefill(M_max, E, I, top_k, fmt) != MOE_FP4_OK) return 0;
  int sms = 0;
  if (device_sms(&sms) != MOE_FP4_OK) return 0;
  return workspace_need(M_max < 1 ? 1 : M_max, E, H, I, top_k, fmt, sms, prefill_mode != MOE_FP4_PREFILL_NVFP4);
}

int moe_fp4_forward_ws(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                       const int32_t* topk_ids, const float* topk_weights, void* out_bf16, int M, int E, int H,
                       int I, int top_k, int fmt, void* workspace, size_t workspace_bytes, void* stream) {
  return moe_fp4_forward_ex(x_bf16, w13, s13, w2, s2, topk_ids, topk_weights, out_bf16, M, E, H, I, top_k, fmt,
                            nullptr, workspace, workspace_bytes, stream);
}

int moe_fp4_forward(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                    const int32_t* topk_ids, const float* topk_weights, void* out_bf16, int M, int E, int H, int I,
                    int top_k, int fmt, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= 64) return MOE_FP4_EUNSUPPORTED;
  void* ptr;
  size_t bytes;
  {
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    ptr = g_ws[dev].ptr;
    bytes = g_ws[dev].bytes;
  }
  if (M > 0 && !ptr) return MOE_FP4_EWORKSPACE;
  return moe_fp4_forward_ws(x_bf16, w13, s13, w2, s2, topk_ids, topk_weights, out_bf16, M, E, H, I, top_k, fmt, ptr,
                            bytes, stream);
}

size_t moe_fp4_host_workspace_bytes(int M_max, int E, int H, int I, int top_k, int fmt) {
  if (check_shape(E, H, I, top_k, fmt) != MOE_FP4_OK || M_max <= 0) return 0;
  if (M_max > MOE_FP4_DECODE_MAX_M && check_prefill(M_max, E, I, top_k, fmt) != MOE_FP4_OK) return 0;
  int sms = 0;
  if (device_sms(&sms) != MOE_FP4_OK) return 0;
  // both parts grow with M, so the M_max layout covers every smaller batch
  return align256(workspace_need(M_max, E, H, I, top_k, fmt, sms)) + host_stage(M_max, H, top_k).total;
}

int moe_fp4_forward_host(const void* x_bf16, const void* w13, const void* s13, const void* w2, const void* s2,
                         const int32_t* topk_ids, const float* topk_weights, void* out_bf16, int M, int E, int H,
                         int I, int top_k, int fmt, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_shape(E, H, I, top_k, fmt);
  if (st != MOE_FP4_OK) return st;
  if (M < 0) return MOE_FP4_EINVAL;
  if (M == 0) return MOE_FP4_OK;
  if (!x_bf16 || !topk_ids || !topk_weights || !out_bf16) return MOE_FP4_EINVAL;
  if (M > MOE_FP4_DECODE_MAX_M) {
    st = check_prefill(M, E, I, top_k, fmt);
    if (st != MOE_FP4_OK) return st;
  }
  if (!workspace || ((uintptr_t)workspace & 255u)) return MOE_FP4_EWORKSPACE;
  int sms = 0;
  st = device_sms(&sms);
  if (st != MOE_FP4_OK) return st;
  const size_t base = align256(workspace_need(M, E, H, I, top_k, fmt, sms));
  const HostStage hs = host_stage(M, H, top_k);
  if (base + hs.total >= kMaxWorkspace || workspace_bytes < base + hs.total) return MOE_FP4_EWORKSPACE;
  char* stage = static_cast<char*>(workspace) + base;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)M * H * 2, rb = (size_t)M * top_k * 4;
  // On the decode-band kernels (and their chunks), buffers the GPU can
  // address (page-locked host memory, mapped into the device's address space
  // over the CPU-GPU link) are read and written in place by the kernels: a
  // few KB each, where a copy's fixed cost would exceed the layer's.
  // Everything else, and the prefill band's large tensors, go through the
  // staging area.
  const bool decode = M <= MOE_FP4_DECODE_MAX_M || mid_band_chunks(M);
  void* xd = decode ? device_view(x_bf16) : nullptr;
  void* idd = decode ? device_view(topk_ids) : nullptr;
  void* twd = decode ? device_view(topk_weights) : nullptr;
  void* od = decode ? device_view(out_bf16) : nullptr;
  cudaError_t e = cudaSuccess;
  if (!xd) {
    xd = stage + hs.x;
    e = cudaMemcpyAsync(xd, x_bf16, xb, cudaMemcpyDefault, s);
  }
  if (!idd && e == cudaSuccess) {
    idd = stage + hs.ids;
    e = cudaMemcpyAsync(idd, topk_ids, rb, cudaMemcpyDefault, s);
  }
  if (!twd && e == cudaSuccess) {
    twd = stage + hs.tw;
    e = cudaMemcpyAsync(twd, topk_weights, rb, cudaMemcpyDefault, s);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  const bool out_direct = od != nullptr;
  if (!out_direct) od = stage + hs.out;
  st = moe_fp4_forward_ws(xd, w13, s13, w2, s2, static_cast<const int32_t*>(idd), static_cast<const float*>(twd), od,
                          M, E, H, I, top_k, fmt, workspace, base, stream);
  if (st != MOE_FP4_OK || out_direct) return st;
  e = cudaMemcpyAsync(out_bf16, od, xb, cudaMemcpyDefault, s);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_workspace_status(const void* workspace, uint32_t* flags, int clear, void* stream) {
  if (!flags) return MOE_FP4_EINVAL;
  void* ws = const_cast<void*>(workspace);
  if (!ws) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= 64) return MOE_FP4_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    ws = g_ws[dev].ptr;
  }
  if (!ws) return MOE_FP4_EWORKSPACE;
  if ((uintptr_t)ws & 255u) return MOE_FP4_EWORKSPACE;
  return read_status_word(ws, flags, clear, static_cast<cudaStream_t>(stream));
}

int moe_fp4_debug_wait_timeout(void* status_word, unsigned polls, void* stream) {
  if (!status_word || ((uintptr_t)status_word & 3u)) return MOE_FP4_EINVAL;
  if (polls == 0 || polls > (1u << 20)) return MOE_FP4_EINVAL;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(status_word), polls);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_debug_set_decode_family(int family, int* previous) {
  if (family < 0 || family > 3) return MOE_FP4_EINVAL;
  const int old = g_decode_family.exchange(family);
  if (previous) *previous = old;
  return MOE_FP4_OK;
}

int moe_fp4_debug_set_mid_band(int mode, int* previous) {
  if (mode < 0 || mode > 3) return MOE_FP4_EINVAL;
  const int old = g_mid_band.exchange(mode);
  if (previous) *previous = old;
  return MOE_FP4_OK;
}

int moe_fp4_debug_decode_family_of(int M, int E, int H, int I, int top_k) {
  if (M < 1 || M > MOE_FP4_DECODE_MAX_M || check_shape(E, H, I, top_k, MOE_FP4_NVFP4) != MOE_FP4_OK) return 0;
  return decode_family_of(M, E, H, I, top_k);
}

int moe_fp4_debug_decode_plan(int M, int E, int H, int I, int top_k, int* plan) {
  if (!plan) return MOE_FP4_EINVAL;
  plan[0] = plan[1] = plan[2] = plan[3] = 0;
  if (M < 1 || M > MOE_FP4_DECODE_MAX_M) return MOE_FP4_EINVAL;
  const int st = check_shape(E, H, I, top_k, MOE_FP4_NVFP4);
  if (st != MOE_FP4_OK) return st;
  int C = 0, s1 = 0, Q = 0, cap = 0;
  if (decode_fused_plan(M, H, I, top_k, &C, &s1, &Q, &cap)) {
    plan[0] = C;
    plan[1] = s1;
    plan[2] = Q;
    plan[3] = cap;
  }
  return MOE_FP4_OK;
}

int moe_fp4_debug_decode_gemv_fits(int M, int E, int H, int I, int top_k) {
  return decode_gemv_fits(M, E, H, I, top_k) ? 1 : 0;
}

int moe_fp4_debug_decode_launches(int M, int E, int H, int I, int top_k) {
  if (M < 1 || check_shape(E, H, I, top_k, MOE_FP4_NVFP4) != MOE_FP4_OK) return 0;
  if (M <= MOE_FP4_DECODE_MAX_M) return decode_launches(M, E, H, I, top_k);
  if (!mid_band_chunks(M)) return 0;
  const int n = (M + MOE_FP4_DECODE_MAX_M - 1) / MOE_FP4_DECODE_MAX_M;
  int total = 0;
  for (int c = 0, m0 = 0; c < n; ++c) {
    const int mc = (M - m0) / (n - c);
    total += decode_launches(mc, E, H, I, top_k);
    m0 += mc;
  }
  return total;
}

int moe_fp4_debug_mid_band_of(int M, int E, int H, int I, int top_k) {
  if (M <= MOE_FP4_DECODE_MAX_M || check_shape(E, H, I, top_k, MOE_FP4_NVFP4) != MOE_FP4_OK) return 0;
  if (mid_band_chunks(M)) return 2;
  return mid_band_swap(M, E, I, top_k) ? 3 : 1;
}

int moe_fp4_debug_dequant(const void* w, const void* s, int which, int expert, int E, int H, int I, int fmt,
                          float* out_f32, void* stream) {
  int st = check_shape(E, H, I, 1, fmt);
  if (st != MOE_FP4_OK) return st;
  if (!w || !s || !out_f32 || which < 0 || which > 2 || expert < 0 || expert >= E) return MOE_FP4_EINVAL;
  cudaError_t e = launch_debug_dequant(w, s, which, expert, E, H, I, fmt, out_f32, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_debug_gemm(const void* a_q, const void* a_sf, const void* b_q, const void* b_sf, float* d, int M_rows,
                       int N_rows, int K, int fmt, uint32_t* status, void* stream) {
  if (fmt != MOE_FP4_NVFP4 && fmt != MOE_FP4_MXFP4) return MOE_FP4_EINVAL;
  if (fmt != MOE_FP4_NVFP4) return MOE_FP4_EUNSUPPORTED;
  if (!a_q || !a_sf || !b_q || !b_sf || !d || !status) return MOE_FP4_EINVAL;
  if (M_rows <= 0 || N_rows <= 0 || K <= 0) return MOE_FP4_EINVAL;
  if (M_rows % 128 || N_rows % 256 || K % 256) return MOE_FP4_EUNSUPPORTED;
  if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(a_sf) || !aligned16(b_sf) || !aligned16(d))
    return MOE_FP4_EINVAL;
  int cu = 0;
  cudaError_t e = launch_debug_gemm(a_q, a_sf, b_q, b_sf, d, M_rows, N_rows, K, status,
                                    static_cast<cudaStream_t>(stream), &cu);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_debug_route(const int32_t* topk_ids, int M, int E, int top_k, int32_t* perm, int32_t* expert_offset,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!topk_ids || !perm || !expert_offset || M <= 0 || E <= 0 || top_k <= 0) return MOE_FP4_EINVAL;
  if (E > 4096 || top_k > 16) return MOE_FP4_EUNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < debug_route_workspace_bytes(M, E, top_k))
    return MOE_FP4_EWORKSPACE;
  cudaError_t e = launch_debug_route(topk_ids, M, E, top_k, perm, expert_offset, workspace,
                                     static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_debug_route_small(const int32_t* topk_ids, int M, int E, int top_k, int32_t* perm,
                              int32_t* expert_offset, void* workspace, size_t workspace_bytes, void* stream) {
  if (!topk_ids || !perm || !expert_offset || M <= 0 || E <= 0 || top_k <= 0) return MOE_FP4_EINVAL;
  if (E > 4096 || top_k > 16 || (int64_t)M * top_k > 8192) return MOE_FP4_EUNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < debug_route_workspace_bytes(M, E, top_k))
    return MOE_FP4_EWORKSPACE;
  cudaError_t e = launch_debug_route(topk_ids, M, E, top_k, perm, expert_offset, workspace,
                                     static_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

size_t moe_fp4_debug_route_workspace_bytes(int M, int E, int top_k) {
  if (M <= 0 || E <= 0 || top_k <= 0 || E > 4096 || top_k > 16) return 0;
  return debug_route_workspace_bytes(M, E, top_k);
}

int moe_fp4_debug_quant_rows(const float* in, int rows, int K, uint8_t* q, uint8_t* s, float* G, void* stream) {
  if (!in || !q || !s || !G || rows <= 0 || K <= 0) return MOE_FP4_EINVAL;
  if (K % 16 != 0) return MOE_FP4_EUNSUPPORTED;
  if (((uintptr_t)q & 7u) || ((uintptr_t)in & 3u)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_debug_quant(in, rows, K, q, s, G, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

int moe_fp4_debug_quant_mxfp8_rows(const float* in, int rows, int K, uint8_t* q, uint8_t* s, void* stream) {
  if (!in || !q || !s || rows <= 0 || K <= 0) return MOE_FP4_EINVAL;
  if (K % 32 != 0) return MOE_FP4_EUNSUPPORTED;
  if (((uintptr_t)q & 15u) || ((uintptr_t)in & 3u)) return MOE_FP4_EINVAL;
  cudaError_t e = launch_debug_quant_mxfp8(in, rows, K, q, s, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_FP4_OK : fail_cuda(e);
}

}  // extern "C"
