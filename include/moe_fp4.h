/*
 * moe_fp4.h — C ABI of libmoe_fp4.so, a fused mixture-of-experts layer over
 * 4-bit E2M1 expert weights with block scales, for one NVIDIA GB300 GPU
 * (sm_103a).
 *
 * The layer (b12x PR #22, "rp-native tiny-decode kernel for w4a8_mx (M=1)",
 * section What): for every token t and each of its top-k slots j with a valid
 * expert id e,
 *     gate_n = x_t . W13[e][n],  up_n = x_t . W13[e][I+n]      (FC1, FP32)
 *     h_n    = SiLU(gate_n) * up_n
 *     y_m    = W2[e][m] . h                                     (FC2)
 *     out_t  = sum_j topk_weights[t][j] * y                     (BF16 output)
 * Activations are BF16 and are not quantised in the decode band (same
 * section: "Activations stay BF16").  A slot whose id is < 0 or >= E
 * contributes exactly zero (b12x PR #311, conversation: invalid routes get an
 * exact-zero effective weight and caller tensors are never mutated).
 *
 * Formats (fmt):
 *   MOE_FP4_MXFP4 — E2M1 elements, one UE8M0 scale byte per 32 K-elements
 *                   (flashinfer PR #4285, scale_format_e8m0_k32).
 *   MOE_FP4_NVFP4 — E2M1 elements, one E4M3 scale byte per 16 K-elements,
 *                   times an FP32 per-tensor multiplier (b12x PR #459,
 *                   "Reduce NVFP4-CSF scale reconstruction overhead":
 *                   FP32 calibration kept with the scale bytes).
 *
 * Conventions for every function:
 *   - All array arguments are DEVICE pointers on the current CUDA device,
 *     unless stated as host.  They are owned by the caller; the library never
 *     frees or retains them past the call (except the library workspace of
 *     moe_fp4_reserve_workspace, which the library owns).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising.
 *   - Every function returns a moe_fp4_status; nothing throws.  Argument
 *     errors are reported before any work is enqueued.  MOE_FP4_ECUDA means a
 *     CUDA launch or API call failed; moe_fp4_last_cuda_error() gives the
 *     cudaError_t value.
 *   - Shape limits: H % 256 == 0, I % 64 == 0, 1 <= top_k <= 16,
 *     1 <= E <= 65536, 2I * H <= 2^31; violating shapes return
 *     MOE_FP4_EUNSUPPORTED.
 */
#ifndef MOE_FP4_H
#define MOE_FP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_FP4_API __attribute__((visibility("default")))
#else
#define MOE_FP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MOE_FP4_MXFP4 = 0, MOE_FP4_NVFP4 = 1 } moe_fp4_fmt;

typedef enum {
    MOE_FP4_OK = 0,
    MOE_FP4_EINVAL = 1,       /* null pointer, negative size, unknown fmt */
    MOE_FP4_EUNSUPPORTED = 2, /* shape outside the supported limits */
    MOE_FP4_ECUDA = 3,        /* a CUDA call failed */
    MOE_FP4_EWORKSPACE = 4    /* workspace missing or too small, or >= 2^31 bytes */
} moe_fp4_status;

/* Largest token count handled by one pass of the decode band (HBM-bound
 * weight-streaming kernels).  Larger batches run the mid band (the grouped
 * block-scaled GEMMs with the weights on the MMA's 128-row side) while the
 * experts average at most 28 routed rows (36 with I <= 384), else the
 * prefill band (the grouped block-scaled GEMMs with the routed rows on that
 * side). */
#define MOE_FP4_DECODE_MAX_M 8

/* Human-readable name of a status code (static string, never NULL). */
MOE_FP4_API const char *moe_fp4_status_string(int status);

/* cudaError_t of the most recent MOE_FP4_ECUDA on the calling host thread. */
MOE_FP4_API int moe_fp4_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
MOE_FP4_API int moe_fp4_version(void);

/*
 * Sizes in bytes of the four resident (prepared) weight buffers for E
 * experts of shape (H, I) in format fmt.  Host pointers out; any may be NULL.
 *
 * Resident layout (written by moe_fp4_prepare_weights):
 *   w13: [E][2I][H/2] bytes.  Rows are the logical gate/up rows interleaved
 *        in groups of 64: resident rows 128j..128j+63 are gate rows
 *        64j..64j+63 and resident rows 128j+64..128j+127 are up rows
 *        64j..64j+63, so each 128-row tile holds matching gate and up rows.
 *        Byte order within a row is the logical one (low nibble = even K).
 *   w2:  [E][H][I/2] bytes, the logical layout.
 *   s13, s2: E4M3 scale bytes, one per 16 K-elements for both formats, in
 *        512-byte chunks, one per (expert, 128-row tile, group of 4
 *        consecutive 16-element K-blocks); inside a chunk the byte of row r
 *        (0..127 within the tile) and K-block b (0..3 within the group) is at
 *        (r % 32) * 16 + (r / 32) * 4 + b.  Chunks are ordered expert, row
 *        tile, K-block group.  After the chunks, s13 holds FP32 multipliers
 *        [E][2] (gate, up) and s2 holds [E].  NVFP4: the checkpoint's scale
 *        bytes and per-tensor multipliers.  MXFP4: each UE8M0 block scale
 *        2^(e-127) becomes the E4M3 power of two 2^(e-127-b) for both of its
 *        16-element halves, with the projection multiplier 2^b, b = (largest
 *        block exponent of that expert's projection) - 127 - 8; block scales
 *        more than 2^17 below the projection's largest are stored as 0 (their
 *        weights read as zero), all others exactly.
 */
MOE_FP4_API int moe_fp4_prepared_sizes(int E, int H, int I, int fmt, size_t *w13_bytes, size_t *s13_bytes, size_t *w2_bytes,
                           size_t *s2_bytes);

/*
 * Repack logical checkpoint tensors into the resident layout (one-time,
 * outside the hot path).  Inputs (device):
 *   w13_logical [E][2I][H/2] u8 — rows 0..I-1 gate, I..2I-1 up; low nibble =
 *                                 even K index
 *   s13_logical [E][2I][H/B] u8 — one scale byte per (row, K-block of B)
 *   g13         [E][2] f32      — NVFP4 gate/up multipliers (NULL for MXFP4)
 *   w2_logical  [E][H][I/2] u8, s2_logical [E][H][I/B] u8, g2 [E] f32 (NVFP4)
 * Outputs (device, sizes from moe_fp4_prepared_sizes): w13, s13, w2, s2.
 * Inputs and outputs must not overlap.
 */
MOE_FP4_API int moe_fp4_prepare_weights(const void *w13_logical, const void *s13_logical, const float *g13,
                            const void *w2_logical, const void *s2_logical, const float *g2, int E, int H, int I,
                            int fmt, void *w13, void *s13, void *w2, void *s2, void *stream);

/* Inverse of moe_fp4_prepare_weights (test support): resident -> logical. */
MOE_FP4_API int moe_fp4_unprepare_weights(const void *w13, const void *s13, const void *w2, const void *s2, int E, int H, int I,
                              int fmt, void *w13_logical, void *s13_logical, float *g13, void *w2_logical,
                              void *s2_logical, float *g2, void *stream);

/*
 * Workspace bytes needed by moe_fp4_forward_ws for up to M_max tokens.
 * Returns 0 for invalid arguments.  Workspaces of 2^31 bytes or more are
 * rejected by the forward calls (MOE_FP4_EWORKSPACE).
 */
MOE_FP4_API size_t moe_fp4_workspace_bytes(int M_max, int E, int H, int I, int top_k, int fmt);

/*
 * Allocate (cudaMalloc) and zero a library-owned workspace on the current
 * device, sized for moe_fp4_workspace_bytes(M_max, ...).  A later call with
 * larger sizes grows it; smaller calls keep it.  Call it before capturing
 * moe_fp4_forward in a CUDA graph: moe_fp4_forward itself never allocates.
 * moe_fp4_release_workspace frees it.
 */
MOE_FP4_API int moe_fp4_reserve_workspace(int M_max, int E, int H, int I, int top_k, int fmt, void *stream);
MOE_FP4_API int moe_fp4_release_workspace(void);

/*
 * The fused MoE layer, using the reserved library workspace
 * (MOE_FP4_EWORKSPACE if none is reserved or it is too small).
 *   x_bf16       [M][H] bf16 activations
 *   w13, s13, w2, s2  resident weights from moe_fp4_prepare_weights
 *   topk_ids     [M][top_k] int32 expert ids (ids < 0 or >= E are ignored)
 *   topk_weights [M][top_k] f32 router weights
 *   out_bf16     [M][H] bf16, fully overwritten (tokens with no valid slot
 *                get +0.0); must not overlap any input.
 * M = 0 is a no-op.  Inputs are never written.  Decode-band results (M <=
 * 8) are bitwise deterministic; the mid and prefill bands sum routed rows
 * into an FP32 token accumulator with atomic adds, so their low-order bits
 * may vary run to run.
 *
 * Mid and prefill bands (M > 8): E <= 4096 (else MOE_FP4_EUNSUPPORTED).
 * Activations are quantised to NVFP4 per row (x per token, h =
 * SiLU(gate)*up per routed row after BF16 staging) so both GEMMs run on the
 * FP4 tensor cores; the two bands compute the same products.
 */
MOE_FP4_API int moe_fp4_forward(const void *x_bf16, const void *w13, const void *s13, const void *w2, const void *s2,
                    const int32_t *topk_ids, const float *topk_weights, void *out_bf16, int M, int E, int H, int I,
                    int top_k, int fmt, void *stream);

/*
 * Same as moe_fp4_forward with an explicit caller-owned workspace of at
 * least moe_fp4_workspace_bytes(M, E, H, I, top_k, fmt) bytes (256-byte
 * aligned).  Before its first use the first
 * moe_fp4_workspace_zero_bytes(E, H, I, top_k, fmt) bytes of a workspace
 * (the status word and the synchronisation words) must be zero (cudaMemset;
 * the rest is scratch that needs no initialisation, and zero-filling the
 * whole workspace is fine too); every call leaves its synchronisation words
 * at zero again, so later calls need no re-zeroing.  Calls sharing one
 * workspace must be ordered (same stream or explicit dependencies).  One
 * workspace serves every batch size up to the M it was sized for, in both
 * bands, for one (E, H, I, top_k, fmt).
 */
MOE_FP4_API size_t moe_fp4_workspace_zero_bytes(int E, int H, int I, int top_k, int fmt);
MOE_FP4_API int moe_fp4_forward_ws(const void *x_bf16, const void *w13, const void *s13, const void *w2, const void *s2,
                       const int32_t *topk_ids, const float *topk_weights, void *out_bf16, int M, int E, int H,
                       int I, int top_k, int fmt, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Workspace bytes needed by moe_fp4_forward_host for up to M_max tokens: the
 * layer's own workspace plus a staging area for the inputs and the output.
 * Returns 0 for invalid or unsupported arguments.  Queries the current
 * device's SM count.
 */
MOE_FP4_API size_t moe_fp4_host_workspace_bytes(int M_max, int E, int H, int I, int top_k, int fmt);

/*
 * The fused MoE layer with its per-call tensors in HOST memory:
 *   x_bf16       [M][H] bf16, host
 *   topk_ids     [M][top_k] int32, host
 *   topk_weights [M][top_k] f32, host
 *   out_bf16     [M][H] bf16, host, fully overwritten
 *   w13, s13, w2, s2  resident weights on the device (moe_fp4_prepare_weights)
 *   workspace    device memory of moe_fp4_host_workspace_bytes(M, ...) bytes
 *                or more, 256-byte aligned, zero-filled before its first use
 * Enqueues on `stream` the layer (the kernels of moe_fp4_forward_ws) and
 * the transfers of its per-call tensors.  In the decode band
 * (M <= MOE_FP4_DECODE_MAX_M) a 16-byte-aligned buffer that the current
 * device can address (page-locked host memory from cudaHostAlloc or
 * cudaHostRegister, mapped over the CPU-GPU link; or memory of the current
 * device) is read or written in place by the kernels.  Any other buffer, and
 * every buffer in the prefill band, goes through the workspace's staging
 * area: one host-to-device copy per input before the layer, one
 * device-to-host copy of the output after it.  Returns once everything is
 * enqueued: out_bf16 holds the result when the stream has reached that point
 * (cudaStreamSynchronize or an event), and the host buffers must stay valid
 * and unmodified until then.  Pageable buffers work, but their copies may
 * block the calling thread.  Results, M = 0 and the error codes
 * are those of moe_fp4_forward_ws; a workspace that is too small gives
 * MOE_FP4_EWORKSPACE before anything is enqueued.  Calls sharing a workspace
 * must be ordered.  The pages have no counterpart of this entry point: it is
 * the library's end-to-end call for callers whose tensors live on the host.
 */
MOE_FP4_API int moe_fp4_forward_host(const void *x_bf16, const void *w13, const void *s13, const void *w2,
                                     const void *s2, const int32_t *topk_ids, const float *topk_weights,
                                     void *out_bf16, int M, int E, int H, int I, int top_k, int fmt, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * Device status of a workspace.  Every wait inside the kernels is bounded:
 * a wait that has not completed after its poll limit (about a second) gives
 * up, the kernel sets one of the bits below in the status word of the
 * workspace it ran on (the first 4 bytes; 0 when the workspace is fresh) and
 * goes on without waiting, so the GPU is never hung; the outputs of such a
 * call are not valid.  The bits are sticky: they stay set for every later
 * call until cleared.  A wait can give up only when the launch's CTAs cannot
 * make progress together: the single-launch decode kernel needs its whole
 * grid resident at once, which concurrent work on the same GPU (other
 * streams, other processes) can prevent (flashinfer PR #4285, "sync SM12x
 * NVFP4 fused-MoE kernels": a cooperative kernel deadlocks when concurrent
 * work keeps part of its grid off the GPU).
 *
 * moe_fp4_workspace_status copies the status word of `workspace` (device
 * memory passed to moe_fp4_forward_ws, _ex, _ex_i64 or _host; NULL: the
 * library workspace of moe_fp4_reserve_workspace on the current device) into
 * *flags (host), after everything enqueued on `stream` before it, and if
 * `clear` is nonzero sets it back to 0.  It synchronises `stream` (call it
 * outside stream capture).  MOE_FP4_EWORKSPACE if workspace is NULL and none
 * is reserved, or not 256-byte aligned.  moe_fp4_noalloc_status does the same
 * for the scratch array of moe_fp4_forward_noalloc on the current device.
 */
#define MOE_FP4_STATUS_OK 0u
#define MOE_FP4_STATUS_TEST_WAIT 8192u /* set only by moe_fp4_debug_wait_timeout */
MOE_FP4_API int moe_fp4_workspace_status(const void *workspace, uint32_t *flags, int clear, void *stream);
MOE_FP4_API int moe_fp4_noalloc_status(uint32_t *flags, int clear, void *stream);
/*
 * Test support: one GPU thread waits on a barrier that nothing completes,
 * with a poll limit of `polls` (1 .. 2^20) instead of the kernels' own, so
 * that the bounded wait gives up and sets MOE_FP4_STATUS_TEST_WAIT in the
 * 32-bit word at `status_word` (device, 4-byte aligned; e.g. a workspace's
 * first word).  Nothing else is touched.  MOE_FP4_EINVAL for a null or
 * misaligned pointer or a limit out of range.
 */
MOE_FP4_API int moe_fp4_debug_wait_timeout(void *status_word, unsigned polls, void *stream);

/*
 * Gated activations of FC1's (gate, up) pair.  MOE_FP4_ACT_SILU,
 * SiLU(gate) * up, is the layer's own (and the default of every other
 * entry point).  The SM12x sync PR's kernels also take "gelu_tanh" and
 * "swigluoai_uninterleave":
 *   MOE_FP4_ACT_GELU_TANH  0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) u
 *   MOE_FP4_ACT_SWIGLUOAI  g' = min(g, limit), u' = min(max(u, -limit), limit),
 *                          (u' + beta) g' sigmoid(alpha g')
 * with g and u the dequantised FC1 outputs (per-tensor multipliers applied).
 * alpha, beta and limit are read for MOE_FP4_ACT_SWIGLUOAI only.
 */
#define MOE_FP4_ACT_SILU 0
#define MOE_FP4_ACT_GELU_TANH 1
#define MOE_FP4_ACT_SWIGLUOAI 2
#define MOE_FP4_ACT_RELU2 3 /* non-gated experts: see moe_fp4_prepare_weights_relu2 */
typedef struct moe_fp4_activation {
  int kind;
  float alpha, beta, limit;
} moe_fp4_activation;

/*
 * moe_fp4_forward_ws with a chosen activation (act == NULL: SiLU).  Same
 * arguments, workspace, results and errors otherwise; MOE_FP4_EINVAL for an
 * unknown kind, or for SwiGLU-OAI with a non-finite alpha or beta or a
 * limit that is not a positive number.  With MOE_FP4_ACT_RELU2 the experts
 * are non-gated and w13, s13 are the w1, s1 of moe_fp4_prepare_weights_relu2.
 */
MOE_FP4_API int moe_fp4_forward_ex(const void *x_bf16, const void *w13, const void *s13, const void *w2,
                                   const void *s2, const int32_t *topk_ids, const float *topk_weights, void *out_bf16,
                                   int M, int E, int H, int I, int top_k, int fmt, const moe_fp4_activation *act,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * The activation precision of batches past the decode band (M >
 * MOE_FP4_DECODE_MAX_M):
 *   MOE_FP4_PREFILL_NVFP4  (default of every other entry point) x per token
 *                          and h per routed row quantised to NVFP4, both
 *                          GEMMs on the FP4 tensor cores (kind::mxf4nvf4)
 *   MOE_FP4_PREFILL_BF16   exact numerics: x in BF16 against the weights
 *                          decoded to BF16 (exact: an E2M1 value times its
 *                          E4M3 block scale has at most six significant
 *                          bits), FP32 sums on the BF16 tensor cores
 *                          (kind::f16), h staged in BF16 for FC2; the layer
 *                          of the plain definition up to FP32/BF16 rounding,
 *                          at the BF16 tensor-core rate.
 *   MOE_FP4_PREFILL_W4A8_MX  MXFP8 activations (b12x PR #22, section What:
 *                          the w4a8_mx variant; flashinfer PR #4285,
 *                          Description: scale_format_e8m0_k32): x quantised
 *                          per token and h (staged in BF16) per routed row,
 *                          E4M3 elements with one UE8M0 scale per 32, block
 *                          exponent ceil(log2(amax / 448)); MXFP4 weights and
 *                          gated activations only (MOE_FP4_EUNSUPPORTED
 *                          otherwise).  Where I % 128 == 0 on the FP8 tensor
 *                          cores (tcgen05.mma kind::mxf8f6f4: E4M3 x E2M1
 *                          with UE8M0 scales per 32, the weights' MXFP4
 *                          scales taken exactly); otherwise on the 16-bit
 *                          engine of the previous mode (every MXFP8 value is
 *                          exact in row-scaled FP16 within 2^31 of its row's
 *                          largest).  Either way the FP32 sums are those of
 *                          the MXFP8 x MXFP4 products.
 * Batches past the decode band always take the prefill band in the BF16 and
 * W4A8-MX modes (neither the mid band nor decode-kernel chunks); batches of
 * at most MOE_FP4_DECODE_MAX_M tokens run the decode band in every mode
 * (BF16 activations, as the pages' w4a8_mx tiny-decode kernel keeps them).
 * The pages' decode keeps BF16 activations for accuracy (b12x PR #22, "rp-
 * native tiny-decode kernel for w4a8_mx (M=1)", section Measured: cosine
 * 0.999980 with BF16 activations against 0.9990 with MXFP8 ones).
 *
 * moe_fp4_forward_mode: moe_fp4_forward_ex (ids_int64 = 0) or _ex_i64
 * (ids_int64 = 1, ids 8-byte aligned) with a prefill precision; the
 * workspace must hold moe_fp4_workspace_bytes_mode(M, ..., prefill_mode)
 * bytes (the BF16 and W4A8-MX bands add x's BF16 image per routed row; a
 * workspace sized for either serves every mode; moe_fp4_workspace_bytes_mode
 * returns 0 for an unknown mode or a mode the format does not support).
 * MOE_FP4_EINVAL for an unknown mode.
 */
/* Test support: the W4A8-MX engine, 1 (default) = the FP8 tensor cores
 * (tcgen05.mma kind::mxf8f6f4 on the MXFP8 activations and the MXFP4 weights
 * as stored) wherever I % 128 == 0, 0 = always the 16-bit engine (the same
 * products).  Process-wide; returns the previous setting. */
MOE_FP4_API int moe_fp4_debug_set_w4a8_engine(int fp8);

#define MOE_FP4_PREFILL_NVFP4 0
#define MOE_FP4_PREFILL_BF16 1
#define MOE_FP4_PREFILL_W4A8_MX 2
MOE_FP4_API size_t moe_fp4_workspace_bytes_mode(int M_max, int E, int H, int I, int top_k, int fmt,
                                                int prefill_mode);
MOE_FP4_API int moe_fp4_forward_mode(const void *x_bf16, const void *w13, const void *s13, const void *w2,
                                     const void *s2, const void *topk_ids, int ids_int64, const float *topk_weights,
                                     void *out_bf16, int M, int E, int H, int I, int top_k, int fmt,
                                     const moe_fp4_activation *act, int prefill_mode, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * Non-gated experts with the squared ReLU: "relu2" of flashinfer PR #4285
 * ("sync SM12x NVFP4 fused-MoE kernels"), which names it among the
 * activations and keeps the exact activation quantiser for it (its outputs
 * are squares, not a gated product).  FC1 has I rows:
 *     h_n = max(x_t . W1[e][n], 0)^2
 * then FC2 and the router-weighted sum as for the gated layer.  Logical
 * inputs (device): w1 [E][I][H/2] u8 (low nibble = even K), s1 [E][I][H/B]
 * u8, g1 [E] f32 (NVFP4 only, else NULL), and w2, s2, g2 as for
 * moe_fp4_prepare_weights.  Resident layout: w1 rows in logical order; s1
 * scale chunks as for w13 (moe_fp4_prepared_sizes) with each expert's rows
 * padded to a multiple of 128 (padding rows' scales are zero), then the FP32
 * multipliers [E] (NVFP4: g1; MXFP4: the power of two of the re-expressed
 * block scales, as for w13); w2, s2 as for the gated layer.  Run the layer
 * with moe_fp4_forward_ex or moe_fp4_forward_ex_i64 and act kind
 * MOE_FP4_ACT_RELU2, w1 and s1 in place of w13 and s13 (the same shape
 * limits and workspace sizes; the decode band runs the tcgen05 launch chain,
 * the prefill band quantises h = max(u, 0)^2 after BF16 staging with the
 * same exact row quantiser).
 */
MOE_FP4_API int moe_fp4_prepared_sizes_relu2(int E, int H, int I, int fmt, size_t *w1_bytes, size_t *s1_bytes,
                                             size_t *w2_bytes, size_t *s2_bytes);
MOE_FP4_API int moe_fp4_prepare_weights_relu2(const void *w1_logical, const void *s1_logical, const float *g1,
                                              const void *w2_logical, const void *s2_logical, const float *g2, int E,
                                              int H, int I, int fmt, void *w1, void *s1, void *w2, void *s2,
                                              void *stream);
/* Inverse of moe_fp4_prepare_weights_relu2 (test support). */
MOE_FP4_API int moe_fp4_unprepare_weights_relu2(const void *w1, const void *s1, const void *w2, const void *s2, int E,
                                                int H, int I, int fmt, void *w1_logical, void *s1_logical, float *g1,
                                                void *w2_logical, void *s2_logical, float *g2, void *stream);

/*
 * moe_fp4_forward_ex with int64 routing ids (topk_ids int64 [M][top_k],
 * row-major, device memory, 8-byte aligned).  The b12x PR #459 page (Reduce
 * NVFP4-CSF scale reconstruction overhead, its commit list) keeps kernels
 * for both integer types of the routing ids; here the same kernels read
 * either width.  Every id outside [0, E) is invalid and contributes exactly
 * zero, including values that do not fit in 32 bits (they are never
 * truncated into a valid expert).  Same arguments, workspace, results and
 * errors as moe_fp4_forward_ex otherwise, plus MOE_FP4_EINVAL for a
 * topk_ids pointer that is not 8-byte aligned.  For ids that are all in
 * [-2^31, 2^31) the result is that of moe_fp4_forward_ex on the same ids as
 * int32: bitwise on the decode kernels, which are deterministic, and up to
 * the prefill band's run-to-run summation order there.
 */
MOE_FP4_API int moe_fp4_forward_ex_i64(const void *x_bf16, const void *w13, const void *s13, const void *w2,
                                       const void *s2, const int64_t *topk_ids, const float *topk_weights,
                                       void *out_bf16, int M, int E, int H, int I, int top_k, int fmt,
                                       const moe_fp4_activation *act, void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * The decode-band layer (M <= MOE_FP4_DECODE_MAX_M) without any device
 * allocation, for callers that cannot call cudaMalloc where they run the
 * layer: inside a stream capture, under a runtime that owns all device memory
 * through its own pool, or on a latency-critical path that cannot afford an
 * allocation's implicit synchronisation.  The pages have no counterpart of
 * this entry point; it is an addition of this library.
 *
 * Arguments, layouts and results are those of moe_fp4_forward (same
 * kernels, bitwise the same output).  Instead of a workspace it uses one
 * fixed scratch array in the library's device image (laid out as a decode
 * workspace: the 256-byte status block, the single-launch kernel's
 * synchronisation words, the intermediate; MOE_FP4_NOALLOC_SCRATCH_BYTES +
 * 256 bytes in all), which every GPU that loads the library's device code
 * keeps until the process exits.  Shapes whose scratch need
 * (moe_fp4_workspace_bytes(M, ...)) exceeds MOE_FP4_NOALLOC_SCRATCH_BYTES +
 * 256 return MOE_FP4_EWORKSPACE; M > MOE_FP4_DECODE_MAX_M returns
 * MOE_FP4_EUNSUPPORTED; other shape limits as moe_fp4_forward.  The first
 * call on each device looks up the array's device address while that device
 * is current; make that first call outside any stream capture.  All calls on
 * a device share the one array: calls that may overlap on the GPU (different
 * streams without ordering between them) race and corrupt each other's
 * results, so order them.  The synchronisation words must be zero when a
 * call starts: the array is zero when the device code is loaded and every
 * completed call leaves them at zero; the intermediate needs no clearing.
 * moe_fp4_noalloc_status reads the array's status word.
 */
#define MOE_FP4_NOALLOC_SCRATCH_BYTES (16u << 20)
MOE_FP4_API int moe_fp4_forward_noalloc(const void *x_bf16, const void *w13, const void *s13, const void *w2,
                                        const void *s2, const int32_t *topk_ids, const float *topk_weights,
                                        void *out_bf16, int M, int E, int H, int I, int top_k, int fmt, void *stream);

/*
 * Test support: choose the kernel family of the decode band (M <=
 * MOE_FP4_DECODE_MAX_M) for every later call in the process.
 *   family 0  by shape (default): the streaming GEMV kernels for one token
 *             with at most 4 MB of routed weights, else the tcgen05 launch
 *             chain
 *   family 1  the streaming GEMV kernels where the shape fits them
 *   family 2  the tcgen05 launch chain (x pre-pass, FC1, h pre-pass from
 *             M = 2, FC2)
 *   family 3  the tcgen05 single launch where it fits (the whole grid
 *             resident at once on this device), else the chain
 * All compute the same layer and agree within the parity bound; they are not
 * bitwise equal in general (the GEMV family sums in a different order, and
 * the two tcgen05 plans may split FC1's K range differently).  *previous
 * (if non-null) receives the old setting.  MOE_FP4_EINVAL for other values.
 * moe_fp4_debug_decode_gemv_fits returns 1 if the GEMV kernels take the
 * shape (their shared memory holds all tokens' activations and every routed
 * pair's h), else 0.
 */
MOE_FP4_API int moe_fp4_debug_set_decode_family(int family, int *previous);
/*
 * Test support: the kernels of batches past the decode band
 * (M > MOE_FP4_DECODE_MAX_M) under MOE_FP4_PREFILL_NVFP4 for every later
 * call in the process.
 *   mode 0  by shape (default): the mid band's GEMMs while the experts
 *           average at most 28 routed rows (M * top_k <= 28 E; 36 rows with
 *           I <= 384, where the prefill band's FC2 has little K), else the
 *           prefill band's
 *   mode 1  the prefill band's GEMMs (routed rows on the MMA's 128-row
 *           side)
 *   mode 2  the decode-band kernels on balanced chunks of at most
 *           MOE_FP4_DECODE_MAX_M tokens, one chunk after another (up to
 *           3 * MOE_FP4_DECODE_MAX_M tokens; larger batches as mode 0)
 *   mode 3  the mid band's GEMMs (weights on the MMA's 128-row side, an
 *           expert's routed rows on its N side), any batch size
 * The prefill and mid bands compute the same layer (NVFP4 activations).
 * *previous (if non-null) receives the old setting.  MOE_FP4_EINVAL for
 * other values.
 */
MOE_FP4_API int moe_fp4_debug_set_mid_band(int mode, int *previous);
MOE_FP4_API int moe_fp4_debug_decode_gemv_fits(int M, int E, int H, int I, int top_k);
/* The plan the current setting picks for a decode-band shape on the current
 * device (1 streaming GEMV, 2 tcgen05 launch chain, 3 tcgen05 single
 * launch); 0 for M outside 1..MOE_FP4_DECODE_MAX_M or invalid arguments. */
MOE_FP4_API int moe_fp4_debug_decode_family_of(int M, int E, int H, int I, int top_k);
/* The single-launch plan's geometry for a decode-band shape on the current
 * device, into plan[4] (host): cluster size C, FC1 K ranges per w13 tile,
 * clusters launched, and the clusters of that size the device can hold
 * resident at once; all zero if the shape has no single-launch plan there
 * (it then runs as the launch chain).  MOE_FP4_EINVAL for M outside
 * 1..MOE_FP4_DECODE_MAX_M or a null plan. */
MOE_FP4_API int moe_fp4_debug_decode_plan(int M, int E, int H, int I, int top_k, int *plan);
/* Kernel launches one decode-band layer of this shape makes under the
 * current family and mid-band settings (2 streaming GEMV; 1 tcgen05 single
 * launch; 3, or 4 from M = 2, tcgen05 chain; the sum over the chunks of a
 * batch that mode 2 of moe_fp4_debug_set_mid_band runs in chunks); 0 for
 * shapes that take the mid or prefill band, or invalid arguments. */
MOE_FP4_API int moe_fp4_debug_decode_launches(int M, int E, int H, int I, int top_k);
/* The kernels the current moe_fp4_debug_set_mid_band setting picks for a
 * batch past the decode band under MOE_FP4_PREFILL_NVFP4 (1 the prefill
 * band's GEMMs, 2 decode-band chunks, 3 the mid band's GEMMs); 0 for
 * M <= MOE_FP4_DECODE_MAX_M or invalid shape arguments. */
MOE_FP4_API int moe_fp4_debug_mid_band_of(int M, int E, int H, int I, int top_k);

/*
 * Test support: dequantise one expert's projection from the resident layout
 * into out_f32 [rows][K] in LOGICAL row order, each element computed as the
 * kernels use it: RN_fp32((e2m1 * e4m3) * g) (one rounding; exact for MXFP4,
 * whose e4m3 and g are powers of two).  which = 0: w13 (rows 2I, K = H, gate
 * rows first), which = 1: w2 (rows H, K = I), which = 2: the w1 of
 * moe_fp4_prepare_weights_relu2 (rows I, K = H).
 */
MOE_FP4_API int moe_fp4_debug_dequant(const void *w, const void *s, int which, int expert, int E, int H, int I, int fmt,
                          float *out_f32, void *stream);

/*
 * Test support: the prefill band's block-scaled FP4 GEMM on one pair of
 * matrices, D[m][n] = sum_k A[m][k] * B[n][k] in FP32 (no per-tensor
 * multipliers).  a_q [M_rows][K/2] and b_q [N_rows][K/2] packed E2M1 (low
 * nibble = even k); a_sf, b_sf their E4M3 scales (one per 16 K-elements) in
 * the resident 512-byte chunk layout of moe_fp4_prepared_sizes (rows in
 * 128-row tiles); d [M_rows][N_rows] FP32.  status: one device word, zeroed
 * by the caller; nonzero afterwards means an internal wait timed out.
 * M_rows % 128 == 0, N_rows % 256 == 0, K % 256 == 0; NVFP4 only.
 */
MOE_FP4_API int moe_fp4_debug_gemm(const void *a_q, const void *a_sf, const void *b_q, const void *b_sf, float *d,
                                   int M_rows, int N_rows, int K, int fmt, uint32_t *status, void *stream);

/*
 * Test support: the prefill band's routing compaction.  Routed rows (t, j)
 * with a valid id are grouped by expert (ascending), then token, then slot:
 * perm[r] = t*top_k + j for grouped row r, and expert_offset[e] ..
 * expert_offset[e+1] delimit expert e's rows (expert_offset has E+1
 * entries).  perm has M*top_k entries; those past expert_offset[E] are -1.
 * Uses `workspace` of moe_fp4_debug_route_workspace_bytes(M, E, top_k)
 * bytes.  E <= 4096.
 */
MOE_FP4_API int moe_fp4_debug_route(const int32_t *topk_ids, int M, int E, int top_k, int32_t *perm,
                                    int32_t *expert_offset, void *workspace, size_t workspace_bytes, void *stream);
MOE_FP4_API size_t moe_fp4_debug_route_workspace_bytes(int M, int E, int top_k);
/*
 * Test support: the same compaction as the layers of at most 8192 routing
 * entries compute it (one CTA; each expert's rows in the order its entries
 * won a shared-memory counter, not necessarily token order).  Same arguments
 * and outputs as moe_fp4_debug_route; expert_offset is the same, and perm
 * holds the same entries per expert.  MOE_FP4_EUNSUPPORTED for
 * M * top_k > 8192.
 */
MOE_FP4_API int moe_fp4_debug_route_small(const int32_t *topk_ids, int M, int E, int top_k, int32_t *perm,
                                          int32_t *expert_offset, void *workspace, size_t workspace_bytes,
                                          void *stream);

/*
 * Test support: the prefill band's NVFP4 activation quantiser on FP32 rows
 * in[rows][K] (K % 16 == 0): q [rows][K/2] packed E2M1 (low nibble = even
 * element), s [rows][K/16] E4M3 scale bytes, G [rows] FP32 multipliers, by
 *   G = amax/(6*448) (1 for an all-zero row), s = e4m3_rn_satfinite(bmax/(6G)),
 *   q = e2m1_rn_satfinite(a/(s*G)) (0 where s*G == 0),
 * each step an IEEE FP32 operation.
 */
MOE_FP4_API int moe_fp4_debug_quant_rows(const float *in, int rows, int K, uint8_t *q, uint8_t *s, float *G,
                                         void *stream);

/*
 * Test support: the MXFP8 activation quantiser of the W4A8-MX variant on
 * rows x K FP32 values in device memory (K % 32 == 0): q [rows][K] E4M3
 * bytes (16-byte aligned), s [rows][K/32] UE8M0 bytes.  Per 32-block the
 * scale is 2^ceil(log2(amax/448)) (2^0 for an all-zero block, exponent
 * clamped to [-127, 127]) and each element e4m3_rn(a / scale); the sign of a
 * value that rounds to zero is kept.  The pages name MXFP8 activations with
 * UE8M0 scales per 32 (b12x PR #22, "rp-native tiny-decode kernel for
 * w4a8_mx (M=1)"; flashinfer PR #4285, scale_format_e8m0_k32) without the
 * scale rule; this is the MX weight rule with 448 in place of 6.
 * MOE_FP4_EINVAL for null or misaligned pointers, MOE_FP4_EUNSUPPORTED for
 * K % 32 != 0.
 */
MOE_FP4_API int moe_fp4_debug_quant_mxfp8_rows(const float *in, int rows, int K, uint8_t *q, uint8_t *s,
                                               void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP4_H */
