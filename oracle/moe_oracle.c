/*
 * Oracle for the fused FP4-weight MoE layer: plain, slow, FP64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * What it computes (the plain definition of the layer):
 *   - E2M1 element: sign * {0, .5, 1, 1.5, 2, 3, 4, 6}[code & 7]
 *     (the pages name "native E2M1 experts" and "fp4 nibbles" but print no
 *     table; the grid is the OCP E2M1 definition: 1 sign, 2 exponent bits
 *     with bias 1, 1 mantissa bit, exponent 0 subnormal).
 *   - Block scales: MXFP4 = UE8M0 byte e -> 2^(e-127) (255 is NaN) per 32
 *     K-elements; NVFP4 = E4M3 byte per 16 K-elements times an FP32
 *     per-tensor multiplier (b12x PR #459, "Reduce NVFP4-CSF scale
 *     reconstruction overhead": FP32 calibration kept beside the scale bytes;
 *     flashinfer PR #4285 "sync SM12x NVFP4 fused-MoE kernels":
 *     scale_format_e8m0_k32 for the MX case).
 *   - FC1: gate and up dot products of the token's activation with the
 *     expert's rows; SiLU(gate) * up; FC2 (down); router-weighted sum over
 *     the token's top-k slots (b12x PR #22, "rp-native tiny-decode kernel
 *     for w4a8_mx (M=1)", section What: FC1 gate+up dots into an fp32
 *     intermediate, FC2 inline SiLU and router-weighted scatter-add into the
 *     bf16 output, activations stay BF16).
 *   - A slot whose expert id is < 0 or >= E contributes exactly zero and is
 *     never dereferenced (b12x PR #311, conversation: invalid routes carry an
 *     exact-zero effective weight; caller tensors are not mutated).
 *   - Prefill band mirror: activations quantised per row to NVFP4 with an
 *     FP32 row multiplier, then the same FP64 layer from the dequantised
 *     values (flashinfer PR #4285: W4A4 NVFP4 prefill with a fast FP4
 *     quantiser restricted to gated activations).
 *   - W4A8-MX mirror: MXFP4 weights with activations quantised to MXFP8
 *     (E4M3 elements, a UE8M0 scale per 32), then the same FP64 layer.
 *   - Non-gated experts with the squared ReLU: FC1 of I rows, h = max(u, 0)^2.
 *
 * Build: plain C99, -O2 -fno-fast-math -ffp-contract=off, optional OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MXFP4 0
#define ORACLE_NVFP4 1

/* ---------------------------------------------------------------- formats */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. */
double moe_oracle_e2m1(unsigned code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7u];
    return (code & 8u) ? -v : v;
}

/* UE8M0: 2^(e-127); 0xFF encodes NaN. */
double moe_oracle_ue8m0(unsigned b)
{
    b &= 0xFFu;
    if (b == 0xFFu) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* E4M3 (FN variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities. */
double moe_oracle_e4m3(unsigned b)
{
    b &= 0xFFu;
    int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

double moe_oracle_scale(int fmt, unsigned b)
{
    return fmt == ORACLE_MXFP4 ? moe_oracle_ue8m0(b) : moe_oracle_e4m3(b);
}

static int block_of(int fmt) { return fmt == ORACLE_MXFP4 ? 32 : 16; }

static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Element (r, k) of one projection stored as nibbles [rows][K/2] and scale
 * bytes [rows][K/B], times the FP32 multiplier g (1 for MXFP4). */
static double weight_at(const uint8_t *nib, const uint8_t *sc, int K, int fmt, double g, int r, int k)
{
    int B = block_of(fmt);
    uint8_t byte = nib[(size_t)r * (K / 2) + k / 2];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    double s = moe_oracle_scale(fmt, sc[(size_t)r * (K / B) + k / B]);
    return moe_oracle_e2m1(code) * s * g;
}

/* Dequantise `rows` rows of one projection into out[rows][K] (FP64). */
void moe_oracle_dequant(const uint8_t *nib, const uint8_t *sc, int rows, int K, int fmt, double g, double *out)
{
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < K; ++k) out[(size_t)r * K + k] = weight_at(nib, sc, K, fmt, g, r, k);
}

/* ---------------------------------------------------------------- layer */

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* The gated activation applied to FC1's (gate, up) pair.  SiLU is the
 * layer's own (tiny-decode PR, What); the SM12x sync PR's kernels also take
 * "gelu_tanh" and "swigluoai_uninterleave" with parameters alpha, beta
 * (default 1.0) and limit:
 *   GELU, tanh form:  h = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) u
 *   SwiGLU-OAI:       g' = min(g, limit), u' = min(max(u, -limit), limit),
 *                     h = (u' + beta) g' sigmoid(alpha g')                 */
#define ORACLE_ACT_SILU 0
#define ORACLE_ACT_GELU_TANH 1
#define ORACLE_ACT_SWIGLUOAI 2
typedef struct {
    int kind;
    double alpha, beta, limit;
} oracle_act;

static double gated_other(double gate, double up, const oracle_act *a)
{
    if (a->kind == ORACLE_ACT_GELU_TANH) {
        double c = sqrt(2.0 / acos(-1.0));
        return 0.5 * gate * (1.0 + tanh(c * (gate + 0.044715 * gate * gate * gate))) * up;
    }
    double g = gate < a->limit ? gate : a->limit;
    double u = up < -a->limit ? -a->limit : (up > a->limit ? a->limit : up);
    return (u + a->beta) * g / (1.0 + exp(-a->alpha * g));
}

/* h_n = act(x . W13[e][n], x . W13[e][I+n]) for one intermediate index n < I
 * (SiLU(gate) * up by default). */
static double expert_fc1_row(const double *x, const uint8_t *w13, const uint8_t *s13, const float *g13, int e,
                             int H, int I, int fmt, const oracle_act *act, int n)
{
    int B = block_of(fmt);
    const uint8_t *nib = w13 + (size_t)e * 2 * I * (H / 2);
    const uint8_t *sc = s13 + (size_t)e * 2 * I * (H / B);
    double gg = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 0] : 1.0;
    double gu = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 1] : 1.0;
    double gate = 0.0, up = 0.0;
    for (int k = 0; k < H; ++k) {
        gate += x[k] * weight_at(nib, sc, H, fmt, gg, n, k);
        up += x[k] * weight_at(nib, sc, H, fmt, gu, I + n, k);
    }
    if (act->kind == ORACLE_ACT_SILU) return silu(gate) * up;
    return gated_other(gate, up, act);
}

/* h[n] for every n < I. */
static void expert_fc1(const double *x, const uint8_t *w13, const uint8_t *s13, const float *g13, int e, int H,
                       int I, int fmt, const oracle_act *act, double *h)
{
    for (int n = 0; n < I; ++n) h[n] = expert_fc1_row(x, w13, s13, g13, e, H, I, fmt, act, n);
}

/* y_m = W2[e][m] . h for one output row m < H. */
static double expert_fc2_row(const double *h, const uint8_t *w2, const uint8_t *s2, const float *g2, int e, int H,
                             int I, int fmt, int m)
{
    int B = block_of(fmt);
    const uint8_t *nib = w2 + (size_t)e * H * (I / 2);
    const uint8_t *sc = s2 + (size_t)e * H * (I / B);
    double gd = fmt == ORACLE_NVFP4 ? (double)g2[e] : 1.0;
    double acc = 0.0;
    for (int n = 0; n < I; ++n) acc += weight_at(nib, sc, I, fmt, gd, m, n) * h[n];
    return acc;
}

/* y[m] for every m < H. */
static void expert_fc2(const double *h, const uint8_t *w2, const uint8_t *s2, const float *g2, int e, int H, int I,
                       int fmt, double *y)
{
    for (int m = 0; m < H; ++m) y[m] = expert_fc2_row(h, w2, s2, g2, e, H, I, fmt, m);
}

/* A routing id names an expert only inside [0, E); any other id is an
 * invalid route with an exact-zero contribution (never dereferenced). */
static int valid_route(int e, int E) { return e >= 0 && e < E; }

/* Full layer for the tokens listed in `tokens` (n_tok entries; NULL = all M
 * tokens in order), activation `act_kind` with parameters alpha, beta, limit
 * (SwiGLU-OAI only).  out is [n_tok][H] FP64.  Returns 0 on success.
 *
 *   out[t][m] = sum over valid slots j of w[t][j] * (W2[e] . h_tj)[m],
 *   h_tj[n]   = act(x_t . W13[e][n], x_t . W13[e][I+n]),  e = ids[t][j].
 *
 * With OpenMP the work is spread over (token, slot, intermediate row) for
 * FC1 and over (token, output row) for FC2; each sum runs in the same order
 * as with one thread (K index, then intermediate index, then slot), so the
 * result does not depend on the thread count. */
int moe_oracle_forward_act(const uint16_t *x_bf16, const uint8_t *w13, const uint8_t *s13, const float *g13,
                           const uint8_t *w2, const uint8_t *s2, const float *g2, const int32_t *topk_ids,
                           const float *topk_w, int M, int E, int H, int I, int top_k, int fmt, const int32_t *tokens,
                           int n_tok, double *out, int nthreads, int act_kind, double alpha, double beta,
                           double limit)
{
    oracle_act act = {act_kind, alpha, beta, limit};
    if (act_kind < ORACLE_ACT_SILU || act_kind > ORACLE_ACT_SWIGLUOAI) return 1;
    if (M < 0 || E <= 0 || H <= 0 || I <= 0 || top_k <= 0) return 1;
    if (fmt != ORACLE_MXFP4 && fmt != ORACLE_NVFP4) return 1;
    if (H % block_of(fmt) || I % block_of(fmt)) return 1;
    if (!tokens) n_tok = M;
    double *x = (double *)malloc(sizeof(double) * ((size_t)n_tok * H + 1));
    double *h = (double *)malloc(sizeof(double) * ((size_t)n_tok * top_k * I + 1));
    if (!x || !h) {
        free(x);
        free(h);
        return 2;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    /* the activations, exactly, as FP64 */
    for (int i = 0; i < n_tok; ++i) {
        int t = tokens ? tokens[i] : i;
        for (int k = 0; k < H; ++k) x[(size_t)i * H + k] = bf16_to_double(x_bf16[(size_t)t * H + k]);
    }
    /* FC1 and the activation for every valid (token, slot) */
    long n1 = (long)n_tok * top_k * I;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (long u = 0; u < n1; ++u) {
        int i = (int)(u / ((long)top_k * I)), j = (int)(u / I % top_k), n = (int)(u % I);
        int t = tokens ? tokens[i] : i;
        int e = topk_ids[(size_t)t * top_k + j];
        if (!valid_route(e, E)) continue;
        h[u] = expert_fc1_row(x + (size_t)i * H, w13, s13, g13, e, H, I, fmt, &act, n);
    }
    /* FC2 and the router-weighted sum over the slots, per output element */
    long n2 = (long)n_tok * H;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (long v = 0; v < n2; ++v) {
        int i = (int)(v / H), m = (int)(v % H);
        int t = tokens ? tokens[i] : i;
        const int32_t *ids = topk_ids + (size_t)t * top_k;
        const float *tw = topk_w + (size_t)t * top_k;
        double o = 0.0; /* overwrite: out = the sum over valid slots */
        for (int j = 0; j < top_k; ++j) {
            int e = ids[j];
            if (!valid_route(e, E)) continue; /* invalid route: exact-zero contribution */
            double w = (double)tw[j];
            o += w * expert_fc2_row(h + ((size_t)i * top_k + j) * I, w2, s2, g2, e, H, I, fmt, m);
        }
        out[v] = o;
    }
    free(x);
    free(h);
    (void)nthreads;
    return 0;
}

/* The layer with its own activation (SiLU). */
int moe_oracle_forward(const uint16_t *x_bf16, const uint8_t *w13, const uint8_t *s13, const float *g13,
                       const uint8_t *w2, const uint8_t *s2, const float *g2, const int32_t *topk_ids,
                       const float *topk_w, int M, int E, int H, int I, int top_k, int fmt, const int32_t *tokens,
                       int n_tok, double *out, int nthreads)
{
    return moe_oracle_forward_act(x_bf16, w13, s13, g13, w2, s2, g2, topk_ids, topk_w, M, E, H, I, top_k, fmt, tokens,
                                  n_tok, out, nthreads, ORACLE_ACT_SILU, 0.0, 0.0, 0.0);
}

/* FC1 stage alone for one (token, expert): gate[n], up[n] for n < I. */
int moe_oracle_fc1(const uint16_t *x_row, const uint8_t *w13, const uint8_t *s13, const float *g13, int e, int H,
                   int I, int fmt, double *gate, double *up)
{
    int B = block_of(fmt);
    const uint8_t *nib = w13 + (size_t)e * 2 * I * (H / 2);
    const uint8_t *sc = s13 + (size_t)e * 2 * I * (H / B);
    double gg = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 0] : 1.0;
    double gu = fmt == ORACLE_NVFP4 ? (double)g13[2 * e + 1] : 1.0;
    for (int n = 0; n < I; ++n) {
        double a = 0.0, b = 0.0;
        for (int k = 0; k < H; ++k) {
            double xv = bf16_to_double(x_row[k]);
            a += xv * weight_at(nib, sc, H, fmt, gg, n, k);
            b += xv * weight_at(nib, sc, H, fmt, gu, I + n, k);
        }
        gate[n] = a;
        up[n] = b;
    }
    return 0;
}

/* ------------------------------------------------- prefill activation quantiser
 *
 * Row-wise NVFP4 quantisation in IEEE FP32 (every operation correctly
 * rounded, no contraction):
 *   amax = max|a|;  G = amax / (6*448)  (G = 1 if amax == 0)
 *   per 16-block:   s = e4m3_rn_satfinite(amax_blk / (6*G))
 *   per element:    q = e2m1_rn_satfinite(a / (s*G))  (q = 0 if s*G == 0)
 */

/* Round a non-negative finite float to the E4M3 grid, nearest-even,
 * saturating at 448.  Returns the byte (sign bit clear). */
static uint8_t e4m3_from_float_pos(float v)
{
    if (!(v > 0.0f)) return 0;
    if (v >= 448.0f) return 0x7E; /* 1111.110 = 448 */
    /* scan all 127 finite non-negative codes for the nearest, ties to even code */
    double dv = (double)v;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(moe_oracle_e4m3((unsigned)c) - dv);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            bestd = d;
            best = c;
        }
    }
    return (uint8_t)best;
}

/* Round to the E2M1 grid, nearest-even on the code, saturating at +-6.
 * Like IEEE rounding it keeps the input's sign, so a negative value that
 * rounds to zero gives -0 (code 8).  Returns the 4-bit code. */
static uint8_t e2m1_from_float(float v)
{
    double dv = fabs((double)v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(moe_oracle_e2m1((unsigned)c) - dv);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            bestd = d;
            best = c;
        }
    }
    if (signbit(v)) best |= 8; /* the sign survives rounding: small negatives give -0 */
    return (uint8_t)best;
}

uint8_t moe_oracle_e4m3_round(float v) { return e4m3_from_float_pos(v); }
uint8_t moe_oracle_e2m1_round(float v) { return e2m1_from_float(v); }

/* Quantise one row a[K] (K % 16 == 0): q[K/2] packed nibbles (low nibble =
 * even index), s[K/16] E4M3 bytes, *G the FP32 multiplier. */
void moe_oracle_quant_nvfp4_row(const float *a, int K, uint8_t *q, uint8_t *s, float *G)
{
    volatile float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
        float v = fabsf(a[k]);
        if (v > amax) amax = v;
    }
    volatile float six448 = 6.0f * 448.0f;
    volatile float g = amax / six448;
    if (amax == 0.0f) g = 1.0f;
    *G = g;
    volatile float six_g = 6.0f * g;
    for (int b = 0; b < K / 16; ++b) {
        volatile float bmax = 0.0f;
        for (int k = 0; k < 16; ++k) {
            float v = fabsf(a[b * 16 + k]);
            if (v > bmax) bmax = v;
        }
        volatile float sf = bmax / six_g;
        uint8_t sb = e4m3_from_float_pos(sf);
        s[b] = sb;
        volatile float sdec = (float)moe_oracle_e4m3(sb);
        volatile float sg = sdec * g;
        for (int k = 0; k < 16; k += 2) {
            uint8_t c0 = 0, c1 = 0;
            if (sg != 0.0f) {
                volatile float r0 = a[b * 16 + k] / sg;
                volatile float r1 = a[b * 16 + k + 1] / sg;
                c0 = e2m1_from_float(r0);
                c1 = e2m1_from_float(r1);
            }
            q[(b * 16 + k) / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

/* Round an FP32 value to the nearest BF16 (ties to even), returned as FP32.
 * The prefill band stages h = SiLU(gate)*up in BF16 between FC1 and the h
 * quantiser; the mirror takes the same rounding from an FP32 value. */
static float bf16_round(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) return v; /* inf / nan unchanged */
    uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7fffu + lsb) & 0xffff0000u;
    memcpy(&v, &u, 4);
    return v;
}

/* Dequantise a quantised row back to FP64: q * s * G. */
static void dequant_nvfp4_row(const uint8_t *q, const uint8_t *s, float G, int K, double *out)
{
    for (int k = 0; k < K; ++k) {
        uint8_t byte = q[k / 2];
        unsigned code = (k & 1) ? (byte >> 4) : (byte & 0xF);
        out[k] = moe_oracle_e2m1(code) * moe_oracle_e4m3(s[k / 16]) * (double)G;
    }
}

/* Prefill band (mirrored quantisation), for the tokens listed (NULL = all):
 *   x_q = quant(x_t); for each valid slot: g,u = FC1(dequant(x_q)) in FP64;
 *   h = act(g, u) (SiLU(g)*u by default) rounded to FP32, then to BF16;
 *   h_q = quant(h);
 *   y = FC2(dequant(h_q));
 *   out_t = sum_j w_j y.
 * Also returns (optionally) the quantised x rows of the listed tokens. */
int moe_oracle_forward_prefill_act(const uint16_t *x_bf16, const uint8_t *w13, const uint8_t *s13,
                                   const float *g13, const uint8_t *w2, const uint8_t *s2, const float *g2,
                                   const int32_t *topk_ids, const float *topk_w, int M, int E, int H, int I,
                                   int top_k, int fmt, const int32_t *tokens, int n_tok, double *out,
                                   uint8_t *xq_out, uint8_t *xs_out, float *xg_out, int nthreads, int act_kind,
                                   double alpha, double beta, double limit)
{
    oracle_act act = {act_kind, alpha, beta, limit};
    if (act_kind < ORACLE_ACT_SILU || act_kind > ORACLE_ACT_SWIGLUOAI) return 1;
    if (fmt != ORACLE_NVFP4 && fmt != ORACLE_MXFP4) return 1;
    if (H % block_of(fmt) || I % block_of(fmt) || H % 16 || I % 16) return 1;
    if (!tokens) n_tok = M;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        float *xf = (float *)malloc(sizeof(float) * (size_t)H);
        uint8_t *xq = (uint8_t *)malloc((size_t)H / 2);
        uint8_t *xs = (uint8_t *)malloc((size_t)H / 16);
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        float *hf = (float *)malloc(sizeof(float) * (size_t)I);
        uint8_t *hq = (uint8_t *)malloc((size_t)I / 2);
        uint8_t *hs = (uint8_t *)malloc((size_t)I / 16);
        double *hd = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < n_tok; ++i) {
            int t = tokens ? tokens[i] : i;
            for (int k = 0; k < H; ++k) xf[k] = (float)bf16_to_double(x_bf16[(size_t)t * H + k]);
            float xG;
            moe_oracle_quant_nvfp4_row(xf, H, xq, xs, &xG);
            if (xq_out) memcpy(xq_out + (size_t)i * (H / 2), xq, (size_t)H / 2);
            if (xs_out) memcpy(xs_out + (size_t)i * (H / 16), xs, (size_t)H / 16);
            if (xg_out) xg_out[i] = xG;
            dequant_nvfp4_row(xq, xs, xG, H, xd);
            double *o = out + (size_t)i * H;
            for (int m = 0; m < H; ++m) o[m] = 0.0;
            for (int j = 0; j < top_k; ++j) {
                int e = topk_ids[(size_t)t * top_k + j];
                if (e < 0 || e >= E) continue;
                expert_fc1(xd, w13, s13, g13, e, H, I, fmt, &act, h);
                for (int n = 0; n < I; ++n) hf[n] = bf16_round((float)h[n]);
                float hG;
                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);
                dequant_nvfp4_row(hq, hs, hG, I, hd);
                expert_fc2(hd, w2, s2, g2, e, H, I, fmt, y);
                double w = (double)topk_w[(size_t)t * top_k + j];
                for (int m = 0; m < H; ++m) o[m] += w * y[m];
            }
        }
        free(xf); free(xq); free(xs); free(xd); free(h); free(hf); free(hq); free(hs); free(hd); free(y);
    }
    (void)nthreads;
    return 0;
}

/* The prefill band with the layer's own activation (SiLU). */
int moe_oracle_forward_prefill(const uint16_t *x_bf16, const uint8_t *w13, const uint8_t *s13, const float *g13,
                               const uint8_t *w2, const uint8_t *s2, const float *g2, const int32_t *topk_ids,
                               const float *topk_w, int M, int E, int H, int I, int top_k, int fmt,
                               const int32_t *tokens, int n_tok, double *out, uint8_t *xq_out, uint8_t *xs_out,
                               float *xg_out, int nthreads)
{
    return moe_oracle_forward_prefill_act(x_bf16, w13, s13, g13, w2, s2, g2, topk_ids, topk_w, M, E, H, I, top_k,
                                          fmt, tokens, n_tok, out, xq_out, xs_out, xg_out, nthreads,
                                          ORACLE_ACT_SILU, 0.0, 0.0, 0.0);
}

/* --------------------------------------------- non-gated experts (ReLU^2) */

/*
 * Non-gated experts with the squared ReLU ("relu2" of the SM12x sync PR,
 * flashinfer PR #4285, which keeps the exact activation quantiser for it
 * because its squared outputs are not a gated product): FC1 has I rows,
 * w1 [E][I][H/2] with s1 [E][I][H/B] (and for NVFP4 one multiplier g1[e]),
 *   h[n] = max(x . W1[e][n], 0)^2
 * then FC2 and the router-weighted sum as for the gated layer.  For the
 * tokens listed (NULL = all M); out is [n_tok][H] FP64.                     */
int moe_oracle_forward_relu2(const uint16_t *x_bf16, const uint8_t *w1, const uint8_t *s1, const float *g1,
                             const uint8_t *w2, const uint8_t *s2, const float *g2, const int32_t *topk_ids,
                             const float *topk_w, int M, int E, int H, int I, int top_k, int fmt,
                             const int32_t *tokens, int n_tok, double *out, int nthreads)
{
    if (fmt != ORACLE_NVFP4 && fmt != ORACLE_MXFP4) return 1;
    int B = block_of(fmt);
    if (H % B || I % B) return 1;
    if (!tokens) n_tok = M;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < n_tok; ++i) {
            int t = tokens ? tokens[i] : i;
            for (int k = 0; k < H; ++k) x[k] = bf16_to_double(x_bf16[(size_t)t * H + k]);
            double *o = out + (size_t)i * H;
            for (int m = 0; m < H; ++m) o[m] = 0.0;
            for (int j = 0; j < top_k; ++j) {
                int e = topk_ids[(size_t)t * top_k + j];
                if (e < 0 || e >= E) continue;
                const uint8_t *nib = w1 + (size_t)e * I * (H / 2);
                const uint8_t *sc = s1 + (size_t)e * I * (H / B);
                double g = fmt == ORACLE_NVFP4 ? (double)g1[e] : 1.0;
                for (int n = 0; n < I; ++n) {
                    double u = 0.0;
                    for (int k = 0; k < H; ++k) u += x[k] * weight_at(nib, sc, H, fmt, g, n, k);
                    double r = u > 0.0 ? u : 0.0;
                    h[n] = r * r;
                }
                expert_fc2(h, w2, s2, g2, e, H, I, fmt, y);
                double w = (double)topk_w[(size_t)t * top_k + j];
                for (int m = 0; m < H; ++m) o[m] += w * y[m];
            }
        }
        free(x); free(h); free(y);
    }
    (void)nthreads;
    return 0;
}

/* ------------------------------------------- W4A8-MX activations (MXFP8) */

/*
 * MXFP8 quantiser of one row a[K] (K % 32 == 0): E4M3 elements with one
 * UE8M0 scale per 32 K-elements, the activation format of the W4A8-MX
 * variant (b12x PR #22, "rp-native tiny-decode kernel for w4a8_mx (M=1)":
 * MXFP8 activations on the prefill side; flashinfer PR #4285:
 * scale_format_e8m0_k32).  The pages do not print the rule; the reading
 * follows the MX weight recipe of the synthetic checkpoints with E4M3's
 * largest finite value 448 in place of E2M1's 6:
 *   per 32-block:  e = ceil(log2(amax_blk / 448))  (e = 0 if amax_blk == 0),
 *                  clamped to [-127, 127]; scale byte e + 127
 *   per element:   q = e4m3_rn(a / 2^e), |a / 2^e| <= 448 by construction
 * The sign survives rounding (a small negative value gives -0, byte 0x80).
 * q[K] E4M3 bytes, s[K/32] UE8M0 bytes.
 */
void moe_oracle_quant_mxfp8_row(const float *a, int K, uint8_t *q, uint8_t *s)
{
    for (int b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int k = 0; k < 32; ++k) {
            double v = fabs((double)a[b * 32 + k]);
            if (v > amax) amax = v;
        }
        int e = 0;
        if (amax > 0.0) {
            int ex;
            double m = frexp(amax / 448.0, &ex); /* amax/448 = m * 2^ex, m in [0.5, 1) */
            e = (m == 0.5) ? ex - 1 : ex;         /* ceil(log2(amax/448)) */
        }
        if (e < -127) e = -127;
        if (e > 127) e = 127;
        s[b] = (uint8_t)(e + 127);
        double scale = ldexp(1.0, e);
        for (int k = 0; k < 32; ++k) {
            float v = a[b * 32 + k];
            float r = (float)((double)v / scale); /* a power-of-two division: exact unless it underflows */
            uint8_t c = e4m3_from_float_pos(fabsf(r));
            if (signbit(v)) c |= 0x80;
            q[b * 32 + k] = c;
        }
    }
}

/* Dequantise an MXFP8 row back to FP64: e4m3(q) * 2^(s - 127). */
static void dequant_mxfp8_row(const uint8_t *q, const uint8_t *s, int K, double *out)
{
    for (int k = 0; k < K; ++k) {
        double v = moe_oracle_e4m3(q[k] & 0x7F);
        if (q[k] & 0x80) v = -v;
        out[k] = v * ldexp(1.0, (int)s[k / 32] - 127);
    }
}

/* W4A8-MX layer (MXFP4 weights, MXFP8 activations, mirrored), for the
 * tokens listed (NULL = all):
 *   x_q = mxfp8(x_t); for each valid slot: g,u = FC1(dequant(x_q)) in FP64;
 *   h = act(g, u) rounded to FP32, then to BF16 (staged like the NVFP4
 *   prefill band's h); h_q = mxfp8(h); y = FC2(dequant(h_q));
 *   out_t = sum_j w_j y.                                                    */
int moe_oracle_forward_w4a8_act(const uint16_t *x_bf16, const uint8_t *w13, const uint8_t *s13,
                                const uint8_t *w2, const uint8_t *s2, const int32_t *topk_ids, const float *topk_w,
                                int M, int E, int H, int I, int top_k, const int32_t *tokens, int n_tok,
                                double *out, int nthreads, int act_kind, double alpha, double beta, double limit)
{
    oracle_act act = {act_kind, alpha, beta, limit};
    if (act_kind < ORACLE_ACT_SILU || act_kind > ORACLE_ACT_SWIGLUOAI) return 1;
    if (H % 32 || I % 32) return 1;
    if (!tokens) n_tok = M;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        float *xf = (float *)malloc(sizeof(float) * (size_t)H);
        uint8_t *xq = (uint8_t *)malloc((size_t)H);
        uint8_t *xs = (uint8_t *)malloc((size_t)H / 32);
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        float *hf = (float *)malloc(sizeof(float) * (size_t)I);
        uint8_t *hq = (uint8_t *)malloc((size_t)I);
        uint8_t *hs = (uint8_t *)malloc((size_t)I / 32);
        double *hd = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < n_tok; ++i) {
            int t = tokens ? tokens[i] : i;
            for (int k = 0; k < H; ++k) xf[k] = (float)bf16_to_double(x_bf16[(size_t)t * H + k]);
            moe_oracle_quant_mxfp8_row(xf, H, xq, xs);
            dequant_mxfp8_row(xq, xs, H, xd);
            double *o = out + (size_t)i * H;
            for (int m = 0; m < H; ++m) o[m] = 0.0;
            for (int j = 0; j < top_k; ++j) {
                int e = topk_ids[(size_t)t * top_k + j];
                if (e < 0 || e >= E) continue;
                expert_fc1(xd, w13, s13, NULL, e, H, I, ORACLE_MXFP4, &act, h);
                for (int n = 0; n < I; ++n) hf[n] = bf16_round((float)h[n]);
                moe_oracle_quant_mxfp8_row(hf, I, hq, hs);
                dequant_mxfp8_row(hq, hs, I, hd);
                expert_fc2(hd, w2, s2, NULL, e, H, I, ORACLE_MXFP4, y);
                double w = (double)topk_w[(size_t)t * top_k + j];
                for (int m = 0; m < H; ++m) o[m] += w * y[m];
            }
        }
        free(xf); free(xq); free(xs); free(xd); free(h); free(hf); free(hq); free(hs); free(hd); free(y);
    }
    (void)nthreads;
    return 0;
}

/* The prefill band's mirror for non-gated experts (squared ReLU): x
 * quantised per token to NVFP4 and dequantised, u = x . W1[e][n] in FP64,
 * h = max(u, 0)^2 rounded to FP32 then BF16 (the same staging as the gated
 * mirror), h quantised per routed row with the same row quantiser and
 * dequantised, then FC2 and the router-weighted sum in FP64.  w1, s1, g1 as
 * for moe_oracle_forward_relu2. */
int moe_oracle_forward_prefill_relu2(const uint16_t *x_bf16, const uint8_t *w1, const uint8_t *s1, const float *g1,
                                     const uint8_t *w2, const uint8_t *s2, const float *g2,
                                     const int32_t *topk_ids, const float *topk_w, int M, int E, int H, int I,
                                     int top_k, int fmt, const int32_t *tokens, int n_tok, double *out,
                                     int nthreads)
{
    if (fmt != ORACLE_NVFP4 && fmt != ORACLE_MXFP4) return 1;
    int B = block_of(fmt);
    if (H % B || I % B || H % 16 || I % 16) return 1;
    if (!tokens) n_tok = M;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        float *xf = (float *)malloc(sizeof(float) * (size_t)H);
        uint8_t *xq = (uint8_t *)malloc((size_t)H / 2);
        uint8_t *xs = (uint8_t *)malloc((size_t)H / 16);
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        float *hf = (float *)malloc(sizeof(float) * (size_t)I);
        uint8_t *hq = (uint8_t *)malloc((size_t)I / 2);
        uint8_t *hs = (uint8_t *)malloc((size_t)I / 16);
        double *hd = (double *)malloc(sizeof(double) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < n_tok; ++i) {
            int t = tokens ? tokens[i] : i;
            for (int k = 0; k < H; ++k) xf[k] = (float)bf16_to_double(x_bf16[(size_t)t * H + k]);
            float xG;
            moe_oracle_quant_nvfp4_row(xf, H, xq, xs, &xG);
            dequant_nvfp4_row(xq, xs, xG, H, xd);
            double *o = out + (size_t)i * H;
            for (int m = 0; m < H; ++m) o[m] = 0.0;
            for (int j = 0; j < top_k; ++j) {
                int e = topk_ids[(size_t)t * top_k + j];
                if (e < 0 || e >= E) continue;
                const uint8_t *nib = w1 + (size_t)e * I * (H / 2);
                const uint8_t *sc = s1 + (size_t)e * I * (H / B);
                double g = fmt == ORACLE_NVFP4 ? (double)g1[e] : 1.0;
                for (int n = 0; n < I; ++n) {
                    double u = 0.0;
                    for (int k = 0; k < H; ++k) u += xd[k] * weight_at(nib, sc, H, fmt, g, n, k);
                    double r = u > 0.0 ? u : 0.0;
                    hf[n] = bf16_round((float)(r * r));
                }
                float hG;
                moe_oracle_quant_nvfp4_row(hf, I, hq, hs, &hG);
                dequant_nvfp4_row(hq, hs, hG, I, hd);
                expert_fc2(hd, w2, s2, g2, e, H, I, fmt, y);
                double w = (double)topk_w[(size_t)t * top_k + j];
                for (int m = 0; m < H; ++m) o[m] += w * y[m];
            }
        }
        free(xf); free(xq); free(xs); free(xd); free(hf); free(hq); free(hs); free(hd); free(y);
    }
    (void)nthreads;
    return 0;
}

/* ------------------------------------------------- routing / compaction */

/* Stable grouping of routed rows by expert: rows (t, j) with a valid id are
 * ordered by expert ascending, then token, then slot.  perm[r] = t*top_k + j
 * for the r-th grouped row; expert_offset[e] .. expert_offset[e+1] are expert
 * e's rows.  Returns the number of valid rows. */
int moe_oracle_route(const int32_t *topk_ids, int M, int E, int top_k, int32_t *perm, int32_t *expert_offset)
{
    int r = 0;
    for (int e = 0; e < E; ++e) {
        expert_offset[e] = r;
        for (int t = 0; t < M; ++t)
            for (int j = 0; j < top_k; ++j)
                if (topk_ids[(size_t)t * top_k + j] == e) perm[r++] = t * top_k + j;
    }
    expert_offset[E] = r;
    return r;
}

int moe_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
