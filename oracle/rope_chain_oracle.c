/*
 * rope_chain_oracle.c -- CPU oracle of the speculative draft's context K/V
 * chain (MuseSparkDSparkModel.precompute_and_store_context_kv).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline legs load this library.  The product path (the CUDA library
 * under rope_chain_gb300/) never calls it and shares no code with it.
 *
 * Sources (web pages; cited by page title and symbol):
 *   [ctx]  "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context"
 *   [rt]   "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft"
 *   [bnd]  "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.common.draft_boundary"
 *
 * The chain is specified bit for bit: every FP32 operation is one IEEE
 * binary32 operation rounded to nearest even, and nothing is contracted
 * ([ctx], module docstring).  This file is built with -ffp-contract=off and
 * without -ffast-math, so each C operator below is exactly one such
 * operation; fmaf() is the one fused multiply-add the pages write.
 *
 * Readings where the pages are silent:
 *   R1  The order of the 8192-wide sum of squares ("row_norm.py" is not on
 *       the pages): thread t < 256 holds columns 2048k + 8t + i (k < 4,
 *       i < 8) as the norms kernel maps them ([ctx] _ContextNormsKernel);
 *       each thread sums its 32 squares in (k, i) order, each warp of 32
 *       threads folds its partials by a xor butterfly (offsets 16, 8, 4, 2,
 *       1), and the 8 warp sums are added left to right.
 *   R2  rsqrt_approx_ftz is a hardware approximation that cannot be
 *       restated without NVIDIA's internals; the inverse RMS here is the
 *       correctly rounded 1 / sqrt(v) (IEEE sqrt, then IEEE divide) with
 *       v = fma(S, 1/width, eps) as the pages write it.
 *   R3  Norm gains scale the output unless the norm is input-scaled (R14):
 *       y = (x * r) * gamma ([bnd] boundary_fragments order); a weightless
 *       norm is y = x * r.
 *   R4  NaN rounds to the canonical bf16 NaN 0x7FFF.
 *   R5  A slot >= num_blocks*block_size, or (with RoPE) a position outside
 *       [0, max_position), skips its row and counts it in *err.
 *   R13 A gain center is added to the weight only when it is non-zero: the
 *       stock norm with center 0 multiplies by the weight itself, so a -0.0
 *       weight keeps its sign ([ctx] _ContextNormsKernel adds it always).
 *   R15 The decode QKV front ([rt] _fused_qkv_projection, _attention,
 *       may_fuse_qkv_front): its output row is [Q | K | V | O-gate] with
 *       q_size = 64 * num_heads and kv_size = 64 * num_kv_heads (the split
 *       _attention makes); the QK-norm of every Q and K head is the same
 *       weightless 64-wide RMSNorm as the context K-norm (same order, same
 *       eps), then GPT-J RoPE on Q and K; K and V go into the cache as the
 *       context store inserts them; V and the gate pass through.  A row whose
 *       slot is past the cache or whose position is outside the table is
 *       counted in *err and inserts nothing; its Q and K are normed but not
 *       rotated when the position is out of range.  A negative slot inserts
 *       nothing and is not an error.
 *   R14 An input-scale weight multiplies the input before the sum of
 *       squares and nothing after it, in the order of [bnd]
 *       boundary_fragments; the hidden norm's output is still rounded to
 *       bf16 before the layer norm reads it.
 *
 * Parity pins: every function here is checked by the "not gpu" tests
 * against closed forms, invariants, brute force or library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define RCO_D 8192
#define RCO_HEAD 64

#if defined(__FLT_EVAL_METHOD__) && __FLT_EVAL_METHOD__ != 0
#error "the oracle needs FLT_EVAL_METHOD == 0 (binary32 arithmetic evaluated in binary32)"
#endif

/* ---------------------------------------------------------------- bf16 */

/* Exact widening of a bf16 bit pattern ([ctx]: bf16x2_to_f32x2,
   load_bf16x8_as_f32). */
float rco_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest even ([ctx]: round_bf16,
   pack_bf16x2_rn, store_bf16x8_rn).  Adding 0x7FFF plus the kept LSB to the
   bit pattern and truncating is RNE for every finite value, subnormals
   included, and carries into Inf on overflow.  NaN -> 0x7FFF (R4). */
uint16_t rco_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)0x7FFFu;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* binary64 -> bf16, round to nearest even directly (no intermediate
   binary32 rounding): used to round the float64 projection reference. */
uint16_t rco_bf16_rn_f64(double d)
{
    if (isnan(d))
        return (uint16_t)0x7FFFu;
    uint16_t sign = signbit(d) ? (uint16_t)0x8000u : (uint16_t)0u;
    double a = fabs(d);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    int e;
    (void)frexp(a, &e);              /* a = m * 2^e, 0.5 <= m < 1 */
    int qe = e - 8;                  /* bf16 keeps 8 significant bits */
    if (qe < -133)
        qe = -133;                   /* subnormal spacing 2^-133 */
    double r = ldexp(nearbyint(ldexp(a, -qe)), qe);
    if (r >= 0x1p128)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;              /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void rco_bf16_rn_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = rco_bf16_rn(in[i]);
}

void rco_bf16_rn_f64_array(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = rco_bf16_rn_f64(in[i]);
}

/* ------------------------------------------------------------- reductions */

/* Fold 32 lane values by a xor butterfly: at each offset o in 16, 8, 4, 2, 1
   lane j becomes q[j] + q[j ^ o] (a warp shuffle-xor reduction); every lane
   ends with the same value because IEEE addition is commutative. */
static float butterfly32(const float *in)
{
    float q[32], n[32];
    memcpy(q, in, sizeof q);
    for (int o = 16; o >= 1; o >>= 1) {
        for (int j = 0; j < 32; ++j)
            n[j] = q[j] + q[j ^ o];
        memcpy(q, n, sizeof q);
    }
    return q[0];
}

/* Sum of squares of one 8192-wide row in the order of reading R1. */
float rco_row_sumsq(const float *v)
{
    float lane[256];
    for (int t = 0; t < 256; ++t) {
        float p = 0.0f;
        for (int k = 0; k < 4; ++k)
            for (int i = 0; i < 8; ++i) {
                float e = v[2048 * k + 8 * t + i];
                float sq = e * e;
                p = p + sq;
            }
        lane[t] = p;
    }
    float s = butterfly32(&lane[0]);
    for (int w = 1; w < 8; ++w) {
        float ws = butterfly32(&lane[32 * w]);
        s = s + ws;
    }
    return s;
}

/* x.pow(2).sum(-1) of one 64-wide key head as [ctx] _sum_squares_64 computes
   it with lane j holding the pair (2j, 2j+1): the even squares and the odd
   squares are each folded by the xor butterfly, then even + odd. */
float rco_head_sumsq(const float *k)
{
    float ev[32], od[32];
    for (int j = 0; j < 32; ++j) {
        ev[j] = k[2 * j] * k[2 * j];
        od[j] = k[2 * j + 1] * k[2 * j + 1];
    }
    float e = butterfly32(ev);
    float o = butterfly32(od);
    return e + o;
}

/* Inverse RMS: 1 / sqrt(fma(S, 1/width, eps)) (R2; the fma and the exact
   power-of-two 1/width are the pages'). */
float rco_inv_rms(float sumsq, float inv_width, float eps)
{
    float v = fmaf(sumsq, inv_width, eps);
    float root = sqrtf(v);
    return 1.0f / root;
}

/* GPT-J rotation of one pair as [ctx] _rope writes it:
   (fma(x, c, -(y*s)), fma(y, c, x*s)). */
void rco_rope(float x, float y, float c, float s, float *xo, float *yo)
{
    float ys = y * s;
    float xs = x * s;
    *xo = fmaf(x, c, -ys);
    *yo = fmaf(y, c, xs);
}

static int pick_threads(int32_t threads)
{
#ifdef _OPENMP
    return threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

int32_t rco_max_threads(void) { return pick_threads(0); }

/* --------------------------------------------------------------- a1 + a2 */

/* out[l, t, :] = bf16(pre_norm_l(bf16(hidden_norm(x[t, :])))) for every
   layer l: [ctx] ContextNorms / _ContextNormsKernel (the hidden norm's
   output rounded to BF16 before the layer norm reads it) and [rt]
   ContextKV._project (the stack over layers).  hidden_w [D] and pre_w [L, D]
   may be NULL (weightless norms).  Each layer's norm is computed from its
   definition, so the per-layer inverse RMS is recomputed per layer.
   Returns 0, or 1 for unsupported arguments. */
int32_t rco_context_norms(const uint16_t *x, int64_t T, int32_t D,
                          const uint16_t *hidden_w, const uint16_t *pre_w,
                          int32_t L, float eps, uint16_t *out, int32_t threads)
{
    if (D != RCO_D || T < 0 || L < 1 || !x || !out)
        return 1;
    const float inv_d = 1.0f / 8192.0f;   /* exact: 2^-13 */
#pragma omp parallel for schedule(static) num_threads(pick_threads(threads))
    for (int64_t t = 0; t < T; ++t) {
        float *v = (float *)malloc(2 * RCO_D * sizeof(float));
        float *z = v + RCO_D;
        const uint16_t *xr = x + t * (int64_t)RCO_D;
        for (int c = 0; c < RCO_D; ++c)
            v[c] = rco_f32(xr[c]);
        /* a1: hidden RMSNorm, rounded to bf16 */
        float r = rco_inv_rms(rco_row_sumsq(v), inv_d, eps);
        for (int c = 0; c < RCO_D; ++c) {
            float y = v[c] * r;
            if (hidden_w)
                y = y * rco_f32(hidden_w[c]);
            z[c] = rco_f32(rco_bf16_rn(y));
        }
        /* a2: each layer's input RMSNorm of z, stacked at [l, t] */
        for (int32_t l = 0; l < L; ++l) {
            float r2 = rco_inv_rms(rco_row_sumsq(z), inv_d, eps);
            uint16_t *o = out + ((int64_t)l * T + t) * RCO_D;
            const uint16_t *g = pre_w ? pre_w + (int64_t)l * RCO_D : NULL;
            for (int c = 0; c < RCO_D; ++c) {
                float y = z[c] * r2;
                if (g)
                    y = y * rco_f32(g[c]);
                o[c] = rco_bf16_rn(y);
            }
        }
        free(v);
    }
    return 0;
}

/* One norm of the chain with every option [ctx] ContextNorms binds
   (ContextNormConstants and the call's eps and gain centers):
     weight       NULL (weightless), else [D] (hidden) or [L, D] (pre);
     fp32         the weight's dtype: 1 FP32, 0 BF16;
     input_scale  1: the weight scales the input before the norm, 0: the
                  norm's output (R3);
     center       the gain center, added to each weight element (R13);
     eps          this norm's own eps. */
typedef struct {
    const void *weight;
    int32_t fp32;
    int32_t input_scale;
    float center;
    float eps;
} rco_norm;

/* gamma_c of the weight row at `offset` (R13: the center is added only when non-zero, so
   that a center of 0 leaves the weight's bits, -0.0 included, unchanged). */
static float norm_gain(const rco_norm *n, int64_t offset, int32_t c)
{
    float g;
    if (n->fp32)
        g = ((const float *)n->weight)[offset + c];
    else
        g = rco_f32(((const uint16_t *)n->weight)[offset + c]);
    if (n->center != 0.0f)
        g = g + n->center;
    return g;
}

/* The RMSNorm of one 8192-wide row v (binary32 values) as [bnd]
   boundary_fragments writes each of its two norms: with an input-scale
   weight u = gamma * v first, else u = v; S = sum of squares of u (R1);
   r = 1 / sqrt(fma(S, 2^-13, eps)) (R2); y = u * r, times gamma when the
   weight scales the output.  `offset` selects the weight row. */
static void norm_row(const float *v, const rco_norm *n, int64_t offset, float *y)
{
    const int weighted = n->weight != NULL;
    const int pre_scale = weighted && n->input_scale;
    float *u = y;                         /* y doubles as the scaled input */
    for (int c = 0; c < RCO_D; ++c)
        u[c] = pre_scale ? norm_gain(n, offset, c) * v[c] : v[c];
    const float r = rco_inv_rms(rco_row_sumsq(u), 1.0f / 8192.0f, n->eps);
    for (int c = 0; c < RCO_D; ++c) {
        float t = u[c] * r;
        if (weighted && !pre_scale)
            t = t * norm_gain(n, offset, c);
        y[c] = t;
    }
}

/* rco_context_norms with every variant of ContextNormConstants: the hidden
   norm (weight [D]) of each row, rounded to bf16, then each layer's input
   norm (weight row l of [L, D]) of that, stacked at out[l, t, :] in bf16.
   Each norm has its own eps, gain center, weight dtype and scale side.
   Returns 0, or 1 for unsupported arguments. */
int32_t rco_context_norms_ex(const uint16_t *x, int64_t T, int32_t D,
                             const rco_norm *hidden, const rco_norm *pre,
                             int32_t L, uint16_t *out, int32_t threads)
{
    if (D != RCO_D || T < 0 || L < 1 || !x || !out || !hidden || !pre)
        return 1;
#pragma omp parallel for schedule(static) num_threads(pick_threads(threads))
    for (int64_t t = 0; t < T; ++t) {
        float *v = (float *)malloc(3 * RCO_D * sizeof(float));
        float *z = v + RCO_D, *y = z + RCO_D;
        const uint16_t *xr = x + t * (int64_t)RCO_D;
        for (int c = 0; c < RCO_D; ++c)
            v[c] = rco_f32(xr[c]);
        /* a1: the hidden norm, its output rounded to bf16 */
        norm_row(v, hidden, 0, y);
        for (int c = 0; c < RCO_D; ++c)
            z[c] = rco_f32(rco_bf16_rn(y[c]));
        /* a2: layer l's input norm of z, stacked at [l, t] */
        for (int32_t l = 0; l < L; ++l) {
            norm_row(z, pre, (int64_t)l * RCO_D, y);
            uint16_t *o = out + ((int64_t)l * T + t) * RCO_D;
            for (int c = 0; c < RCO_D; ++c)
                o[c] = rco_bf16_rn(y[c]);
        }
        free(v);
    }
    return 0;
}

/* ------------------------------------------------------------------- a3 */

/* Float64 reference of the K/V projection ([rt] ContextKV._project:
   torch.bmm(per_layer, W^T)): for the selected rows rows[i] of each layer,
     out[l, i, n]    = sum_k f32(normed[l, rows[i], k]) * f32(W_l[k, n])
     absout[l, i, n] = sum_k |f32(normed[l, rows[i], k]) * f32(W_l[k, n])|
   summed in ascending k in binary64 (each bf16 x bf16 product is exact in
   binary64).  W is [L, D, N] (N contiguous) when w_nd == 0, or [L, N, D]
   (the nn.Linear layout the pages store) when w_nd == 1.  rows == NULL
   selects rows 0..nrows-1.  absout may be NULL.  Returns 0 or 1. */
int32_t rco_kv_project(const uint16_t *normed, const uint16_t *W, int32_t w_nd,
                       int32_t L, int64_t T, int32_t D, int32_t N,
                       const int64_t *rows, int64_t nrows,
                       double *out, double *absout, int32_t threads)
{
    if (!normed || !W || !out || L < 1 || T < 0 || D < 1 || N < 1 || nrows < 0)
        return 1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= T))
            return 1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(pick_threads(threads))
    for (int32_t l = 0; l < L; ++l) {
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t t = rows ? rows[i] : i;
            const uint16_t *a = normed + ((int64_t)l * T + t) * D;
            double *o = out + ((int64_t)l * nrows + i) * N;
            double *ab = absout ? absout + ((int64_t)l * nrows + i) * N : NULL;
            for (int32_t n = 0; n < N; ++n) {
                o[n] = 0.0;
                if (ab)
                    ab[n] = 0.0;
            }
            if (w_nd == 0) {
                const uint16_t *w = W + (int64_t)l * D * N;
                for (int32_t k = 0; k < D; ++k) {
                    double ak = (double)rco_f32(a[k]);
                    const uint16_t *wk = w + (int64_t)k * N;
                    for (int32_t n = 0; n < N; ++n) {
                        double p = ak * (double)rco_f32(wk[n]);
                        o[n] = o[n] + p;
                        if (ab)
                            ab[n] = ab[n] + fabs(p);
                    }
                }
            } else {
                const uint16_t *w = W + (int64_t)l * N * D;
                for (int32_t n = 0; n < N; ++n) {
                    const uint16_t *wn = w + (int64_t)n * D;
                    double acc = 0.0, aacc = 0.0;
                    for (int32_t k = 0; k < D; ++k) {
                        double p = (double)rco_f32(a[k]) * (double)rco_f32(wn[k]);
                        acc = acc + p;
                        aacc = aacc + fabs(p);
                    }
                    o[n] = acc;
                    if (ab)
                        ab[n] = aacc;
                }
            }
        }
    }
    return 0;
}

/* -------------------------------------------------------------- a4 - a8 */

/* The chain after the projection for L layers ([ctx] ContextKvStore and
   _ContextKvStoreKernel; [rt] ContextKV.store):
     for every layer l with slots[l] != NULL and every row t < rows:
       s = slots[l][t]; s < 0 skips the row;
       K-norm of each head h of k[l, t, h, :] (weightless, eps),
       the bf16 key, GPT-J RoPE at positions[t] from cos_sin when it is not
       NULL (cos in columns 0..31, sin in 32..63), the bf16 result;
       cache_l[s / block_size, h, s % block_size, 0:64]   <- the key,
       cache_l[s / block_size, h, s % block_size, 64:128] <- v[l, t, h, :].
   k and v are addressed as base + l*layer_stride + t*row_stride + h*64 + e
   (elements).  caches[l] is a contiguous bf16 [num_blocks, H, block_size,
   128].  Rows skipped under R5 add one to *err (when err != NULL).
   Returns 0, or 1 for unsupported arguments. */
int32_t rco_kv_store(const uint16_t *k, const uint16_t *v,
                     int64_t k_layer_stride, int64_t k_row_stride,
                     int64_t v_layer_stride, int64_t v_row_stride,
                     const int64_t *positions, const int64_t *const *slots,
                     const uint16_t *cos_sin, int64_t max_position,
                     uint16_t *const *caches, int32_t num_blocks,
                     int32_t block_size, int32_t H, int32_t L, float eps,
                     int64_t rows, int32_t *err, int32_t threads)
{
    if (!k || !v || !slots || !caches || H < 1 || L < 1 || rows < 0 ||
        num_blocks < 1 || block_size < 1 || (cos_sin && !positions))
        return 1;
    const int64_t capacity = (int64_t)num_blocks * block_size;
    const float inv_hd = 1.0f / 64.0f;   /* exact: 2^-6 */
    int64_t skipped = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (!slots[l])
            continue;
        if (!caches[l])
            return 1;
#pragma omp parallel for schedule(static) reduction(+ : skipped) num_threads(pick_threads(threads))
        for (int64_t t = 0; t < rows; ++t) {
            int64_t s = slots[l][t];
            if (s < 0)
                continue;
            if (s >= capacity) {
                skipped += 1;
                continue;
            }
            int64_t pos = 0;
            if (cos_sin) {
                pos = positions[t];
                if (pos < 0 || pos >= max_position) {
                    skipped += 1;
                    continue;
                }
            }
            int64_t blk = s / block_size, page = s % block_size;
            for (int32_t h = 0; h < H; ++h) {
                const uint16_t *kh = k + l * k_layer_stride + t * k_row_stride + (int64_t)h * RCO_HEAD;
                const uint16_t *vh = v + l * v_layer_stride + t * v_row_stride + (int64_t)h * RCO_HEAD;
                uint16_t *dst = caches[l] + (((blk * H) + h) * block_size + page) * (2 * RCO_HEAD);
                float kf[RCO_HEAD];
                for (int e = 0; e < RCO_HEAD; ++e)
                    kf[e] = rco_f32(kh[e]);
                /* a5: weightless K-norm, then the bf16 key */
                float r = rco_inv_rms(rco_head_sumsq(kf), inv_hd, eps);
                for (int j = 0; j < RCO_HEAD / 2; ++j) {
                    float y0 = kf[2 * j] * r;
                    float y1 = kf[2 * j + 1] * r;
                    float n0 = rco_f32(rco_bf16_rn(y0));
                    float n1 = rco_f32(rco_bf16_rn(y1));
                    /* a6: GPT-J RoPE on the pair (2j, 2j+1) */
                    if (cos_sin) {
                        float c = rco_f32(cos_sin[pos * RCO_HEAD + j]);
                        float sn = rco_f32(cos_sin[pos * RCO_HEAD + RCO_HEAD / 2 + j]);
                        float xo, yo;
                        rco_rope(n0, n1, c, sn, &xo, &yo);
                        n0 = xo;
                        n1 = yo;
                    }
                    /* a7: the insert; V is copied bit for bit */
                    dst[2 * j] = rco_bf16_rn(n0);
                    dst[2 * j + 1] = rco_bf16_rn(n1);
                }
                memcpy(dst + RCO_HEAD, vh, RCO_HEAD * sizeof(uint16_t));
            }
        }
    }
    if (err)
        *err += (int32_t)skipped;
    return 0;
}

/* ---------------------------------------------------------- decode front */

/* The QKV front after its projection (R15; [rt] _fused_qkv_projection and
   _attention): raw is the bf16 projection [M, Nqkv] of M decode tokens,
   Nqkv = 64 * (2 * num_heads + 2 * num_kv_heads), columns [Q | K | V | gate].
     out[m, Q and K heads] = RoPE(bf16(head * r)), r the head's weightless
                             inverse RMS (rco_head_sumsq order, eps), RoPE at
                             positions[m] from cos_sin when it is not NULL;
     out[m, V and gate]    = raw[m, V and gate];
     cache[s / bs, h, s % bs, 0:64]   = out[m, K head h],
     cache[s / bs, h, s % bs, 64:128] = raw[m, V head h]   for s = slots[m] >= 0;
   a row whose slot is >= num_blocks * block_size or (with a table) whose
   position is outside [0, max_position) adds one to *err and inserts
   nothing (R15).  slots may be NULL (nothing inserted).
   cache is bf16 [num_blocks, num_kv_heads, block_size, 128].  Returns 0, or 1
   for unsupported arguments. */
int32_t rco_qkv_front_post(const uint16_t *raw, int32_t M, int32_t num_heads, int32_t num_kv_heads,
                           const int64_t *positions, const uint16_t *cos_sin, int64_t max_position,
                           const int64_t *slots, uint16_t *cache, int32_t num_blocks,
                           int32_t block_size, float eps, uint16_t *out, int32_t *err)
{
    if (!raw || !out || M < 0 || num_heads < 1 || num_kv_heads < 1 || num_blocks < 1 ||
        block_size < 1 || (cos_sin && !positions) || (slots && !cache))
        return 1;
    const int32_t q_size = RCO_HEAD * num_heads, kv_size = RCO_HEAD * num_kv_heads;
    const int32_t N = 2 * q_size + 2 * kv_size;
    const int64_t capacity = (int64_t)num_blocks * block_size;
    const float inv_hd = 1.0f / 64.0f;
    for (int32_t m = 0; m < M; ++m) {
        const uint16_t *rr = raw + (int64_t)m * N;
        uint16_t *o = out + (int64_t)m * N;
        int64_t pos = 0;
        int bad_pos = 0;
        if (cos_sin) {
            pos = positions[m];
            bad_pos = pos < 0 || pos >= max_position;
        }
        const int rotate = cos_sin != NULL && !bad_pos;
        const int64_t s = slots ? slots[m] : -1;
        const int bad_slot = s >= capacity;
        if ((bad_pos || bad_slot) && err)
            *err += 1;
        const int insert = s >= 0 && !bad_slot && !bad_pos;
        /* Q and K heads: QK-norm, then RoPE */
        for (int32_t h = 0; h < num_heads + num_kv_heads; ++h) {
            const int32_t c0 = h * RCO_HEAD;
            float kf[RCO_HEAD];
            for (int e = 0; e < RCO_HEAD; ++e)
                kf[e] = rco_f32(rr[c0 + e]);
            float r = rco_inv_rms(rco_head_sumsq(kf), inv_hd, eps);
            for (int j = 0; j < RCO_HEAD / 2; ++j) {
                float n0 = rco_f32(rco_bf16_rn(kf[2 * j] * r));
                float n1 = rco_f32(rco_bf16_rn(kf[2 * j + 1] * r));
                if (rotate) {
                    float c = rco_f32(cos_sin[pos * RCO_HEAD + j]);
                    float sn = rco_f32(cos_sin[pos * RCO_HEAD + RCO_HEAD / 2 + j]);
                    float xo, yo;
                    rco_rope(n0, n1, c, sn, &xo, &yo);
                    n0 = xo;
                    n1 = yo;
                }
                o[c0 + 2 * j] = rco_bf16_rn(n0);
                o[c0 + 2 * j + 1] = rco_bf16_rn(n1);
            }
        }
        /* V and the gate pass through */
        memcpy(o + q_size + kv_size, rr + q_size + kv_size, (size_t)(kv_size + q_size) * sizeof(uint16_t));
        if (insert) {
            const int64_t blk = s / block_size, page = s % block_size;
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                uint16_t *dst = cache + ((blk * num_kv_heads + h) * block_size + page) * (2 * RCO_HEAD);
                memcpy(dst, o + q_size + h * RCO_HEAD, RCO_HEAD * sizeof(uint16_t));
                memcpy(dst + RCO_HEAD, rr + q_size + kv_size + h * RCO_HEAD, RCO_HEAD * sizeof(uint16_t));
            }
        }
    }
    return 0;
}
