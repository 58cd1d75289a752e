/*
 * h3qk oracle: a plain, slow, single-threaded CPU statement of the fused
 * QK-prep path of the MiniMax-H3 video VAE decoder and DiT attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA path.
 *
 * Pages this file follows (cited below by the tag in brackets):
 *   [P2] TensorRT-LLM pull request #21485, "cuDNN FP8 attention path for
 *        MiniMax-H3 on SM107 under Ulysses": the Summary's second bullet and
 *        the commits that add the fused QK-norm + RoPE + FP8 cast, its
 *        single-tensor norm_rope_tensor variant, the valid-length exclusion
 *        from the amax and the custom-op aliasing fix.
 *   [P3] vllm-omni pull request #6607, MiniMax-H3 VAE decoder eager
 *        operators: the "Operations" table, row "Q/K normalization + RoPE".
 *   [P5] stable-diffusion.cpp pull request #19, "MiniMax-H3: sage takes the
 *        fused RoPE op, faster video and audio VAE decode": the commits on
 *        the fused q/k/v path of the decoder attention and on the fused
 *        per-head norm (ggml patch 0005).
 *
 * What the pages fix: per-head RMS normalisation of Q and K, a partial
 * rotary embedding, the permute of the packed QKV projection to head-major
 * Q/K/V, and an optional per-tensor e4m3 cast with one amax pass and one
 * cast pass, dynamic or static scales, padded rows left out of the amax.
 * They also fix the precision policy: FP32 accumulation in a fixed reduction
 * order with explicit 16-bit rounding points, bit-exact to an unfused chain
 * [P3 Operations; P5 patch 0005 commit].  They do NOT print the rounding
 * points, the reduction tree, the rotary pairing or the axis split.  Where
 * they are silent this file takes one plain reading and says so in a
 * "Reading:" note beside the step.
 *
 * Arithmetic: every float operation is one IEEE binary32 operation rounded
 * to nearest-even.  The file must be compiled with -ffp-contract=off (no
 * silent multiply-add fusion); the only fused multiply-adds are the explicit
 * fmaf calls of the sine/cosine routine.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Largest H*D of one tensor row and largest rotary_dim / 2 (stack buffers). */
#define H3O_MAX_HD 16384
#define H3O_MAX_PAIRS 128

/* ------------------------------------------------------------------------ */
/* Problem description (the oracle's own; the CUDA path has its own header). */
/* ------------------------------------------------------------------------ */

enum { H3O_FP16 = 1, H3O_BF16 = 2 };
enum { H3O_OUT_16B = 0, H3O_OUT_E4M3 = 1 };
enum { H3O_SCALE_NONE = 0, H3O_SCALE_DYNAMIC = 1, H3O_SCALE_STATIC = 2 };

typedef struct {
    int64_t batch;        /* B: independent items (tiles)                     */
    int64_t seq;          /* S: rows per item; rows r = b*S + s               */
    int64_t valid_len;    /* rows s >= valid_len of every item are skipped    */
    int64_t row_stride;   /* elements between packed QKV rows (>= 3*H*D)      */
    int32_t heads;        /* H                                                */
    int32_t head_dim;     /* D, a multiple of 8, at most 256                  */
    int32_t rotary_dim;   /* R <= D, rotated leading channels                 */
    int32_t n_axes;       /* 1 (1-D positions) or 3 (t,h,w)                   */
    int32_t axis_dims[3]; /* even widths summing to R                         */
    int32_t in_dtype;     /* H3O_FP16 or H3O_BF16                             */
    int32_t out_kind;     /* H3O_OUT_16B or H3O_OUT_E4M3                      */
    int32_t scale_mode;   /* H3O_SCALE_*                                      */
    float eps;            /* RMSNorm epsilon                                  */
    float static_scales[3]; /* descales for STATIC mode (q, k, v)             */
    double theta;         /* rotary base                                      */
    int32_t out_layout;   /* 0: head-major [B, H, S, D]; 1: token-major [B, S, H, D] */
    int32_t pad_;
    const int32_t* valid_lens; /* per-item valid lengths (clamped to [0, S]) or NULL */
} h3o_problem;

/* ------------------------------------------------------------------------ */
/* Number formats, written from the format definitions (IEEE 754 binary16,  */
/* bfloat16 = the upper half of binary32, OCP 8-bit E4M3FN).                */
/* ------------------------------------------------------------------------ */

/* Round |a| (finite, > 0) to a format with `mbits` stored mantissa bits,
 * minimum normal exponent `emin`: returns the integer significand m and the
 * exponent E with value m * 2^(E - mbits); m < 2^mbits means subnormal.
 * Scaling by a power of two is exact and rintf rounds half to even, so this
 * is round-to-nearest-even by construction. */
static void h3o_round_sig(float a, int mbits, int emin, int* E_out, uint32_t* m_out)
{
    int e;
    (void)frexpf(a, &e);         /* a = f * 2^e, f in [0.5, 1)              */
    int E = e - 1;               /* 2^E <= a < 2^(E+1)                      */
    if (E < emin) E = emin;      /* subnormal range keeps the fixed quantum */
    float n = ldexpf(a, mbits - E);   /* exact: a / 2^(E - mbits)           */
    uint32_t m = (uint32_t)rintf(n);
    if (m == (2u << mbits)) {    /* rounded up to the next binade           */
        m = 1u << mbits;
        E += 1;
    }
    *E_out = E;
    *m_out = m;
}

/* binary32 -> binary16, round to nearest even, subnormals kept, overflow to
 * infinity, NaN to a quiet NaN with the sign kept. */
uint16_t h3o_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    float a = fabsf(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0f) return sign;
    int E;
    uint32_t m;
    h3o_round_sig(a, 10, -14, &E, &m);
    if (m < (1u << 10)) return (uint16_t)(sign | m);          /* subnormal */
    if (E > 15) return (uint16_t)(sign | 0x7C00u);             /* overflow  */
    return (uint16_t)(sign | ((uint32_t)(E + 15) << 10) | (m - (1u << 10)));
}

float h3o_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    float v;
    if (ex == 0x1F) v = man ? NAN : INFINITY;
    else if (ex == 0) v = ldexpf((float)man, -24);
    else v = ldexpf((float)(man | 0x400), ex - 25);
    return sign ? -v : v;
}

/* binary32 -> bfloat16 (8-bit exponent, 7 stored mantissa bits), round to
 * nearest even, subnormals kept, overflow to infinity, NaN quiet. */
uint16_t h3o_f32_to_bf16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    float a = fabsf(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0f) return sign;
    int E;
    uint32_t m;
    h3o_round_sig(a, 7, -126, &E, &m);
    if (m < (1u << 7)) return (uint16_t)(sign | m);
    if (E > 127) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | ((uint32_t)(E + 127) << 7) | (m - (1u << 7)));
}

float h3o_bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float v;
    memcpy(&v, &bits, sizeof v);
    return v;
}

/* binary32 -> E4M3FN (bias 7, 3 mantissa bits, no infinity, 0x7F/0xFF NaN),
 * round to nearest even with saturation: every |x| >= 448 (infinity too)
 * gives the largest finite code 0x7E (0xFE when negative). */
uint8_t h3o_f32_to_e4m3(float x)
{
    uint8_t sign = signbit(x) ? 0x80u : 0u;
    if (isnan(x)) return (uint8_t)(sign | 0x7Fu);
    float a = fabsf(x);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7Eu);
    if (a == 0.0f) return sign;
    int E;
    uint32_t m;
    h3o_round_sig(a, 3, -6, &E, &m);
    if (m < 8u) return (uint8_t)(sign | m);                   /* subnormal */
    return (uint8_t)(sign | ((uint32_t)(E + 7) << 3) | (m - 8u));
}

float h3o_e4m3_to_f32(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int ex = (c >> 3) & 0xF;
    int man = c & 7;
    float v;
    if (ex == 0xF && man == 7) v = NAN;
    else if (ex == 0) v = ldexpf((float)man, -9);
    else v = ldexpf((float)(man | 8), ex - 10);
    return sign ? -v : v;
}

static float h3o_widen(int dtype, uint16_t h)
{
    return dtype == H3O_FP16 ? h3o_f16_to_f32(h) : h3o_bf16_to_f32(h);
}

static uint16_t h3o_round16(int dtype, float x)
{
    return dtype == H3O_FP16 ? h3o_f32_to_f16(x) : h3o_f32_to_bf16(x);
}

/* ------------------------------------------------------------------------ */
/* Sine and cosine.  The pages give no formula for the rotary tables; the   */
/* path needs sin and cos of a binary32 angle that a CPU and a GPU can both */
/* evaluate identically, so this is a routine of our own, from two          */
/* published methods:                                                       */
/*  - Cody & Waite, "Software Manual for the Elementary Functions" (1980):  */
/*    additive argument reduction a = j*pi/2 + r with pi/2 split into three */
/*    binary32 parts, each subtraction one fused multiply-add;              */
/*  - the Taylor series of sin (to r^11) and cos (to r^12) on |r| <= pi/4,  */
/*    evaluated in Horner form with fused multiply-adds.                    */
/* Constants (hex binary32 literals):                                       */
/*  2/pi rounded; P1 = pi/2 rounded; P2 = (pi/2 - P1) rounded;              */
/*  P3 = (pi/2 - P1 - P2) rounded; Sn, Cn = +-1/n! rounded.                 */
/* ------------------------------------------------------------------------ */

static const float H3O_TWO_OVER_PI = 0x1.45f306p-1f;
static const float H3O_PIO2_1 = 0x1.921fb6p+0f;
static const float H3O_PIO2_2 = -0x1.777a5cp-25f;
static const float H3O_PIO2_3 = -0x1.ee59dap-50f;

static const float H3O_S3 = -0x1.555556p-3f;   /* -1/3!  */
static const float H3O_S5 = 0x1.111112p-7f;    /* +1/5!  */
static const float H3O_S7 = -0x1.a01a02p-13f;  /* -1/7!  */
static const float H3O_S9 = 0x1.71de3ap-19f;   /* +1/9!  */
static const float H3O_S11 = -0x1.ae6456p-26f; /* -1/11! */
static const float H3O_C2 = -0x1.000000p-1f;   /* -1/2!  */
static const float H3O_C4 = 0x1.555556p-5f;    /* +1/4!  */
static const float H3O_C6 = -0x1.6c16c2p-10f;  /* -1/6!  */
static const float H3O_C8 = 0x1.a01a02p-16f;   /* +1/8!  */
static const float H3O_C10 = -0x1.27e4fcp-22f; /* -1/10! */
static const float H3O_C12 = 0x1.1eed8ep-29f;  /* +1/12! */

void h3o_sincos(float a, float* s_out, float* c_out)
{
    /* Reduction: j = nearest integer to a*(2/pi), ties to even. */
    float j = rintf(a * H3O_TWO_OVER_PI);
    float r = fmaf(-j, H3O_PIO2_1, a);
    r = fmaf(-j, H3O_PIO2_2, r);
    r = fmaf(-j, H3O_PIO2_3, r);
    float r2 = r * r;
    /* sin r = r + r^3 (S3 + r^2 (S5 + r^2 (S7 + r^2 (S9 + r^2 S11)))) */
    float ps = fmaf(H3O_S11, r2, H3O_S9);
    ps = fmaf(ps, r2, H3O_S7);
    ps = fmaf(ps, r2, H3O_S5);
    ps = fmaf(ps, r2, H3O_S3);
    float r3 = r2 * r;
    float sr = fmaf(ps, r3, r);
    /* cos r = 1 + r^2 (C2 + r^2 (C4 + r^2 (C6 + r^2 (C8 + r^2 (C10 + r^2 C12))))) */
    float pc = fmaf(H3O_C12, r2, H3O_C10);
    pc = fmaf(pc, r2, H3O_C8);
    pc = fmaf(pc, r2, H3O_C6);
    pc = fmaf(pc, r2, H3O_C4);
    pc = fmaf(pc, r2, H3O_C2);
    float cr = fmaf(pc, r2, 1.0f);
    /* Quadrant: sin(j*pi/2 + r), cos(j*pi/2 + r) for j mod 4. */
    int q = ((int)j) & 3;
    float s, c;
    switch (q) {
    case 0: s = sr; c = cr; break;
    case 1: s = cr; c = -sr; break;
    case 2: s = -sr; c = -cr; break;
    default: s = -cr; c = sr; break;
    }
    *s_out = s;
    *c_out = c;
}

/* Rotary inverse frequencies of one axis of width d (even):
 * inv_freq[i] = theta^(-2i/d), i < d/2, evaluated in double and rounded to
 * binary32 once.
 * Reading: the pages name a partial (t,h,w) RoPE [P5, decoder-attention
 * commit] but print no frequency formula; this is the standard rotary
 * ladder, one per axis over that axis's own width. */
void h3o_inv_freq(double theta, int d, float* inv_freq)
{
    for (int i = 0; i < d / 2; ++i) {
        double expo = -(2.0 * (double)i) / (double)d;
        inv_freq[i] = (float)pow(theta, expo);
    }
}

/* ------------------------------------------------------------------------ */
/* Per-head RMS normalisation [P2 fused-cast commit; P3 Operations; P5      */
/* patch 0005 commit].                                                      */
/* ------------------------------------------------------------------------ */

/* Sum of squares of one head row in the fixed order.
 * Reading: the pages only say the reduction order is fixed ("the reference
 * RMS reduction tree" [P3], "the same block reduction as the standalone
 * norm" [P5]).  The order taken here: split the D channels into C = D/8
 * chunks of 8 neighbours; each chunk sums its squares left to right
 * (((x0*x0 + x1*x1) + x2*x2) + ... + x7*x7), every product and every sum
 * rounded; the C chunk sums (padded with zeros to a power of two P) are
 * then added by a halving tree: for o = P/2, P/4, ..., 1, p[i] = p[i] +
 * p[i + o] for every i < o; the sum is p[0]. */
float h3o_sumsq(const float* x, int D)
{
    int C = D / 8;
    int P = 1;
    while (P < C) P <<= 1;
    float p[32];
    for (int c = 0; c < P; ++c) p[c] = 0.0f;
    for (int c = 0; c < C; ++c) {
        const float* xc = x + 8 * c;
        float acc = xc[0] * xc[0];
        for (int k = 1; k < 8; ++k) {
            float sq = xc[k] * xc[k];
            acc = acc + sq;
        }
        p[c] = acc;
    }
    for (int o = P / 2; o >= 1; o /= 2)
        for (int i = 0; i < o; ++i) p[i] = p[i] + p[i + o];
    return p[0];
}

/* The reciprocal RMS of one head row: inv = 1 / sqrt(ss/D + eps).
 * Reading: eps inside the square root (the usual RMSNorm); a correctly
 * rounded division, a correctly rounded square root and a correctly rounded
 * reciprocal (never an approximate reciprocal square root), because the
 * pages require results bit-identical to an unfused chain [P3]. */
float h3o_rms_inv(const float* x, int D, float eps)
{
    float ss = h3o_sumsq(x, D);
    float ms = ss / (float)D;
    float t = ms + eps;
    float rt = sqrtf(t);
    return 1.0f / rt;
}

/* Normalise one head row in binary32: y[d] = (x[d] * inv) * w[d], two
 * rounded products in that order. */
void h3o_norm_head_f32(const float* x, const float* w, int D, float eps, float* y)
{
    float inv = h3o_rms_inv(x, D, eps);
    for (int d = 0; d < D; ++d) {
        float xn = x[d] * inv;
        y[d] = xn * w[d];
    }
}

/* Normalise one head row and round it to the 16-bit type:
 * n[d] = round16((x[d] * inv) * w[d]), two rounded products in that order.
 * Reading: one rounding point after the norm, as an unfused norm kernel
 * that writes its 16-bit result in place on the projection has [P5,
 * decoder-attention commit: "normalise q/k in place on the projection"]. */
void h3o_norm_head(int dtype, const float* x, const float* w, int D, float eps, uint16_t* n)
{
    float y[256];
    h3o_norm_head_f32(x, w, D, eps, y);
    for (int d = 0; d < D; ++d) n[d] = h3o_round16(dtype, y[d]);
}

/* ------------------------------------------------------------------------ */
/* Partial multi-axis rotary embedding [P5 decoder-attention commit:        */
/* "partial RoPE"; P2 fused-cast commit: Q and K are rotated].              */
/* ------------------------------------------------------------------------ */

/* The rotation in binary32: (u, v) -> (u*c - v*s, u*s + v*c), every product
 * rounded, then one rounded subtract or add (no fusion). */
void h3o_rotate_f32(float c, float s, float u, float v, float* u_out, float* v_out)
{
    float uc = u * c;
    float vs = v * s;
    float us = u * s;
    float vc = v * c;
    *u_out = uc - vs;
    *v_out = us + vc;
}

/* Rotate one pair (u, v) by the angle whose cosine and sine are (c, s):
 *   u' = round16(u*c - v*s),  v' = round16(u*s + v*c),
 * every product rounded, then one rounded add or subtract (no fusion). */
void h3o_rotate_pair(int dtype, float c, float s, uint16_t u16, uint16_t v16,
                     uint16_t* u_out, uint16_t* v_out)
{
    float a, b;
    h3o_rotate_f32(c, s, h3o_widen(dtype, u16), h3o_widen(dtype, v16), &a, &b);
    *u_out = h3o_round16(dtype, a);
    *v_out = h3o_round16(dtype, b);
}

/* Cosines and sines of one token's rotary angles, listed pair by pair over
 * the leading R channels.
 * Readings (the pages are silent on all of these):
 *  - channels [0, R) are cut into n_axes consecutive segments of the given
 *    widths, in (t, h, w) order for three axes;
 *  - segment a rotates its pairs (2i, 2i+1), interleaved neighbours, by
 *    angle pos[a] * inv_freq_a[i], the product rounded once;
 *  - channels [R, D) pass through unrotated. */
static void h3o_token_angles(const h3o_problem* pb, const int32_t* tok_pos,
                             const float* inv_freq, float* cs, float* sn)
{
    int pair = 0;
    for (int a = 0; a < pb->n_axes; ++a) {
        int da = pb->axis_dims[a];
        float p = (float)tok_pos[a];
        for (int i = 0; i < da / 2; ++i, ++pair) {
            float ang = p * inv_freq[pair];
            h3o_sincos(ang, &sn[pair], &cs[pair]);
        }
    }
}

/* Build the per-pair inverse-frequency list for all axes of a problem. */
static void h3o_problem_inv_freq(const h3o_problem* pb, float* inv_freq)
{
    int pair = 0;
    for (int a = 0; a < pb->n_axes; ++a) {
        h3o_inv_freq(pb->theta, pb->axis_dims[a], inv_freq + pair);
        pair += pb->axis_dims[a] / 2;
    }
}

/* Norm and rotation of one Q or K head row: D 16-bit codes in, D out.
 * Rotated pairs use the token's cos/sin lists; channels >= R pass through
 * normalised but unrotated. */
static void h3o_head16(const h3o_problem* pb, const uint16_t* src, const float* w, const float* cs,
                       const float* sn, uint16_t* dst)
{
    const int D = pb->head_dim, R = pb->rotary_dim;
    float x[256];
    uint16_t n[256];
    for (int d = 0; d < D; ++d) x[d] = h3o_widen(pb->in_dtype, src[d]);
    h3o_norm_head(pb->in_dtype, x, w, D, pb->eps, n);
    for (int i = 0; i < R / 2; ++i)
        h3o_rotate_pair(pb->in_dtype, cs[i], sn[i], n[2 * i], n[2 * i + 1],
                        &dst[2 * i], &dst[2 * i + 1]);
    for (int d = R; d < D; ++d) dst[d] = n[d];
}

/* ------------------------------------------------------------------------ */
/* One packed QKV row -> the 16-bit Q, K and V values of every head.        */
/* ------------------------------------------------------------------------ */

/* Layout of the input [P2 fused-cast commit: "the packed QKV projection";
 * P5 decoder-attention commit: q/k/v "chunk-copied ... out of the fused
 * projection"].  Reading: row r holds [Q | K | V], each H*D values with
 * head h's D channels contiguous at h*D.
 * Outputs yq, yk, yv: H*D 16-bit codes each, in (head, channel) order.
 * V is passed through unchanged [P2 norm_rope_tensor commit: "identity
 * for V"]. */
static void h3o_row16_with(const h3o_problem* pb, const uint16_t* qkv, const float* wq,
                           const float* wk, const int32_t* pos, const float* inv_freq, int64_t r,
                           uint16_t* yq, uint16_t* yk, uint16_t* yv)
{
    const int H = pb->heads, D = pb->head_dim;
    const int64_t HD = (int64_t)H * D;
    const uint16_t* row = qkv + r * pb->row_stride;
    float cs[H3O_MAX_PAIRS], sn[H3O_MAX_PAIRS];

    h3o_token_angles(pb, pos + r * pb->n_axes, inv_freq, cs, sn);

    for (int part = 0; part < 2; ++part) {
        const float* w = part == 0 ? wq : wk;
        uint16_t* y = part == 0 ? yq : yk;
        for (int h = 0; h < H; ++h)
            h3o_head16(pb, row + part * HD + (int64_t)h * D, w, cs, sn, y + (int64_t)h * D);
    }
    const uint16_t* vsrc = row + 2 * HD;
    for (int64_t e = 0; e < HD; ++e) yv[e] = vsrc[e];
}

/* Public per-row entry: the 16-bit Q, K, V of row r (any row, valid or not;
 * the caller decides).  Used to check sampled rows of a full-size run. */
void h3o_row16(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
               const int32_t* pos, int64_t r, uint16_t* yq, uint16_t* yk, uint16_t* yv)
{
    float inv_freq[H3O_MAX_PAIRS];
    h3o_problem_inv_freq(pb, inv_freq);
    h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, yq, yk, yv);
}

/* Row r = b*S + s is kept when s < the item's valid length: valid_lens[b]
 * (clamped to [0, S]) when given, else valid_len [P2 valid-length commit:
 * the per-item valid length leaves padded rows out]. */
static int h3o_row_valid(const h3o_problem* pb, int64_t r)
{
    int64_t b = r / pb->seq, s = r % pb->seq;
    int64_t vl = pb->valid_len;
    if (pb->valid_lens) {
        vl = pb->valid_lens[b];
        if (vl < 0) vl = 0;
        if (vl > pb->seq) vl = pb->seq;
    }
    return s < vl;
}

/* Offset of (row r, head h, channel 0) in a head-major [B, H, S, D] tensor
 * [P5 first commit: ggml_rope_pe_permute writes [head_dim, tokens, heads,
 * batch], innermost first], or in a token-major [B, S, H, D] one (the layout
 * the cuDNN path reads [P2 norm_rope_tensor commit: [B, S, H, D]]). */
static int64_t h3o_head_major(const h3o_problem* pb, int64_t r, int h)
{
    int64_t b = r / pb->seq, s = r % pb->seq;
    if (pb->out_layout == 1) return ((b * pb->seq + s) * pb->heads + h) * pb->head_dim;  /* [B, S, H, D] */
    return ((b * pb->heads + h) * pb->seq + s) * pb->head_dim;
}

/* 16-bit output: write the head-major Q, K, V of the valid rows in
 * [row0, row1); padded rows are not written [P2 valid-length commit]. */
void h3o_prepare16_rows(const h3o_problem* pb, const uint16_t* qkv, const float* wq,
                        const float* wk, const int32_t* pos, int64_t row0, int64_t row1,
                        uint16_t* out_q, uint16_t* out_k, uint16_t* out_v)
{
    const int H = pb->heads, D = pb->head_dim;
    float inv_freq[H3O_MAX_PAIRS];
    uint16_t yq[H3O_MAX_HD], yk[H3O_MAX_HD], yv[H3O_MAX_HD];
    h3o_problem_inv_freq(pb, inv_freq);
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, yq, yk, yv);
        for (int h = 0; h < H; ++h) {
            int64_t o = h3o_head_major(pb, r, h);
            memcpy(out_q + o, yq + (int64_t)h * D, sizeof(uint16_t) * D);
            memcpy(out_k + o, yk + (int64_t)h * D, sizeof(uint16_t) * D);
            memcpy(out_v + o, yv + (int64_t)h * D, sizeof(uint16_t) * D);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Per-tensor e4m3 cast [P2 Summary bullet 2 and fused-cast commit: one     */
/* amax pass and one cast pass; dynamic scales by default, a static scale   */
/* table as an option; Q, K and V each get a per-tensor descale].           */
/* ------------------------------------------------------------------------ */

/* amax pass: amax[t] = max |y| over the valid rows in [row0, row1), every
 * head and channel, of tensor t in (Q, K, V), where y is the 16-bit value
 * the 16-bit path would write.  Padded rows are left out [P2 valid-length
 * commit].  NaN values are skipped (a comparison with NaN is false).
 * Reading: the amax is taken on the 16-bit rounded values, as the unfused
 * chain the fused op replaces ("the compiled norm + RoPE pair and three
 * per-tensor scale kernels" [P2 Summary]) would see them. */
void h3o_amax_rows(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                   const int32_t* pos, int64_t row0, int64_t row1, float* amax)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    float inv_freq[H3O_MAX_PAIRS];
    uint16_t y[3][H3O_MAX_HD];
    h3o_problem_inv_freq(pb, inv_freq);
    float m[3] = {0.0f, 0.0f, 0.0f};
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, y[0], y[1], y[2]);
        for (int t = 0; t < 3; ++t)
            for (int64_t e = 0; e < HD; ++e) {
                float a = fabsf(h3o_widen(pb->in_dtype, y[t][e]));
                if (a > m[t]) m[t] = a;
            }
    }
    for (int t = 0; t < 3; ++t) amax[t] = m[t];
}

/* A scale usable as a divisor: a finite normal positive binary32. */
static int h3o_scale_ok(float s)
{
    return s >= FLT_MIN && s <= FLT_MAX;
}

/* Scales of the cast.  scale[t] is the descale the consumer multiplies by,
 * inv[t] the factor the cast multiplies by.
 *   dynamic: scale = amax / 448, inv = 448 / amax (448 = largest e4m3);
 *   static:  scale = table[t],   inv = 1 / table[t]  [P2 Summary bullet 2].
 * Reading (the pages are silent): when amax (or a table entry) is zero,
 * subnormal, infinite or NaN, scale = inv = 1. */
void h3o_scales(const h3o_problem* pb, const float* amax, float* scale, float* inv)
{
    for (int t = 0; t < 3; ++t) {
        float s, i;
        if (pb->scale_mode == H3O_SCALE_STATIC) {
            float tab = pb->static_scales[t];
            if (h3o_scale_ok(tab)) {
                s = tab;
                i = 1.0f / tab;
            } else {
                s = 1.0f;
                i = 1.0f;
            }
        } else {
            float a = amax[t];
            if (h3o_scale_ok(a)) {
                s = a / 448.0f;
                i = 448.0f / a;
            } else {
                s = 1.0f;
                i = 1.0f;
            }
        }
        scale[t] = s;
        inv[t] = i;
    }
}

/* Cast n 16-bit values of tensor t: code = e4m3(y * inv), one rounded
 * product then the saturating round-to-nearest-even e4m3 conversion.
 * Reading: multiply by the reciprocal rather than divide every element,
 * and cast from the 16-bit rounded value. */
static void h3o_cast_values(int dtype, const uint16_t* y, int64_t n, float inv, uint8_t* out)
{
    for (int64_t e = 0; e < n; ++e) {
        float v = h3o_widen(dtype, y[e]);
        float z = v * inv;
        out[e] = h3o_f32_to_e4m3(z);
    }
}

/* Per-row cast entry: the e4m3 codes of row r (H*D per tensor, in (head,
 * channel) order) under the factors inv[3]. */
void h3o_cast_row(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                  const int32_t* pos, int64_t r, const float* inv, uint8_t* cq, uint8_t* ck,
                  uint8_t* cv)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    uint16_t y[3][H3O_MAX_HD];
    uint8_t* outs[3] = {cq, ck, cv};
    h3o_row16(pb, qkv, wq, wk, pos, r, y[0], y[1], y[2]);
    for (int t = 0; t < 3; ++t) h3o_cast_values(pb->in_dtype, y[t], HD, inv[t], outs[t]);
}

/* cast pass: recompute the 16-bit values of the valid rows in [row0, row1)
 * and write their e4m3 codes head-major; padded rows are not written. */
void h3o_cast_rows(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                   const int32_t* pos, int64_t row0, int64_t row1, const float* inv,
                   uint8_t* out_q, uint8_t* out_k, uint8_t* out_v)
{
    const int H = pb->heads, D = pb->head_dim;
    float inv_freq[H3O_MAX_PAIRS];
    uint16_t y[3][H3O_MAX_HD];
    uint8_t* outs[3] = {out_q, out_k, out_v};
    h3o_problem_inv_freq(pb, inv_freq);
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, y[0], y[1], y[2]);
        for (int t = 0; t < 3; ++t)
            for (int h = 0; h < H; ++h)
                h3o_cast_values(pb->in_dtype, y[t] + (int64_t)h * D, D, inv[t],
                                outs[t] + h3o_head_major(pb, r, h));
    }
}

/* The whole path on one thread: 16-bit out, or the amax pass (dynamic),
 * the scales and the cast pass.  out_scales receives the three descales
 * in e4m3 mode and is not touched in 16-bit mode. */
void h3o_prepare(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                 const int32_t* pos, void* out_q, void* out_k, void* out_v, float* out_scales)
{
    int64_t N = pb->batch * pb->seq;
    if (pb->out_kind == H3O_OUT_16B) {
        h3o_prepare16_rows(pb, qkv, wq, wk, pos, 0, N, (uint16_t*)out_q, (uint16_t*)out_k,
                           (uint16_t*)out_v);
        return;
    }
    float amax[3] = {0.0f, 0.0f, 0.0f}, scale[3], inv[3];
    if (pb->scale_mode == H3O_SCALE_DYNAMIC) h3o_amax_rows(pb, qkv, wq, wk, pos, 0, N, amax);
    h3o_scales(pb, amax, scale, inv);
    h3o_cast_rows(pb, qkv, wq, wk, pos, 0, N, inv, (uint8_t*)out_q, (uint8_t*)out_k,
                  (uint8_t*)out_v);
    for (int t = 0; t < 3; ++t) out_scales[t] = scale[t];
}

/* Saturation count [P2 commit adding H3_FP8_SAT_LOG: the elements clipped at
 * the E4M3 range, per tensor]: counts[t] += the number of valid-row values
 * of tensor t whose scaled value y * inv[t] has magnitude above 448, the
 * largest e4m3 code.  Reading: "clipped" means beyond the largest finite
 * code; NaN is not counted. */
void h3o_sat_rows(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                  const int32_t* pos, int64_t row0, int64_t row1, const float* inv, uint32_t* counts)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    float inv_freq[H3O_MAX_PAIRS];
    uint16_t y[3][H3O_MAX_HD];
    h3o_problem_inv_freq(pb, inv_freq);
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, y[0], y[1], y[2]);
        for (int t = 0; t < 3; ++t)
            for (int64_t e = 0; e < HD; ++e) {
                float z = h3o_widen(pb->in_dtype, y[t][e]) * inv[t];
                if (fabsf(z) > 448.0f) counts[t] += 1;
            }
    }
}

/* ------------------------------------------------------------------------ */
/* Single-tensor variant [P2 norm_rope_tensor commit: one [B, S, H, D]       */
/* tensor, norm + RoPE for Q / K, identity for V, to 16 bits or e4m3 with   */
/* its own per-tensor descale].  x holds rows of H*D values (row stride     */
/* pb->row_stride); kind 0 = Q, 1 = K (normalised with w, rotated), 2 = V   */
/* (copied).  The output is token-major [B, S, H, D], the layout of the     */
/* input.                                                                   */
/* ------------------------------------------------------------------------ */

/* The 16-bit values of row r of the tensor (H*D, head by head). */
void h3o_tensor_row16(const h3o_problem* pb, int kind, const uint16_t* x, const float* w,
                      const int32_t* pos, int64_t r, uint16_t* y)
{
    const int H = pb->heads, D = pb->head_dim;
    const uint16_t* row = x + r * pb->row_stride;
    if (kind == 2) {
        for (int64_t e = 0; e < (int64_t)H * D; ++e) y[e] = row[e];
        return;
    }
    float inv_freq[H3O_MAX_PAIRS], cs[H3O_MAX_PAIRS], sn[H3O_MAX_PAIRS];
    h3o_problem_inv_freq(pb, inv_freq);
    h3o_token_angles(pb, pos + r * pb->n_axes, inv_freq, cs, sn);
    for (int h = 0; h < H; ++h) h3o_head16(pb, row + (int64_t)h * D, w, cs, sn, y + (int64_t)h * D);
}

/* 16-bit output of the valid rows in [row0, row1), token-major. */
void h3o_tensor16_rows(const h3o_problem* pb, int kind, const uint16_t* x, const float* w,
                       const int32_t* pos, int64_t row0, int64_t row1, uint16_t* out)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    for (int64_t r = row0; r < row1; ++r)
        if (h3o_row_valid(pb, r)) h3o_tensor_row16(pb, kind, x, w, pos, r, out + r * HD);
}

/* amax over the valid rows in [row0, row1) of the tensor's 16-bit values. */
float h3o_tensor_amax_rows(const h3o_problem* pb, int kind, const uint16_t* x, const float* w,
                           const int32_t* pos, int64_t row0, int64_t row1)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    uint16_t y[H3O_MAX_HD];
    float m = 0.0f;
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_tensor_row16(pb, kind, x, w, pos, r, y);
        for (int64_t e = 0; e < HD; ++e) {
            float a = fabsf(h3o_widen(pb->in_dtype, y[e]));
            if (a > m) m = a;
        }
    }
    return m;
}

/* e4m3 codes of the valid rows in [row0, row1), token-major, under factor inv. */
void h3o_tensor_cast_rows(const h3o_problem* pb, int kind, const uint16_t* x, const float* w,
                          const int32_t* pos, int64_t row0, int64_t row1, float inv, uint8_t* out)
{
    const int64_t HD = (int64_t)pb->heads * pb->head_dim;
    uint16_t y[H3O_MAX_HD];
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        h3o_tensor_row16(pb, kind, x, w, pos, r, y);
        h3o_cast_values(pb->in_dtype, y, HD, inv, out + r * HD);
    }
}

/* ------------------------------------------------------------------------ */
/* Sage-attention outputs [P5 first commit: the fused RoPE / permute op     */
/* writes head-major [head_dim, tokens, heads, batch] tensors for the sage  */
/* kernel: F32 Q, F32 K * kv_scale and F16 V * kv_scale, with the rounding  */
/* points of the unfused sage chain].                                       */
/* Readings: the projection is 16-bit here (the rest of the path reads      */
/* 16-bit rows), widened exactly; from there every step stays binary32, as  */
/* in an all-F32 chain: the normalised value is NOT rounded to 16 bits      */
/* before the rotation, and Q and K are written unrounded; K is scaled      */
/* after the rotation by one rounded product with kv_scale; V is widened,   */
/* multiplied by kv_scale (one rounded product) and rounded to binary16     */
/* (nearest even, overflow to infinity).  No valid-prefix rule differs from */
/* the 16-bit path.                                                         */
/* ------------------------------------------------------------------------ */

/* Norm and rotation of one Q or K head row in binary32: D 16-bit codes in,
 * D binary32 values out; channels >= R pass through normalised. */
static void h3o_head_f32(const h3o_problem* pb, const uint16_t* src, const float* w, const float* cs,
                         const float* sn, float* dst)
{
    const int D = pb->head_dim, R = pb->rotary_dim;
    float x[256], n[256];
    for (int d = 0; d < D; ++d) x[d] = h3o_widen(pb->in_dtype, src[d]);
    h3o_norm_head_f32(x, w, D, pb->eps, n);
    for (int i = 0; i < R / 2; ++i)
        h3o_rotate_f32(cs[i], sn[i], n[2 * i], n[2 * i + 1], &dst[2 * i], &dst[2 * i + 1]);
    memcpy(dst + R, n + R, sizeof(float) * (size_t)(D - R));
}

/* Sage outputs of the valid rows in [row0, row1), head-major [B, H, S, D]
 * (or token-major, pb->out_layout): out_q, out_k binary32, out_v binary16
 * codes.  Padded rows are not written. */
void h3o_sage_rows(const h3o_problem* pb, const uint16_t* qkv, const float* wq, const float* wk,
                   const int32_t* pos, float kv_scale, int64_t row0, int64_t row1, float* out_q,
                   float* out_k, uint16_t* out_v)
{
    const int H = pb->heads, D = pb->head_dim;
    const int64_t HD = (int64_t)H * D;
    float inv_freq[H3O_MAX_PAIRS], cs[H3O_MAX_PAIRS], sn[H3O_MAX_PAIRS];
    float y[256];
    h3o_problem_inv_freq(pb, inv_freq);
    for (int64_t r = row0; r < row1; ++r) {
        if (!h3o_row_valid(pb, r)) continue;
        const uint16_t* row = qkv + r * pb->row_stride;
        h3o_token_angles(pb, pos + r * pb->n_axes, inv_freq, cs, sn);
        for (int h = 0; h < H; ++h) {
            const int64_t o = h3o_head_major(pb, r, h);
            h3o_head_f32(pb, row + (int64_t)h * D, wq, cs, sn, out_q + o);
            h3o_head_f32(pb, row + HD + (int64_t)h * D, wk, cs, sn, y);
            for (int d = 0; d < D; ++d) out_k[o + d] = y[d] * kv_scale;
            const uint16_t* v = row + 2 * HD + (int64_t)h * D;
            for (int d = 0; d < D; ++d) {
                float sv = h3o_widen(pb->in_dtype, v[d]) * kv_scale;
                out_v[o + d] = h3o_f32_to_f16(sv);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Adjacent VAE-block operations [P3 Operations table, rows "SwiGLU" (SiLU  */
/* and multiply after the FP16 w1 output) and "Scaled residual" (FP32       */
/* residual + FP16 branch * FP32 scale, with contraction disabled)].        */
/* ------------------------------------------------------------------------ */

/* e^x: the library's own routine (the pages give no exp; both the CPU and
 * the GPU evaluate this one, so SiLU agrees bit for bit).  Cody & Waite
 * reduction x = k*ln2 + r with ln2 split in two binary32 parts (each step a
 * fused multiply-add), the Taylor series of e^r to r^8 in Horner form, then
 * one rounded product with 2^k (k = 128 as 2^127 then 2).  Domain handling:
 * NaN returns NaN, x > 89 returns +inf, and results below 2^-126 (x < -87.4,
 * where 1 + e^x already rounds to 1) return 0. */
static const float H3O_LOG2E = 0x1.715476p+0f;
static const float H3O_LN2_HI = 0x1.62e430p-1f;
static const float H3O_LN2_LO = -0x1.05c610p-29f;
static const float H3O_E2 = 0x1.000000p-1f;   /* 1/2! */
static const float H3O_E3 = 0x1.555556p-3f;   /* 1/3! */
static const float H3O_E4 = 0x1.555556p-5f;   /* 1/4! */
static const float H3O_E5 = 0x1.111112p-7f;   /* 1/5! */
static const float H3O_E6 = 0x1.6c16c2p-10f;  /* 1/6! */
static const float H3O_E7 = 0x1.a01a02p-13f;  /* 1/7! */
static const float H3O_E8 = 0x1.a01a02p-16f;  /* 1/8! */

float h3o_exp(float x)
{
    if (x != x) return x;
    if (x > 89.0f) return INFINITY;
    if (x < -104.0f) return 0.0f;
    float k = rintf(x * H3O_LOG2E);
    float r = fmaf(-k, H3O_LN2_HI, x);
    r = fmaf(-k, H3O_LN2_LO, r);
    float p = fmaf(H3O_E8, r, H3O_E7);
    p = fmaf(p, r, H3O_E6);
    p = fmaf(p, r, H3O_E5);
    p = fmaf(p, r, H3O_E4);
    p = fmaf(p, r, H3O_E3);
    p = fmaf(p, r, H3O_E2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ki = (int)k;
    if (ki < -126) return 0.0f;
    /* k = 128 (x near the overflow bound): 2^128 is not a binary32, so scale
     * by 2^127 and then by 2; both products are exact until overflow. */
    int k1 = ki > 127 ? 127 : ki;
    uint32_t bits = (uint32_t)(k1 + 127) << 23;
    float two_k;
    memcpy(&two_k, &bits, sizeof two_k);
    float y = p * two_k;
    if (ki > 127) y = y * 2.0f;
    return y;
}

/* SiLU(g) = g / (1 + e^-g): one rounded sum, one correctly rounded division.
 * Reading: the fp32 form of the reused SiluAndMul operator. */
float h3o_silu(float g)
{
    float e = h3o_exp(-g);
    float d = 1.0f + e;
    return g / d;
}

/* SwiGLU rows: x is [rows, row_stride] 16-bit with gate = x[:, 0:f] and
 * up = x[:, f:2f]; out[r, j] = round16(silu(gate) * up), one rounded product
 * then the 16-bit rounding; out is [rows, f]. */
void h3o_silu_and_mul_rows(int dtype, const uint16_t* x, int64_t rows, int f, int64_t row_stride,
                           uint16_t* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int j = 0; j < f; ++j) {
            float g = h3o_widen(dtype, x[r * row_stride + j]);
            float u = h3o_widen(dtype, x[r * row_stride + f + j]);
            float s = h3o_silu(g);
            float y = s * u;
            out[r * f + j] = h3o_round16(dtype, y);
        }
}

/* Scaled residual: out[i] = residual[i] + branch[i] * scale[c], c = i mod
 * channels (scale_len == channels) or 0 (scale_len == 1); the product is
 * rounded to binary32 on its own ("contraction disabled"), then the sum. */
void h3o_scaled_residual(int dtype, const float* residual, const uint16_t* branch, const float* scale,
                         int64_t rows, int channels, int scale_len, float* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < channels; ++c) {
            int64_t i = r * channels + c;
            float b = h3o_widen(dtype, branch[i]);
            float sc = scale[scale_len == 1 ? 0 : c];
            float t = b * sc;
            out[i] = residual[i] + t;
        }
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the tests (element-wise loops over the scalar steps).  */
/* ------------------------------------------------------------------------ */

void h3o_f32_to_f16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = h3o_f32_to_f16(x[i]);
}

void h3o_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = h3o_f32_to_bf16(x[i]);
}

void h3o_f32_to_e4m3_array(const float* x, uint8_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = h3o_f32_to_e4m3(x[i]);
}

void h3o_sincos_array(const float* a, float* s, float* c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h3o_sincos(a[i], &s[i], &c[i]);
}

/* Angles the path evaluates for positions pos (n_tok tokens, n_axes each):
 * out[t * (R/2) + pair] = pos[t][axis(pair)] * inv_freq[pair] (one rounded
 * product), the argument list the sine/cosine pin covers. */
void h3o_angles_array(const h3o_problem* pb, const int32_t* pos, int64_t n_tok, float* out)
{
    float inv_freq[H3O_MAX_PAIRS];
    h3o_problem_inv_freq(pb, inv_freq);
    int64_t npair = pb->rotary_dim / 2;
    for (int64_t t = 0; t < n_tok; ++t) {
        int pair = 0;
        for (int a = 0; a < pb->n_axes; ++a) {
            float p = (float)pos[t * pb->n_axes + a];
            for (int i = 0; i < pb->axis_dims[a] / 2; ++i, ++pair)
                out[t * npair + pair] = p * inv_freq[pair];
        }
    }
}

void h3o_problem_inv_freq_public(const h3o_problem* pb, float* inv_freq)
{
    h3o_problem_inv_freq(pb, inv_freq);
}

void h3o_exp_array(const float* x, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = h3o_exp(x[i]);
}
