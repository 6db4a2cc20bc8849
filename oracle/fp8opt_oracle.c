/*
 * fp8opt oracle: a plain, slow, scalar CPU implementation of the scaled FP8
 * cast, of the local reduction of FP8 shards, and of the FP8-state AdamW step
 * (MS-AMP levels O1, O2 and O3).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may load or call this file.  It shares no code with the
 * CUDA library: its own codecs, its own loops, its own scalar set-up.
 *
 * Sources.  MS-AMP documentation, "Optimization Level" page: O1 keeps weight
 * gradients in FP8; O2 keeps the Adam/AdamW first moment in FP8 and the second
 * moment in FP16 with FP16 weights; O3 adds an FP16 master weight and an FP8
 * regular weight (the level table).  MS-AMP README, "Usage": the GradScaler
 * loop (scale, backward, step), and the two torch optimizers it supports,
 * Adam and AdamW.  TransformerEngine issue #131: the two FP8 formats
 * E4M3 and E5M2.  The pages give neither bit layouts nor a scaling rule nor an
 * update order; the readings used here are:
 *   - E4M3 / E5M2 are the OCP 8-bit floating-point formats (E4M3: bias 7, no
 *     infinity, NaN = S.1111.111, max 448; E5M2: bias 15, IEEE-like, max
 *     57344).  Encoding rounds to nearest, ties to even, and saturates finite
 *     overflow to +-max.  A NaN input gives code 0x7F; an infinite input gives
 *     0x7F in E4M3 and the signed infinity code in E5M2.
 *   - The per-tensor scale is fp8_max / amax, computed just in time from the
 *     tensor being encoded, as one fp32 IEEE division; it is 1.0 when amax is
 *     zero or not finite, or when the quotient is not finite.
 *   - amax orders NaN above +inf above every finite |x|; a NaN amax is
 *     returned as the quiet NaN 0x7FC00000.
 *   - The AdamW update is torch.optim.AdamW's (decoupled weight decay applied
 *     as w * (1 - lr * wd), eps added after the bias-corrected square root),
 *     evaluated in fp32 in the order written in oracle_adamw_step below.  The
 *     bias corrections enter as two per-call scalars computed in double and
 *     rounded once: step_size = lr / (1 - beta1^t) and inv_sbc2 =
 *     1 / sqrt(1 - beta2^t), with beta^t by binary exponentiation in double
 *     (oracle_bias_power).  Dequantization and the GradScaler unscale are
 *     one per-tensor factor k = inv_loss_scale / g_scale.  Where the order
 *     below writes fmaf, the product and sum are rounded once (IEEE fused
 *     multiply-add); every other product and sum is rounded on its own.
 *   - found_inf is set when any unscaled gradient element is not finite; then
 *     no state element changes.
 *   - The first moment is re-encoded from the fp32 value of this step, with a
 *     scale taken from this step's amax; the O3 weight copy is encoded from the
 *     FP16-rounded master.
 *   - Optional per-tensor scaled second moment (the O2 paragraph's "FP16"
 *     state, kept clear of FP16 underflow): a per-tensor bound B on max v
 *     follows B_new = fma(beta2, B_old, (1 - beta2) * gmax^2), gmax = max |g|
 *     of this step; v is stored as FP16 of v * 2^14 / B_new and read back as
 *     FP16 value * B_old * 2^-14.  B = 0 means v = 0.
 *   - Optional Adam with L2 weight decay (torch.optim.Adam, the other
 *     recognised optimizer): g = fma(wd, w, g) before the moments, and the
 *     weight itself is not decayed.
 *   - The global gradient norm for clipping (the run script's --clip-grad):
 *     the L2 norm of the unscaled gradient, taken from the codes with each
 *     tensor's sum of squares exact and the tensors combined in double in
 *     order; clipping multiplies each tensor's dequantization factor by
 *     max_norm / (norm + 1e-6) (torch's clip_grad_norm_ coefficient) when
 *     that is below 1.
 *   - The local reduction of an FP8 all-reduce (the O1 paragraph's FP8
 *     AllReduce communication of weight gradients): k shards of one tensor,
 *     shard j encoded with its own scale s_j, are dequantized as code value
 *     times (1 / s_j), summed in fp32 in shard order, multiplied by a
 *     caller-given factor (1 for a sum, 1 / k for a mean), and cast back to
 *     FP8 with a just-in-time scale like any other tensor.
 *
 * Floating point: compiled with -ffp-contract=off and no fast-math, so every
 * float expression below is evaluated as written in IEEE binary32 with
 * round-to-nearest-even (C float arithmetic with FLT_EVAL_METHOD 0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_E4M3 = 0, OR_E5M2 = 1 };
enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* ---------------------------------------------------------------- formats */

typedef struct {
    int mbits;       /* explicit mantissa bits */
    int bias;        /* exponent bias */
    double maxval;   /* largest finite magnitude */
    int has_inf;     /* all-ones exponent with zero mantissa is infinity */
} or_format;

/* E4M3, E5M2 (OCP 8-bit formats), and IEEE binary16 for the FP16 state. */
static const or_format OR_FMT[2] = {
    {3, 7, 448.0, 0},
    {2, 15, 57344.0, 1},
};
static const or_format OR_HALF = {10, 15, 65504.0, 1};

static float or_bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Largest finite magnitude of an FP8 format (448 or 57344). */
double oracle_fp8_max(int fmt) { return OR_FMT[fmt].maxval; }

/* Value of an FP8 code by the format definition: (-1)^s * 2^(E-bias) *
 * (1 + M/2^mbits) for a nonzero exponent field, (-1)^s * 2^(1-bias) *
 * M/2^mbits for a zero one; E4M3's S.1111.111 is NaN, E5M2's all-ones
 * exponent is infinity (M = 0) or NaN. */
float oracle_fp8_decode(uint8_t c, int fmt)
{
    const or_format *f = &OR_FMT[fmt];
    int ebits = 7 - f->mbits;
    int s = c >> 7;
    int e = (c >> f->mbits) & ((1 << ebits) - 1);
    int m = c & ((1 << f->mbits) - 1);
    int eall = (1 << ebits) - 1;
    double v;
    if (!f->has_inf && e == eall && m == (1 << f->mbits) - 1)
        return or_bits_f32(0x7FC00000u);
    if (f->has_inf && e == eall) {
        if (m != 0) return or_bits_f32(0x7FC00000u);
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, 1 - f->bias - f->mbits);
    } else {
        v = ldexp(1.0 + ldexp((double)m, -f->mbits), e - f->bias);
    }
    return (float)(s ? -v : v);   /* exact: at most 4 significant bits */
}

/* Round |a| (finite, >= 0) to the nearest value of format f with an
 * unbounded exponent range above, ties to even.  The spacing of f's values in
 * the binade of a is 2^(lead - mbits), lead = max(floor(log2 a), 1 - bias);
 * a / spacing is exact in double and rint() rounds it half-to-even. */
static double or_round_rne(double a, const or_format *f)
{
    int emin = 1 - f->bias;
    int lead = emin;
    if (a > 0.0) {
        int e;
        frexp(a, &e);           /* a = fr * 2^e, fr in [0.5, 1) */
        lead = e - 1;
        if (lead < emin) lead = emin;
    }
    double q = ldexp(1.0, lead - f->mbits);
    return rint(a / q) * q;
}

/* Bit fields of a representable magnitude r of format f (no sign). */
static uint32_t or_fields(double r, const or_format *f)
{
    if (r == 0.0) return 0;
    int emin = 1 - f->bias;
    int e;
    frexp(r, &e);
    int lead = e - 1;
    if (lead < emin)   /* subnormal: exponent field 0, M = r / 2^(emin-mbits) */
        return (uint32_t)(r / ldexp(1.0, emin - f->mbits));
    uint32_t M = (uint32_t)((r / ldexp(1.0, lead) - 1.0) * (double)(1 << f->mbits));
    return ((uint32_t)(lead + f->bias) << f->mbits) | M;
}

/* FP8 code of x: round to nearest even, saturate finite overflow to +-max. */
uint8_t oracle_fp8_encode(float x, int fmt)
{
    const or_format *f = &OR_FMT[fmt];
    if (isnan(x)) return 0x7F;
    int neg = signbit(x) != 0;
    if (isinf(x)) return f->has_inf ? (neg ? 0xFC : 0x7C) : 0x7F;
    double r = or_round_rne(fabs((double)x), f);
    if (r > f->maxval) r = f->maxval;
    uint32_t code = or_fields(r, f);
    return (uint8_t)(neg ? (code | 0x80u) : code);
}

/* IEEE binary16 bits of x: round to nearest even; overflow gives infinity
 * (a value that rounds above 65504 is out of range); NaN gives 0x7E00. */
uint16_t oracle_f32_to_f16(float x)
{
    if (isnan(x)) return 0x7E00;
    int neg = signbit(x) != 0;
    uint32_t bits;
    if (isinf(x)) {
        bits = 0x7C00;
    } else {
        double r = or_round_rne(fabs((double)x), &OR_HALF);
        bits = (r > OR_HALF.maxval) ? 0x7C00u : or_fields(r, &OR_HALF);
    }
    return (uint16_t)(neg ? (bits | 0x8000u) : bits);
}

/* Value of IEEE binary16 bits. */
float oracle_f16_to_f32(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0x1F) {
        if (m) return or_bits_f32(0x7FC00000u);
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -24);
    } else {
        v = ldexp(1.0 + ldexp((double)m, -10), e - 15);
    }
    return (float)(s ? -v : v);
}

/* bfloat16 is the upper half of a binary32 pattern. */
float oracle_bf16_to_f32(uint16_t h) { return or_bits_f32((uint32_t)h << 16); }

/* ------------------------------------------------------------ amax, scale */

/* Running amax with NaN above +inf above every finite magnitude. */
typedef struct { int nan; int inf; float fin; } or_amax;

static void or_amax_add(or_amax *a, float x)
{
    if (isnan(x)) a->nan = 1;
    else if (isinf(x)) a->inf = 1;
    else if (fabsf(x) > a->fin) a->fin = fabsf(x);
}

static float or_amax_value(const or_amax *a)
{
    if (a->nan) return or_bits_f32(0x7FC00000u);
    if (a->inf) return INFINITY;
    return a->fin;
}

/* Just-in-time per-tensor scale fp8_max / amax, one fp32 division; 1.0 when
 * amax is zero or not finite, or when the quotient is not finite. */
float oracle_scale_from_amax(float amax, int fmt)
{
    if (!(amax > 0.0f) || !isfinite(amax)) return 1.0f;
    float q = (float)OR_FMT[fmt].maxval / amax;
    if (!isfinite(q)) return 1.0f;
    return q;
}

static float or_load(const void *src, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32: return ((const float *)src)[i];
    case OR_BF16: return oracle_bf16_to_f32(((const uint16_t *)src)[i]);
    default: return oracle_f16_to_f32(((const uint16_t *)src)[i]);
    }
}

/* ------------------------------------------------------------------- cast */

/* The encode of a cast: each element multiplied by the scale in fp32 and
 * encoded; a non-finite element keeps its own code. */
static void or_cast_encode(const void *src, int dtype, int64_t numel, int fmt,
                           float scale, uint8_t *codes)
{
    for (int64_t i = 0; i < numel; ++i) {
        float x = or_load(src, dtype, i);
        if (!isfinite(x)) { codes[i] = oracle_fp8_encode(x, fmt); continue; }
        float t = x * scale;
        codes[i] = oracle_fp8_encode(t, fmt);
    }
}

/* Scaled FP8 cast of one tensor (weight gradients from wider types to FP8,
 * MS-AMP O1): amax over the tensor, scale = fp8_max / amax, then each element
 * is multiplied by the scale in fp32 and encoded.  Returns 0, or -1 on a bad
 * argument. */
int oracle_cast_scaled(const void *src, int dtype, int64_t numel, int fmt,
                       uint8_t *codes, float *amax_out, float *scale_out)
{
    if (numel < 0 || fmt < 0 || fmt > 1 || dtype < 0 || dtype > 2) return -1;
    or_amax a = {0, 0, 0.0f};
    for (int64_t i = 0; i < numel; ++i) or_amax_add(&a, or_load(src, dtype, i));
    float amax = or_amax_value(&a);
    float scale = oracle_scale_from_amax(amax, fmt);
    or_cast_encode(src, dtype, numel, fmt, scale, codes);
    *amax_out = amax;
    *scale_out = scale;
    return 0;
}

/* ------------------------------------------------------------------- step */

typedef struct {
    int64_t numel;
    const uint8_t *g;      /* gradient codes */
    float g_scale;         /* scale the gradient codes were encoded with */
    int g_fmt;             /* OR_E4M3 or OR_E5M2 */
    uint8_t *m;            /* first moment, E4M3 codes (in/out) */
    float *m_scale;        /* its scale (in/out) */
    uint16_t *v;           /* second moment, FP16 bits (in/out) */
    uint16_t *w;           /* O2: FP16 weight; O3: FP16 master (in/out) */
    uint8_t *w8;           /* O3 only: E4M3 weight copy (out), else NULL */
    float *w8_scale;       /* O3 only: its scale (out) */
    float *w8_amax;        /* O3 only: amax of the FP16 master (out) */
    float *v_bound;        /* scaled second moment only (in/out), else NULL */
} oracle_param;

/* Largest value a scaled second moment is stored at (as FP16 of v * scale). */
#define OR_V_TARGET 16384.0f

/* Scale of a scaled second moment from its bound: 2^14 / B, one fp32
 * division; 1.0 when B is zero or not finite, or the quotient is not finite. */
float oracle_v_scale_from_bound(float b)
{
    if (!(b > 0.0f) || !isfinite(b)) return 1.0f;
    float q = OR_V_TARGET / b;
    return isfinite(q) ? q : 1.0f;
}

/* beta^t in double by binary exponentiation: from the lowest bit of t up,
 * r = r * b when the bit is set, then b = b * b, each product rounded to
 * double.  (libm's pow is not specified to the bit, and platforms differ;
 * this form gives the same bits wherever double products round to nearest.) */
double oracle_bias_power(double b, int64_t t)
{
    double r = 1.0;
    while (t > 0) {
        if (t & 1) r = r * b;
        b = b * b;
        t >>= 1;
    }
    return r;
}

/* Per-call scalars.  The bias corrections 1 - beta^t are evaluated in double
 * and enter only through step_size = lr / bc1 and inv_sbc2 = 1 / sqrt(bc2),
 * each rounded to float once. */
typedef struct {
    float step_size, inv_sbc2, omb1, omb2, decay;
} or_scalars;

static or_scalars or_make_scalars(float lr, float beta1, float beta2,
                                  float wd, int64_t step, int l2)
{
    or_scalars s;
    double bc1 = 1.0 - oracle_bias_power((double)beta1, step);
    double bc2 = 1.0 - oracle_bias_power((double)beta2, step);
    s.step_size = (float)((double)lr / bc1);
    s.inv_sbc2 = (float)(1.0 / sqrt(bc2));
    s.omb1 = 1.0f - beta1;
    s.omb2 = 1.0f - beta2;
    s.decay = l2 ? 1.0f : 1.0f - lr * wd;
    return s;
}

/* The per-tensor factor that dequantizes a gradient code and undoes the loss
 * scale at once: k = inv_loss_scale / g_scale. */
static float or_grad_factor(const oracle_param *p, float inv_loss_scale)
{
    return inv_loss_scale / p->g_scale;
}

/* Unscaled gradient: the code's value times k. */
static float or_grad(const oracle_param *p, float k, int64_t i)
{
    return oracle_fp8_decode(p->g[i], p->g_fmt) * k;
}

/* New first moment in fp32: beta1 * m_prev + (1 - beta1) * g, with the
 * previous moment dequantized as code value times 1 / m_scale. */
static float or_m_new(const oracle_param *p, float minv, float g, float beta1,
                      const or_scalars *s, int64_t i)
{
    float mp = oracle_fp8_decode(p->m[i], OR_E4M3) * minv;
    return fmaf(beta1, mp, s->omb1 * g);
}

/* Gradient after the optional L2 decay term: fma(wd, w, g). */
static float or_grad_l2(const oracle_param *p, float g, int l2, float wd,
                        int64_t i)
{
    return l2 ? fmaf(wd, oracle_f16_to_f32(p->w[i]), g) : g;
}

/* ------------------------------------------------------ step, by phases
 *
 * A step's per-tensor quantities are maxima over the tensor's elements: the
 * amax of this step's fp32 first moment (its new scale), max |g| (a scaled
 * second moment's bound) and, for O3, the amax of the new FP16 master (the
 * weight copy's scale).  Everything else is elementwise.  The phases below
 * compute the maxima, or take them as given: oracle_adam_step runs them in
 * turn over whole tensors, and a tensor cut into pieces (element ranges with
 * the tensor's scales and bounds) gives the same elements when every piece
 * takes the whole tensor's maxima. */

/* The phases' argument check: a list length and a step count (from 1). */
static int or_bad_step(int n, int64_t step)
{
    return n < 0 || step < 1;
}

/* The factor the moments use: k = inv_loss_scale / g_scale, times the
 * clip coefficient when the step clips (clip != 1).  found_inf is decided on
 * the unclipped k. */
static float or_step_factor(const oracle_param *p, float inv_loss_scale,
                            float clip)
{
    float k = or_grad_factor(p, inv_loss_scale);
    if (clip != 1.0f) k = k * clip;
    return k;
}

static int or_adam_step(const oracle_param *p, int n, int l2, float lr,
                        float beta1, float beta2, float eps, float wd,
                        int64_t step, float inv_loss_scale, float clip);

/* One multi-tensor Adam step with FP8 first moment and FP16 second moment:
 * l2 = 0 is AdamW (decoupled decay), l2 = 1 is Adam with L2 decay.  Returns 1
 * when found_inf (nothing written), 0 after an update, -1 on a bad argument. */
int oracle_adam_step(const oracle_param *p, int n, int l2, float lr, float beta1,
                     float beta2, float eps, float wd, int64_t step,
                     float inv_loss_scale)
{
    return or_adam_step(p, n, l2, lr, beta1, beta2, eps, wd, step,
                        inv_loss_scale, 1.0f);
}

/* One tensor's maxima: the amax of this step's fp32 first moment and, for a
 * scaled second moment, max |g| (else 0). */
static void or_tensor_maxima(const oracle_param *q, int l2, float beta1,
                             float wd, const or_scalars *sc, float k,
                             float *amax_m, float *gmax)
{
    const or_scalars s = *sc;
    float minv = 1.0f / *q->m_scale;
    int scaled_v = q->v_bound != NULL;
    or_amax am = {0, 0, 0.0f}, ag = {0, 0, 0.0f};
    for (int64_t i = 0; i < q->numel; ++i) {
        float g = or_grad_l2(q, or_grad(q, k, i), l2, wd, i);
        or_amax_add(&am, or_m_new(q, minv, g, beta1, &s, i));
        if (scaled_v) or_amax_add(&ag, g);
    }
    *amax_m = or_amax_value(&am);
    *gmax = or_amax_value(&ag);
}

/* One tensor's update from its given maxima: the first moment re-encoded
 * with the scale of amax_m, v (scaled by the bound that gmax gives), the
 * FP16 weight or master; returns the amax of the new FP16 master. */
static float or_tensor_update(const oracle_param *q, int l2, float beta1,
                              float beta2, float eps, float wd,
                              const or_scalars *sc, float k, float amax_m,
                              float gmax)
{
    const or_scalars s = *sc;
    float minv = 1.0f / *q->m_scale;
    int scaled_v = q->v_bound != NULL;
    float m_scale_new = oracle_scale_from_amax(amax_m, OR_E4M3);
    float vinv = 1.0f, b_new = 0.0f, v_scale_new = 1.0f;
    if (scaled_v) {
        vinv = *q->v_bound * 0x1p-14f;
        b_new = fmaf(beta2, *q->v_bound, s.omb2 * (gmax * gmax));
        v_scale_new = oracle_v_scale_from_bound(b_new);
    }

    or_amax aw = {0, 0, 0.0f};
    for (int64_t i = 0; i < q->numel; ++i) {
        float g = or_grad_l2(q, or_grad(q, k, i), l2, wd, i);
        float m = or_m_new(q, minv, g, beta1, &s, i);
        float vp = oracle_f16_to_f32(q->v[i]);
        if (scaled_v) vp = vp * vinv;
        float wp = oracle_f16_to_f32(q->w[i]);
        float v = fmaf(beta2, vp, s.omb2 * (g * g));
        float denom = fmaf(sqrtf(v), s.inv_sbc2, eps);
        float upd = m / denom;
        float w = fmaf(-s.step_size, upd, wp * s.decay);
        q->m[i] = oracle_fp8_encode(m * m_scale_new, OR_E4M3);
        q->v[i] = oracle_f32_to_f16(scaled_v ? v * v_scale_new : v);
        q->w[i] = oracle_f32_to_f16(w);
        if (q->w8) or_amax_add(&aw, oracle_f16_to_f32(q->w[i]));
    }
    *q->m_scale = m_scale_new;
    if (scaled_v) *q->v_bound = b_new;
    return or_amax_value(&aw);
}

/* One tensor's O3 FP8 weight copy, encoded from the FP16 master with the
 * scale of the given master amax. */
static void or_tensor_copy(const oracle_param *q, float amax_w)
{
    float w8_scale = oracle_scale_from_amax(amax_w, OR_E4M3);
    for (int64_t i = 0; i < q->numel; ++i)
        q->w8[i] = oracle_fp8_encode(oracle_f16_to_f32(q->w[i]) * w8_scale,
                                     OR_E4M3);
    *q->w8_scale = w8_scale;
    *q->w8_amax = amax_w;
}

/* Phase 1: found_inf, the GradScaler check over every record (on the
 * unscaled gradients, before any decay term and any clipping), and when it
 * is clear each record's maxima (amax_m[t], gmax[t]; the factor k times
 * clip).  Writes no state.  Returns 1 when found_inf (the maxima are then
 * not written), 0, or -1 on a bad argument. */
int oracle_step_maxima(const oracle_param *p, int n, int l2, float lr,
                       float beta1, float beta2, float wd, int64_t step,
                       float inv_loss_scale, float clip, float *amax_m,
                       float *gmax)
{
    if (or_bad_step(n, step)) return -1;
    or_scalars s = or_make_scalars(lr, beta1, beta2, wd, step, l2);

    /* GradScaler check over every tensor before any state changes (on the
     * unscaled gradients, before any decay term). */
    for (int t = 0; t < n; ++t) {
        float k = or_grad_factor(&p[t], inv_loss_scale);
        for (int64_t i = 0; i < p[t].numel; ++i)
            if (!isfinite(or_grad(&p[t], k, i))) return 1;
    }
    for (int t = 0; t < n; ++t)
        or_tensor_maxima(&p[t], l2, beta1, wd, &s,
                         or_step_factor(&p[t], inv_loss_scale, clip),
                         &amax_m[t], &gmax[t]);
    return 0;
}

/* Phase 2: each record's update from the given maxima (phase 1's, or the
 * whole tensor's for a piece); master_amax[t] receives the amax of record
 * t's new FP16 master (may be NULL).  Returns 0, or -1 on a bad argument. */
int oracle_step_update(const oracle_param *p, int n, int l2, float lr,
                       float beta1, float beta2, float eps, float wd,
                       int64_t step, float inv_loss_scale, float clip,
                       const float *amax_m, const float *gmax,
                       float *master_amax)
{
    if (or_bad_step(n, step)) return -1;
    or_scalars s = or_make_scalars(lr, beta1, beta2, wd, step, l2);
    for (int t = 0; t < n; ++t) {
        float aw = or_tensor_update(&p[t], l2, beta1, beta2, eps, wd, &s,
                                    or_step_factor(&p[t], inv_loss_scale, clip),
                                    amax_m[t], gmax[t]);
        if (master_amax != NULL) master_amax[t] = aw;
    }
    return 0;
}

/* Phase 3: the O3 weight copy of each O3 record from the given master amax.
 * Returns 0, or -1 on a bad argument. */
int oracle_weight_copy(const oracle_param *p, int n, const float *master_amax)
{
    if (n < 0) return -1;
    for (int t = 0; t < n; ++t)
        if (p[t].w8) or_tensor_copy(&p[t], master_amax[t]);
    return 0;
}

static int or_adam_step(const oracle_param *p, int n, int l2, float lr,
                        float beta1, float beta2, float eps, float wd,
                        int64_t step, float inv_loss_scale, float clip)
{
    if (or_bad_step(n, step)) return -1;
    size_t bytes = (size_t)(n > 0 ? n : 1) * sizeof(float);
    float *am = malloc(bytes), *gm = malloc(bytes), *wm = malloc(bytes);
    int rc = -1;
    if (am != NULL && gm != NULL && wm != NULL) {
        rc = oracle_step_maxima(p, n, l2, lr, beta1, beta2, wd, step,
                                inv_loss_scale, clip, am, gm);
        if (rc == 0)
            rc = oracle_step_update(p, n, l2, lr, beta1, beta2, eps, wd, step,
                                    inv_loss_scale, clip, am, gm, wm);
        if (rc == 0) rc = oracle_weight_copy(p, n, wm);
    }
    free(am);
    free(gm);
    free(wm);
    return rc;
}

/* AdamW: oracle_adam_step with decoupled weight decay. */
int oracle_adamw_step(const oracle_param *p, int n, float lr, float beta1,
                      float beta2, float eps, float wd, int64_t step,
                      float inv_loss_scale)
{
    return oracle_adam_step(p, n, 0, lr, beta1, beta2, eps, wd, step,
                            inv_loss_scale);
}

/* --------------------------------------------------------- FP8 reduction */

/* Local reduction of k FP8 shards of one tensor.  Shard j is the numel codes
 * at src + j * stride (format in_fmt, encoded with scale scales[j]).  Each
 * element's reduced value is
 *     y = (((x_0 + x_1) + x_2) + ... + x_{k-1}) * post,
 *     x_j = decode(code_j) * (1 / s_j),
 * every product and sum rounded to fp32 on its own; then y is cast to out_fmt
 * exactly as oracle_cast_scaled casts an fp32 tensor.  Returns 0, or -1 on a
 * bad argument. */
static int or_reduce_values(const uint8_t *src, int64_t numel, int64_t stride,
                            const float *scales, int k, int in_fmt, int out_fmt,
                            float post, float *y)
{
    if (numel < 0 || k < 1 || k > 64 || stride < numel || in_fmt < 0 ||
        in_fmt > 1 || out_fmt < 0 || out_fmt > 1)
        return -1;
    float r[64];
    for (int j = 0; j < k; ++j) r[j] = 1.0f / scales[j];
    for (int64_t i = 0; i < numel; ++i) {
        float acc = oracle_fp8_decode(src[i], in_fmt) * r[0];
        for (int j = 1; j < k; ++j)
            acc = acc + oracle_fp8_decode(src[(int64_t)j * stride + i], in_fmt) * r[j];
        y[i] = acc * post;
    }
    return 0;
}

int oracle_reduce_scaled(const uint8_t *src, int64_t numel, int64_t stride,
                         const float *scales, int k, int in_fmt, int out_fmt,
                         float post, uint8_t *codes, float *amax_out,
                         float *scale_out)
{
    float *y = malloc((size_t)(numel > 0 ? numel : 1) * sizeof(float));
    if (y == NULL) return -1;
    int rc = or_reduce_values(src, numel, stride, scales, k, in_fmt, out_fmt,
                              post, y);
    if (rc == 0)
        rc = oracle_cast_scaled(y, OR_F32, numel, out_fmt, codes, amax_out,
                                scale_out);
    free(y);
    return rc;
}

/* The reduction above with its output scale taken from a given amax instead
 * of the codes' own: scale = fp8_max(out_fmt) / amax with the cast's
 * guards.  A tensor reduced in pieces (element ranges of every shard) gives
 * the whole tensor's codes when each piece takes the whole tensor's amax,
 * the largest of the pieces' own.  Returns 0, or -1 on a bad argument. */
int oracle_reduce_scaled_given(const uint8_t *src, int64_t numel, int64_t stride,
                               const float *scales, int k, int in_fmt,
                               int out_fmt, float post, float amax,
                               uint8_t *codes, float *scale_out)
{
    float *y = malloc((size_t)(numel > 0 ? numel : 1) * sizeof(float));
    if (y == NULL) return -1;
    int rc = or_reduce_values(src, numel, stride, scales, k, in_fmt, out_fmt,
                              post, y);
    if (rc == 0) {
        *scale_out = oracle_scale_from_amax(amax, out_fmt);
        or_cast_encode(y, OR_F32, numel, out_fmt, *scale_out, codes);
    }
    free(y);
    return rc;
}

/* Exact sum of the squared values of n FP8 codes, in units of 2^-32, as a
 * 128-bit integer: out[0] the low and out[1] the high 64 bits.  Every code
 * value is a multiple of 2^-16, so each square is an integer count of
 * 2^-32.  Non-finite codes count 0 (they set found_inf instead). */
void oracle_fp8_sq_sum(const uint8_t *codes, int64_t n, int fmt, uint64_t *out)
{
    unsigned __int128 acc = 0;
    for (int64_t i = 0; i < n; ++i) {
        float x = oracle_fp8_decode(codes[i], fmt);
        if (!isfinite(x)) continue;
        uint64_t r = (uint64_t)ldexp(fabs((double)x), 16);   /* exact */
        acc += (unsigned __int128)r * r;
    }
    out[0] = (uint64_t)acc;
    out[1] = (uint64_t)(acc >> 64);
}

/* ------------------------------------------------ gradient norm, clipping */

/* The per-tensor terms of the norm below: terms[t] = k_t^2 * S_t rounded
 * to double once (k_t^2 is exact in double; S_t, the exact sum of squared
 * code values, is rounded to double first).  Returns 1 when found_inf (some
 * unscaled g not finite; the terms are then not meaningful), else 0; -1 on
 * a bad argument. */
int oracle_grad_norm_terms(const oracle_param *p, int n, float inv_loss_scale,
                           double *terms)
{
    if (n < 0) return -1;
    int found = 0;
    for (int t = 0; t < n; ++t) {
        float k = or_grad_factor(&p[t], inv_loss_scale);
        unsigned __int128 sum = 0;
        for (int64_t i = 0; i < p[t].numel; ++i) {
            if (!isfinite(or_grad(&p[t], k, i))) { found = 1; continue; }
            double d = fabs((double)oracle_fp8_decode(p[t].g[i], p[t].g_fmt));
            uint64_t q = (uint64_t)ldexp(d, 16);           /* exact integer */
            sum += (unsigned __int128)q * q;
        }
        double kk = (double)k * (double)k;
        terms[t] = kk * ldexp((double)sum, -32);
    }
    return found;
}

/* Global L2 norm of the unscaled gradient of a step call, the quantity a
 * training loop clips (torch.nn.utils.clip_grad_norm_ in the run script's
 * --clip-grad).  Element i of tensor t is g = decode(code) * k_t, k_t the
 * step's factor inv_loss_scale / g_scale.  The norm is
 *     sqrt( sum over t, in tensor order, of k_t^2 * S_t ),
 *     S_t = sum over i of decode(code_i)^2, taken exactly,
 * where each k_t^2 * S_t is rounded to double once (k_t^2 is exact in double
 * and S_t is rounded to double first), each sum in tensor order is rounded to
 * double, and the root is the correctly rounded double root.  Decoded codes
 * are integer multiples of 2^-16, so S_t is an integer count of 2^-32 held
 * here in 128 bits.  Returns 1 with *norm = +inf when found_inf (some g not
 * finite, the step's test), else 0; -1 on a bad argument. */
int oracle_grad_norm(const oracle_param *p, int n, float inv_loss_scale,
                     double *norm)
{
    if (n < 0) return -1;
    double *terms = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (terms == NULL) return -1;
    int found = oracle_grad_norm_terms(p, n, inv_loss_scale, terms);
    double total = 0.0;
    for (int t = 0; t < n; ++t) total = total + terms[t];
    free(terms);
    if (found != 0) { *norm = INFINITY; return found; }
    *norm = sqrt(total);
    return 0;
}

/* Clip coefficient of a global norm: max_norm / (norm + 1e-6) in double,
 * rounded to float, when that is below 1; 1 (no clipping) otherwise or when
 * max_norm <= 0. */
float oracle_clip_coef(double norm, float max_norm)
{
    if (!(max_norm > 0.0f)) return 1.0f;
    double c = (double)max_norm / (norm + 1e-6);
    return c < 1.0 ? (float)c : 1.0f;
}

/* The Adam / AdamW step with global gradient-norm clipping: the norm of the
 * unscaled gradient (oracle_grad_norm) gives the coefficient c
 * (oracle_clip_coef), and every tensor's factor becomes k_t * c, rounded to
 * float, when c < 1.  found_inf is decided on the unclipped gradient.  *norm
 * receives the norm (+inf when found_inf).  Returns as oracle_adam_step. */
int oracle_adam_step_clipped(const oracle_param *p, int n, int l2, float lr,
                             float beta1, float beta2, float eps, float wd,
                             int64_t step, float inv_loss_scale,
                             float max_norm, double *norm)
{
    if (n < 0 || step < 1) return -1;
    int found = oracle_grad_norm(p, n, inv_loss_scale, norm);
    if (found != 0) return found;
    return or_adam_step(p, n, l2, lr, beta1, beta2, eps, wd, step,
                        inv_loss_scale, oracle_clip_coef(*norm, max_norm));
}

/* The step with a given clip coefficient (oracle_adam_step_clipped after
 * the norm): every tensor's factor becomes k_t * clip when clip != 1. */
int oracle_adam_step_coef(const oracle_param *p, int n, int l2, float lr,
                          float beta1, float beta2, float eps, float wd,
                          int64_t step, float inv_loss_scale, float clip)
{
    return or_adam_step(p, n, l2, lr, beta1, beta2, eps, wd, step,
                        inv_loss_scale, clip);
}

/* Optimizer-state bytes per parameter for a level of the MS-AMP table:
 * first moment + second moment.  FP32+FP32 for FP16 AMP and O1 (level 0, 1),
 * FP8+FP16 for O2 and O3 (level 2, 3); -1 for another level. */
int oracle_state_bytes(int level)
{
    switch (level) {
    case 0: case 1: return (int)(sizeof(float) + sizeof(float));
    case 2: case 3: return (int)(sizeof(uint8_t) + sizeof(uint16_t));
    default: return -1;
    }
}

/* ------------------------------------------------------ array entry points */

/* Element-wise forms of the codecs above, for tests over many values. */
void oracle_fp8_encode_array(const float *x, int64_t n, int fmt, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_encode(x[i], fmt);
}

void oracle_fp8_decode_array(const uint8_t *c, int64_t n, int fmt, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_decode(c[i], fmt);
}

void oracle_f32_to_f16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f16_to_f32_array(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(h[i]);
}
