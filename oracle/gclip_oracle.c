/*
 * gclip_oracle.c -- CPU oracle for global L2-norm gradient clipping.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only at the seeded input generators.
 *
 * What it computes, and where that is defined:
 *
 *  - "Grow a language model: gradient clipping" (unhomeschool.com, Russian),
 *    section "Mathematics": the global norm is the square root of the sum of
 *    g_i^2 over every element of every parameter; if norm <= max_norm the
 *    gradients pass unchanged, otherwise every element is multiplied by
 *    max_norm / norm.  The section "Why computing the grad norm needs three
 *    kernels" gives the serial form used here: one accumulator, every tensor
 *    in order, every element in order, then one square root.
 *  - "Gradient Clipping" (paweldubiel.com glossary), section "Mechanism and
 *    details", the piecewise equation: g~ = g when ||g||_2 <= c, and
 *    c g / ||g||_2 when ||g||_2 > c, for c > 0.  The comparison is strict.
 *  - Same glossary page, section "Order changes the result": with loss
 *    scaling the gradients are unscaled first, so the threshold refers to
 *    their true size; with accumulation the clip runs on the whole effective
 *    batch.  "Grow a language model: backprop" (unhomeschool.com, Vietnamese),
 *    section "Accumulation across microbatches": the accumulated buffer is
 *    averaged by 1/n_microbatches.  Both factors arrive here as one
 *    multiplier, inv_scale, applied to every element before squaring.
 *  - Glossary page, section "Shorten the arrow, keep the direction": a NaN or
 *    infinity needs diagnosis and an explicit stop of the update.  Reading
 *    taken: a nonfinite element raises the flag and every gradient is left
 *    exactly as it was.
 *
 * Precision: every element is widened exactly to double; the products and the
 * running sum are double; the square root and the division are the IEEE
 * double operations of libm.  Outputs are rounded once, to nearest-even, into
 * the tensor's own storage format.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *  - no epsilon is added to the norm in the divisor (the pages divide by the
 *    norm itself, and the division only happens when norm > max_norm > 0);
 *  - a sum of squares above the largest finite fp32 value counts as
 *    nonfinite, because the product accumulates in fp32 and would hold inf;
 *  - fp16 / bf16 gradients are rewritten in place in their own format.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2

#define OR_DECISION_PASS 0
#define OR_DECISION_CLIP 1
#define OR_DECISION_SKIP 2

typedef struct {
    const void *data;  /* host memory, element type per dtype */
    int64_t numel;
    int32_t dtype;     /* OR_F32, OR_F16, OR_BF16 */
    int32_t pad;
} oracle_tensor;

typedef struct {
    double sumsq;      /* sum of (x * inv_scale)^2 over every element */
    double norm;       /* sqrt(sumsq) */
    double coef;       /* multiplier applied to x * inv_scale (1 on PASS) */
    int32_t nonfinite; /* 1 if an element is NaN/inf or sumsq > FLT_MAX */
    int32_t decision;  /* OR_DECISION_* */
} oracle_result;

/* Planted mistakes for the mutation tests: compiled in only when the test
 * suite rebuilds this file with -DORACLE_MUTANT=<n>, to show that the pins
 * catch each one.  The default build has ORACLE_MUTANT == 0. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ------------------------------------------------------------------------ */
/* Storage formats.  IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10
 * fraction bits.  bfloat16: the upper 16 bits of a binary32. */

static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

static double decode_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

double oracle_decode(const void *data, int64_t i, int32_t dtype)
{
    if (dtype == OR_F32) {
        float x;
        memcpy(&x, (const char *)data + 4 * i, 4);
        return (double)x;
    }
    uint16_t h;
    memcpy(&h, (const char *)data + 2 * i, 2);
    return dtype == OR_F16 ? decode_f16(h) : decode_bf16(h);
}

/* Round |a| (finite, > 0) to nearest-even on the grid of a binary format with
 * p significand bits (hidden bit included) and minimum normal exponent emin.
 * Returns the rounded magnitude as an integer multiple n of the quantum
 * 2^qexp, so that the caller can assemble the bit pattern. */
static void round_grid(double a, int p, int emin, int64_t *n, int *qexp)
{
    int ex;
    frexp(a, &ex);               /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;              /* floor(log2 a) */
    if (e < emin)
        e = emin;                /* subnormal range shares emin's quantum */
    *qexp = e - (p - 1);
    double r = ldexp(a, -*qexp); /* exact: scaling by a power of two */
    double fl = floor(r);
    double d = r - fl;           /* exact: r < 2^(p+1) has few integer bits */
    int64_t k = (int64_t)fl;
    if (d > 0.5 || (d == 0.5 && (k & 1)))
        k += 1;
    *n = k;
}

/* binary16 from double, round to nearest even, with overflow to inf. */
static uint16_t encode_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return sign | 0x7e00;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    /* halfway between 65504 (odd significand) and 2^16 rounds up to inf */
    if (a >= 65520.0)
        return sign | 0x7c00;
    int64_t n;
    int qexp;
    round_grid(a, 11, -14, &n, &qexp);
    /* n * 2^qexp with n < 2^11 after normalisation */
    if (n == 2048) {
        n = 1024;
        qexp += 1;
    }
    if (n < 1024)                       /* subnormal (qexp == -24) or zero */
        return sign | (uint16_t)n;
    int e = qexp + 10;                  /* unbiased exponent of n * 2^qexp */
    return sign | (uint16_t)(((e + 15) << 10) | (n - 1024));
}

/* bfloat16 from double: 8 significand bits, binary32 exponent range. */
static uint16_t encode_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return sign | 0x7fc0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    /* largest finite bf16 is (2 - 2^-7) * 2^127; half a step above it
     * rounds up to inf because that significand is odd */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127))
        return sign | 0x7f80;
    int64_t n;
    int qexp;
    round_grid(a, 8, -126, &n, &qexp);
    if (n == 256) {
        n = 128;
        qexp += 1;
    }
    if (n < 128)                        /* subnormal (qexp == -133) or zero */
        return sign | (uint16_t)n;
    int e = qexp + 7;
    return sign | (uint16_t)(((e + 127) << 7) | (n - 128));
}

/* binary32 from double through the same grid rounding, used by the tests to
 * check round_grid against the C conversion (which is IEEE round-to-nearest
 * under the default rounding mode). */
uint32_t oracle_round_grid_f32_bits(double v)
{
    uint32_t sign = signbit(v) ? 0x80000000u : 0;
    if (isnan(v))
        return sign | 0x7fc00000u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= ldexp(2.0 - ldexp(1.0, -24), 127))
        return sign | 0x7f800000u;
    int64_t n;
    int qexp;
    round_grid(a, 24, -126, &n, &qexp);
    if (n == (1 << 24)) {
        n = 1 << 23;
        qexp += 1;
    }
    if (n < (1 << 23))
        return sign | (uint32_t)n;
    int e = qexp + 23;
    return sign | (uint32_t)(((e + 127) << 23) | (n - (1 << 23)));
}

void oracle_encode(void *data, int64_t i, int32_t dtype, double v)
{
    if (dtype == OR_F32) {
        float x = (float)v;  /* IEEE round to nearest even */
        memcpy((char *)data + 4 * i, &x, 4);
        return;
    }
    uint16_t h = dtype == OR_F16 ? encode_f16(v) : encode_bf16(v);
    memcpy((char *)data + 2 * i, &h, 2);
}

static int elem_size(int32_t dtype) { return dtype == OR_F32 ? 4 : 2; }

static int check_dtype(int32_t dtype)
{
    return dtype == OR_F32 || dtype == OR_F16 || dtype == OR_BF16;
}

/* ------------------------------------------------------------------------ */
/* The serial sum of squares (the three-kernel page's naive loop, in double).
 * Returns 0, or -1 for a malformed descriptor. */
int oracle_sumsq(const oracle_tensor *ts, int32_t n_tensors, double inv_scale,
                 double *out_sumsq, int32_t *out_elem_nonfinite)
{
    double total = 0.0;
    int32_t nf = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (ts[t].numel < 0 || !check_dtype(ts[t].dtype))
            return -1;
        for (int64_t i = 0; i < ts[t].numel; ++i) {
            double x = oracle_decode(ts[t].data, i, ts[t].dtype);
            if (!isfinite(x))
                nf = 1;
#if ORACLE_MUTANT == 1
            double y = x;                      /* mistake: unscale dropped */
#elif ORACLE_MUTANT == 2
            double y = x * inv_scale * inv_scale; /* mistake: scale twice */
#else
            double y = x * inv_scale;
#endif
#if ORACLE_MUTANT == 3
            total += fabs(y);                  /* mistake: L1, not L2 */
#elif ORACLE_MUTANT == 4
            if (i + 1 < ts[t].numel)           /* mistake: last elem dropped */
                total += y * y;
#else
            total += y * y;
#endif
        }
#if ORACLE_MUTANT == 5
        break;                                 /* mistake: first tensor only */
#endif
    }
    *out_sumsq = total;
    *out_elem_nonfinite = nf;
    return 0;
}

/* The decision: sum of squares, norm, nonfinite flag, clip or pass, and the
 * multiplier.  Returns 0, or -1 for bad arguments (c <= 0 or nonfinite,
 * inv_scale <= 0 or nonfinite, malformed descriptors). */
static int decide(const oracle_tensor *in, int32_t n_tensors, double max_norm,
                  double inv_scale, oracle_result *res)
{
    if (!(max_norm > 0.0) || !isfinite(max_norm) || !(inv_scale > 0.0) ||
        !isfinite(inv_scale) || n_tensors < 0)
        return -1;
    double s;
    int32_t nf;
    if (oracle_sumsq(in, n_tensors, inv_scale, &s, &nf) != 0)
        return -1;
    if (s > (double)FLT_MAX)
        nf = 1;
    double norm = sqrt(s);

    int32_t decision;
    double coef;
    if (nf) {
        decision = OR_DECISION_SKIP;
        coef = 1.0;
#if ORACLE_MUTANT == 6
    } else if (norm >= max_norm) {             /* mistake: boundary clips */
#else
    } else if (norm > max_norm) {
#endif
        decision = OR_DECISION_CLIP;
#if ORACLE_MUTANT == 7
        coef = norm / max_norm;                /* mistake: ratio inverted */
#elif ORACLE_MUTANT == 8
        coef = max_norm / s;                   /* mistake: no square root */
#else
        coef = max_norm / norm;
#endif
    } else {
        decision = OR_DECISION_PASS;
        coef = 1.0;
    }
    res->sumsq = s;
    res->norm = norm;
    res->coef = coef;
    res->nonfinite = nf;
    res->decision = decision;
    return 0;
}

/* The clipped value of one element, before rounding to its format. */
static double clipped_value(double x, double inv_scale, double coef)
{
#if ORACLE_MUTANT == 9
    return x * coef;                           /* mistake: output not unscaled */
#elif ORACLE_MUTANT == 10
    return -x * inv_scale * coef;              /* mistake: sign flipped */
#else
    return x * inv_scale * coef;
#endif
}

/* Global-norm clip.  `in` and `out` describe the same shapes and dtypes;
 * out[t].data is writable host memory (it may equal in[t].data).  On SKIP
 * the input bits are copied unchanged; on PASS and CLIP every element is
 * rewritten as round(x * inv_scale * coef) in its own format.
 * Returns 0, or -1 for bad arguments. */
int oracle_clip(const oracle_tensor *in, const oracle_tensor *out,
                int32_t n_tensors, double max_norm, double inv_scale,
                oracle_result *res)
{
    for (int32_t t = 0; t < n_tensors; ++t)
        if (out[t].numel != in[t].numel || out[t].dtype != in[t].dtype)
            return -1;
    if (decide(in, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;

    for (int32_t t = 0; t < n_tensors; ++t) {
        int64_t n = in[t].numel;
        int32_t dt = in[t].dtype;
        if (res->decision == OR_DECISION_SKIP) {
            if (out[t].data != in[t].data)
                memcpy((void *)out[t].data, in[t].data,
                       (size_t)n * (size_t)elem_size(dt));
            continue;
        }
        for (int64_t i = 0; i < n; ++i) {
            double x = oracle_decode(in[t].data, i, dt);
            oracle_encode((void *)out[t].data, i, dt,
                          clipped_value(x, inv_scale, res->coef));
        }
    }
    return 0;
}

/* The same clip with the outputs of only `k` chosen elements: element
 * elem[j] of tensor tensor[j] is written, in its tensor's storage format, to
 * out_storage at byte offset 4*j (fp32) or 2*j (fp16/bf16 use the low half
 * of a 4-byte slot).  For sets too large to rewrite whole in the tests.
 * Returns 0, or -1 for bad arguments or an index out of range. */
int oracle_clip_sample(const oracle_tensor *in, int32_t n_tensors,
                       double max_norm, double inv_scale,
                       const int32_t *tensor, const int64_t *elem, int64_t k,
                       void *out_storage, oracle_result *res)
{
    if (decide(in, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;
    for (int64_t j = 0; j < k; ++j) {
        int32_t t = tensor[j];
        if (t < 0 || t >= n_tensors || elem[j] < 0 || elem[j] >= in[t].numel)
            return -1;
        int32_t dt = in[t].dtype;
        char *slot = (char *)out_storage + 4 * j;
        if (res->decision == OR_DECISION_SKIP) {
            memcpy(slot, (const char *)in[t].data + elem_size(dt) * elem[j],
                   (size_t)elem_size(dt));
            continue;
        }
        double x = oracle_decode(in[t].data, elem[j], dt);
        oracle_encode(slot, 0, dt, clipped_value(x, inv_scale, res->coef));
    }
    return 0;
}

/* Gradient accumulation, the last microbatch: every element of acc[t]
 * becomes acc + add, the sum of the two stored values rounded once to nearest
 * even in the tensor's own format.  "Grow a language model: backprop"
 * (unhomeschool.com, Vietnamese), section "Accumulation across
 * microbatches": the backward kernels add their contribution into the
 * gradient buffer (+=), which holds the running sum until zero_grads.  The
 * sum is formed in double and rounded once; double carries more than twice
 * the significand bits of each format plus two, so this is the correctly
 * rounded sum of the format.  Returns 0, or -1 for mismatched descriptors. */
int oracle_accumulate(const oracle_tensor *acc, const oracle_tensor *add, int32_t n_tensors)
{
    for (int32_t t = 0; t < n_tensors; ++t)
        if (acc[t].numel != add[t].numel || acc[t].dtype != add[t].dtype ||
            acc[t].numel < 0 || !check_dtype(acc[t].dtype))
            return -1;
    for (int32_t t = 0; t < n_tensors; ++t) {
        int32_t dt = acc[t].dtype;
        for (int64_t i = 0; i < acc[t].numel; ++i) {
            double a = oracle_decode(acc[t].data, i, dt);
            double b = oracle_decode(add[t].data, i, dt);
#if ORACLE_MUTANT == 16
            double v = a - b;                  /* mistake: addend subtracted */
#else
            double v = a + b;
#endif
            oracle_encode((void *)acc[t].data, i, dt, v);
        }
    }
    return 0;
}

/* The last microbatch's accumulation followed by the clip of the whole
 * buffer, in that order (the glossary page, "Order changes the result": with
 * accumulation the clip acts on the whole effective batch).  acc[t] is
 * rewritten in place: first with the rounded sums, then, on PASS or CLIP,
 * with the clipped values.  On SKIP the sums stay (the accumulation is not
 * part of the stopped update).  Returns 0, or -1 for bad arguments. */
int oracle_clip_accumulate(const oracle_tensor *acc, const oracle_tensor *add,
                           int32_t n_tensors, double max_norm, double inv_scale,
                           oracle_result *res)
{
    if (!(max_norm > 0.0) || !isfinite(max_norm) || !(inv_scale > 0.0) ||
        !isfinite(inv_scale) || n_tensors < 0)
        return -1;
#if ORACLE_MUTANT == 17
    /* mistake: each contribution clipped before it is added */
    if (oracle_clip(acc, acc, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;
    return oracle_accumulate(acc, add, n_tensors);
#else
    if (oracle_accumulate(acc, add, n_tensors) != 0)
        return -1;
    return oracle_clip(acc, acc, n_tensors, max_norm, inv_scale, res);
#endif
}

/* Out-of-place clip into fp32 buffers: the same decision as oracle_clip, and
 * every element x becomes round_fp32(x * inv_scale * coef) in out[t] (fp32
 * host arrays of the tensors' numel); on SKIP the outputs are not written.
 * The gradients are not modified.  For fp16/bf16 gradients under loss
 * scaling this keeps the unscaled values that binary16 could only hold as
 * subnormals (the glossary page, "Order changes the result": unscale before
 * the threshold; the backprop page, "Where gradients live": FP16 gradient
 * buffers). */
int oracle_clip_to_f32(const oracle_tensor *in, void *const *out,
                       int32_t n_tensors, double max_norm, double inv_scale,
                       oracle_result *res)
{
    if (decide(in, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;
    if (res->decision == OR_DECISION_SKIP)
        return 0;
    for (int32_t t = 0; t < n_tensors; ++t)
        for (int64_t i = 0; i < in[t].numel; ++i) {
            double x = oracle_decode(in[t].data, i, in[t].dtype);
#if ORACLE_MUTANT == 19
            oracle_encode(out[t], i, OR_F32, x * inv_scale);  /* mistake: clip factor lost */
#else
            oracle_encode(out[t], i, OR_F32, clipped_value(x, inv_scale, res->coef));
#endif
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Clip, then one AdamW step on the clipped gradients.
 *
 * Order: "Grow a language model: gradient clipping" (unhomeschool.com),
 * section "Order matters: Pre-Adam": the clip runs before the AdamW moments
 * m, v and the weights are updated, so a spike never enters m and v.  Section
 * "ANDREA-120M v1 ... Stability v2": v2 uses AdamW with clipping; section
 * "Adjacent activities": AdamW keeps m and v.  "Grow a language model:
 * backprop", section "Optimizer state": one m and one v per weight.
 *
 * The pages do not write the AdamW update out; the reading taken is the
 * published algorithm with decoupled weight decay and bias correction:
 *   g^ = x * inv_scale * coef             (the clipped, unscaled gradient)
 *   m  = beta1 * m + (1 - beta1) * g^
 *   v  = beta2 * v + (1 - beta2) * g^ * g^
 *   w  = w - lr * wd * w - lr * (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 * w, m, v are fp32 arrays; every value is widened exactly to double and each
 * result is rounded once to fp32.  On SKIP (a nonfinite gradient) nothing is
 * updated and the gradients are not touched.  With zero_grads the gradients
 * are set to +0 after use (the backprop page, "Accumulation across
 * microbatches": zero_grads() resets the buffers after the optimizer step). */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;      /* 1-based */
    int32_t zero_grads;
    int32_t pad;
} oracle_adamw_params;

typedef struct {
    void *w, *m, *v;   /* fp32, numel of the matching gradient tensor */
} oracle_adamw_state;

static float ld_f32(const void *p, int64_t i)
{
    float x;
    memcpy(&x, (const char *)p + 4 * i, 4);
    return x;
}

static void st_f32(void *p, int64_t i, double v)
{
    float x = (float)v;
    memcpy((char *)p + 4 * i, &x, 4);
}

int oracle_clip_adamw(const oracle_tensor *g, const oracle_adamw_state *st,
                      int32_t n_tensors, double max_norm, double inv_scale,
                      const oracle_adamw_params *p, oracle_result *res)
{
    if (p->step < 1 || !(p->lr >= 0.0) || !(p->eps > 0.0) ||
        !(p->beta1 >= 0.0 && p->beta1 < 1.0) ||
        !(p->beta2 >= 0.0 && p->beta2 < 1.0))
        return -1;
    if (decide(g, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;
    if (res->decision == OR_DECISION_SKIP)
        return 0;
    double bc1 = 1.0 - pow(p->beta1, (double)p->step);
    double bc2 = 1.0 - pow(p->beta2, (double)p->step);
    for (int32_t t = 0; t < n_tensors; ++t) {
        for (int64_t i = 0; i < g[t].numel; ++i) {
            double x = oracle_decode(g[t].data, i, g[t].dtype);
#if ORACLE_MUTANT == 14
            double gh = x * inv_scale;         /* mistake: Adam sees the raw gradient */
#else
            double gh = clipped_value(x, inv_scale, res->coef);
#endif
            double w = ld_f32(st[t].w, i);
            double m = ld_f32(st[t].m, i);
            double v = ld_f32(st[t].v, i);
#if ORACLE_MUTANT == 13
            gh += p->weight_decay * w;         /* mistake: L2 decay, not decoupled */
#endif
            m = p->beta1 * m + (1.0 - p->beta1) * gh;
#if ORACLE_MUTANT == 15
            v = p->beta1 * v + (1.0 - p->beta1) * gh * gh;  /* mistake: beta1 in v */
#else
            v = p->beta2 * v + (1.0 - p->beta2) * gh * gh;
#endif
#if ORACLE_MUTANT == 11
            double mh = m, vh = v;             /* mistake: no bias correction */
#else
            double mh = m / bc1, vh = v / bc2;
#endif
#if ORACLE_MUTANT == 12
            double upd = mh / sqrt(vh + p->eps);   /* mistake: eps inside sqrt */
#else
            double upd = mh / (sqrt(vh) + p->eps);
#endif
#if ORACLE_MUTANT == 13
            w = w - p->lr * upd;
#else
            w = w - p->lr * p->weight_decay * w - p->lr * upd;
#endif
            st_f32(st[t].w, i, w);
            st_f32(st[t].m, i, m);
            st_f32(st[t].v, i, v);
            if (p->zero_grads)
                oracle_encode((void *)g[t].data, i, g[t].dtype, 0.0);
        }
    }
    return 0;
}

/* Per-coordinate (value) clipping to [-c, c], the contrast drawn on the
 * glossary page, section "Shorten the arrow, keep the direction": each
 * element is clamped on its own, which can change the direction.  Used only
 * by the tests, never offered by the library. */
void oracle_value_clip(const double *x, int64_t n, double c, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = x[i] > c ? c : (x[i] < -c ? -c : x[i]);
}

/* Per-tensor clipping, the alternative named in the gradient-clipping page's
 * section "Per-Tensor or Global": each tensor is clipped by its own norm.
 * Same conventions as oracle_clip, one result per tensor. */
int oracle_clip_per_tensor(const oracle_tensor *in, const oracle_tensor *out,
                           int32_t n_tensors, double max_norm,
                           double inv_scale, oracle_result *res)
{
#if ORACLE_MUTANT == 18
    /* mistake: the global clip applied to the whole set, its record copied */
    if (oracle_clip(in, out, n_tensors, max_norm, inv_scale, res) != 0)
        return -1;
    for (int32_t t = 1; t < n_tensors; ++t)
        res[t] = res[0];
    return 0;
#else
    for (int32_t t = 0; t < n_tensors; ++t)
        if (oracle_clip(in + t, out + t, 1, max_norm, inv_scale, res + t) != 0)
            return -1;
    return 0;
#endif
}
