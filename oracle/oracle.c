/*
 * oracle.c -- plain fp64 CPU definition of the fused optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this.  The product library never
 * does, and this file shares no code, header or constant with it.
 *
 * What it computes (SomaSpeed page, "Robot learning, at a different pace",
 * its two optimizer paragraphs: the first lists what a step does to each
 * gradient, the second how the work is batched over the tensor list):
 *
 *   1. normalize every gradient for the effective batch: g / d, where d is
 *      the step's divisor or, if its group sets one, the group's own (the
 *      veRL write-up divides the loss by the number of accumulated
 *      micro-batches, 4.2 PPO Update; groups accumulated over different
 *      counts divide by different numbers);
 *   2. measure one global L2 norm of the normalized gradients, where each
 *      owned shard counts once (non-owned, i.e. replicated, tensors do not
 *      enter the sum) and frozen tensors do not enter at all;
 *   3. take one clipping decision from that norm, with the coefficient of
 *      torch.nn.utils.clip_grad_norm_ as called in the veRL write-up
 *      ("veRL Training Process", 4.2 PPO Update, gradient clipping and
 *      optimizer step; max_norm 1.0 in "PPO Update Summary"):
 *          c = min(1, max_norm / (norm + 1e-6));
 *   4. AdamW with decoupled weight decay and bias correction on every
 *      trainable tensor, owned or not, reading g * c / d; the stored
 *      gradient is never written and frozen tensors are never touched.
 *      Weights and moments are kept in fp64 here (the RLinf page, "Retaining
 *      Low-Precision Gradients", converts gradients to FP32 for the update
 *      and keeps FP32 optimizer state; fp64 is the exact-arithmetic stand-in).
 *
 * AdamW is taken in the form of torch.optim.AdamW (non-amsgrad): decay the
 * weight by (1 - lr*wd) first, then
 *     m = b1*m + (1-b1)*g,   v = b2*v + (1-b2)*g^2,
 *     p = p - lr * (m / bc1) / (sqrt(v / bc2) + eps),
 * with bc_k = 1 - b_k^t and t the group's step count after incrementing.
 *
 * Gradients are read in their stored type (fp32, or bf16 or fp16 bits); all
 * convert to fp64 exactly.  fp16 gradients are the compute-dtype gradients
 * of an fp16 policy (RLinf page, "Retaining Low-Precision Gradients").
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_GRAD_F32 0
#define ORACLE_GRAD_BF16 1
#define ORACLE_GRAD_F16 2

typedef struct {
    double *param;      /* fp64 weights, updated in place                */
    const void *grad;   /* stored gradient (fp32 or bf16 bits), read only */
    int32_t grad_dtype; /* ORACLE_GRAD_F32 or ORACLE_GRAD_BF16            */
    int32_t group;      /* index into the group array                    */
    double *exp_avg;    /* fp64 first moment m                           */
    double *exp_avg_sq; /* fp64 second moment v                          */
    int64_t numel;
    int32_t trainable;  /* 0: frozen, skipped entirely                   */
    int32_t owned;      /* 0: replicated, updated but not in the norm    */
} oracle_tensor;

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;   /* steps this group has taken so far */
    double divisor; /* this group's effective-batch divisor; 0 = the step's */
} oracle_group;

/* IEEE 754 binary16 word -> exact fp64: 1 sign bit, 5 exponent bits (bias
 * 15), 10 fraction bits; exponent 0 is subnormal, 31 is inf/NaN. */
static double half_to_double(uint16_t w)
{
    int sign = (w >> 15) & 1, e = (w >> 10) & 0x1f, f = w & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* One stored gradient element as an exact fp64 value.  bf16 is the upper
 * half of an IEEE binary32, so widening it is a 16-bit shift. */
static double grad_element(const void *grad, int32_t dtype, int64_t i)
{
    if (dtype == ORACLE_GRAD_F32)
        return (double)((const float *)grad)[i];
    if (dtype == ORACLE_GRAD_F16)
        return half_to_double(((const uint16_t *)grad)[i]);
    uint32_t bits = ((uint32_t)((const uint16_t *)grad)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Exposed for the decoder's pin: n binary16 words to fp64. */
void oracle_f16_to_f64(const uint16_t *w, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = half_to_double(w[i]);
}

/* Sum over one tensor of the squared normalized gradient, (g_i / d)^2. */
double oracle_tensor_sqsum(const void *grad, int32_t dtype, int64_t numel, double divisor)
{
    double s = 0.0;
    for (int64_t i = 0; i < numel; ++i) {
        double g = grad_element(grad, dtype, i) / divisor;
        s += g * g;
    }
    return s;
}

/* Global L2 norm over trainable, owned tensors (step 2). */
double oracle_global_norm(const oracle_tensor *ts, int64_t n, double divisor)
{
    double total = 0.0;
    for (int64_t k = 0; k < n; ++k) {
        if (!ts[k].trainable || !ts[k].owned)
            continue;
        total += oracle_tensor_sqsum(ts[k].grad, ts[k].grad_dtype, ts[k].numel, divisor);
    }
    return sqrt(total);
}

/* Clip coefficient (step 3).  A NaN norm gives a NaN coefficient, as
 * clip_grad_norm_'s clamp does; an infinite norm gives 0. */
double oracle_clip_coef(double norm, double max_norm)
{
    double c = max_norm / (norm + 1e-6);
    if (isnan(c))
        return c;
    return c < 1.0 ? c : 1.0;
}

/* AdamW on `numel` elements of one tensor at the group's step count `step`
 * (already incremented for this step), reading g * c / d (step 4). */
void oracle_adamw_update(double *p, const void *grad, int32_t dtype, double *m, double *v,
                         int64_t numel, double lr, double beta1, double beta2, double eps,
                         double weight_decay, int64_t step, double c, double divisor)
{
    double bc1 = 1.0 - pow(beta1, (double)step);
    double bc2 = 1.0 - pow(beta2, (double)step);
    for (int64_t i = 0; i < numel; ++i) {
        double g = grad_element(grad, dtype, i) / divisor * c;
        p[i] = p[i] * (1.0 - lr * weight_decay);
        m[i] = beta1 * m[i] + (1.0 - beta1) * g;
        v[i] = beta2 * v[i] + (1.0 - beta2) * g * g;
        double m_hat = m[i] / bc1;
        double v_hat = v[i] / bc2;
        p[i] = p[i] - lr * m_hat / (sqrt(v_hat) + eps);
    }
}

/* One whole step over a tensor list.  Returns 0, or -1 if a trainable
 * tensor names a group outside [0, ngroups); nothing is changed then. */
int oracle_step(oracle_tensor *ts, int64_t n, oracle_group *groups, int32_t ngroups,
                double divisor, double max_norm, double *norm_out, double *coef_out)
{
    for (int64_t k = 0; k < n; ++k)
        if (ts[k].trainable && (ts[k].group < 0 || ts[k].group >= ngroups))
            return -1;

    /* Step 2 with each tensor normalized by its group's divisor (the step's
     * divisor unless the group sets its own). */
    double total = 0.0;
    for (int64_t k = 0; k < n; ++k) {
        if (!ts[k].trainable || !ts[k].owned)
            continue;
        double dk = groups[ts[k].group].divisor > 0.0 ? groups[ts[k].group].divisor : divisor;
        total += oracle_tensor_sqsum(ts[k].grad, ts[k].grad_dtype, ts[k].numel, dk);
    }
    double norm = sqrt(total);
    double c = oracle_clip_coef(norm, max_norm);

    /* A group takes a step when it has at least one trainable tensor. */
    for (int32_t q = 0; q < ngroups; ++q) {
        int present = 0;
        for (int64_t k = 0; k < n && !present; ++k)
            present = ts[k].trainable && ts[k].group == q;
        if (present)
            groups[q].step += 1;
    }

    for (int64_t k = 0; k < n; ++k) {
        if (!ts[k].trainable)
            continue;
        const oracle_group *gp = &groups[ts[k].group];
        oracle_adamw_update(ts[k].param, ts[k].grad, ts[k].grad_dtype, ts[k].exp_avg,
                            ts[k].exp_avg_sq, ts[k].numel, gp->lr, gp->beta1, gp->beta2,
                            gp->eps, gp->weight_decay, gp->step, c,
                            gp->divisor > 0.0 ? gp->divisor : divisor);
    }
    if (norm_out)
        *norm_out = norm;
    if (coef_out)
        *coef_out = c;
    return 0;
}
