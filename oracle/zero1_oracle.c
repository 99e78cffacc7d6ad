/*
 * zero1_oracle.c -- plain, slow, scalar CPU oracle for the ZeRO-1 local-shard
 * optimizer step (accumulate -> global L2 norm + clip -> AdamW -> bf16 copy).
 *
 * TEST INFRASTRUCTURE ONLY.  It is used by tests/, by the package smoke check
 * and by the CPU-baseline leg of the benchmark.  The product path never
 * calls, links or loads it, and it shares no code, header or constant table
 * with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off matters: GCC contracts a*b+c into an FMA by default on
 * Arm, and every fp32 operation below must round exactly once.
 *
 * Arithmetic types: the pages fix fp32 for the optimizer state (master, m, v)
 * and bf16 for the compute weights ("Nanotron Guide", section "Memory &
 * Optimization / 1. ZeRO-1 Optimizer State Partitioning"; "Distributed
 * Training", section 0 "what does training actually need in memory?").  So
 * the element-wise step is fp32 with every operation rounded; the gradient
 * norm, a reduction the pages leave unspecified, is summed in double.
 *
 * Every array here is the local shard list in plan order with no padding:
 * tensor 0's shard, then tensor 1's shard, and so on.
 *
 * Pins: every function below is pinned by a test under tests/ against
 * something other than itself (a library routine, a closed form, a value the
 * pages print, brute force).  None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Shard split.                                                             */
/* "ZeRO-1 风格的 Distributed Optimizer", section 6.3: every parameter is cut  */
/* on its own (not flattened into one blob), its total numel divided evenly */
/* over the dp_size ranks; each rank keeps fp32 master/m/v for its 1/N.     */
/* The page does not say where a remainder goes.  Reading taken: shards are */
/* contiguous and in rank order, and the first (n mod dp) ranks hold one    */
/* extra element (so an n < dp tensor leaves some ranks empty).             */
/* ------------------------------------------------------------------------ */
void oracle_shard_range(int64_t n, int32_t dp, int32_t r, int64_t *start, int64_t *count)
{
    int64_t q = n / dp;
    int64_t rem = n % dp;
    int64_t extra_before = (r < rem) ? r : rem; /* ranks before r that got +1 */
    *count = q + ((r < rem) ? 1 : 0);
    *start = (int64_t)r * q + extra_before;
}

/* Shard every tensor of a list for rank r.  Returns the local element count
 * (the sum of the shard sizes). */
int64_t oracle_plan(const int64_t *numels, int32_t n_tensors, int32_t dp, int32_t r,
                    int64_t *shard_start, int64_t *shard_count)
{
    int64_t local = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        oracle_shard_range(numels[i], dp, r, &shard_start[i], &shard_count[i]);
        local += shard_count[i];
    }
    return local;
}

/* ------------------------------------------------------------------------ */
/* Memory accounting, bytes held by one data-parallel rank.                 */
/* "Distributed Training", section 0: 2 (bf16 weights) + 2 (bf16 grads) +   */
/* 12 (fp32 master, m, v) = 16 bytes per parameter.  "Nanotron Guide",      */
/* section "1. ZeRO-1 Optimizer State Partitioning" itemises a 4-byte       */
/* gradient instead (2+4+4+4+4, i.e. 18).  "ZeRO-1 风格的 Distributed        */
/* Optimizer", sections 6.1 and 6.3: ZeRO-1 keeps the full bf16 weights and  */
/* gradient buffer on every rank and shards only the 12 bytes of optimizer  */
/* state.  out = {weights, grads, optimizer state, total}.                  */
/* ------------------------------------------------------------------------ */
void oracle_zero1_bytes(int64_t total_numel, int64_t local_numel, int32_t grad_bytes,
                        int64_t out[4])
{
    out[0] = 2 * total_numel;
    out[1] = (int64_t)grad_bytes * total_numel;
    out[2] = 12 * local_numel; /* fp32 master + m + v of the local shard */
    out[3] = out[0] + out[1] + out[2];
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32.                                                            */
/* ------------------------------------------------------------------------ */
static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 is the top half of an IEEE binary32, so widening is exact. */
float oracle_bf16_to_f32(uint16_t b)
{
    return f32_from_bits((uint32_t)b << 16);
}

/* Round-to-nearest, ties-to-even, from binary32 to bf16.  The pages do not
 * name a rounding mode for the bf16 weight copy; IEEE's default is taken.
 * The low 16 bits are dropped after adding half an ulp of bf16 minus one,
 * plus the kept LSB (so an exact half rounds towards the even result).  A
 * carry out of the mantissa moves into the exponent, which turns the largest
 * finite values into infinity exactly as RNE requires.  NaN keeps its sign
 * and top payload bits and is forced quiet. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept_lsb = (u >> 16) & 1u;
    u += 0x7fffu + kept_lsb;
    return (uint16_t)(u >> 16);
}

void oracle_bf16_rne_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = oracle_bf16_rne(x[j]);
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation.                                                    */
/* "ZeRO-1 风格的 Distributed Optimizer", section 6.7, and "Distributed       */
/* Training", section 2: K micro-batches run one after another and their    */
/* gradients are added into .grad; "accumulate_grad_in_fp32: true" in the  */
/* "Nanotron Guide" YAML config puts that buffer in fp32.  Reading taken: a  */
/* plain sum in micro-batch order, no division by K (loss scaling belongs   */
/* upstream).  One micro-batch per call, as backward passes arrive; with    */
/* overwrite set, the buffer is assigned (not 0 + g, which would turn a     */
/* -0.0 gradient into +0.0).                                                 */
/* ------------------------------------------------------------------------ */
void oracle_accumulate(float *grad, const uint16_t *micro, int64_t n, int32_t overwrite)
{
    for (int64_t j = 0; j < n; ++j) {
        float g = oracle_bf16_to_f32(micro[j]);
        grad[j] = overwrite ? g : grad[j] + g;
    }
}

/* The average over data-parallel ranks ("TorchTitan 生产级预训练方案",       */
/* appendix B.1: FSDP2 runs a single divide kernel that divides the local   */
/* fp32 reduce-scattered gradient by the world size).  grad[j] = grad[j] /  */
/* divisor, one IEEE fp32 division per element, after the last addition.    */
void oracle_divide(float *grad, int64_t n, float divisor)
{
    for (int64_t j = 0; j < n; ++j)
        grad[j] = grad[j] / divisor;
}

/* ------------------------------------------------------------------------ */
/* Sum of squares for the L2 gradient norm ("ZeRO-1 风格的 Distributed        */
/* Optimizer", section 6.6: clip_grad 1.0; the norm type is not stated, L2  */
/* is taken).  The value wanted is the exact sum of the squares: the clip   */
/* coefficient is rounded once to fp32 from it, so it must not depend on a  */
/* summation order.  The product of two floats is exact in double; the      */
/* running sum is double in index order with a Neumaier compensation term,  */
/* which keeps the result within a few double ulps of the exact sum for any */
/* length (a plain double sum drifts by up to n ulps).                       */
/* ------------------------------------------------------------------------ */
double oracle_sumsq(const float *grad, int64_t n)
{
    double s = 0.0;
    double comp = 0.0; /* the low-order parts lost by the additions to s */
    for (int64_t j = 0; j < n; ++j) {
        double x = (double)grad[j];
        double sq = x * x;
        double t = s + sq;
        if (fabs(s) >= fabs(sq))
            comp += (s - t) + sq;
        else
            comp += (sq - t) + s;
        s = t;
    }
    return s + comp;
}

/* ------------------------------------------------------------------------ */
/* Clip coefficient.  The global norm is sqrt(local sumsq + the other ranks' */
/* sumsq).  Reading taken (the pages give only "clip_grad: 1.0"): the      */
/* gradient is scaled by clip / (norm + 1e-6) when that is below 1, and not  */
/* at all when clip <= 0.  A non-finite norm reports 0 and the step must be  */
/* skipped.  Computed in double, rounded once to float.                      */
/* ------------------------------------------------------------------------ */
int32_t oracle_clip_coef(double sumsq_total, double clip, double *norm_out, float *coef_out)
{
    double norm = sqrt(sumsq_total);
    *norm_out = norm;
    *coef_out = 1.0f;
    if (!isfinite(norm))
        return 0;
    if (clip > 0.0) {
        double q = clip / (norm + 1e-6);
        if (q < 1.0)
            *coef_out = (float)q;
    }
    return 1;
}

/* ------------------------------------------------------------------------ */
/* AdamW on the fp32 master weights, then the bf16 copy.                     */
/* "ZeRO-1 风格的 Distributed Optimizer", section 6.6: adam_w with beta1 0.9, */
/* beta2 0.95, eps 1e-8, weight_decay 0.1 (no formula printed); section 6.2  */
/* and 6.3: each rank steps only its own shard, then ships the updated bf16  */
/* weights in an all-gather.  Reading taken: decoupled weight decay         */
/* (Loshchilov & Hutter) applied to p before the Adam update, bias-corrected */
/* moments, eps added outside the square root.  Step-size scalars are       */
/* computed once in double and rounded once to float:                        */
/*     bc1 = 1 - beta1^t,  stepsize = lr / bc1,  sqrtbc2 = sqrt(1 - beta2^t) */
/*     dfac = 1 - lr*wd (decayed tensors) or 1 (excluded tensors)            */
/* and per element, each fp32 operation rounded:                             */
/*     g = grad*coef;  p = p*dfac;  m = b1*m + (1-b1)*g;                     */
/*     v = b2*v + (1-b2)*(g*g);  d = sqrt(v)/sqrtbc2 + eps;                  */
/*     p = p - stepsize*(m/d);  w = bf16_rne(p)                              */
/* The clipped gradient is used, not written back.                           */
/* ------------------------------------------------------------------------ */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
} oracle_adamw_hp;

/* AdamW with a learning-rate and a weight-decay multiplier per tensor (the
 * "Nanotron Guide", "3. Spectral muTransfer": learning rates scaled per
 * layer class, e.g. eta_hidden = eta_0 / d_model).  Tensor i steps with
 * lr_i = lr * lr_scale[i] and wd_i = weight_decay * wd_scale[i]; every
 * scalar derived from them is computed in double and rounded once, then the
 * per-element update is the one of oracle_adamw below. */
void oracle_adamw_scaled(float *p, float *m, float *v, const float *grad, uint16_t *w,
                         const int64_t *counts, const double *lr_scale, const double *wd_scale,
                         int32_t n_tensors, const oracle_adamw_hp *hp, int64_t t, float coef)
{
    double bc1 = 1.0 - pow(hp->beta1, (double)t);
    double bc2 = 1.0 - pow(hp->beta2, (double)t);
    const float sqrtbc2 = (float)sqrt(bc2);
    const float b1 = (float)hp->beta1;
    const float b2 = (float)hp->beta2;
    const float omb1 = (float)(1.0 - hp->beta1);
    const float omb2 = (float)(1.0 - hp->beta2);
    const float eps = (float)hp->eps;

    int64_t j = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const double lr_i = hp->lr * lr_scale[i];
        const double wd_i = hp->weight_decay * wd_scale[i];
        const float stepsize = (float)(lr_i / bc1);
        const float dfac = (float)(1.0 - lr_i * wd_i);
        for (int64_t e = 0; e < counts[i]; ++e, ++j) {
            float g = grad[j] * coef;
            float pj = p[j] * dfac;
            float mj = b1 * m[j] + omb1 * g;
            float gg = g * g;
            float vj = b2 * v[j] + omb2 * gg;
            float d = sqrtf(vj) / sqrtbc2 + eps;
            float upd = mj / d;
            pj = pj - stepsize * upd;
            p[j] = pj;
            m[j] = mj;
            v[j] = vj;
            if (w)
                w[j] = oracle_bf16_rne(pj);
        }
    }
}

void oracle_adamw(float *p, float *m, float *v, const float *grad, uint16_t *w,
                  const int64_t *counts, const uint8_t *no_decay, int32_t n_tensors,
                  const oracle_adamw_hp *hp, int64_t t, float coef)
{
    double bc1 = 1.0 - pow(hp->beta1, (double)t);
    double bc2 = 1.0 - pow(hp->beta2, (double)t);
    const float stepsize = (float)(hp->lr / bc1);
    const float sqrtbc2 = (float)sqrt(bc2);
    const float b1 = (float)hp->beta1;
    const float b2 = (float)hp->beta2;
    const float omb1 = (float)(1.0 - hp->beta1);
    const float omb2 = (float)(1.0 - hp->beta2);
    const float eps = (float)hp->eps;
    const float dfac_decay = (float)(1.0 - hp->lr * hp->weight_decay);

    int64_t j = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const float dfac = no_decay[i] ? 1.0f : dfac_decay;
        for (int64_t e = 0; e < counts[i]; ++e, ++j) {
            float g = grad[j] * coef;
            float pj = p[j] * dfac;
            float mj = b1 * m[j] + omb1 * g;
            float gg = g * g;
            float vj = b2 * v[j] + omb2 * gg;
            float d = sqrtf(vj) / sqrtbc2 + eps;
            float upd = mj / d;
            pj = pj - stepsize * upd;
            p[j] = pj;
            m[j] = mj;
            v[j] = vj;
            if (w)
                w[j] = oracle_bf16_rne(pj);
        }
    }
}
