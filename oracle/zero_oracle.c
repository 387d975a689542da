/*
 * Oracle for the ZeRO stage-1/2/3 sharded mixed-precision optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, scalar CPU statement of
 * what the sharded step computes.  It exists so that tests, the smoke check and
 * the CPU-baseline leg of the benchmark have something obviously correct to
 * compare the CUDA library against.  Nothing on the product path may link,
 * load or call it, and it shares no code, header or constant with the CUDA
 * library.  Build flags: -O2 -ffp-contract=off, so every fp32 operation below
 * is rounded on its own (no fused multiply-add), in the order written.
 *
 * Sources (the pages this follows):
 *  - "ZeRO and FSDP" (zerotofrontier.app), section "The idea, one stage at a
 *    time": flatten all parameters into one vector, cut it into n_dp equal
 *    contiguous shards, rank r owns shard r; stage 1 reduce-scatters so rank r
 *    receives the averaged gradient of shard r, updates its fp32 master shard,
 *    casts to bf16 and all-gathers.
 *  - same page, exercise "A sharded Adam step": Adam with bias correction at
 *    step t (t starts at 1), epsilon added outside the square root.
 *  - "DeepSpeed ZeRO" (ozercemkelahmet.com), "The configuration file", and
 *    "ZeRO Optimizer, in depth" (aicassindra.com), "Running it with DeepSpeed":
 *    the optimizer is AdamW with a weight_decay parameter (decoupled decay).
 *  - "ZeRO and FSDP", "The idea, one stage at a time", paragraph on gradient
 *    accumulation: stage 1 adds each micro-batch's full local gradient into a
 *    full buffer and communicates once; stage 2 reduce-scatters after every
 *    micro-batch.
 *  - "ZeRO and FSDP", "FSDP, ZeRO-3 inside PyTorch": each unit is flattened
 *    into one contiguous buffer, gathering a unit is one all-gather.
 *
 * Readings taken where the pages are silent (each one also listed in the
 * design notes):
 *  - shards are equal; the flat vector is padded at its tail so that the shard
 *    length S is a multiple of an alignment a: S = round_up(ceil(N/n_dp), a);
 *  - the gradient mean sums in fp32, ranks in ascending order, starting from
 *    +0.0f, then divides once by the divisor;
 *  - AdamW: m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g); mh = m/bc1;
 *    vh = v/bc2; w = w - (lr*wd)*w; w = w - lr*(mh/(sqrt(vh)+eps)); every
 *    hyper-parameter is an fp32 value; bc1 = 1-b1^t and bc2 = 1-b2^t are
 *    evaluated in fp64 from those fp32 values and rounded once to fp32;
 *    (1-b1), (1-b2) and lr*wd are formed in fp32;
 *  - bf16 cast: round to nearest, ties to even; a NaN stays a NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper half of an fp32 bit pattern, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to the even neighbour.
 * The kept part is the upper 16 bits; the dropped part is the lower 16 bits,
 * compared against one half of the kept part's last place (0x8000).  Adding
 * one to the kept part carries into the exponent by itself, so the largest
 * finite values round up to infinity when they should. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint32_t exponent = (u >> 23) & 0xffu;
    uint32_t mantissa = u & 0x7fffffu;
    if (exponent == 0xffu && mantissa != 0u) {
        /* NaN: keep the sign and the top payload bits, force it quiet. */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u) {
        kept += 1u;
    } else if (dropped == 0x8000u) {
        if (kept & 1u) kept += 1u;
    }
    return (uint16_t)kept;
}

void oracle_cast_bf16(const float* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Layout: flatten, pad, shard, bucket                                       */
/* ------------------------------------------------------------------------ */

/* "ZeRO and FSDP", "The idea, one stage at a time": all parameters are
 * flattened into one vector cut into n_dp equal contiguous shards, rank r
 * owning shard r (equal shards with tail padding: the reading taken above).
 * out[0] = N (real elements), out[1] = S (shard length), out[2] = P = n_dp*S
 * (padded length), out[3] = bucket length rounded up to a multiple of a,
 * out[4] = number of buckets covering [0, P).  offsets (may be NULL) receives
 * each tensor's start in the flat vector: the tensors are laid end to end in
 * the order given, with no padding between them.  Returns 0, or -1 for an
 * argument no layout exists for, or -2 when a size does not fit in int64. */
int oracle_layout(const int64_t* numel, int32_t n_tensors, int32_t n_dp,
                  int64_t align, int64_t bucket, int64_t* offsets, int64_t* out)
{
    if (n_tensors < 0 || n_dp < 1 || align < 1 || bucket < 1 || out == NULL) return -1;
    if (n_tensors > 0 && numel == NULL) return -1;
    int64_t total = 0;
    for (int32_t i = 0; i < n_tensors; ++i) {
        if (numel[i] < 0) return -1;
        if (offsets) offsets[i] = total;
        if (numel[i] > INT64_MAX / 4 - total) return -2;
        total += numel[i];
    }
    int64_t per_rank = total / n_dp;
    if (per_rank * n_dp < total) per_rank += 1;           /* ceil(N / n_dp) */
    int64_t shard = per_rank / align;
    if (shard * align < per_rank) shard += 1;
    if (shard > INT64_MAX / 4 / align) return -2;
    shard *= align;                                        /* round up to a */
    if (shard > INT64_MAX / 4 / n_dp) return -2;
    int64_t padded = shard * n_dp;
    int64_t bq = bucket / align;
    if (bq * align < bucket) bq += 1;
    if (bq > INT64_MAX / 4 / align) return -2;
    bq *= align;
    int64_t nb = padded / bq;
    if (nb * bq < padded) nb += 1;
    out[0] = total;
    out[1] = shard;
    out[2] = padded;
    out[3] = bq;
    out[4] = nb;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Reduce-scatter as a mean                                                  */
/* ------------------------------------------------------------------------ */

/* "ZeRO and FSDP", "The idea, one stage at a time" (stage 1: rank r receives
 * the average over ranks of shard r of the gradients) and exercise "A sharded
 * Adam step", step (1).
 * g[i] = (sum over r = 0..n_src-1 of src[r*ld + i]) / divisor, fp32, ranks in
 * ascending order.  src rows are bf16 bit patterns. */
void oracle_reduce_mean_bf16(const uint16_t* src, int32_t n_src, int64_t ld, int64_t n,
                             float divisor, float* g)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_src; ++r) s = s + oracle_bf16_to_f32(src[(int64_t)r * ld + i]);
        g[i] = s / divisor;
    }
}

/* The same with fp32 rows (accumulated gradients). */
void oracle_reduce_mean_f32(const float* src, int32_t n_src, int64_t ld, int64_t n,
                            float divisor, float* g)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_src; ++r) s = s + src[(int64_t)r * ld + i];
        g[i] = s / divisor;
    }
}

/* ------------------------------------------------------------------------ */
/* AdamW on one shard                                                        */
/* ------------------------------------------------------------------------ */

/* "ZeRO and FSDP", exercise "A sharded Adam step", step (2): the bias
 * corrections 1 - beta1^t and 1 - beta2^t at step t >= 1 (fp64 from the fp32
 * betas, rounded once to fp32: the reading taken above). */
void oracle_bias_corrections(float b1, float b2, int64_t t, float* bc1, float* bc2)
{
    *bc1 = (float)(1.0 - pow((double)b1, (double)t));
    *bc2 = (float)(1.0 - pow((double)b2, (double)t));
}

/* One AdamW step at step t (t >= 1) on n elements, in place on w, m, v:
 * Adam as in "ZeRO and FSDP", exercise "A sharded Adam step", step (2), with
 * the decoupled weight decay of the "AdamW" optimizer blocks ("DeepSpeed
 * ZeRO", "The configuration file"). */
void oracle_adamw(float* w, float* m, float* v, const float* g, int64_t n,
                  float lr, float b1, float b2, float eps, float wd, int64_t t)
{
    float bc1, bc2;
    oracle_bias_corrections(b1, b2, t, &bc1, &bc2);
    float one_minus_b1 = 1.0f - b1;
    float one_minus_b2 = 1.0f - b2;
    float lr_wd = lr * wd;
    for (int64_t i = 0; i < n; ++i) {
        float gi = g[i];
        float mi = b1 * m[i] + one_minus_b1 * gi;
        float vi = b2 * v[i] + one_minus_b2 * (gi * gi);
        float m_hat = mi / bc1;
        float v_hat = vi / bc2;
        float wi = w[i];
        wi = wi - lr_wd * wi;                              /* decoupled decay */
        wi = wi - lr * (m_hat / (sqrtf(v_hat) + eps));     /* Adam step */
        m[i] = mi;
        v[i] = vi;
        w[i] = wi;
    }
}

/* ------------------------------------------------------------------------ */
/* The ZeRO-1/2 step over n_dp simulated ranks                               */
/* ------------------------------------------------------------------------ */

/* grads:   n_dp rows of P = n_dp*S bf16, row r = rank r's full local gradient.
 * w/m/v:   n_dp rows of S fp32, row o = rank o's shard of the master weights
 *          and moments (updated in place).
 * full_w:  n_copies rows of P bf16; after the all-gather every rank holds the
 *          full bf16 weights, so every row is written with the same vector
 *          (n_copies = n_dp reproduces every rank's copy; 1 keeps one).
 * Steps ("ZeRO and FSDP", exercise "A sharded Adam step"): (1) reduce-scatter:
 * rank o receives the mean over ranks of shard o; (2) AdamW on rank o's own
 * shard only; (3) cast to bf16 and all-gather. */
int oracle_zero_step(const uint16_t* grads, int32_t n_dp, int64_t shard,
                     float* w, float* m, float* v, uint16_t* full_w, int32_t n_copies,
                     float lr, float b1, float b2, float eps, float wd, int64_t t)
{
    if (n_dp < 1 || shard < 0 || t < 1) return -1;
    int64_t padded = shard * n_dp;
    float* g = (float*)malloc(sizeof(float) * (size_t)(shard > 0 ? shard : 1));
    if (!g) return -3;
    for (int32_t o = 0; o < n_dp; ++o) {
        /* (1) rank o's piece of the reduce-scatter */
        oracle_reduce_mean_bf16(grads + (int64_t)o * shard, n_dp, padded, shard,
                                (float)n_dp, g);
        /* (2) update rank o's shard */
        oracle_adamw(w + (int64_t)o * shard, m + (int64_t)o * shard, v + (int64_t)o * shard,
                     g, shard, lr, b1, b2, eps, wd, t);
    }
    free(g);
    /* (3) all-gather of the bf16 casts: each rank receives every shard */
    for (int32_t c = 0; c < n_copies; ++c)
        for (int32_t o = 0; o < n_dp; ++o)
            for (int64_t i = 0; i < shard; ++i)
                full_w[(int64_t)c * padded + (int64_t)o * shard + i] =
                    oracle_f32_to_bf16(w[(int64_t)o * shard + i]);
    return 0;
}

/* Plain data parallelism ("ZeRO and FSDP", "The idea, one stage at a time":
 * stages 1 and 2 compute exactly what data parallelism computes, a ring
 * all-reduce being a reduce-scatter followed by an all-gather), for the
 * invariant that a ZeRO-1/2 step equals it:
 * all-reduce the gradients as a mean (same order), then every rank runs the
 * full AdamW step on its own full copy of the state (n_dp rows of P fp32) and
 * casts its full weights (n_dp rows of P bf16). */
int oracle_dp_step(const uint16_t* grads, int32_t n_dp, int64_t padded,
                   float* w, float* m, float* v, uint16_t* full_w,
                   float lr, float b1, float b2, float eps, float wd, int64_t t)
{
    if (n_dp < 1 || padded < 0 || t < 1) return -1;
    float* g = (float*)malloc(sizeof(float) * (size_t)(padded > 0 ? padded : 1));
    if (!g) return -3;
    oracle_reduce_mean_bf16(grads, n_dp, padded, padded, (float)n_dp, g);
    for (int32_t r = 0; r < n_dp; ++r) {
        oracle_adamw(w + (int64_t)r * padded, m + (int64_t)r * padded, v + (int64_t)r * padded,
                     g, padded, lr, b1, b2, eps, wd, t);
        oracle_cast_bf16(w + (int64_t)r * padded, full_w + (int64_t)r * padded, padded);
    }
    free(g);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation                                                     */
/* ------------------------------------------------------------------------ */

/* "ZeRO and FSDP", "The idea, one stage at a time", paragraph on gradient
 * accumulation.
 * Stage 1: a rank adds one micro-batch's full local bf16 gradient into its
 * full fp32 buffer (first = 1 starts the buffer with this micro-batch). */
void oracle_accumulate_local(float* acc, const uint16_t* g, int64_t n, int32_t first)
{
    for (int64_t i = 0; i < n; ++i) {
        float x = oracle_bf16_to_f32(g[i]);
        acc[i] = first ? x : acc[i] + x;
    }
}

/* Stage 2 (and the stage-3 layer reduce-scatter): the owner adds the sum over
 * ranks of one micro-batch's slice into its fp32 shard buffer.  src: n_src
 * rows of bf16 with row stride ld. */
void oracle_accumulate_reduce(float* acc, const uint16_t* src, int32_t n_src, int64_t ld,
                              int64_t n, int32_t first)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_src; ++r) s = s + oracle_bf16_to_f32(src[(int64_t)r * ld + i]);
        acc[i] = first ? s : acc[i] + s;
    }
}

/* ------------------------------------------------------------------------ */
/* All-gather (stage 3 per-unit gather, and the stage-1/2 weight gather)      */
/* ------------------------------------------------------------------------ */

/* "ZeRO and FSDP", stage 1's all-gather and "FSDP, ZeRO-3 inside PyTorch"
 * (gathering a unit is one all-gather of its flat buffer):
 * full[o*S + i] = shards[o*S + i], the concatenation of the n_dp shards. */
void oracle_all_gather_bf16(const uint16_t* shards, int32_t n_dp, int64_t shard, uint16_t* full)
{
    for (int32_t o = 0; o < n_dp; ++o)
        for (int64_t i = 0; i < shard; ++i)
            full[(int64_t)o * shard + i] = shards[(int64_t)o * shard + i];
}

/* ------------------------------------------------------------------------ */
/* Clipping by the global gradient norm                                     */
/* ------------------------------------------------------------------------ */

/* The configurations of "DeepSpeed ZeRO" ("The configuration file") and "ZeRO
 * Optimizer, in depth" ("Running it with DeepSpeed") set gradient_clipping to
 * 1.0: the gradient is scaled so that its global L2 norm does not exceed it.
 * Reading taken (the pages give no formula): the global norm is the L2 norm of
 * the mean gradient over all elements, ||g|| = sqrt(sum g_i^2); the scale is
 * min(1, max_norm / (||g|| + 1e-6)), applied as one fp32 multiply.  Each
 * square of an fp32 value is exact in fp64; the squares are summed in fp64
 * with Neumaier's compensation (A. Neumaier, "Rundungsfehleranalyse einiger
 * Verfahren zur Summation endlicher Summen", ZAMM 54, 1974): the running sum
 * plus a running correction that collects every addition's rounding error, so
 * that for these non-negative terms the result is within a few units in the
 * last place of the exact sum whatever the number of terms (a plain running
 * fp64 sum drifts by up to about n units).  The quotient is taken in fp64 and
 * rounded once to fp32. */

typedef struct {
    double sum, comp;
} oracle_csum;

static void oracle_csum_add(oracle_csum* k, double x)
{
    double t = k->sum + x;
    if (fabs(k->sum) >= fabs(x))
        k->comp = k->comp + ((k->sum - t) + x);
    else
        k->comp = k->comp + ((x - t) + k->sum);
    k->sum = t;
}

static double oracle_csum_value(const oracle_csum* k)
{
    return k->sum + k->comp;
}

double oracle_grad_norm_sq_bf16(const uint16_t* src, int32_t n_src, int64_t ld, int64_t n,
                                float divisor)
{
    oracle_csum acc = {0.0, 0.0};
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_src; ++r) s = s + oracle_bf16_to_f32(src[(int64_t)r * ld + i]);
        double g = (double)(s / divisor);
        oracle_csum_add(&acc, g * g);
    }
    return oracle_csum_value(&acc);
}

double oracle_grad_norm_sq_f32(const float* src, int32_t n_src, int64_t ld, int64_t n,
                               float divisor)
{
    oracle_csum acc = {0.0, 0.0};
    for (int64_t i = 0; i < n; ++i) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_src; ++r) s = s + src[(int64_t)r * ld + i];
        double g = (double)(s / divisor);
        oracle_csum_add(&acc, g * g);
    }
    return oracle_csum_value(&acc);
}

float oracle_clip_coef(double norm_sq, float max_norm)
{
    float c = (float)((double)max_norm / (sqrt(norm_sq) + 1e-6));
    return c < 1.0f ? c : 1.0f;
}

void oracle_scale(float* g, int64_t n, float coef)
{
    for (int64_t i = 0; i < n; ++i) g[i] = g[i] * coef;
}

/* ------------------------------------------------------------------------ */
/* 8-bit quantized weight gather (ZeRO++)                                    */
/* ------------------------------------------------------------------------ */

/* "ZeRO Optimizer, in depth" ("Offload and ZeRO++": zero_quantized_weights
 * quantises the weight all-gather) and "ZeRO and FSDP" ("Fewer bytes on the
 * wire": the weight all-gather quantized to 8 bits).  Reading taken (the
 * pages give no format): each owner quantizes its own bf16 shard in blocks of
 * `block` consecutive elements (the last block of a shard may be shorter);
 * symmetric int8 with one fp32 scale per block, scale = max|w| / 127; each
 * weight is multiplied by the block's inverse scale inv = 127 / max|w| (both
 * one fp32 division per block) and rounded to the nearest integer, ties to
 * even, clamped to [-127, 127]; an all-zero block has scale 0 and q = 0.  A
 * receiver rebuilds bf16 weights as the RNE bf16 cast of the fp32 product
 * q * scale.  Weights must be finite. */

void oracle_quantize_int8(const uint16_t* w, int64_t n, int32_t block, int8_t* q, float* scales)
{
    int64_t nb = n / block;
    if (nb * block < n) nb += 1;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t lo = b * block;
        int64_t hi = lo + block < n ? lo + block : n;
        float amax = 0.0f;
        for (int64_t i = lo; i < hi; ++i) {
            float a = fabsf(oracle_bf16_to_f32(w[i]));
            if (a > amax) amax = a;
        }
        scales[b] = amax / 127.0f;
        if (amax == 0.0f) {
            for (int64_t i = lo; i < hi; ++i) q[i] = 0;
            continue;
        }
        float inv = 127.0f / amax;
        for (int64_t i = lo; i < hi; ++i) {
            float r = nearbyintf(oracle_bf16_to_f32(w[i]) * inv);   /* ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[i] = (int8_t)r;
        }
    }
}

void oracle_dequantize_int8(const int8_t* q, const float* scales, int64_t n, int32_t block,
                            uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16((float)q[i] * scales[i / block]);
}

/* ------------------------------------------------------------------------ */
/* 8-bit quantized gradient reduce-scatter (ZeRO++)                          */
/* ------------------------------------------------------------------------ */

/* "ZeRO Optimizer, in depth" ("Offload and ZeRO++": zero_quantized_gradients
 * quantises the gradient reduce-scatter) and "ZeRO and FSDP" ("Fewer bytes on
 * the wire": gradients quantized during the reduce-scatter).  Reading taken
 * (the pages give neither the format nor the bit width): each rank quantizes
 * the slice of its bf16 gradient that goes to owner o -- the elements
 * [o*S, (o+1)*S) -- in the 8-bit block format of the weight gather above
 * (oracle_quantize_int8 over that slice).  The owner turns every received
 * code back into an fp32 gradient value, the code times its block's scale
 * rounded once to fp32 (no bf16 rounding in between), and then takes the same
 * fp32 mean over ranks as for bf16 gradients (oracle_reduce_mean_f32). */
void oracle_dequantize_grad_int8(const int8_t* codes, const float* block_scales, int64_t n,
                                 int32_t block, float* out)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = (float)codes[k] * block_scales[k / block];
}
