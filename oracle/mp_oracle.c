/*
 * mp_oracle.c — plain CPU oracle of the mixed-precision AdamW + stochastic
 * rounding step. TEST INFRASTRUCTURE ONLY (see mp_oracle.h): used by the
 * tests, the smoke check and the benchmark's CPU baseline, never by the
 * product. Written for a reader to check against the pages by eye: one
 * element at a time, in the order the pages give the operations.
 */
#include "mp_oracle.h"

#include <math.h>
#include <string.h>

/* bf16 is the top half of an fp32 bit pattern ([LLMC] §2.1: floatX = bf16,
 * same exponent as fp32, 7-bit mantissa), so widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t float_to_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* ---- Rounding randomness ----------------------------------------------
 * [LLMC] §2.3 and §7: the rounding draws come from SquirrelNoise5 through
 * its 2D entry (Get2dNoiseUint), which makes every draw a pure function of
 * its coordinates and the seed. SquirrelNoise5 is Squirrel Eiserloh's
 * published noise hash: multiply by a constant, add the seed, then four
 * rounds alternating an xor with a right shift (9, 11, 13, 15, 17) and an
 * add or multiply by a further constant. Its 2D form folds y into x with
 * the prime 198491317. Here the coordinates are the low and high 32 bits
 * of the global element index. */
uint32_t oracle_noise_u32(uint64_t k, uint32_t seed)
{
    const uint32_t x = (uint32_t)(k & 0xFFFFFFFFu);
    const uint32_t y = (uint32_t)(k >> 32);
    uint32_t bits = x + 198491317u * y;

    bits *= 0xD2A80A3Fu;
    bits += seed;
    bits ^= bits >> 9;
    bits += 0xA884F197u;
    bits ^= bits >> 11;
    bits *= 0x6C736F4Bu;
    bits ^= bits >> 13;
    bits += 0xB79F3ABBu;
    bits ^= bits >> 15;
    bits *= 0x1B56C4F5u;
    bits ^= bits >> 17;
    return bits;
}

void oracle_noise_fill(uint32_t* out, uint64_t first, uint64_t n, uint32_t seed)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = oracle_noise_u32(first + i, seed);
}

/* ---- Stochastic rounding -------------------------------------------------
 * [LLMC] §2.3: keep the top 16 bits of the fp32 pattern; the low 16 bits are
 * the discarded fraction of one bf16 step. Round to the neighbour away from
 * zero ("ceil" of the magnitude) when that fraction exceeds a uniform 16-bit
 * draw, else truncate ("floor"): the probability of going up is lo16/65536,
 * so the result equals the input in expectation. Incrementing the 16-bit
 * pattern carries into the exponent correctly. NaN maps to the canonical
 * quiet NaN, since truncating a NaN with only low mantissa bits set would
 * give an infinity. */
uint16_t oracle_sr_with_rand(float x, uint32_t rand16)
{
    if (isnan(x))
        return 0x7FC0u;
    const uint32_t b = float_to_bits(x);
    const uint32_t lo16 = b & 0xFFFFu;
    const uint32_t truncated = b >> 16;
    if (lo16 > rand16)
        return (uint16_t)(truncated + 1u);
    return (uint16_t)truncated;
}

uint16_t oracle_sr(float x, uint64_t k, uint32_t seed)
{
    return oracle_sr_with_rand(x, oracle_noise_u32(k, seed) & 0xFFFFu);
}

void oracle_stochastic_round(uint16_t* out, const float* in,
                             uint64_t global_offset, uint64_t n, uint32_t seed)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = oracle_sr(in[i], global_offset + i, seed);
}

/* ---- Stochastic rounding to fp16 -------------------------------------------
 * [LLMC] §6 notes that fp16 stochastic rounding is unfinished upstream. Read
 * here as [LLMC] §2.3's rule on fp16's grid: between the fp16 neighbour a
 * toward zero and the next one b away from zero (b = a + one fp16 step, the
 * step past the largest finite value giving infinity), round away from zero
 * when the discarded fraction f = (|x| - |a|) / (|b| - |a|), cut to 16 bits
 * (floor(f * 65536)), exceeds the 16-bit draw. For fp16 normal values the
 * fraction has 13 bits, so the rounding is unbiased exactly; for fp16
 * subnormal values it is cut to 16 bits. Magnitudes of 65536 and above
 * become infinity (they lie beyond the step after the largest finite fp16),
 * NaN the canonical quiet NaN 0x7E00; the sign is kept. Computed here in
 * double from the values, not from bit patterns. */
static double fp16_value(uint16_t h) /* a finite non-negative pattern */
{
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    return e == 0 ? ldexp((double)m, -24) : ldexp(1024.0 + m, e - 25);
}

uint16_t oracle_sr_fp16_with_rand(float x, uint32_t rand16)
{
    if (isnan(x))
        return 0x7E00u;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    const double ax = fabs((double)x);
    if (ax >= 65536.0)
        return (uint16_t)(sign | 0x7C00u);
    /* a: the largest fp16 pattern whose value is <= |x| (a binary search over
     * the ordered non-negative finite patterns 0x0000 .. 0x7BFF) */
    uint32_t lo = 0, hi = 0x7BFF;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) / 2;
        if (fp16_value((uint16_t)mid) <= ax)
            lo = mid;
        else
            hi = mid - 1;
    }
    const double a = fp16_value((uint16_t)lo);
    const double step = lo == 0x7BFF ? 32.0 : fp16_value((uint16_t)(lo + 1)) - a;
    const double f = (ax - a) / step; /* exact: step is a power of two */
    const uint32_t frac16 = (uint32_t)floor(f * 65536.0);
    const uint32_t up = frac16 > rand16 ? 1u : 0u;
    return (uint16_t)(sign | (lo + up)); /* 0x7BFF + 1 = 0x7C00, infinity */
}

void oracle_stochastic_round_fp16(uint16_t* out, const float* in, uint64_t global_offset, uint64_t n,
                                  uint32_t seed)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = oracle_sr_fp16_with_rand(in[i], oracle_noise_u32(global_offset + i, seed) & 0xFFFFu);
}

/* ---- Accumulation with stochastic rounding -------------------------------
 * [LLMC] §2.3: the same rounding also writes the embedding gradients of the
 * encoder's backward pass (dwte, dwpe): the stored bf16 gradient is widened
 * to fp32, the new fp32 contribution added, and the sum written back to bf16
 * by stochastic rounding, so small contributions are kept in expectation
 * instead of being rounded away. Keyed on (global index, seed) like every
 * other draw here. */
void oracle_accumulate_sr(uint16_t* acc, const float* delta, uint64_t global_offset, uint64_t n,
                          uint32_t seed)
{
    for (uint64_t i = 0; i < n; ++i) {
        const float sum = bf16_bits_to_float(acc[i]) + delta[i];
        acc[i] = oracle_sr(sum, global_offset + i, seed);
    }
}

/* ---- Gradient norm ---------------------------------------------------------
 * [LLMC] §4: the global norm of all gradients, then the clip scale
 * min(1, 1.0 / grad_norm). The threshold 1.0 is an argument here. */
double oracle_sumsq_from(double s, const uint16_t* grads, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) {
        const double g = (double)bf16_bits_to_float(grads[i]);
        s += g * g;
    }
    return s;
}

double oracle_sumsq(const uint16_t* grads, uint64_t n)
{
    return oracle_sumsq_from(0.0, grads, n);
}

float oracle_clip_scale(float norm, float clip)
{
    if (!isfinite(norm))
        return NAN; /* the step must refuse to run on a non-finite norm */
    const float q = clip / norm; /* norm == 0 gives +Inf, so the min is 1 */
    return q < 1.0f ? q : 1.0f;
}

void oracle_grad_norm(const uint16_t* grads, uint64_t n, float clip,
                      double* sumsq, float* norm, float* scale)
{
    const double s = oracle_sumsq(grads, n);
    const float nf = (float)sqrt(s);
    if (sumsq)
        *sumsq = s;
    if (norm)
        *norm = nf;
    if (scale)
        *scale = oracle_clip_scale(nf, clip);
}

/* ---- ZeRO-1 norm --------------------------------------------------------
 * [LLMC] §4: under ZeRO-1 each rank takes the sum of squares of its own
 * shard only, and the per-rank sums are combined across ranks into the
 * global norm. Reading taken here: the `count` per-rank sums are added in
 * rank order, left to right, in fp64; the norm and clip scale then follow
 * oracle_grad_norm. With one part this is oracle_grad_norm's result. */
void oracle_norm_from_parts(const double* parts, int32_t count, float clip,
                            double* sumsq, float* norm, float* scale)
{
    double s = 0.0;
    for (int32_t r = 0; r < count; ++r)
        s += parts[r];
    const float root = (float)sqrt(s);
    if (sumsq)
        *sumsq = s;
    if (norm)
        *norm = root;
    if (scale)
        *scale = oracle_clip_scale(root, clip);
}

/* ---- Learning-rate schedules ----------------------------------------------
 * [LLMC] §4 names four schedules (cosine, linear, constant, WSD) without
 * formulas. Reading taken here, for the 1-based step t the update uses:
 *   warm-up (t <= warmup): lr_max * t / warmup
 *   afterwards, with p = (t - warmup) / (total - warmup) clamped to [0, 1]:
 *     constant  lr_max
 *     cosine    lr_min + (lr_max - lr_min) * (1 + cos(pi * p)) / 2
 *     linear    lr_max - (lr_max - lr_min) * p
 *     WSD       lr_max while p <= 1 - f (warm-up, stable), then linear from
 *               lr_max to lr_min over the last fraction f of the steps:
 *               lr_max - (lr_max - lr_min) * (p - (1 - f)) / f
 * all in double, rounded to float once. Returns NaN for t < 1 or an invalid
 * schedule (unknown kind, warmup < 0, total <= warmup for a decaying kind,
 * f outside (0, 1] for WSD). */
float oracle_lr(int32_t kind, int64_t warmup, int64_t total, float lr_max, float lr_min,
                float decay_frac, int64_t t)
{
    if (t < 1 || warmup < 0 || kind < 0 || kind > 3)
        return NAN;
    if (kind != 0 && total <= warmup)
        return NAN;
    if (kind == 3 && !(decay_frac > 0.0f && decay_frac <= 1.0f))
        return NAN;
    const double hi = (double)lr_max, lo = (double)lr_min;
    if (t <= warmup)
        return (float)(hi * (double)t / (double)warmup);
    if (kind == 0)
        return lr_max;
    double p = (double)(t - warmup) / (double)(total - warmup);
    if (p > 1.0)
        p = 1.0;
    double lr;
    if (kind == 1) {
        const double pi = 3.14159265358979323846; /* the double nearest pi */
        lr = lo + (hi - lo) * (1.0 + cos(pi * p)) / 2.0;
    } else if (kind == 2) {
        lr = hi - (hi - lo) * p;
    } else {
        const double f = (double)decay_frac;
        lr = (p <= 1.0 - f) ? hi : hi - (hi - lo) * (p - (1.0 - f)) / f;
    }
    return (float)lr;
}

/* ---- Bias correction ----------------------------------------------------
 * [LLMC] §2.2 divides m and v by their bias corrections (m_hat, v_hat) and
 * §4 passes t = step + 1; [CMU13] §1.7: the moments start at zero, so their
 * averages are pulled towards zero by the factor 1 - beta^t. */
void oracle_bias_corrections(float beta1, float beta2, int32_t t,
                             float* bc1, float* bc2)
{
    *bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    *bc2 = (float)(1.0 - pow((double)beta2, (double)t));
}

/* lerp(start, end, w) = start + w * (end - start) as two FMAs, as [LLMC]
 * §2.2 says the kernel does: w * end + (start - w * start). */
static float lerp_two_fma(float start, float end, float w)
{
    return fmaf(w, end, fmaf(-w, start, start));
}

/* ---- The AdamW step ------------------------------------------------------
 * [LLMC] §2.2, per parameter, in fp32:
 *   grad = grad_scale * (float)grads[i]
 *   m = lerp(grad, m, beta1);  v = lerp(grad*grad, v, beta2)
 *   old = master ? master[i] : (float)params[i]
 *   p = old - lr * (m_hat / (sqrt(v_hat) + eps) + wd * old)
 *   params[i] = stochastic_round(p);  master[i] = p
 * with wd applied only to tensors that decay (§2.2: matrices and embeddings,
 * not LayerNorm weights or biases) — [CMU13] §1.7's decoupled decay. */
int oracle_adamw_step(uint16_t* params, const uint16_t* grads, float* master,
                      float* m, float* v,
                      uint64_t global_offset, uint64_t n,
                      const oracle_tensor* table, int32_t n_tensors,
                      float lr, float beta1, float beta2, float eps,
                      float weight_decay, float scale,
                      int32_t t, uint32_t seed)
{
    if (!isfinite(scale))
        return 5;

    /* The tensors must cover every element of the range. */
    uint64_t covered = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
        const uint64_t lo = table[k].offset;
        const uint64_t hi = table[k].offset + table[k].size;
        const uint64_t a = lo > global_offset ? lo : global_offset;
        const uint64_t b = hi < global_offset + n ? hi : global_offset + n;
        if (b > a)
            covered += b - a;
    }
    if (covered != n)
        return -1;

    float bc1, bc2;
    oracle_bias_corrections(beta1, beta2, t, &bc1, &bc2);

    for (int32_t k = 0; k < n_tensors; ++k) {
        const float wd = table[k].decay ? weight_decay : 0.0f;
        const uint64_t lo = table[k].offset;
        const uint64_t hi = table[k].offset + table[k].size;
        const uint64_t a = lo > global_offset ? lo : global_offset;
        const uint64_t b = hi < global_offset + n ? hi : global_offset + n;
        for (uint64_t gi = a; gi < b; ++gi) {
            const uint64_t i = gi - global_offset;

            const float grad = scale * bf16_bits_to_float(grads[i]);
            const float m_new = lerp_two_fma(grad, m[i], beta1);
            const float gg = grad * grad;
            const float v_new = lerp_two_fma(gg, v[i], beta2);
            const float m_hat = m_new / bc1;
            const float v_hat = v_new / bc2;

            const float old = master ? master[i] : bf16_bits_to_float(params[i]);
            const float denom = sqrtf(v_hat) + eps;
            const float update = m_hat / denom + wd * old;
            const float p = old - lr * update;

            m[i] = m_new;
            v[i] = v_new;
            params[i] = oracle_sr(p, gi, seed);
            if (master)
                master[i] = p;
        }
    }
    return 0;
}

/* ---- Outlier skip --------------------------------------------------------
 * [LLMC] §4: before the update, the train step feeds the grad norm to an
 * outlier detector holding a window of 128 past values; if the norm's
 * z-score is above a threshold the update is skipped. Reading taken here:
 * z = (x - mean) / std over the 128 most recent finite norms (population
 * standard deviation, both sums in array-slot order), z is NaN while fewer
 * than 128 norms have been seen, the check happens before x joins the
 * window, a threshold <= 0 never skips, and a non-finite norm never enters
 * the window (the step is refused for it anyway). */
int oracle_outlier_check(oracle_outlier* st, float norm, float z_threshold,
                         float* scale, double* z)
{
    const double x = (double)norm;
    double zz = NAN;
    if (st->count >= ORACLE_OUTLIER_WINDOW) {
        double sum = 0.0;
        for (int i = 0; i < ORACLE_OUTLIER_WINDOW; ++i)
            sum += st->window[i];
        const double mean = sum / ORACLE_OUTLIER_WINDOW;
        double ss = 0.0;
        for (int i = 0; i < ORACLE_OUTLIER_WINDOW; ++i) {
            const double d = st->window[i] - mean;
            ss += d * d;
        }
        const double sd = sqrt(ss / ORACLE_OUTLIER_WINDOW);
        zz = (x - mean) / sd;
    }
    *z = zz;
    int status = 0;
    if (z_threshold > 0.0f && zz > (double)z_threshold) {
        *scale = NAN;
        status = 8;
    }
    if (isfinite(x)) {
        st->window[st->count % ORACLE_OUTLIER_WINDOW] = x;
        st->count += 1;
    }
    return status;
}
