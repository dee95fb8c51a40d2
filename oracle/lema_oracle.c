/*
 * lema_oracle.c -- CPU oracle for the selective-full-fine-tuning optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, scalar reference that
 * the CUDA path is checked against.  Only the test suite, the package smoke test
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library, and it includes nothing from it.
 *
 * What it computes, and where the pages say so
 * (page "LEMA: Layer-wise Efficient Memory Abstraction"):
 *   - Section "Selective Full Fine-Tuning": the optimizer states and the gradient
 *     accumulators are fp32; AdamW runs layer by layer; checkpoints hold the fp32
 *     difference between the updated and the original weights.
 *   - Section "Quick Start": the optimizer named is torch.optim.AdamW, so the update
 *     follows that convention: decoupled weight decay applied to the weight before
 *     the Adam update, bias correction on both moments, eps added outside the
 *     square root of the bias-corrected second moment.
 *   - Section "Features" / "TensorStore": fp32 optimizer states live in RAM and are
 *     streamed like the weights (that residency does not change the arithmetic).
 * The pages print no formula and no values for the step; the fixed operation order
 * below is this project's reading (each operation rounded to fp32, round to
 * nearest even, no fused multiply-add, subnormals kept).
 *
 * Build: plain C, -O2 -ffp-contract=off -fno-fast-math -fno-tree-vectorize.
 * The optional OpenMP pragmas only split the element loops (and, for 8-bit
 * states, the loops over 256-element blocks) across threads, for the timed CPU
 * baseline and to check whole workloads in reasonable time; every element (every
 * block) is independent, so results are identical for any thread count.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 ---- */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, sizeof u); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, sizeof x); return x; }

/* bf16 is the top half of an fp32 bit pattern, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round an fp32 value to the nearest bf16, ties to even.
 * Finite values: add 0x7FFF plus the lowest kept bit, keep the top 16 bits; a carry
 * out of the mantissa bumps the exponent, and past the largest finite bf16 it lands
 * on the infinity pattern.  Infinities pass through unchanged.  Any NaN becomes the
 * canonical quiet NaN 0x7FC0 (sign dropped), the convention of PyTorch's CPU
 * conversion. */
uint16_t oracle_f32_to_bf16_rne(float x)
{
    if (isnan(x)) return (uint16_t)0x7FC0u;
    uint32_t u = f32_bits(x);
    uint32_t lsb = (u >> 16) & 1u;
    u = u + 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16_rne(x[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* h, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(h[i]);
}

/* ------------------------------------------------- gradient accumulation ---- */

/* One micro-step of fp32 gradient accumulation: acc[i] = acc[i] + (fp32) g[i].
 * Section "Selective Full Fine-Tuning": gradient accumulation is fp32. */
void oracle_accum(float* acc, const uint16_t* g_bf16, int64_t n, int threads)
{
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t i = 0; i < n; ++i) {
        float g = oracle_bf16_to_f32(g_bf16[i]);
        acc[i] = acc[i] + g;
    }
}

/* ------------------------------------------------ per-call fp32 scalars ---- */

typedef struct {
    float decay;           /* (fp32)(1 - lr*wd)                     */
    float beta1;           /* (fp32) beta1                          */
    float one_minus_beta1; /* (fp32)(1 - beta1), formed in fp64     */
    float beta2;           /* (fp32) beta2                          */
    float one_minus_beta2; /* (fp32)(1 - beta2), formed in fp64     */
    float step_size;       /* (fp32)(lr / (1 - beta1^t))            */
    float bc2_sqrt;        /* (fp32) sqrt(1 - beta2^t)              */
    float eps;             /* (fp32) eps                            */
    float accum_steps;     /* (fp32) K, the number of micro-steps   */
} oracle_scalars;

/* Hyperparameters arrive as fp64.  beta^t is the product of t factors of beta,
 * multiplied one at a time in fp64; each derived scalar is formed in fp64 and
 * rounded once to fp32.  The step counter t is 1-based.
 * Returns 0, or -1 for arguments outside the method's domain. */
int oracle_make_scalars(int64_t step, double lr, double beta1, double beta2,
                        double eps, double weight_decay, int32_t accum_steps,
                        oracle_scalars* s)
{
    if (step < 1 || accum_steps < 1) return -1;
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0)) return -1;
    if (!(eps > 0.0) || !(lr >= 0.0) || !(weight_decay >= 0.0)) return -1;
    if (!(lr * weight_decay < 1.0)) return -1;

    double beta1_pow_t = 1.0, beta2_pow_t = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        beta1_pow_t = beta1_pow_t * beta1;
        beta2_pow_t = beta2_pow_t * beta2;
    }
    double bias_correction1 = 1.0 - beta1_pow_t;
    double bias_correction2 = 1.0 - beta2_pow_t;

    s->decay = (float)(1.0 - lr * weight_decay);
    s->beta1 = (float)beta1;
    s->one_minus_beta1 = (float)(1.0 - beta1);
    s->beta2 = (float)beta2;
    s->one_minus_beta2 = (float)(1.0 - beta2);
    s->step_size = (float)(lr / bias_correction1);
    s->bc2_sqrt = (float)sqrt(bias_correction2);
    s->eps = (float)eps;
    s->accum_steps = (float)accum_steps;
    return 0;
}

/* ---------------------------------------------------------- AdamW step ---- */

/* One bias-corrected AdamW step with decoupled weight decay on fp32 master
 * weights and fp32 moments, for n elements.  Per element, in this order, every
 * operation rounded to fp32:
 *   g     = acc / K                      mean of the K accumulated micro-batch grads
 *   w     = master * decay               decoupled weight decay
 *   m     = beta1*m + (1-beta1)*g        first moment
 *   v     = beta2*v + (1-beta2)*(g*g)    second moment
 *   den   = sqrt(v) / sqrt(bc2) + eps
 *   w     = w - step_size * (m / den)
 *   delta = w - (fp32) orig              cumulative change since the original weight
 *   w_bf16 = round_to_nearest_even_bf16(w)
 * Outputs may alias the matching inputs (master_out == master_in etc.). */
void oracle_adamw_step(int64_t n,
                       const float* master_in, const float* m_in, const float* v_in,
                       const float* acc, const uint16_t* orig_bf16,
                       float* master_out, float* m_out, float* v_out,
                       float* delta, uint16_t* w_bf16,
                       const oracle_scalars* s, int threads)
{
    const float decay = s->decay;
    const float b1 = s->beta1, omb1 = s->one_minus_beta1;
    const float b2 = s->beta2, omb2 = s->one_minus_beta2;
    const float step_size = s->step_size, bc2_sqrt = s->bc2_sqrt;
    const float eps = s->eps, K = s->accum_steps;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t i = 0; i < n; ++i) {
        float g = acc[i] / K;

        float w = master_in[i] * decay;

        float m_old_part = b1 * m_in[i];
        float m_new_part = omb1 * g;
        float m = m_old_part + m_new_part;

        float g_sq = g * g;
        float v_old_part = b2 * v_in[i];
        float v_new_part = omb2 * g_sq;
        float v = v_old_part + v_new_part;

        float root_v = sqrtf(v);
        float root_v_hat = root_v / bc2_sqrt;
        float den = root_v_hat + eps;

        float ratio = m / den;
        float update = step_size * ratio;
        w = w - update;

        float orig = oracle_bf16_to_f32(orig_bf16[i]);
        float d = w - orig;

        master_out[i] = w;
        m_out[i] = m;
        v_out[i] = v;
        delta[i] = d;
        w_bf16[i] = oracle_f32_to_bf16_rne(w);
    }
}

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ============================================ int8 states (8-bit format) ==== */
/*
 * Section "Quantization" of the same page: Adam moments and gradient accumulators
 * may be kept as 8-bit integers (opt_state_bits = 8, grad_acc_bits = 8) and are
 * expanded to full precision only within each layer's AdamW update.  The page does
 * not fix the format; this project's reading:
 *   - blocks of Q8_BLOCK = 256 consecutive elements of a tensor (the last one
 *     ragged), one fp32 scale per block;
 *   - signed fields (m, the accumulator): code q in [-127, 127], stored scale
 *     s = absmax / 127; q = nearest-even integer to x * (127 / absmax), the
 *     reciprocal formed once per block (all codes 0 when absmax or s is 0);
 *     value q * s;
 *   - the second moment is stored as r = sqrt(v): code c in [0, 255], stored scale
 *     t = rmax / 255, c = min(ceil(r * (255 / rmax)), 255) (rounded up, so the
 *     stored second moment does not understate the true one beyond rounding),
 *     value r = c * t, v = r * r;
 *   - a block whose largest magnitude is below 2^-100 is stored as all zeros with
 *     scale 0 (such moments change no update; it keeps 127/absmax finite).
 * Every division, product and square root is one fp32 operation.
 */
#define Q8_BLOCK 256

static int64_t q8_blocks(int64_t n) { return (n + Q8_BLOCK - 1) / Q8_BLOCK; }

/* Quantize one block of nb signed values. */
static void q8_encode_signed(const float* x, int64_t nb, int8_t* q, float* scale)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < nb; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    if (amax < 0x1p-100f) amax = 0.0f;
    float s = amax / 127.0f;
    *scale = s;
    float inv = s == 0.0f ? 0.0f : 127.0f / amax;
    for (int64_t i = 0; i < nb; ++i) {
        if (s == 0.0f) { q[i] = 0; continue; }
        float k = rintf(x[i] * inv);
        if (k > 127.0f) k = 127.0f;
        if (k < -127.0f) k = -127.0f;
        q[i] = (int8_t)k;
    }
}

/* Quantize one block of nb non-negative roots, rounding codes up. */
static void q8_encode_root(const float* r, int64_t nb, uint8_t* c, float* scale)
{
    float rmax = 0.0f;
    for (int64_t i = 0; i < nb; ++i)
        if (r[i] > rmax) rmax = r[i];
    if (rmax < 0x1p-100f) rmax = 0.0f;
    float t = rmax / 255.0f;
    *scale = t;
    float inv = t == 0.0f ? 0.0f : 255.0f / rmax;
    for (int64_t i = 0; i < nb; ++i) {
        if (t == 0.0f) { c[i] = 0; continue; }
        float k = ceilf(r[i] * inv);
        if (k > 255.0f) k = 255.0f;
        c[i] = (uint8_t)k;
    }
}

void oracle_q8_encode_signed(const float* x, int64_t n, int8_t* q, float* scale)
{
    for (int64_t b = 0; b < q8_blocks(n); ++b) {
        int64_t lo = b * Q8_BLOCK, nb = n - lo < Q8_BLOCK ? n - lo : Q8_BLOCK;
        q8_encode_signed(x + lo, nb, q + lo, scale + b);
    }
}

void oracle_q8_decode_signed(const int8_t* q, const float* scale, int64_t n, float* x)
{
    for (int64_t i = 0; i < n; ++i) x[i] = (float)q[i] * scale[i / Q8_BLOCK];
}

void oracle_q8_encode_root(const float* r, int64_t n, uint8_t* c, float* scale)
{
    for (int64_t b = 0; b < q8_blocks(n); ++b) {
        int64_t lo = b * Q8_BLOCK, nb = n - lo < Q8_BLOCK ? n - lo : Q8_BLOCK;
        q8_encode_root(r + lo, nb, c + lo, scale + b);
    }
}

void oracle_q8_decode_root(const uint8_t* c, const float* scale, int64_t n, float* r)
{
    for (int64_t i = 0; i < n; ++i) r[i] = (float)c[i] * scale[i / Q8_BLOCK];
}

/* One micro-step into an 8-bit accumulator: per block, decode (or start from +0
 * when first != 0), add the fp32 grads, encode again.  Blocks are independent; the
 * OpenMP pragma only splits the block loop over `threads` host cores. */
void oracle_accum_q8(int8_t* acc_q, float* acc_scale, const uint16_t* g_bf16, int64_t n,
                     int first, int threads)
{
    const int64_t n_blocks = q8_blocks(n);
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t b = 0; b < n_blocks; ++b) {
        float tmp[Q8_BLOCK];
        int64_t lo = b * Q8_BLOCK, nb = n - lo < Q8_BLOCK ? n - lo : Q8_BLOCK;
        for (int64_t i = 0; i < nb; ++i) {
            float a = first ? 0.0f : (float)acc_q[lo + i] * acc_scale[b];
            tmp[i] = a + oracle_bf16_to_f32(g_bf16[lo + i]);
        }
        q8_encode_signed(tmp, nb, acc_q + lo, acc_scale + b);
    }
}

/* The AdamW step on 8-bit moments: decode m, v (from its root) and the
 * accumulated grads, run the fp32 update of oracle_adamw_step element by element,
 * encode m and sqrt(v) again per block.  When grad_last is given it is the K-th
 * micro-batch grad, added to the decoded accumulator (acc_q may then be NULL for
 * K = 1); the accumulator itself is not written.  Blocks are independent; the
 * OpenMP pragma only splits the block loop over `threads` host cores. */
void oracle_adamw_step_q8(int64_t n, const float* master_in,
                          const int8_t* m_q_in, const float* m_scale_in,
                          const uint8_t* r_q_in, const float* r_scale_in,
                          const int8_t* acc_q, const float* acc_scale,
                          const uint16_t* grad_last, const uint16_t* orig_bf16,
                          float* master_out, int8_t* m_q_out, float* m_scale_out,
                          uint8_t* r_q_out, float* r_scale_out,
                          float* delta, uint16_t* w_bf16, const oracle_scalars* s,
                          int threads)
{
    const float decay = s->decay;
    const float b1 = s->beta1, omb1 = s->one_minus_beta1;
    const float b2 = s->beta2, omb2 = s->one_minus_beta2;
    const float step_size = s->step_size, bc2_sqrt = s->bc2_sqrt;
    const float eps = s->eps, K = s->accum_steps;
    const int64_t n_blocks = q8_blocks(n);
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t b = 0; b < n_blocks; ++b) {
        float m_new[Q8_BLOCK], r_new[Q8_BLOCK];
        int64_t lo = b * Q8_BLOCK, nb = n - lo < Q8_BLOCK ? n - lo : Q8_BLOCK;
        for (int64_t j = 0; j < nb; ++j) {
            int64_t i = lo + j;
            float sum = acc_q ? (float)acc_q[i] * acc_scale[b] : 0.0f;
            if (grad_last) sum = sum + oracle_bf16_to_f32(grad_last[i]);
            float g = sum / K;

            float w = master_in[i] * decay;

            float m_old = (float)m_q_in[i] * m_scale_in[b];
            float m_old_part = b1 * m_old;
            float m_new_part = omb1 * g;
            float m = m_old_part + m_new_part;

            float r_old = (float)r_q_in[i] * r_scale_in[b];
            float v_old = r_old * r_old;
            float g_sq = g * g;
            float v_old_part = b2 * v_old;
            float v_new_part = omb2 * g_sq;
            float v = v_old_part + v_new_part;

            float root_v = sqrtf(v);
            float root_v_hat = root_v / bc2_sqrt;
            float den = root_v_hat + eps;

            float ratio = m / den;
            float update = step_size * ratio;
            w = w - update;

            master_out[i] = w;
            delta[i] = w - oracle_bf16_to_f32(orig_bf16[i]);
            w_bf16[i] = oracle_f32_to_bf16_rne(w);
            m_new[j] = m;
            r_new[j] = root_v;
        }
        q8_encode_signed(m_new, nb, m_q_out + lo, m_scale_out + b);
        q8_encode_root(r_new, nb, r_q_out + lo, r_scale_out + b);
    }
}

/* ================================================================ merge ==== */
/* Section "Selective Full Fine-Tuning", its paragraph on checkpoints and serving:
 * a servable model is the base model plus the saved fp32 delta.  Per element:
 * merged = round_to_nearest_even_bf16((fp32) base + delta), one fp32 add. */
void oracle_merge_delta(const uint16_t* base_bf16, const float* delta, int64_t n,
                        uint16_t* merged_bf16)
{
    for (int64_t i = 0; i < n; ++i) {
        float sum = oracle_bf16_to_f32(base_bf16[i]) + delta[i];
        merged_bf16[i] = oracle_f32_to_bf16_rne(sum);
    }
}
