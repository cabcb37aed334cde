/*
 * oracle.c -- plain CPU fp64 oracle of one grouped-query-attention decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference legs load this library; the product path never does.
 * It shares no code with the CUDA library.
 *
 * Every function is the plain definition it cites, in the pages' order:
 * explicit rotation of each pair, a full softmax over all visible keys, no
 * splitting, no blocking, no fusion. Floating point is fp64 throughout except
 * where the method fixes a precision: bf16 storage (round to nearest even) and
 * the vq8 quantiser, which is defined in fp32 and is done in fp32 here. Build
 * without fast-math and with -ffp-contract=off so the fp32 steps are IEEE.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

static const double kTwoPi = 6.283185307179586476925286766559;

/* ------------------------------------------------------------------ bf16 */

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* bf16 keeps 8 significant bits and the fp32 exponent range. Scale x so the
 * last kept bit has weight 1, round half to even with nearbyint (default
 * rounding mode), scale back. Below 2^-126 the bit spacing stays 2^-133. */
uint16_t oracle_bf16_from_double(double x)
{
    if (isnan(x)) return 0x7FC0;
    if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    int e;
    frexp(x, &e); /* |x| = m 2^e, 0.5 <= m < 1 */
    int q = e - 8;
    if (q < -133) q = -133;
    double r = ldexp(nearbyint(ldexp(x, -q)), q);
    const double bf16_max = 3.38953138925153547590470800371487866880e38; /* (2 - 2^-7) 2^127 */
    if (fabs(r) > bf16_max) return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

/* ------------------------------------------------------------------ RoPE */

/*
 * Inverse frequencies theta_p = base^(-2p/D), p = 0 .. D/2-1, over the D rotated
 * dims of a head (its rotary_dim, else head_dim), then the scaling rule
 * (huggingface_decoder_completeness.md, P0.2 "RoPE scaling"):
 *
 * llama3 (Llama-3.1 frequency interpolation; its four parameters factor, low 1,
 * high 4, original 8192 are the ones FreeToken PR #722 "Changes" recovers):
 *   wavelength l = 2 pi / theta.
 *   l < original / high          : theta unchanged (high frequency)
 *   l > original / low           : theta / factor  (low frequency)
 *   otherwise, with smooth = (original / l - low) / (high - low):
 *                                  (1 - smooth) theta / factor + smooth theta
 *
 * yarn (named for gpt-oss on llamay "Architectures"; the pages give no formula,
 * so this is YaRN as published, Peng et al. 2023, with the ramp linear in the
 * pair index as the method's released code has it):
 *   correction index c(n) = D ln(original / (2 pi n)) / (2 ln base) is the pair
 *   whose wavelength fits n times into the original context.
 *   lo = c(beta_fast), hi = c(beta_slow) (not rounded),
 *   ramp_p = clamp((p - lo) / (hi - lo), 0, 1),
 *   theta'_p = theta_p / factor * ramp_p + theta_p * (1 - ramp_p),
 *   cos and sin are multiplied by attn_factor (default 0.1 ln(factor) + 1).
 *
 * linear: theta_p / factor.
 */
/* Rotated dims of a head: rotary_dim, or the whole head (decoder page, P1.5:
 * rotary_dim = head_dim * partial_rotary_factor; the frequencies follow the
 * rotated dims). */
static int rotary_dims(const oracle_desc* d)
{
    return d->rotary_dim > 0 ? d->rotary_dim : d->head_dim;
}

void oracle_rope_inv_freq(const oracle_desc* d, double* inv_freq, double* mscale)
{
    const int D = rotary_dims(d), half = D / 2;
    const double base = d->rope_theta;
    *mscale = 1.0;
    for (int p = 0; p < d->head_dim / 2; ++p) inv_freq[p] = 0.0;
    for (int p = 0; p < half; ++p)
        inv_freq[p] = pow(base, -2.0 * (double)p / (double)D);

    if (d->rope_scaling == ORACLE_SCALING_LLAMA3) {
        const double orig = (double)d->original_max_pos;
        const double low = d->low_freq_factor, high = d->high_freq_factor;
        const double long_wavelength = orig / low;   /* beyond it: divide by factor */
        const double short_wavelength = orig / high; /* below it: unchanged */
        for (int p = 0; p < half; ++p) {
            const double theta = inv_freq[p];
            const double wavelength = kTwoPi / theta;
            if (wavelength < short_wavelength) {
                /* unchanged */
            } else if (wavelength > long_wavelength) {
                inv_freq[p] = theta / d->factor;
            } else {
                const double smooth = (orig / wavelength - low) / (high - low);
                inv_freq[p] = (1.0 - smooth) * theta / d->factor + smooth * theta;
            }
        }
    } else if (d->rope_scaling == ORACLE_SCALING_YARN) {
        const double orig = (double)d->original_max_pos;
        const double lo = (double)D * log(orig / (kTwoPi * d->beta_fast)) / (2.0 * log(base));
        const double hi = (double)D * log(orig / (kTwoPi * d->beta_slow)) / (2.0 * log(base));
        for (int p = 0; p < half; ++p) {
            double ramp = (hi > lo) ? ((double)p - lo) / (hi - lo) : ((double)p >= lo ? 1.0 : 0.0);
            if (ramp < 0.0) ramp = 0.0;
            if (ramp > 1.0) ramp = 1.0;
            const double theta = inv_freq[p];
            inv_freq[p] = theta / d->factor * ramp + theta * (1.0 - ramp);
        }
        if (d->attn_factor > 0.0)
            *mscale = d->attn_factor;
        else
            *mscale = d->factor > 1.0 ? 0.1 * log(d->factor) + 1.0 : 1.0;
    } else if (d->rope_scaling == ORACLE_SCALING_LINEAR) {
        /* linear: every frequency divided by factor, i.e. positions divided by
         * it (support-matrix page, "Structural fact requirements": the gemma3
         * lane's global layers) */
        for (int p = 0; p < half; ++p) inv_freq[p] /= d->factor;
    }
}

/* RMSNorm over one head row (decoder page, P1.1: offset 0, or 1 where the
 * weight is stored as a delta, x * rsqrt * (1 + w); P1.2: over the last axis of
 * each q and k head). */
void oracle_rms_norm(const double* x, const float* w, int n, double eps, double w_offset, double* y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * ((double)w[i] + w_offset);
}

/* Pair p is (p, p + D/2) for NeoX halves (the qwen convention), (2p, 2p+1) for
 * interleaved pairs (the llama convention): llamay "Architectures"; FreeToken
 * PR #722 "Changes" for the row permutation that maps one onto the other. */
void oracle_rope_rotate(const oracle_desc* d, const double* inv_freq, double mscale,
                        long pos, const double* x, double* y)
{
    const int D = rotary_dims(d), half = D / 2;
    for (int i = D; i < d->head_dim; ++i) y[i] = x[i];  /* not rotated */
    for (int p = 0; p < half; ++p) {
        const int ia = d->rope_style == ORACLE_ROPE_NEOX ? p : 2 * p;
        const int ib = d->rope_style == ORACLE_ROPE_NEOX ? p + half : 2 * p + 1;
        const double angle = (double)pos * inv_freq[p];
        const double c = cos(angle) * mscale, s = sin(angle) * mscale;
        const double a = x[ia], b = x[ib];
        y[ia] = a * c - b * s;
        y[ib] = a * s + b * c;
    }
}

/* ------------------------------------------------------------------ vq8 */

/* llamay "The KV cache, in three precisions": vq8 quantises values to 8 bits
 * and keeps keys exact. The scale is one fp32 per token and head, max|v| / 127;
 * codes are v / s rounded half to even, so |code| <= 127. An all-zero row has
 * scale 0 and codes 0. */
void oracle_vq8_quantize_row(const float* v, int n, int8_t* codes, float* scale)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        const float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float r = rintf(v[i] / s);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
}

/* ------------------------------------------------------------------ loads */

static double load_io(const void* base, int dtype, size_t i)
{
    return dtype == ORACLE_F32 ? (double)((const float*)base)[i]
                               : oracle_bf16_to_double(((const uint16_t*)base)[i]);
}

/* Key j, element dd: stored as given (f32, bf16), or code times the row's scale (q8). */
static double load_key(const void* rows, const float* scale_rows, int kv_dtype, size_t j, int D, int dd)
{
    const size_t i = j * (size_t)D + (size_t)dd;
    if (kv_dtype == ORACLE_F32) return (double)((const float*)rows)[i];
    if (kv_dtype == ORACLE_Q8) return (double)((const int8_t*)rows)[i] * (double)scale_rows[j];
    return oracle_bf16_to_double(((const uint16_t*)rows)[i]);
}

static double load_value(const void* rows, const float* scale_rows, int kv_dtype, size_t j,
                         int D, int dd)
{
    const size_t i = j * (size_t)D + (size_t)dd;
    if (kv_dtype == ORACLE_F32) return (double)((const float*)rows)[i];
    if (kv_dtype == ORACLE_BF16) return oracle_bf16_to_double(((const uint16_t*)rows)[i]);
    return (double)((const int8_t*)rows)[i] * (double)scale_rows[j];
}

static double softmax_scale(const oracle_desc* d)
{
    return d->scale > 0.0 ? d->scale : 1.0 / sqrt((double)d->head_dim);
}

/* ------------------------------------------------------------------ append */

/* Normalise (optional) and rotate one head row at position pos. */
static void norm_and_rotate(const oracle_desc* d, const double* inv_freq, double mscale,
                            long pos, const float* norm_w, double* x, double* tmp)
{
    const int D = d->head_dim;
    if (d->qk_norm) {
        oracle_rms_norm(x, norm_w, D, d->norm_eps, d->norm_offset ? 1.0 : 0.0, tmp);
        memcpy(x, tmp, sizeof(double) * (size_t)D);
    }
    oracle_rope_rotate(d, inv_freq, mscale, pos, x, tmp);
    memcpy(x, tmp, sizeof(double) * (size_t)D);
}

int oracle_append(const oracle_desc* d, int B, const void* q, const void* k_new,
                  const void* v_new, const float* q_norm_w, const float* k_norm_w,
                  void* k_cache, void* v_cache, float* v_scale, float* k_scale, int cap,
                  int32_t* seq_lens, double* q_rot)
{
    const int D = d->head_dim, Hq = d->n_q_heads, Hkv = d->n_kv_heads;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] >= cap) return -1;

    double* inv_freq = (double*)malloc(sizeof(double) * (size_t)(D / 2));
    double* x = (double*)malloc(sizeof(double) * (size_t)D);
    double* tmp = (double*)malloc(sizeof(double) * (size_t)D);
    float* vrow = (float*)malloc(sizeof(float) * (size_t)D);
    double mscale;
    oracle_rope_inv_freq(d, inv_freq, &mscale);

    for (int b = 0; b < B; ++b) {
        const long pos = seq_lens[b]; /* absolute KV index of the new token (decoder page, P1.3) */
        for (int g = 0; g < Hkv; ++g) {
            const size_t in = ((size_t)b * Hkv + g) * (size_t)D;
            const size_t slot = (((size_t)b * Hkv + g) * (size_t)cap + (size_t)pos) * (size_t)D;
            for (int i = 0; i < D; ++i) x[i] = load_io(k_new, d->io_dtype, in + (size_t)i);
            norm_and_rotate(d, inv_freq, mscale, pos, k_norm_w, x, tmp);
            if (d->kv_dtype == ORACLE_Q8) {
                /* q8: the rotated key rounded to fp32, then the vq8 rule (llamay "The
                 * KV cache, in three precisions": q8 quantises keys and values) */
                for (int i = 0; i < D; ++i) vrow[i] = (float)x[i];
                oracle_vq8_quantize_row(vrow, D, (int8_t*)k_cache + slot,
                                        &k_scale[((size_t)b * Hkv + g) * (size_t)cap + (size_t)pos]);
            }
            for (int i = 0; i < D && d->kv_dtype != ORACLE_Q8; ++i) {
                if (d->kv_dtype == ORACLE_F32)
                    ((float*)k_cache)[slot + (size_t)i] = (float)x[i];
                else
                    ((uint16_t*)k_cache)[slot + (size_t)i] = oracle_bf16_from_double(x[i]);
            }
            for (int i = 0; i < D; ++i) x[i] = load_io(v_new, d->io_dtype, in + (size_t)i);
            if (d->kv_dtype == ORACLE_F32) {
                for (int i = 0; i < D; ++i) ((float*)v_cache)[slot + (size_t)i] = (float)x[i];
            } else if (d->kv_dtype == ORACLE_BF16) {
                for (int i = 0; i < D; ++i)
                    ((uint16_t*)v_cache)[slot + (size_t)i] = oracle_bf16_from_double(x[i]);
            } else {
                for (int i = 0; i < D; ++i) vrow[i] = (float)x[i]; /* exact: input is f32 or bf16 */
                oracle_vq8_quantize_row(vrow, D, (int8_t*)v_cache + slot,
                                        &v_scale[((size_t)b * Hkv + g) * (size_t)cap + (size_t)pos]);
            }
        }
        for (int h = 0; h < Hq; ++h) {
            const size_t in = ((size_t)b * Hq + h) * (size_t)D;
            for (int i = 0; i < D; ++i) x[i] = load_io(q, d->io_dtype, in + (size_t)i);
            norm_and_rotate(d, inv_freq, mscale, pos, q_norm_w, x, tmp);
            memcpy(q_rot + in, x, sizeof(double) * (size_t)D);
        }
        seq_lens[b] = (int32_t)(pos + 1);
    }
    free(inv_freq);
    free(x);
    free(tmp);
    free(vrow);
    return 0;
}

/* ------------------------------------------------------------------ attend */

/*
 * One query row against keys [j_lo, j_hi):
 *   s_j = scale * (q . k_j)
 *   softcap c > 0:  s_j = c tanh(s_j / c)      (decoder page, P1.4: logit cap)
 *   p_j = exp(s_j) / (sum_i exp(s_i) + exp(sink))   (sink term only with has_sink;
 *         llamay "Architectures": a per-head sink in the softmax denominator)
 *   o   = sum_j p_j v_j
 * The largest logit (sink included) is subtracted before exponentiating; the
 * quotient is unchanged by it.
 */
void oracle_attend_range(const oracle_desc* d, const double* q_row,
                         const void* k_rows, const void* v_rows, const float* scale_rows,
                         const float* k_scale_rows, long j_lo, long j_hi, int has_sink, double sink,
                         double* o, double* lse)
{
    const int D = d->head_dim;
    const double scale = softmax_scale(d);
    const long n = j_hi > j_lo ? j_hi - j_lo : 0;
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = has_sink ? sink : -INFINITY;
    for (long t = 0; t < n; ++t) {
        const long j = j_lo + t;
        double dot = 0.0;
        for (int i = 0; i < D; ++i)
            dot += q_row[i] * load_key(k_rows, k_scale_rows, d->kv_dtype, (size_t)j, D, i);
        double st = scale * dot;
        if (d->softcap > 0.0) st = d->softcap * tanh(st / d->softcap);
        s[t] = st;
        if (st > m) m = st;
    }
    double den = has_sink ? exp(sink - m) : 0.0;
    for (long t = 0; t < n; ++t) den += exp(s[t] - m);
    for (int i = 0; i < D; ++i) o[i] = 0.0;
    if (den > 0.0) {
        for (long t = 0; t < n; ++t) {
            const double p = exp(s[t] - m) / den;
            for (int i = 0; i < D; ++i)
                o[i] += p * load_value(v_rows, scale_rows, d->kv_dtype, (size_t)(j_lo + t), D, i);
        }
        *lse = m + log(den);
    } else {
        *lse = -INFINITY;
    }
    free(s);
}

typedef struct {
    const oracle_desc* d;
    int B;
    const double* q_rot;
    const float* sink;
    const void* k_cache;
    const void* v_cache;
    const float* v_scale;
    const float* k_scale;
    int cap;
    const int32_t* seq_lens;
    const int32_t* units;
    int n_units;
    double* out;
    int thread;
    int n_threads;
} attend_job;

/* Visible keys of the new token at position n-1: slots [0, n), and with a
 * window W only the last W of them, j > pos - W (decoder page, P1.4). */
static void attend_unit(const attend_job* job, int u)
{
    const oracle_desc* d = job->d;
    const int D = d->head_dim, Hq = d->n_q_heads, Hkv = d->n_kv_heads;
    const int G = Hq / Hkv;
    const int b = job->units ? job->units[2 * u] : u / Hq;
    const int h = job->units ? job->units[2 * u + 1] : u % Hq;
    const int g = h / G; /* kv head g serves query heads g*G .. g*G+G-1 (contiguous groups) */
    const long n = job->seq_lens[b];
    long lo = 0;
    if (d->window > 0 && n - d->window > 0) lo = n - d->window;
    const size_t head = (size_t)b * Hkv + (size_t)g;
    const size_t row0 = head * (size_t)job->cap * (size_t)D;
    const void* k_rows = d->kv_dtype == ORACLE_F32  ? (const void*)((const float*)job->k_cache + row0)
                         : d->kv_dtype == ORACLE_Q8 ? (const void*)((const int8_t*)job->k_cache + row0)
                                                    : (const void*)((const uint16_t*)job->k_cache + row0);
    const void* v_rows;
    if (d->kv_dtype == ORACLE_F32) v_rows = (const float*)job->v_cache + row0;
    else if (d->kv_dtype == ORACLE_BF16) v_rows = (const uint16_t*)job->v_cache + row0;
    else v_rows = (const int8_t*)job->v_cache + row0;
    const int int8_values = d->kv_dtype == ORACLE_VQ8 || d->kv_dtype == ORACLE_Q8;
    const float* scale_rows = int8_values ? job->v_scale + head * (size_t)job->cap : NULL;
    const float* k_scale_rows = d->kv_dtype == ORACLE_Q8 ? job->k_scale + head * (size_t)job->cap : NULL;
    double lse;
    oracle_attend_range(d, job->q_rot + ((size_t)b * Hq + (size_t)h) * (size_t)D, k_rows, v_rows,
                        scale_rows, k_scale_rows, lo, n, d->has_sink, d->has_sink ? (double)job->sink[h] : 0.0,
                        job->out + (size_t)u * (size_t)D, &lse);
}

static void* attend_worker(void* arg)
{
    const attend_job* job = (const attend_job*)arg;
    for (int u = job->thread; u < job->n_units; u += job->n_threads) attend_unit(job, u);
    return NULL;
}

void oracle_attend(const oracle_desc* d, int B, const double* q_rot, const float* sink,
                   const void* k_cache, const void* v_cache, const float* v_scale,
                   const float* k_scale, int cap, const int32_t* seq_lens, const int32_t* units, int n_units,
                   double* out, int n_threads)
{
    if (!units) n_units = B * d->n_q_heads;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_units) n_threads = n_units > 0 ? n_units : 1;
    attend_job* jobs = (attend_job*)malloc(sizeof(attend_job) * (size_t)n_threads);
    pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int t = 0; t < n_threads; ++t) {
        attend_job j = {d, B, q_rot, sink, k_cache, v_cache, v_scale, k_scale, cap, seq_lens,
                        units, n_units, out, t, n_threads};
        jobs[t] = j;
    }
    for (int t = 1; t < n_threads; ++t) pthread_create(&tids[t], NULL, attend_worker, &jobs[t]);
    attend_worker(&jobs[0]);
    for (int t = 1; t < n_threads; ++t) pthread_join(tids[t], NULL);
    free(jobs);
    free(tids);
}

int oracle_decode_step(const oracle_desc* d, int B, const void* q, const void* k_new,
                       const void* v_new, const float* q_norm_w, const float* k_norm_w,
                       const float* sink, void* k_cache, void* v_cache, float* v_scale,
                       float* k_scale, int cap, int32_t* seq_lens, double* out, int n_threads)
{
    double* q_rot = (double*)malloc(sizeof(double) * (size_t)B * (size_t)d->n_q_heads *
                                    (size_t)d->head_dim + 1);
    int rc = oracle_append(d, B, q, k_new, v_new, q_norm_w, k_norm_w, k_cache, v_cache, v_scale,
                           k_scale, cap, seq_lens, q_rot);
    if (rc == 0)
        oracle_attend(d, B, q_rot, sink, k_cache, v_cache, v_scale, k_scale, cap, seq_lens, NULL, 0, out,
                      n_threads);
    free(q_rot);
    return rc;
}
