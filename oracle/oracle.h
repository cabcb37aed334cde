/*
 * oracle.h -- plain CPU fp64 oracle of one grouped-query-attention decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference legs load this library. The CUDA library shares no
 * code, header, table or helper with it, and neither includes the other.
 *
 * What one decode step computes, and where each part is defined:
 *   1. optional per-head RMSNorm of the new q and k rows, before rotation
 *      (huggingface_decoder_completeness.md, P1.2 "Qwen3 QK-norm"; RMSNorm
 *      itself, with Gemma's (1 + w) weight offset: same page, P1.1);
 *   2. rotary position embedding of q and k at the absolute KV index, NeoX
 *      halves or interleaved pairs, plain theta, Llama-3.1 "llama3" scaling,
 *      YaRN or linear scaling, over the whole head or its first rotary_dim
 *      dims (same page, P0.2, P1.3 and P1.5; llamay "Models and formats",
 *      "Architectures"; FreeToken PR #722, "Changes"; YaRN: Peng et al., 2023;
 *      linear: Model support matrix, "Structural fact requirements");
 *   3. append of k and v at slot seq_len, the cache being fp32, bf16, "vq8"
 *      (int8 values with one fp32 scale per token and head, keys exact) or
 *      "q8" (keys too: int8 codes of the rotated key with their own scale)
 *      (llamay "Models and formats", "The KV cache, in three precisions");
 *   4. attention of each query head over its kv head's cache (integral GQA
 *      ratio, Model support matrix, "Structural fact requirements"), with an
 *      optional sliding window and attention-logit softcap (decoder page,
 *      P1.4) and an optional per-head sink logit in the softmax denominator
 *      (llamay "Architectures", gpt-oss row).
 *
 * Layouts (all row-major, caller-owned):
 *   q        [B][Hq][D]    k_new, v_new [B][Hkv][D]      (io_dtype: f32 or bf16)
 *   k_cache  [B][Hkv][cap][D]  (kv_dtype f32 -> float, bf16/vq8 -> uint16 bf16 bits,
 *                               q8 -> int8 codes)
 *   v_cache  [B][Hkv][cap][D]  (f32 -> float, bf16 -> uint16, vq8/q8 -> int8 codes)
 *   v_scale  [B][Hkv][cap]     (vq8 and q8, fp32)
 *   k_scale  [B][Hkv][cap]     (q8 only, fp32)
 *   seq_lens [B] int32: tokens cached before the step; incremented by the append.
 */
#ifndef GQA_ORACLE_H
#define GQA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_ROPE_NEOX = 0, ORACLE_ROPE_INTERLEAVED = 1 };
enum { ORACLE_SCALING_NONE = 0, ORACLE_SCALING_LLAMA3 = 1, ORACLE_SCALING_YARN = 2, ORACLE_SCALING_LINEAR = 3 };
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_VQ8 = 2, ORACLE_Q8 = 3 };

typedef struct {
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    double scale;            /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
    int rope_style;          /* ORACLE_ROPE_* */
    double rope_theta;       /* base of the rotary frequencies */
    int rope_scaling;        /* ORACLE_SCALING_* */
    double factor;           /* llama3 / yarn scaling factor */
    double low_freq_factor;  /* llama3 */
    double high_freq_factor; /* llama3 */
    int original_max_pos;    /* llama3 / yarn original context */
    double beta_fast;        /* yarn: rotations at the high-frequency end of the ramp */
    double beta_slow;        /* yarn: rotations at the low-frequency end of the ramp */
    double attn_factor;      /* yarn: cos/sin multiplier; <= 0 selects 0.1 ln(factor) + 1 */
    int qk_norm;             /* 1: per-head RMSNorm of q and k before rotation */
    double norm_eps;
    int window;              /* 0: none; W: the last W positions are visible */
    double softcap;          /* 0: none; c: s -> c tanh(s / c) */
    int has_sink;            /* 1: one sink logit per query head in the denominator */
    int kv_dtype;            /* ORACLE_F32 / ORACLE_BF16 / ORACLE_VQ8 / ORACLE_Q8 */
    int io_dtype;            /* ORACLE_F32 / ORACLE_BF16 for q, k_new, v_new */
    int rotary_dim;          /* rotated dims of a head (even, <= head_dim); 0: head_dim */
    int norm_offset;         /* 1: the RMSNorm weight is applied as (1 + w) */
} oracle_desc;

/* bf16 <-> fp64. The rounding is round-to-nearest, ties to even, overflow to inf. */
double oracle_bf16_to_double(uint16_t h);
uint16_t oracle_bf16_from_double(double x);

/* Rotary inverse frequencies after scaling ([head_dim/2]; pairs at or beyond
 * rotary_dim/2 are not rotated and get 0) and the cos/sin multiplier. */
void oracle_rope_inv_freq(const oracle_desc* d, double* inv_freq, double* mscale);

/* y = x * (w + w_offset) / sqrt(mean(x^2) + eps) over one row of length n
 * (w_offset 0, or 1 for a weight stored as a delta from one). */
void oracle_rms_norm(const double* x, const float* w, int n, double eps, double w_offset, double* y);

/* Rotate one head row x (length head_dim) to absolute position pos; dims at or
 * beyond rotary_dim are copied unchanged. */
void oracle_rope_rotate(const oracle_desc* d, const double* inv_freq, double mscale,
                        long pos, const double* x, double* y);

/* vq8 storage rule, in fp32 arithmetic: s = max|v| / 127, code = rint(v / s).
 * q8 stores the rotated key row (rounded to fp32) by the same rule. */
void oracle_vq8_quantize_row(const float* v, int n, int8_t* codes, float* scale);

/* Append step for every sequence. Returns 0, or -1 (nothing written) when some
 * seq_lens[b] is negative or >= cap. q_rot receives the normed, rotated q rows
 * in fp64, [B][Hq][D]. */
int oracle_append(const oracle_desc* d, int B, const void* q, const void* k_new,
                  const void* v_new, const float* q_norm_w, const float* k_norm_w,
                  void* k_cache, void* v_cache, float* v_scale, float* k_scale, int cap,
                  int32_t* seq_lens, double* q_rot);

/* Softmax attention of one query row over keys [j_lo, j_hi) of one kv head.
 * k_rows / v_rows / scale_rows (values) / k_scale_rows (q8 keys) point at slot 0
 * of that head's cache rows.
 * sink: the head's sink logit (included in the denominator) when has_sink.
 * o receives the output row, *lse the natural log of the denominator. */
void oracle_attend_range(const oracle_desc* d, const double* q_row,
                         const void* k_rows, const void* v_rows, const float* scale_rows,
                         const float* k_scale_rows, long j_lo, long j_hi, int has_sink, double sink,
                         double* o, double* lse);

/* Attention for (b, h) units after the append. units: n_units pairs (b, h),
 * or NULL for every (b, h) in order. out: [n_units][D] (or [B][Hq][D]). */
void oracle_attend(const oracle_desc* d, int B, const double* q_rot, const float* sink,
                   const void* k_cache, const void* v_cache, const float* v_scale,
                   const float* k_scale, int cap, const int32_t* seq_lens, const int32_t* units, int n_units,
                   double* out, int n_threads);

/* append + attend for the whole batch. Returns the append's status. */
int oracle_decode_step(const oracle_desc* d, int B, const void* q, const void* k_new,
                       const void* v_new, const float* q_norm_w, const float* k_norm_w,
                       const float* sink, void* k_cache, void* v_cache, float* v_scale,
                       float* k_scale, int cap, int32_t* seq_lens, double* out, int n_threads);

#ifdef __cplusplus
}
#endif
#endif
