/*
 * uaa.h -- C ABI of the GB300 (sm_103a) grouped-query-attention decode step.
 *
 * One decode step of one attention layer, for a batch of sequences that each
 * hold a KV cache, with one new token per sequence or a causal chunk of q_len
 * tokens (uaa_step_args.q_len):
 *
 *   1. uaa_rope_qk_norm_append: optional per-head RMSNorm of the new q and k
 *      rows, rotary position embedding at each token's absolute KV index, and
 *      the append of k and v at slots seq_lens[b] .. seq_lens[b] + q_len - 1
 *      (seq_lens[b] then grows by q_len).
 *   2. uaa_decode_attn_partial: split-K flash decoding. A persistent grid of P
 *      CTAs splits the key stages of all units (sequence, kv head, group of
 *      (token, head) query rows) into P contiguous ranges (a stream-K
 *      partition). The tensor-core kernel
 *      sizes the ranges by the speed each CTA slot measured in the previous
 *      launches on the same workspace (the SMs of a GB300 do not all stream
 *      equally fast), so results may differ in rounding from launch to launch;
 *      a desc with reproducible = 1 keeps the ranges uniform instead.
 *      A unit that lies inside one range is finished there and its output rows
 *      written; every other unit leaves one record (normalised output rows and
 *      log-sum-exp) per range it touches in the workspace.
 *   3. uaa_decode_attn_combine: log-sum-exp merge of those records, the sink
 *      logit added to the denominator, the remaining output rows written.
 *   uaa_decode_attn_append_partial runs 1 and 2 (for bf16, vq8 and q8 caches and
 *   one token per sequence in one kernel that forms q', k and v of the new
 *   token itself and attends the new key from shared memory); uaa_decode_attn
 *   runs 1-3 on one stream.

 * Where the method is defined (page title, then section):
 *   - integral GQA ratio, head_dim set, 1/sqrt(head_dim) scale, the split-K
 *     decode and KV-producer paths (prior art):
 *       Model support matrix, "Structural fact requirements", "Kernel path
 *       capabilities"; the typed-refusal convention: "Conformance CLI";
 *   - RoPE scaling (llama3, YaRN), QK-norm before RoPE, RMSNorm (and Gemma's
 *     (1 + w) weight), positions at the absolute KV index, sliding window,
 *     attention-logit softcap, partial rotary:
 *       huggingface_decoder_completeness.md, P0.2, P1.1, P1.2, P1.3, P1.4, P1.5;
 *   - NeoX vs interleaved pairing and the llama3 parameters:
 *       FreeToken PR #722 "serve Llama and Mistral llama-arch GGUF", "Changes";
 *       llamay "Models and formats", "Architectures";
 *   - per-head attention sink in the softmax denominator, YaRN for gpt-oss:
 *       llamay "Models and formats", "Architectures" (gpt-oss row);
 *   - the vq8 cache (int8 values, per-token per-head fp32 scale, keys exact)
 *     and the q8 cache (keys stored the same way as values):
 *       llamay "Models and formats", "The KV cache, in three precisions".
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, owned by the caller, 16-byte
 *     aligned, row-major and dense. The library never allocates device memory,
 *     never synchronises (except uaa_device_status) and launches only on the
 *     given stream.
 *   - Layouts (with q_len = T > 1 every q, k_new, v_new, out and q_rot row set
 *     has a token axis after B, [B][T][H][D]; paged caches: see block_table):
 *     q [B][Hq][D]; k_new, v_new [B][Hkv][D] (io_dtype);
 *     k_cache [B][Hkv][cap][D] (fp32, bf16 for BF16 and VQ8 caches, int8
 *     codes for Q8); v_cache [B][Hkv][cap][D] (fp32, bf16, or int8 codes for
 *     VQ8 and Q8); v_scale [B][Hkv][cap] fp32 (VQ8 and Q8); k_scale
 *     [B][Hkv][cap] fp32 (Q8 only); seq_lens [B] int32;
 *     out [B][Hq][D] (out_dtype). Query head h reads kv head h / (Hq / Hkv).
 *   - Facts outside the supported ranges are refused with a status and a
 *     message naming the fact (uaa_last_error), never approximated.
 *   - A step's entry points must receive the same descriptor and arguments;
 *     partial and combine run after the append of the same step (they read
 *     seq_lens after its increment). The combine may follow either the
 *     separate append + partial or uaa_decode_attn_append_partial.
 */
#ifndef UAA_H
#define UAA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UAA_ABI_VERSION 11

typedef enum {
    UAA_OK = 0,
    UAA_ERR_INVALID_ARGUMENT = 1, /* null or misaligned pointer, workspace too small */
    UAA_ERR_UNSUPPORTED = 2,      /* a fact outside the supported range */
    UAA_ERR_CAPACITY = 3,         /* max_seq_len + 1 does not fit the cache */
    UAA_ERR_CUDA = 4,             /* a CUDA call failed; the message names it */
    UAA_ERR_DEVICE = 5            /* uaa_device_status found a device-side flag */
} uaa_status;

typedef enum { UAA_ROPE_NEOX = 0, UAA_ROPE_INTERLEAVED = 1 } uaa_rope_style;
typedef enum {
    UAA_ROPE_SCALING_NONE = 0,
    UAA_ROPE_SCALING_LLAMA3 = 1,
    UAA_ROPE_SCALING_YARN = 2,
    UAA_ROPE_SCALING_LINEAR = 3
} uaa_rope_scaling;
/* Cache storage: F32, BF16, VQ8 (bf16 keys, int8 value codes + one fp32 scale
 * per token and kv head) or Q8 (keys stored like VQ8 values: the rotated key row
 * as int8 codes + its own scale). Codes follow the rule of uaa_vq8_quantize.
 * With Q8 the key codes meet q' (the normed, rotated q times the logit
 * prescale) as fp16 tensor-core operands: |q'| must stay below 65504. */
typedef enum { UAA_DTYPE_F32 = 0, UAA_DTYPE_BF16 = 1, UAA_DTYPE_VQ8 = 2, UAA_DTYPE_Q8 = 3 } uaa_dtype;

/* Device-side status flags (sticky, in the workspace; read by uaa_device_status). */
#define UAA_DEVFLAG_CAPACITY 0x1u   /* seq_lens[b] >= cache_capacity: that sequence was not appended */
#define UAA_DEVFLAG_LEN_HINT 0x2u   /* seq_lens[b] > max_seq_len at the append (results stay exact) */
#define UAA_DEVFLAG_TIMEOUT 0x4u    /* a bounded wait inside a kernel gave up, or the workspace's
                                       scheduling state was left by such a launch; outputs are
                                       invalid until the workspace is zeroed again */
#define UAA_DEVFLAG_PAGE 0x8u       /* a block_table entry outside [0, n_pages): that row was
                                       neither written nor read (outputs of the sequence invalid) */

/* Rotary embedding of the first R = rotary_dim dims of each head row (R = D when
 * the descriptor's rotary_dim is 0; the other D - R dims pass unchanged: the
 * partial rotary of the decoder-completeness page, P1.5). Pair p < R/2 is
 * (p, p + R/2) for NEOX and (2p, 2p+1) for INTERLEAVED; theta_p = theta^(-2p/R),
 * rotated by angle pos * theta'_p.
 * LLAMA3: Llama-3.1 wavelength interpolation (factor, low_freq_factor,
 *   high_freq_factor, original_max_pos).
 * LINEAR: theta'_p = theta_p / factor (positions divided by factor; the global
 *   layers of the gemma3 lane, support-matrix page, "Structural fact
 *   requirements").
 * YARN: ramp over the pair index between the pairs whose wavelength fits
 *   beta_fast and beta_slow times into original_max_pos (not rounded); theta'
 *   blends theta / factor and theta; cos and sin are multiplied by attn_factor
 *   (<= 0 selects 0.1 ln(factor) + 1).
 * The descriptor is per layer: a model whose layers differ in rotary base,
 *   scaling or window (Gemma 3's local layers with a sliding window and a
 *   second base, its global layers with linear scaling: llamay "Architectures")
 *   passes each layer its own. */
typedef struct {
    int32_t style;            /* uaa_rope_style */
    double theta;             /* base, > 0 */
    int32_t scaling;          /* uaa_rope_scaling */
    double factor;
    double low_freq_factor;
    double high_freq_factor;
    int32_t original_max_pos;
    double beta_fast;
    double beta_slow;
    double attn_factor;
} uaa_rope_params;

typedef struct {
    int32_t n_q_heads;        /* Hq, a positive multiple of n_kv_heads */
    int32_t n_kv_heads;       /* Hkv > 0 */
    int32_t head_dim;         /* D in {64, 128, 256} */
    float scale;              /* softmax scale; 0 selects 1/sqrt(D) */
    uaa_rope_params rope;
    int32_t qk_norm;          /* 1: RMSNorm of each q and k head row before RoPE */
    float norm_eps;           /* RMSNorm epsilon, >= 0 */
    int32_t window;           /* 0: none; W > 0: keys j with pos - W < j <= pos */
    float softcap;            /* 0: none; c > 0: s -> c tanh(s / c), after the scale */
    int32_t has_sink;         /* 1: sink[h] joins the softmax denominator of head h */
    int32_t kv_dtype;         /* UAA_DTYPE_F32, _BF16, _VQ8 or _Q8 */
    int32_t io_dtype;         /* q, k_new, v_new: UAA_DTYPE_F32 or _BF16 */
    int32_t out_dtype;        /* out: UAA_DTYPE_F32 or _BF16 */
    int32_t rotary_dim;       /* rotated dims per head: 0 (all D), or even, 2 <= R <= D */
    int32_t norm_offset;      /* 1: the QK RMSNorm weight applies as (1 + w) (Gemma's
                                 stored delta, decoder-completeness page P1.1); else 0 */
    int32_t reproducible;     /* 1: the tensor-core partial step splits its ranges uniformly
                                 instead of by the slot speeds measured in earlier launches,
                                 so equal inputs give equal bits on every launch; else 0 */
} uaa_attn_desc;

typedef struct {
    int32_t batch;            /* B >= 0 (0 is a no-op) */
    const void* q;            /* [B][Hq][D] io_dtype */
    const void* k_new;        /* [B][Hkv][D] io_dtype */
    const void* v_new;        /* [B][Hkv][D] io_dtype */
    const float* q_norm_w;    /* [D], required when qk_norm */
    const float* k_norm_w;    /* [D], required when qk_norm */
    const float* sink;        /* [Hq], required when has_sink */
    void* k_cache;            /* [B][Hkv][cap][D] */
    void* v_cache;            /* [B][Hkv][cap][D] */
    float* v_scale;           /* [B][Hkv][cap], VQ8 and Q8 */
    int32_t cache_capacity;   /* cap: slots per (sequence, kv head), a multiple of 4 */
    int32_t* seq_lens;        /* [B]: tokens cached before the step; the append adds 1 */
    int32_t max_seq_len;      /* host bound on seq_lens[b] before the step (+1 must fit cap) */
    void* out;                /* [B][Hq][D] out_dtype */
    float* q_rot;             /* optional [B][Hq][D] fp32: the normed, rotated q rows */
    float* k_scale;           /* [B][Hkv][cap], Q8 only: the key rows' scales */
    /* Paged caches (a key and a value per head per position, in pages: llamay
     * "What is refused" on what a KV page holds). block_table NULL: the caches
     * are contiguous, [B][Hkv][cap][...]. Otherwise k_cache / v_cache are pools
     * [n_pages][Hkv][page_size][D], v_scale / k_scale [n_pages][Hkv][page_size],
     * position j of sequence b lives in slot j % page_size of physical page
     * block_table[b][j / page_size], and cap = pages_per_seq * page_size. The
     * table is read, never written; pages may be shared between sequences for
     * reading (a step writes slot seq_lens[b] of its own page only). */
    const int32_t* block_table; /* [B][pages_per_seq] int32, or NULL */
    int32_t page_size;        /* keys per page: a power of two in [16, 4096]; >= 32 for VQ8 / Q8 */
    int32_t pages_per_seq;    /* row length of block_table */
    int32_t n_pages;          /* pages in each pool */
    /* Tokens per sequence in this step, T (0 counts as 1: a decode step). With
     * T > 1 (a prefill chunk, or draft tokens to verify) q, k_new, v_new, out and
     * q_rot hold T rows per sequence, [B][T][H][D]; token t sits at position
     * seq_lens[b] + t, is appended there, and attends the keys up to and
     * including its own (causal within the chunk, and within the window);
     * seq_lens[b] grows by T, and max_seq_len + T must fit cache_capacity. The
     * (token, head) rows of a kv head share every K/V tile the step reads. */
    int32_t q_len;
} uaa_step_args;

/* Scratch memory owned by the caller, at least uaa_workspace_size bytes, zeroed
 * once after allocation. It holds the rotated q rows, the split partials, the
 * device status word, the arrival counter of the append and fused kernels (the
 * last CTA to arrive advances seq_lens) and the range
 * balance state (counters that every completed launch leaves at zero, and the
 * measured slot speeds that carry over to the next launch); it must not be
 * shared by steps that run concurrently. After UAA_DEVFLAG_TIMEOUT zero it
 * again. A workspace may serve descs of different geometry in turn (different
 * P = uaa_workspace_layout.n_ctas); the measured slot speeds then start over
 * at each change of P (uniform ranges for one launch). */
typedef struct {
    void* ptr;
    size_t bytes;
} uaa_workspace;

/* Where each array lives in the workspace, and the split geometry. */
typedef struct {
    int32_t n_ctas;           /* P: persistent CTAs of the partial step (stream-K ranges) */
    int32_t stage_keys;       /* keys per ring stage: 64; 128 for q8 at head_dim 128 / 256;
                                 at head_dim 64 128 (bf16), 256 (vq8, q8) */
    int32_t heads_per_cta;    /* query rows (token, head) of one unit (sequence, kv head, row group) */
    int32_t kernel;           /* 0: fp32 CUDA-core partial, 1: TMA + tensor-core partial,
                                 2: query-tiled prefill on a contiguous cache (bf16 cache,
                                 head_dim 64 / 128, q_len x G >= 128 rows per kv head;
                                 a paged cache of this geometry takes kernel 1, whose
                                 fields the others still describe) */
    int32_t n_slices;         /* partial + combine launches (batch slices) */
    int32_t slice_batch;      /* sequences per slice (the last may hold fewer) */
    int32_t step_kernels;     /* kernels one uaa_decode_attn call launches (contiguous cache) */
    int32_t step_splits;      /* key splits per unit of the fp32 one-launch step, 0 when the
                                 step does not take it (tensor-core caches, chunks, records
                                 beyond 2P, several slices) */
    size_t status_offset;     /* uint32 device flags */
    size_t q_rot_offset;      /* fp32 [B][Hq][D]: rotated q times the kernel's logit prescale */
    size_t prefix_offset;     /* int32 [n_slices][slice_batch + 1]: units x stages, prefix over
                                 the slice's sequences */
    size_t rec_lse_offset;    /* fp32 [n_slices][2P][heads_per_cta]: record log2-sum-exp */
    size_t rec_o_offset;      /* fp32 [n_slices][2P][heads_per_cta][D]: normalised record rows;
                                 record 2c + 0 is CTA c's first segment, 2c + 1 its last */
    size_t prefix_stride;     /* bytes between slices of each of the three arrays above */
    size_t rec_lse_stride;
    size_t rec_o_stride;
    size_t ranges_offset;     /* int64 [n_slices][P' + 1]: start stage of each range of the
                                 last partial launch of the slice (P' = min(P, stages)) */
    size_t ranges_stride;
    size_t owners_offset;     /* uint32 [n_slices][slice_batch][units][2]: first / last range
                                 owning each unit's stages (the combine reads and clears them) */
    size_t owners_stride;
    size_t balance_offset;    /* range-balance state of the tensor-core kernel (opaque), right
                                 after the status word so that it survives a change of batch */
    size_t total_bytes;
} uaa_workspace_layout;

/* Step 1 (append). Writes the k/v rows at slot seq_lens[b], increments seq_lens,
 * and stores the rotated q rows in the workspace (and in args->q_rot if set).
 * A bf16 key element is the exact normalised, rotated value rounded to nearest
 * even: computed in fp32, and recomputed in fp64 where the fp32 result lies
 * within its error bound of a bf16 rounding boundary. */
uaa_status uaa_rope_qk_norm_append(const uaa_attn_desc* desc, const uaa_step_args* args,
                                   const uaa_workspace* ws, cudaStream_t stream);

/* Step 2 (split-K partials) over the visible keys of every sequence; writes the
 * output rows of units finished inside one CTA and records for the others.
 * A long chunk on a contiguous bf16 cache (head_dim 64 or 128, q_len x G >= 128
 * (token, head) rows per kv head; uaa_workspace_layout.kernel == 2) takes the
 * query-tiled prefill kernel instead: a CTA per (sequence, kv head, block of
 * 128 rows) reads each key and value tile its rows see once, and writes the
 * block's output rows itself (sink included); rows of a sequence the append
 * could not take are zero. Step 3 then has nothing to do. */
uaa_status uaa_decode_attn_partial(const uaa_attn_desc* desc, const uaa_step_args* args,
                                   const uaa_workspace* ws, cudaStream_t stream);

/* Step 3 (log-sum-exp combine + sink) of the recorded units into args->out;
 * launches nothing after the query-tiled prefill kernel. */
uaa_status uaa_decode_attn_combine(const uaa_attn_desc* desc, const uaa_step_args* args,
                                   const uaa_workspace* ws, cudaStream_t stream);

/* Steps 1 and 2 on one stream. For bf16, vq8 and q8 caches this is one kernel: each
 * unit normalises and rotates its q rows in registers (the workspace's q rows
 * are not written), the warp that owns slot seq_lens[b] of a unit's last key
 * stage forms the new k and v rows and writes them over that slot of the
 * loaded stage (and, once per kv head, into the cache), and the last CTA to
 * have read the lengths advances seq_lens. Results, cache rows and seq_lens are
 * those of uaa_rope_qk_norm_append followed by uaa_decode_attn_partial, up to
 * fp32 rounding order (bf16 key rows in the cache are the same bits; the step's
 * own attention may use a new key element one bf16 ulp away where its exact
 * rounding is recomputed after the attention; a q8 key code may differ by one
 * where the rotated key lies within fp32 rounding of a rounding tie). For fp32 caches,
 * and for steps of q_len > 1, it is those two launches. Follow it with
 * uaa_decode_attn_combine. */
uaa_status uaa_decode_attn_append_partial(const uaa_attn_desc* desc, const uaa_step_args* args,
                                          const uaa_workspace* ws, cudaStream_t stream);

/* Steps 1-3 on one stream: the whole decode step of one layer
 * (uaa_decode_attn_append_partial, then uaa_decode_attn_combine). An fp32 cache
 * with one token per sequence, a batch of one slice and at most 2P split
 * records (uaa_workspace_layout.step_splits > 0) takes one kernel instead: a
 * CTA per (sequence, kv head, group of up to 8 query heads, split of 512 keys)
 * appends, attends its keys and writes a record, and the last split of each
 * unit to finish merges them (sink included) into the output rows; the results
 * equal those of the three steps up to fp32 rounding order. */
uaa_status uaa_decode_attn(const uaa_attn_desc* desc, const uaa_step_args* args,
                           const uaa_workspace* ws, cudaStream_t stream);

/* Workspace bytes for a step of `batch` sequences of q_len tokens each (0 or 1:
 * decode) whose lengths before the step are at most max_seq_len; a workspace
 * sized for q_len serves every step of at most q_len tokens. n_sm <= 0 queries
 * the current device's SM count; the launches always use the current device's
 * count. Returns 0 on a refused desc. */
size_t uaa_workspace_size(const uaa_attn_desc* desc, int32_t batch, int32_t max_seq_len,
                          int32_t n_sm, int32_t q_len);

/* Number of CTAs P the split-K step runs (each attends one contiguous range of
 * the key stages of all units); 0 on a refused desc. */
int32_t uaa_num_splits(const uaa_attn_desc* desc, int32_t batch, int32_t max_seq_len,
                       int32_t n_sm, int32_t q_len);

/* The workspace layout and split geometry (host only; n_sm as above). */
uaa_status uaa_get_workspace_layout(const uaa_attn_desc* desc, int32_t batch,
                                    int32_t max_seq_len, int32_t n_sm, int32_t q_len,
                                    uaa_workspace_layout* layout);

/* Quantise n_rows rows of head_dim values (fp32 or bf16, v_dtype) to the vq8
 * storage: codes = rint(v / s) with s = max|v| / 127 in fp32 (the append's rule).
 * Used to fill a vq8 cache from existing values, and the keys of a q8 cache. */
uaa_status uaa_vq8_quantize(const void* v, int32_t v_dtype, int64_t n_rows, int32_t head_dim,
                            int8_t* codes, float* scales, cudaStream_t stream);

/* Waits for the stream, reads the device flags (UAA_DEVFLAG_*) of the workspace
 * into *flags, clears them, and returns UAA_ERR_DEVICE if any was set. */
uaa_status uaa_device_status(const uaa_workspace* ws, cudaStream_t stream, uint32_t* flags);

/* The message of the last refused or failed call on this thread. */
const char* uaa_last_error(void);

/* A fixed name for a status code. */
const char* uaa_status_string(uaa_status status);

/* UAA_ABI_VERSION of the built library. */
int32_t uaa_abi_version(void);

/* Bytes of the library's built-in scratch array (see uaa_decode_attn_static). */
#define UAA_STATIC_SCRATCH_BYTES (8u << 20)

/* uaa_decode_attn without a caller workspace. The pages have no counterpart of
 * this entry point: it exists for callers that cannot allocate device memory
 * themselves -- for example a plugin whose host framework owns every device
 * allocation and forbids direct cudaMalloc, or a latency-bound serving loop that
 * must never block on the allocator's implicit device synchronisation.
 *
 * The split partials, rotated q rows and status word then live in one
 * file-scope __device__ array of UAA_STATIC_SCRATCH_BYTES (8 MiB) that every
 * GPU which loads the library holds until the process exits. The caller still
 * passes every input and output in args; this call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *   - A step whose workspace would exceed UAA_STATIC_SCRATCH_BYTES (see
 *     uaa_workspace_size) is refused with UAA_ERR_INVALID_ARGUMENT and a message
 *     giving both sizes; nothing is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *     first call on a device before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents. Each call clears the status word and the arrival counter it
 *     starts from (and, after a call that returned an error between its
 *     partial and combine launches, the range-balance state), so one failed
 *     call leaves nothing that changes the next call's results. Device-side
 *     flags are therefore neither reported nor clearable by the caller: a
 *     sequence without a free slot is silently not appended, and a step whose
 *     bounded wait gave up (UAA_DEVFLAG_TIMEOUT on the workspace entry) goes
 *     unnoticed. Callers that need the flags use uaa_decode_attn with a
 *     workspace and uaa_device_status. Calls whose kernels overlap on the GPU
 *     (two streams, or two threads) race on the array: serialise them.
 * It runs the same kernels as uaa_decode_attn: results equal uaa_decode_attn's
 * for the same desc and args. */
uaa_status uaa_decode_attn_static(const uaa_attn_desc* desc, const uaa_step_args* args,
                                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
