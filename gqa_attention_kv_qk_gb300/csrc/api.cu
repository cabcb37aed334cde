// api.cu -- the C ABI of libuaa: descriptor validation (typed refusals that name
// the fact, the Model support matrix page's "Conformance CLI" convention), the
// split geometry, workspace layout, TMA descriptors and the kernel launches.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "internal.cuh"

namespace {

thread_local char g_err[512] = "";

uaa_status fail(uaa_status st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

uaa_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(UAA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define UAA_TRY(expr)                          \
    do {                                       \
        const uaa_status st_ = (expr);         \
        if (st_ != UAA_OK) return st_;         \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// ---------------------------------------------------------------- descriptor checks

uaa_status check_desc(const uaa_attn_desc* d)
{
    if (!d) return fail(UAA_ERR_INVALID_ARGUMENT, "desc is NULL");
    if (d->n_kv_heads <= 0) return fail(UAA_ERR_UNSUPPORTED, "n_kv_heads=%d is not positive", d->n_kv_heads);
    if (d->n_q_heads <= 0 || d->n_q_heads % d->n_kv_heads != 0)
        return fail(UAA_ERR_UNSUPPORTED,
                    "n_q_heads=%d is not a positive multiple of n_kv_heads=%d (integral GQA ratio required)",
                    d->n_q_heads, d->n_kv_heads);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(UAA_ERR_UNSUPPORTED, "head_dim=%d is not supported (supported: {64, 128, 256})",
                    d->head_dim);
    if (!(d->scale >= 0.f) || !isfinite(d->scale))
        return fail(UAA_ERR_UNSUPPORTED, "scale=%g is not a finite value >= 0", (double)d->scale);
    const uaa_rope_params& r = d->rope;
    if (r.style != UAA_ROPE_NEOX && r.style != UAA_ROPE_INTERLEAVED)
        return fail(UAA_ERR_UNSUPPORTED, "rope.style=%d is not NEOX (0) or INTERLEAVED (1)", r.style);
    if (!(r.theta > 0.0) || !isfinite(r.theta))
        return fail(UAA_ERR_UNSUPPORTED, "rope.theta=%g is not a finite value > 0", r.theta);
    if (r.scaling == UAA_ROPE_SCALING_LLAMA3) {
        if (!(r.factor >= 1.0) || !(r.low_freq_factor > 0.0) || !(r.high_freq_factor > r.low_freq_factor) ||
            r.original_max_pos <= 0)
            return fail(UAA_ERR_UNSUPPORTED,
                        "llama3 rope scaling needs factor>=1, 0<low_freq_factor<high_freq_factor, "
                        "original_max_pos>0 (got %g, %g, %g, %d)",
                        r.factor, r.low_freq_factor, r.high_freq_factor, r.original_max_pos);
    } else if (r.scaling == UAA_ROPE_SCALING_YARN) {
        if (!(r.factor > 0.0) || r.original_max_pos <= 0 || !(r.beta_slow > 0.0) || !(r.beta_fast > r.beta_slow))
            return fail(UAA_ERR_UNSUPPORTED,
                        "yarn rope scaling needs factor>0, original_max_pos>0, beta_fast>beta_slow>0 "
                        "(got %g, %d, %g, %g)",
                        r.factor, r.original_max_pos, r.beta_fast, r.beta_slow);
    } else if (r.scaling == UAA_ROPE_SCALING_LINEAR) {
        if (!(r.factor > 0.0) || !isfinite(r.factor))
            return fail(UAA_ERR_UNSUPPORTED, "linear rope scaling needs a finite factor>0 (got %g)", r.factor);
    } else if (r.scaling != UAA_ROPE_SCALING_NONE) {
        return fail(UAA_ERR_UNSUPPORTED, "rope.scaling=%d is not supported (none, llama3, yarn, linear)",
                    r.scaling);
    }
    if (d->rotary_dim != 0 && (d->rotary_dim < 2 || d->rotary_dim > d->head_dim || d->rotary_dim % 2 != 0))
        return fail(UAA_ERR_UNSUPPORTED, "rotary_dim=%d is not 0 or an even value in [2, head_dim=%d]",
                    d->rotary_dim, d->head_dim);
    if (d->norm_offset != 0 && d->norm_offset != 1)
        return fail(UAA_ERR_UNSUPPORTED, "norm_offset=%d is not 0 or 1", d->norm_offset);
    if (d->reproducible != 0 && d->reproducible != 1)
        return fail(UAA_ERR_UNSUPPORTED, "reproducible=%d is not 0 or 1", d->reproducible);
    if (d->qk_norm != 0 && d->qk_norm != 1)
        return fail(UAA_ERR_UNSUPPORTED, "qk_norm=%d is not 0 or 1", d->qk_norm);
    if (d->qk_norm && (!(d->norm_eps >= 0.f) || !isfinite(d->norm_eps)))
        return fail(UAA_ERR_UNSUPPORTED, "norm_eps=%g is not a finite value >= 0", (double)d->norm_eps);
    if (d->window < 0) return fail(UAA_ERR_UNSUPPORTED, "window=%d is negative", d->window);
    if (!(d->softcap >= 0.f) || !isfinite(d->softcap))
        return fail(UAA_ERR_UNSUPPORTED, "softcap=%g is not a finite value >= 0", (double)d->softcap);
    if (d->has_sink != 0 && d->has_sink != 1)
        return fail(UAA_ERR_UNSUPPORTED, "has_sink=%d is not 0 or 1", d->has_sink);
    if (d->kv_dtype != UAA_DTYPE_F32 && d->kv_dtype != UAA_DTYPE_BF16 && d->kv_dtype != UAA_DTYPE_VQ8 &&
        d->kv_dtype != UAA_DTYPE_Q8)
        return fail(UAA_ERR_UNSUPPORTED, "kv_dtype=%d is not F32, BF16, VQ8 or Q8", d->kv_dtype);
    if (d->io_dtype != UAA_DTYPE_F32 && d->io_dtype != UAA_DTYPE_BF16)
        return fail(UAA_ERR_UNSUPPORTED, "io_dtype=%d is not F32 or BF16", d->io_dtype);
    if (d->out_dtype != UAA_DTYPE_F32 && d->out_dtype != UAA_DTYPE_BF16)
        return fail(UAA_ERR_UNSUPPORTED, "out_dtype=%d is not F32 or BF16", d->out_dtype);
    return UAA_OK;
}

// ---------------------------------------------------------------- split geometry

// Tokens per sequence one step takes at most (a prefill chunk).
constexpr int kMaxQLen = 1024;

struct Plan {
    int G;
    int q_len;           // tokens per sequence (1: decode)
    int kernel;          // 0 CUDA-core, 1 tensor-core
    int heads_per_cta;   // query rows of one unit ((token, head) pairs; heads for a decode step)
    int head_groups;     // units per kv head
    int n_head_tiles;    // 8-head column tiles of the tensor-core kernel
    int mg;              // 64-key tiles per ring stage
    int n_ctas;          // P: persistent CTAs of the partial kernel
    int slice;           // sequences per partial launch
    int n_slices;
    int per_sm;          // resident CTAs per SM
    int prefill;         // a contiguous cache takes the query-tiled prefill kernel (no combine)
    size_t off_status, off_qrot, off_prefix, off_rec_lse, off_rec_o, off_ranges, off_owners, off_balance, total;
    size_t prefix_stride, rec_lse_stride, rec_o_stride, ranges_stride, owners_stride;  // bytes per slice
};

int device_sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < 64) cache[dev] = n;
    return n;
}

// Range-balance state of the tensor-core kernel (BalanceState), at a fixed
// offset after the status word so that it survives changes of batch: header |
// claim[P] (uint64) | rate[P] | weight[P] | cumw[P + 1], each part 256-byte
// aligned.
size_t balance_bytes(int P)
{
    return 256 + align256((size_t)P * 8) + 2 * align256((size_t)P * 4) + align256(((size_t)P + 1) * 4);
}

uaa::BalanceState balance_of(void* ws, const Plan& pl)
{
    char* b = static_cast<char*>(ws) + pl.off_balance;
    const size_t P = (size_t)pl.n_ctas;
    uaa::BalanceState r;
    r.header = reinterpret_cast<unsigned*>(b);
    r.claim = reinterpret_cast<unsigned long long*>(b + 256);
    r.rate = reinterpret_cast<float*>(b + 256 + align256(P * 8));
    r.weight = reinterpret_cast<float*>(b + 256 + align256(P * 8) + align256(P * 4));
    r.cumw = reinterpret_cast<unsigned*>(b + 256 + align256(P * 8) + 2 * align256(P * 4));
    return r;
}

// Geometry of a step. The partial kernels are persistent: P = SMs x resident CTAs
// (4 for the CUDA-core kernel, 2 for the tensor-core kernel, 1 at head_dim 256 or
// with two column tiles),
// each attending one contiguous range of all units' key stages (the stream-K
// partition in internal.cuh), so the split needs no length bound. Batches above
// kMaxSliceBatch sequences are cut into slices (one partial + combine launch each)
// because a CTA keeps the slice's stage prefix in shared memory.
uaa_status make_plan(const uaa_attn_desc* d, int batch, int q_len, int max_len, int n_sm, Plan* pl)
{
    UAA_TRY(check_desc(d));
    if (batch < 0) return fail(UAA_ERR_INVALID_ARGUMENT, "batch=%d is negative", batch);
    if (max_len < 0) return fail(UAA_ERR_INVALID_ARGUMENT, "max_seq_len=%d is negative", max_len);
    if (n_sm <= 0) return fail(UAA_ERR_INVALID_ARGUMENT, "SM count %d is not positive", n_sm);
    if (q_len < 0 || q_len > kMaxQLen)
        return fail(UAA_ERR_UNSUPPORTED, "q_len=%d is not in [0, %d]", q_len, kMaxQLen);
    Plan p{};
    p.G = d->n_q_heads / d->n_kv_heads;
    p.q_len = q_len > 1 ? q_len : 1;
    p.kernel = d->kv_dtype == UAA_DTYPE_F32 ? 0 : 1;
    // a unit's query rows are the (token, head) pairs of one kv head: q_len G of them
    const int rows = p.q_len * p.G;
    if (p.kernel == 0 || d->head_dim == 256 || rows <= 8) {
        p.heads_per_cta = 8;
        p.n_head_tiles = 1;
    } else {
        p.heads_per_cta = 16;
        p.n_head_tiles = 2;
    }
    p.head_groups = (rows + p.heads_per_cta - 1) / p.heads_per_cta;
    p.mg = p.kernel == 1 ? uaa::partial_tc_keys_per_stage(d->head_dim, d->kv_dtype, p.n_head_tiles) / uaa::kTileKeys : 1;
    // tensor-core kernel: two CTAs per SM, one at head_dim 256 and with two column
    // tiles (its eight consumer warps take the registers of two CTAs)
    p.per_sm = p.kernel == 0 ? 4 : (d->head_dim == 256 || p.n_head_tiles == 2 ? 1 : 2);
    p.n_ctas = n_sm * p.per_sm;
    // long chunks on contiguous bf16 caches: whole 64-row blocks of (token, head) rows
    // per CTA, each streaming its keys once (the partial kernel's units hold 16 rows)
    p.prefill = p.kernel == 1 && d->kv_dtype == UAA_DTYPE_BF16 && (d->head_dim == 64 || d->head_dim == 128) &&
                rows >= uaa::kPrefillRows;
    p.slice = batch < uaa::kMaxSliceBatch ? (batch > 0 ? batch : 1) : uaa::kMaxSliceBatch;
    p.n_slices = batch > 0 ? (batch + p.slice - 1) / p.slice : 0;

    const size_t B = (size_t)(batch > 0 ? batch : 0), Hq = d->n_q_heads, D = d->head_dim;
    const size_t HC = (size_t)p.heads_per_cta, P = (size_t)p.n_ctas;
    p.prefix_stride = align256(((size_t)p.slice + 1) * 4);
    p.rec_lse_stride = align256(2 * P * HC * 4);
    p.rec_o_stride = align256(2 * P * HC * D * 4);
    p.ranges_stride = align256((P + 1) * 8);
    p.owners_stride = align256((size_t)p.slice * d->n_kv_heads * p.head_groups * 8);
    p.off_status = 0;
    p.off_balance = 256;
    p.off_qrot = p.off_balance + balance_bytes(p.n_ctas);
    p.off_prefix = p.off_qrot + align256(B * p.q_len * Hq * D * 4);
    p.off_rec_lse = p.off_prefix + p.n_slices * p.prefix_stride;
    p.off_rec_o = p.off_rec_lse + p.n_slices * p.rec_lse_stride;
    p.off_ranges = p.off_rec_o + p.n_slices * p.rec_o_stride;
    p.off_owners = p.off_ranges + p.n_slices * p.ranges_stride;
    p.total = p.off_owners + p.n_slices * p.owners_stride;
    *pl = p;
    return UAA_OK;
}

uaa_status check_args(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, bool need_io)
{
    if (!a) return fail(UAA_ERR_INVALID_ARGUMENT, "args is NULL");
    if (!ws || !ws->ptr) return fail(UAA_ERR_INVALID_ARGUMENT, "workspace is NULL");
    if (!aligned16(ws->ptr)) return fail(UAA_ERR_INVALID_ARGUMENT, "workspace is not 16-byte aligned");
    if (a->batch < 0) return fail(UAA_ERR_INVALID_ARGUMENT, "batch=%d is negative", a->batch);
    if (a->max_seq_len < 0) return fail(UAA_ERR_INVALID_ARGUMENT, "max_seq_len=%d is negative", a->max_seq_len);
    if (a->cache_capacity <= 0 || a->cache_capacity % 4 != 0)
        return fail(UAA_ERR_INVALID_ARGUMENT, "cache_capacity=%d is not a positive multiple of 4",
                    a->cache_capacity);
    const int q_len = a->q_len > 1 ? a->q_len : 1;
    if ((long long)a->max_seq_len + q_len > a->cache_capacity)
        return fail(UAA_ERR_CAPACITY, "max_seq_len=%d + %d new token(s) does not fit cache_capacity=%d",
                    a->max_seq_len, q_len, a->cache_capacity);
    if (a->block_table) {
        const int ps = a->page_size;
        if (ps < 16 || ps > 4096 || (ps & (ps - 1)) != 0)
            return fail(UAA_ERR_UNSUPPORTED, "page_size=%d is not a power of two in [16, 4096]", ps);
        // a page's scales are one TMA box of a stage; its shared-memory destination
        // (4 bytes per key) must start on 128 bytes
        if (ps < 32 && (d->kv_dtype == UAA_DTYPE_VQ8 || d->kv_dtype == UAA_DTYPE_Q8))
            return fail(UAA_ERR_UNSUPPORTED, "page_size=%d is below 32, the smallest page of a vq8 / q8 cache", ps);
        if (a->pages_per_seq <= 0 || (long long)a->pages_per_seq * ps != a->cache_capacity)
            return fail(UAA_ERR_INVALID_ARGUMENT,
                        "cache_capacity=%d is not pages_per_seq=%d x page_size=%d", a->cache_capacity,
                        a->pages_per_seq, ps);
        if (a->n_pages <= 0) return fail(UAA_ERR_INVALID_ARGUMENT, "n_pages=%d is not positive", a->n_pages);
        if ((long long)a->n_pages * d->n_kv_heads * ps > 2147483647LL - 2 * uaa::kTileKeys)
            return fail(UAA_ERR_UNSUPPORTED, "n_pages*n_kv_heads*page_size=%lld exceeds 2^31 cache rows",
                        (long long)a->n_pages * d->n_kv_heads * ps);
        if (!aligned16(a->block_table)) return fail(UAA_ERR_INVALID_ARGUMENT, "block_table is not 16-byte aligned");
    } else if ((long long)a->batch * d->n_kv_heads * a->cache_capacity > 2147483647LL - 2 * uaa::kTileKeys) {
        return fail(UAA_ERR_UNSUPPORTED, "batch*n_kv_heads*cache_capacity=%lld exceeds 2^31 cache rows",
                    (long long)a->batch * d->n_kv_heads * a->cache_capacity);
    }
    struct {
        const void* p;
        const char* name;
        bool needed;
    } ptrs[] = {
        {a->q, "q", need_io},
        {a->k_new, "k_new", need_io},
        {a->v_new, "v_new", need_io},
        {a->k_cache, "k_cache", true},
        {a->v_cache, "v_cache", true},
        {a->seq_lens, "seq_lens", true},
        {a->out, "out", true},
        {a->v_scale, "v_scale", d->kv_dtype == UAA_DTYPE_VQ8 || d->kv_dtype == UAA_DTYPE_Q8},
        {a->k_scale, "k_scale", d->kv_dtype == UAA_DTYPE_Q8},
        {a->q_norm_w, "q_norm_w", need_io && d->qk_norm},
        {a->k_norm_w, "k_norm_w", need_io && d->qk_norm},
        {a->sink, "sink", d->has_sink != 0},
    };
    for (auto& e : ptrs) {
        if (e.needed && !e.p && a->batch > 0)  // a batch of 0 reads and writes nothing
            return fail(d->has_sink && !strcmp(e.name, "sink") ? UAA_ERR_UNSUPPORTED : UAA_ERR_INVALID_ARGUMENT,
                        "%s is NULL%s", e.name,
                        !strcmp(e.name, "sink") ? " while has_sink=1" : "");
        if (e.p && !aligned16(e.p)) return fail(UAA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", e.name);
    }
    if (a->q_rot && !aligned16(a->q_rot)) return fail(UAA_ERR_INVALID_ARGUMENT, "q_rot is not 16-byte aligned");
    return UAA_OK;
}

uaa_status prepare(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, bool need_io,
                   Plan* pl)
{
    UAA_TRY(check_desc(d));
    UAA_TRY(check_args(d, a, ws, need_io));
    const int n_sm = device_sm_count();
    if (n_sm <= 0) return fail(UAA_ERR_CUDA, "no CUDA device: the SM count query failed");
    UAA_TRY(make_plan(d, a->batch, a->q_len, a->max_seq_len, n_sm, pl));
    if (ws->bytes < pl->total)
        return fail(UAA_ERR_INVALID_ARGUMENT, "workspace has %zu bytes, the step needs %zu", ws->bytes,
                    pl->total);
    return UAA_OK;
}

float softmax_scale(const uaa_attn_desc* d)
{
    return d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)d->head_dim);
}

// The prescale of the rotated q rows: logits come out in the log2 domain
// (scale log2 e), or as s / c when a softcap c applies tanh to them first.
// The paging of a step's caches (KvPages in internal.cuh).
uaa::KvPages pages_of(const uaa_step_args* a)
{
    uaa::KvPages pg{};
    if (a->block_table) {
        pg.table = a->block_table;
        int shift = 0;
        while ((1 << shift) < a->page_size) ++shift;
        pg.shift = shift;
        pg.per_seq = a->pages_per_seq;
        pg.n_pages = a->n_pages;
    }
    return pg;
}

float qscale(const uaa_attn_desc* d)
{
    const float scale = softmax_scale(d);
    return d->softcap > 0.f ? scale / d->softcap : scale * uaa::kLog2e;
}

// Rotary frequencies theta'_p / pi in fp64 and the cos/sin multiplier: plain
// base^(-2p/R) over the R rotated dims; llama3 wavelength interpolation; YaRN
// ramp over the pair index between the pairs whose wavelength fits beta_fast /
// beta_slow times into the original context; linear division by the factor
// (huggingface_decoder_completeness.md, P0.2 and P1.5; YaRN as published).
// Entries of pairs beyond R/2 stay 0 (those pairs are not rotated).
int rotary_dims(const uaa_attn_desc* d) { return d->rotary_dim > 0 ? d->rotary_dim : d->head_dim; }

void rope_table(const uaa_attn_desc* d, double* inv_freq_over_pi, float* mscale, double* mscale64 = nullptr)
{
    const int D = rotary_dims(d);
    for (int i = 0; i < d->head_dim / 2; ++i) inv_freq_over_pi[i] = 0.0;
    const double pi = 3.14159265358979323846;
    const uaa_rope_params& r = d->rope;
    double ms = 1.0;
    double lo = 0.0, hi = 0.0;
    if (r.scaling == UAA_ROPE_SCALING_YARN) {
        const double ln_base = log(r.theta);
        lo = D * log(r.original_max_pos / (2.0 * pi * r.beta_fast)) / (2.0 * ln_base);
        hi = D * log(r.original_max_pos / (2.0 * pi * r.beta_slow)) / (2.0 * ln_base);
        ms = r.attn_factor > 0.0 ? r.attn_factor : (r.factor > 1.0 ? 1.0 + 0.1 * log(r.factor) : 1.0);
    }
    for (int i = 0; i < D / 2; ++i) {
        const double f = pow(r.theta, -(2.0 * i) / D);
        double g = f;
        if (r.scaling == UAA_ROPE_SCALING_LLAMA3) {
            const double wl = 2.0 * pi / f;
            const double wl_keep = r.original_max_pos / r.high_freq_factor;
            const double wl_div = r.original_max_pos / r.low_freq_factor;
            if (wl > wl_div) {
                g = f / r.factor;
            } else if (wl >= wl_keep) {
                const double t = (r.original_max_pos / wl - r.low_freq_factor) /
                                 (r.high_freq_factor - r.low_freq_factor);
                g = t * f + (1.0 - t) * f / r.factor;
            }
        } else if (r.scaling == UAA_ROPE_SCALING_YARN) {
            double ramp = hi > lo ? (i - lo) / (hi - lo) : (i >= lo ? 1.0 : 0.0);
            ramp = ramp < 0.0 ? 0.0 : (ramp > 1.0 ? 1.0 : ramp);
            g = ramp * (f / r.factor) + (1.0 - ramp) * f;
        } else if (r.scaling == UAA_ROPE_SCALING_LINEAR) {
            g = f / r.factor;
        }
        inv_freq_over_pi[i] = g / pi;
    }
    *mscale = (float)ms;
    if (mscale64) *mscale64 = ms;
}

// ---------------------------------------------------------------- TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

uaa_status encode_2d(CUtensorMap* tm, CUtensorMapDataType dt, void* ptr, uint64_t inner, uint64_t rows,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw,
                     const char* what)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(UAA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(tm, dt, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(UAA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return UAA_OK;
}

// ---------------------------------------------------------------- the three launches

uaa_status run_append(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                      cudaStream_t s)
{
    if (a->batch == 0) return UAA_OK;
    uaa::AppendParams p{};
    p.B = a->batch;
    p.Hq = d->n_q_heads;
    p.Hkv = d->n_kv_heads;
    p.D = d->head_dim;
    p.q_len = pl.q_len;
    {  // tokens per CTA: one for short steps (parallelism), up to 16 once the grid has ~4 CTAs per SM anyway
        const int n_sm = device_sm_count();
        const long long tokens = (long long)a->batch * pl.q_len;
        long long tpc = n_sm > 0 ? tokens / (4LL * n_sm) : 1;
        p.tokens_per_cta = (int)(tpc < 1 ? 1 : (tpc > 16 ? 16 : tpc));
    }
    p.cap = a->cache_capacity;
    p.max_len = a->max_seq_len;
    p.style = d->rope.style;
    p.half_rot = rotary_dims(d) / 2;
    p.qk_norm = d->qk_norm;
    p.eps = d->norm_eps;
    p.norm_offset = d->norm_offset ? 1.f : 0.f;
    p.qscale = qscale(d);
    p.io_dtype = d->io_dtype;
    p.kv_dtype = d->kv_dtype;
    p.q = a->q;
    p.k_new = a->k_new;
    p.v_new = a->v_new;
    p.q_norm_w = a->q_norm_w;
    p.k_norm_w = a->k_norm_w;
    p.k_cache = a->k_cache;
    p.v_cache = a->v_cache;
    p.v_scale = a->v_scale;
    p.k_scale = a->k_scale;
    p.pages = pages_of(a);
    p.seq_lens = a->seq_lens;
    char* w = static_cast<char*>(ws->ptr);
    p.q_prime = reinterpret_cast<float*>(w + pl.off_qrot);
    p.q_rot_out = a->q_rot;
    p.status = reinterpret_cast<unsigned*>(w + pl.off_status);
    rope_table(d, p.inv_freq_over_pi, &p.mscale, &p.mscale64);
    const cudaError_t e = uaa::launch_append(p, s);
    return e == cudaSuccess ? UAA_OK : cuda_fail(e, "append kernel launch");
}

// The query-tiled prefill kernel takes step 2 of this call (and step 3 has nothing to do).
bool takes_prefill(const uaa_step_args* a, const Plan& pl) { return pl.prefill && !a->block_table; }

uaa_status run_prefill(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                       cudaStream_t s)
{
    char* w = static_cast<char*>(ws->ptr);
    const uint64_t D = d->head_dim;
    const uint64_t rows = (uint64_t)a->batch * d->n_kv_heads * a->cache_capacity;
    CUtensorMap tk, tv;
    UAA_TRY(encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->k_cache, D, rows, D * 2, 64,
                      (uint32_t)uaa::kPrefillKeys, CU_TENSOR_MAP_SWIZZLE_128B, "k_cache"));
    UAA_TRY(encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->v_cache, D, rows, D * 2, 64,
                      (uint32_t)uaa::kPrefillKeys, CU_TENSOR_MAP_SWIZZLE_128B, "v_cache"));
    uaa::PrefillParams p{};
    p.B = a->batch;
    p.Hq = d->n_q_heads;
    p.Hkv = d->n_kv_heads;
    p.D = d->head_dim;
    p.G = pl.G;
    p.q_len = pl.q_len;
    p.cap = a->cache_capacity;
    p.window = d->window;
    p.softcap_log2e = d->softcap > 0.f ? d->softcap * uaa::kLog2e : 0.f;
    p.q_prime = reinterpret_cast<const float*>(w + pl.off_qrot);
    p.seq_lens = a->seq_lens;
    p.sink = d->has_sink ? a->sink : nullptr;
    p.out = a->out;
    p.out_dtype = d->out_dtype;
    p.status = reinterpret_cast<unsigned*>(w + pl.off_status);
    const cudaError_t e = uaa::launch_prefill_umma(p, tk, tv, s);
    return e == cudaSuccess ? UAA_OK : cuda_fail(e, "prefill kernel launch");
}

// fused: the tensor-core kernel also performs the append (steps 1 and 2 in one launch).
uaa_status run_partial(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                       cudaStream_t s, bool fused = false)
{
    if (a->batch == 0) return UAA_OK;
    if (takes_prefill(a, pl)) return run_prefill(d, a, ws, pl, s);
    char* w = static_cast<char*>(ws->ptr);
    const size_t D = d->head_dim, Hq = d->n_q_heads;
    const size_t out_elem = d->out_dtype == UAA_DTYPE_F32 ? 4 : 2;
    uaa::PartialMaps maps{};
    if (pl.kernel == 1) {
        // contiguous caches: one box of a whole stage per row kind (and a second set of
        // 64-key boxes for units' partial last stages); paged caches: the pools, and one
        // box per page-aligned sub-tile of min(64, page_size) keys
        const bool paged = a->block_table != nullptr;
        const uint64_t rows = paged ? (uint64_t)a->n_pages * d->n_kv_heads * a->page_size
                                    : (uint64_t)a->batch * d->n_kv_heads * a->cache_capacity;
        const uint32_t tk_rows =
            paged ? (uint32_t)(a->page_size < uaa::kTileKeys ? a->page_size : uaa::kTileKeys)
                  : (uint32_t)uaa::partial_tc_keys_per_stage(d->head_dim, d->kv_dtype, pl.n_head_tiles);  // box height
        const uint64_t heads = paged ? (uint64_t)a->n_pages * d->n_kv_heads : (uint64_t)a->batch * d->n_kv_heads;
        const uint64_t scale_inner = paged ? (uint64_t)a->page_size : (uint64_t)a->cache_capacity;
        // int8 codes: boxes of box_rows x min(D, 128) bytes, swizzled like the bf16 boxes so
        // the kernel's ldmatrix reads on them are free of bank conflicts; scales: one
        // box_rows-float box per stage
        const uint32_t code_box = D > 128 ? 128u : (uint32_t)D;
        const CUtensorMapSwizzle code_sw = D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
        auto encode_set = [&](uint32_t box_rows, CUtensorMap& tk, CUtensorMap& tv, CUtensorMap& ts,
                              CUtensorMap& tks) -> uaa_status {
            if (d->kv_dtype == UAA_DTYPE_Q8) {
                UAA_TRY(encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->k_cache, D, rows, D, code_box, box_rows,
                                  code_sw, "k_cache codes"));
                UAA_TRY(encode_2d(&tks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->k_scale, scale_inner, heads,
                                  scale_inner * 4, box_rows, 1, CU_TENSOR_MAP_SWIZZLE_NONE, "k_scale"));
            } else {
                UAA_TRY(encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->k_cache, D, rows, D * 2, 64, box_rows,
                                  CU_TENSOR_MAP_SWIZZLE_128B, "k_cache"));
            }
            if (d->kv_dtype == UAA_DTYPE_VQ8 || d->kv_dtype == UAA_DTYPE_Q8) {
                UAA_TRY(encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->v_cache, D, rows, D, code_box, box_rows,
                                  code_sw, "v_cache codes"));
                UAA_TRY(encode_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->v_scale, scale_inner, heads,
                                  scale_inner * 4, box_rows, 1, CU_TENSOR_MAP_SWIZZLE_NONE, "v_scale"));
            } else {
                UAA_TRY(encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->v_cache, D, rows, D * 2, 64, box_rows,
                                  CU_TENSOR_MAP_SWIZZLE_128B, "v_cache"));
                ts = tv;  // unused by the bf16 kernel
            }
            if (d->kv_dtype != UAA_DTYPE_Q8) tks = ts;  // unused without key codes
            return UAA_OK;
        };
        UAA_TRY(encode_set(tk_rows, maps.k, maps.v, maps.s, maps.ks));
        if (!paged && tk_rows > (uint32_t)uaa::kTileKeys) {
            UAA_TRY(encode_set((uint32_t)uaa::kTileKeys, maps.kt, maps.vt, maps.st, maps.kst));
        } else {  // never used: every stage is one 64-key tile, or the pool boxes are sub-tiles already
            maps.kt = maps.k;
            maps.vt = maps.v;
            maps.st = maps.s;
            maps.kst = maps.ks;
        }
    }
    for (int sl = 0; sl < pl.n_slices; ++sl) {
        const int b0 = sl * pl.slice;
        const int nb = a->batch - b0 < pl.slice ? a->batch - b0 : pl.slice;
        uaa::PartialParams p{};
        p.B = nb;
        p.Hq = d->n_q_heads;
        p.Hkv = d->n_kv_heads;
        p.D = d->head_dim;
        p.G = pl.G;
        p.b_off = b0;
        p.heads_per_cta = pl.heads_per_cta;
        p.head_groups = pl.head_groups;
        p.cap = a->cache_capacity;
        p.q_len = pl.q_len;
        p.attn_window = d->window;
        // the partition covers the union of the rows' windows: the first token's
        // window starts q_len - 1 keys before the last one's
        p.window = d->window > 0 ? d->window + pl.q_len - 1 : 0;
        p.mg = pl.mg;
        p.softcap_log2e = d->softcap > 0.f ? d->softcap * uaa::kLog2e : 0.f;
        p.q_prime = reinterpret_cast<const float*>(w + pl.off_qrot) + (size_t)b0 * pl.q_len * Hq * D;
        p.k_cache = a->k_cache;
        p.v_cache = a->v_cache;
        p.v_scale = a->v_scale;
        p.k_scale = a->k_scale;
        p.pages = pages_of(a);
        p.seq_lens = a->seq_lens + b0;
        p.prefix = reinterpret_cast<int*>(w + pl.off_prefix + sl * pl.prefix_stride);
        p.ranges = reinterpret_cast<long long*>(w + pl.off_ranges + sl * pl.ranges_stride);
        p.owners = reinterpret_cast<unsigned*>(w + pl.off_owners + sl * pl.owners_stride);
        if (pl.kernel == 1) {
            p.bal = balance_of(w, pl);
            p.slice = sl;
            p.per_sm = pl.per_sm;
            p.uniform = d->reproducible;
        }
        p.rec_lse = reinterpret_cast<float*>(w + pl.off_rec_lse + sl * pl.rec_lse_stride);
        p.rec_o = reinterpret_cast<float*>(w + pl.off_rec_o + sl * pl.rec_o_stride);
        p.sink = d->has_sink ? a->sink : nullptr;
        p.out = static_cast<char*>(a->out) + (size_t)b0 * pl.q_len * Hq * D * out_elem;
        p.out_dtype = d->out_dtype;
        p.status = reinterpret_cast<unsigned*>(w + pl.off_status);
        if (fused) {
            const size_t io_elem = d->io_dtype == UAA_DTYPE_F32 ? 4 : 2;
            const size_t Hkv = d->n_kv_heads;
            p.fused = 1;
            p.max_len = a->max_seq_len;
            p.arrivals = reinterpret_cast<unsigned*>(w + pl.off_status) + 1;
            p.q = static_cast<const char*>(a->q) + (size_t)b0 * Hq * D * io_elem;  // one token per sequence
            p.k_new = static_cast<const char*>(a->k_new) + (size_t)b0 * Hkv * D * io_elem;
            p.v_new = static_cast<const char*>(a->v_new) + (size_t)b0 * Hkv * D * io_elem;
            p.io_dtype = d->io_dtype;
            p.kv_dtype = d->kv_dtype;
            p.style = d->rope.style;
            p.half_rot = rotary_dims(d) / 2;
            p.qk_norm = d->qk_norm;
            p.eps = d->norm_eps;
            p.norm_offset = d->norm_offset ? 1.f : 0.f;
            p.qscale = qscale(d);
            p.q_norm_w = a->q_norm_w;
            p.k_norm_w = a->k_norm_w;
            p.q_rot_out = a->q_rot ? a->q_rot + (size_t)b0 * Hq * D : nullptr;
            rope_table(d, p.inv_freq_over_pi, &p.mscale, &p.mscale64);
        }
        const cudaError_t e = pl.kernel == 0
                                  ? uaa::launch_partial_simt(p, pl.n_ctas, s)
                                  : uaa::launch_partial_tc(p, maps, d->kv_dtype, pl.n_head_tiles, pl.n_ctas, s);
        if (e != cudaSuccess) return cuda_fail(e, "partial kernel launch");
    }
    return UAA_OK;
}

uaa_status run_combine(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                       cudaStream_t s)
{
    if (a->batch == 0) return UAA_OK;
    if (takes_prefill(a, pl)) return UAA_OK;  // the prefill kernel wrote the output rows
    char* w = static_cast<char*>(ws->ptr);
    const size_t D = d->head_dim, Hq = d->n_q_heads;
    const size_t out_elem = d->out_dtype == UAA_DTYPE_F32 ? 4 : 2;
    for (int sl = 0; sl < pl.n_slices; ++sl) {
        const int b0 = sl * pl.slice;
        const int nb = a->batch - b0 < pl.slice ? a->batch - b0 : pl.slice;
        uaa::CombineParams p{};
        p.B = nb;
        p.Hq = d->n_q_heads;
        p.Hkv = d->n_kv_heads;
        p.D = d->head_dim;
        p.G = pl.G;
        p.heads_per_cta = pl.heads_per_cta;
        p.head_groups = pl.head_groups;
        p.q_len = pl.q_len;
        p.window = d->window > 0 ? d->window + pl.q_len - 1 : 0;
        p.mg = pl.mg;
        p.P = pl.n_ctas;
        p.out_dtype = d->out_dtype;
        p.sink = d->has_sink ? a->sink : nullptr;
        p.seq_lens = a->seq_lens + b0;
        p.prefix = reinterpret_cast<const int*>(w + pl.off_prefix + sl * pl.prefix_stride);
        p.ranges = reinterpret_cast<const long long*>(w + pl.off_ranges + sl * pl.ranges_stride);
        p.owners = reinterpret_cast<unsigned*>(w + pl.off_owners + sl * pl.owners_stride);
        if (pl.kernel == 1) p.bal = balance_of(w, pl);
        p.rec_lse = reinterpret_cast<const float*>(w + pl.off_rec_lse + sl * pl.rec_lse_stride);
        p.rec_o = reinterpret_cast<const float*>(w + pl.off_rec_o + sl * pl.rec_o_stride);
        p.out = static_cast<char*>(a->out) + (size_t)b0 * pl.q_len * Hq * D * out_elem;
        p.status = reinterpret_cast<unsigned*>(w + pl.off_status);
        const cudaError_t e = uaa::launch_combine(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    }
    return UAA_OK;
}

// The whole step: the fp32 one-launch kernel where it applies, else steps 1 and
// 2 (fused for the tensor-core kernel) and the combine.
uaa_status run_step(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                    cudaStream_t s);

// Keys per split of the fp32 one-launch step.
constexpr int kF32SplitKeys = 512;

// Splits per unit of the fp32 one-launch step (step_f32.cu), or 0 when the step
// takes the three-kernel path: it serves fp32 caches with one token per
// sequence in a single batch slice whose split records fit the slice's 2P.
int f32_step_splits(const uaa_attn_desc* d, const uaa_step_args* a, const Plan& pl)
{
    if (pl.kernel != 0 || pl.q_len != 1 || pl.n_slices != 1) return 0;
    const long long S = ((long long)a->max_seq_len + kF32SplitKeys) / kF32SplitKeys;  // keys: max_seq_len + 1
    const long long recs = (long long)a->batch * d->n_kv_heads * pl.head_groups * S;
    if (S > 1 && recs > 2LL * pl.n_ctas) return 0;
    return (int)S;
}

uaa_status run_step_f32(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                        int splits, cudaStream_t s)
{
    if (a->batch == 0) return UAA_OK;
    char* w = static_cast<char*>(ws->ptr);
    uaa::StepF32Params p{};
    p.B = a->batch;
    p.Hq = d->n_q_heads;
    p.Hkv = d->n_kv_heads;
    p.D = d->head_dim;
    p.G = pl.G;
    p.head_groups = pl.head_groups;
    p.cap = a->cache_capacity;
    p.max_len = a->max_seq_len;
    p.window = d->window;
    p.splits = splits;
    p.split_keys = kF32SplitKeys;
    p.style = d->rope.style;
    p.half_rot = rotary_dims(d) / 2;
    p.qk_norm = d->qk_norm;
    p.eps = d->norm_eps;
    p.norm_offset = d->norm_offset ? 1.f : 0.f;
    p.qscale = qscale(d);
    p.softcap_log2e = d->softcap > 0.f ? d->softcap * uaa::kLog2e : 0.f;
    p.io_dtype = d->io_dtype;
    p.out_dtype = d->out_dtype;
    p.q = a->q;
    p.k_new = a->k_new;
    p.v_new = a->v_new;
    p.q_norm_w = a->q_norm_w;
    p.k_norm_w = a->k_norm_w;
    p.sink = d->has_sink ? a->sink : nullptr;
    p.k_cache = static_cast<float*>(a->k_cache);
    p.v_cache = static_cast<float*>(a->v_cache);
    p.pages = pages_of(a);
    p.seq_lens = a->seq_lens;
    p.out = a->out;
    p.q_rot_out = a->q_rot;
    p.rec_o = reinterpret_cast<float*>(w + pl.off_rec_o);
    p.rec_lse = reinterpret_cast<float*>(w + pl.off_rec_lse);
    p.unit_count = reinterpret_cast<unsigned*>(w + pl.off_owners);
    p.arrivals = reinterpret_cast<unsigned*>(w + pl.off_status) + 1;
    p.status = reinterpret_cast<unsigned*>(w + pl.off_status);
    rope_table(d, p.inv_freq_over_pi, &p.mscale);
    const cudaError_t e = uaa::launch_step_f32(p, s);
    return e == cudaSuccess ? UAA_OK : cuda_fail(e, "fp32 step kernel launch");
}

// Steps 1 and 2: one fused launch for the tensor-core kernel, append then
// partial for the fp32 kernel.
uaa_status run_append_partial(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws,
                              const Plan& pl, cudaStream_t s)
{
    // one token per sequence; a chunk's append runs first, a warp per head row (a fused
    // kernel that staged a chunk's rows itself measured slower: its prep warp's
    // start-of-segment work is not hidden at one CTA per SM)
    if (pl.kernel == 1 && pl.q_len == 1) return run_partial(d, a, ws, pl, s, true);
    UAA_TRY(run_append(d, a, ws, pl, s));
    return run_partial(d, a, ws, pl, s);
}

uaa_status run_step(const uaa_attn_desc* d, const uaa_step_args* a, const uaa_workspace* ws, const Plan& pl,
                    cudaStream_t s)
{
    const int splits = f32_step_splits(d, a, pl);
    if (splits > 0) return run_step_f32(d, a, ws, pl, splits, s);
    UAA_TRY(run_append_partial(d, a, ws, pl, s));
    return run_combine(d, a, ws, pl, s);
}

}  // namespace

// ---------------------------------------------------------------- exported C ABI

extern "C" {

uaa_status uaa_rope_qk_norm_append(const uaa_attn_desc* desc, const uaa_step_args* args, const uaa_workspace* ws,
                                   cudaStream_t stream)
{
    Plan pl{};
    UAA_TRY(prepare(desc, args, ws, true, &pl));
    return run_append(desc, args, ws, pl, stream);
}

uaa_status uaa_decode_attn_partial(const uaa_attn_desc* desc, const uaa_step_args* args, const uaa_workspace* ws,
                                   cudaStream_t stream)
{
    Plan pl{};
    UAA_TRY(prepare(desc, args, ws, false, &pl));
    return run_partial(desc, args, ws, pl, stream);
}

uaa_status uaa_decode_attn_combine(const uaa_attn_desc* desc, const uaa_step_args* args, const uaa_workspace* ws,
                                   cudaStream_t stream)
{
    Plan pl{};
    UAA_TRY(prepare(desc, args, ws, false, &pl));
    return run_combine(desc, args, ws, pl, stream);
}

uaa_status uaa_decode_attn_append_partial(const uaa_attn_desc* desc, const uaa_step_args* args,
                                          const uaa_workspace* ws, cudaStream_t stream)
{
    Plan pl{};
    UAA_TRY(prepare(desc, args, ws, true, &pl));
    return run_append_partial(desc, args, ws, pl, stream);
}

uaa_status uaa_decode_attn(const uaa_attn_desc* desc, const uaa_step_args* args, const uaa_workspace* ws,
                           cudaStream_t stream)
{
    Plan pl{};
    UAA_TRY(prepare(desc, args, ws, true, &pl));
    return run_step(desc, args, ws, pl, stream);
}

size_t uaa_workspace_size(const uaa_attn_desc* desc, int32_t batch, int32_t max_seq_len, int32_t n_sm,
                          int32_t q_len)
{
    Plan pl{};
    if (n_sm <= 0) n_sm = device_sm_count();
    if (make_plan(desc, batch, q_len, max_seq_len, n_sm, &pl) != UAA_OK) return 0;
    return pl.total;
}

int32_t uaa_num_splits(const uaa_attn_desc* desc, int32_t batch, int32_t max_seq_len, int32_t n_sm, int32_t q_len)
{
    Plan pl{};
    if (n_sm <= 0) n_sm = device_sm_count();
    if (make_plan(desc, batch, q_len, max_seq_len, n_sm, &pl) != UAA_OK) return 0;
    return pl.n_ctas;
}

uaa_status uaa_get_workspace_layout(const uaa_attn_desc* desc, int32_t batch, int32_t max_seq_len, int32_t n_sm,
                                    int32_t q_len, uaa_workspace_layout* layout)
{
    if (!layout) return fail(UAA_ERR_INVALID_ARGUMENT, "layout is NULL");
    Plan pl{};
    if (n_sm <= 0) n_sm = device_sm_count();
    UAA_TRY(make_plan(desc, batch, q_len, max_seq_len, n_sm, &pl));
    layout->n_ctas = pl.n_ctas;
    layout->stage_keys = pl.mg * uaa::kTileKeys;
    layout->heads_per_cta = pl.heads_per_cta;
    layout->kernel = pl.prefill ? 2 : pl.kernel;
    layout->n_slices = pl.n_slices;
    layout->slice_batch = pl.slice;
    {
        uaa_step_args a{};
        a.batch = batch;
        a.max_seq_len = max_seq_len;
        layout->step_splits = f32_step_splits(desc, &a, pl);
        layout->step_kernels = batch == 0 ? 0
                               : layout->step_splits > 0 ? 1
                               : pl.prefill ? 2
                               : (pl.kernel == 1 && pl.q_len == 1) ? 2 * pl.n_slices
                                                                   : 1 + 2 * pl.n_slices;
    }
    layout->status_offset = pl.off_status;
    layout->q_rot_offset = pl.off_qrot;
    layout->prefix_offset = pl.off_prefix;
    layout->rec_lse_offset = pl.off_rec_lse;
    layout->rec_o_offset = pl.off_rec_o;
    layout->prefix_stride = pl.prefix_stride;
    layout->rec_lse_stride = pl.rec_lse_stride;
    layout->rec_o_stride = pl.rec_o_stride;
    layout->ranges_offset = pl.off_ranges;
    layout->ranges_stride = pl.ranges_stride;
    layout->owners_offset = pl.off_owners;
    layout->owners_stride = pl.owners_stride;
    layout->balance_offset = pl.off_balance;
    layout->total_bytes = pl.total;
    return UAA_OK;
}

uaa_status uaa_vq8_quantize(const void* v, int32_t v_dtype, int64_t n_rows, int32_t head_dim, int8_t* codes,
                            float* scales, cudaStream_t stream)
{
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(UAA_ERR_UNSUPPORTED, "head_dim=%d is not supported (supported: {64, 128, 256})", head_dim);
    if (v_dtype != UAA_DTYPE_F32 && v_dtype != UAA_DTYPE_BF16)
        return fail(UAA_ERR_UNSUPPORTED, "v_dtype=%d is not F32 or BF16", v_dtype);
    if (n_rows < 0) return fail(UAA_ERR_INVALID_ARGUMENT, "n_rows=%lld is negative", (long long)n_rows);
    if (n_rows == 0) return UAA_OK;
    if (!v || !codes || !scales) return fail(UAA_ERR_INVALID_ARGUMENT, "a vq8_quantize pointer is NULL");
    if (!aligned16(v) || !aligned16(codes) || !aligned16(scales))
        return fail(UAA_ERR_INVALID_ARGUMENT, "vq8_quantize pointers must be 16-byte aligned");
    const cudaError_t e = uaa::launch_vq8_quantize(v, v_dtype, n_rows, head_dim, codes, scales, stream);
    return e == cudaSuccess ? UAA_OK : cuda_fail(e, "vq8 quantize kernel launch");
}

uaa_status uaa_device_status(const uaa_workspace* ws, cudaStream_t stream, uint32_t* flags)
{
    if (!ws || !ws->ptr || !flags) return fail(UAA_ERR_INVALID_ARGUMENT, "workspace or flags is NULL");
    uint32_t f = 0;
    cudaError_t e = cudaMemcpyAsync(&f, ws->ptr, sizeof f, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && f) e = cudaMemsetAsync(ws->ptr, 0, sizeof f, stream);
    if (e == cudaSuccess && f) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    *flags = f;
    if (f)
        return fail(UAA_ERR_DEVICE, "device flags 0x%x:%s%s%s", f, (f & UAA_DEVFLAG_CAPACITY) ? " capacity" : "",
                    (f & UAA_DEVFLAG_LEN_HINT) ? " max_seq_len-exceeded" : "",
                    (f & UAA_DEVFLAG_TIMEOUT) ? " wait-timeout" : "");
    return UAA_OK;
}

const char* uaa_last_error(void) { return g_err; }

const char* uaa_status_string(uaa_status s)
{
    switch (s) {
    case UAA_OK: return "UAA_OK";
    case UAA_ERR_INVALID_ARGUMENT: return "UAA_ERR_INVALID_ARGUMENT";
    case UAA_ERR_UNSUPPORTED: return "UAA_ERR_UNSUPPORTED";
    case UAA_ERR_CAPACITY: return "UAA_ERR_CAPACITY";
    case UAA_ERR_CUDA: return "UAA_ERR_CUDA";
    case UAA_ERR_DEVICE: return "UAA_ERR_DEVICE";
    }
    return "UAA_UNKNOWN_STATUS";
}

int32_t uaa_abi_version(void) { return UAA_ABI_VERSION; }

}  // extern "C"

// ---------------------------------------------------------------- built-in scratch
// For callers that cannot allocate device memory: the workspace of
// uaa_decode_attn_static is this array. In host code the name is only a
// host-side stand-in, so the device address is looked up once per device
// (cudaGetSymbolAddress, device current) and handed to the kernels.
static __device__ __align__(256) unsigned char g_static_scratch[UAA_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_static_scratch_mu;
void* g_static_scratch_addr[64] = {};
// per device: a call launched the partial kernel but not the combine that frees
// its range slots, so the next call starts the scheduling state over
bool g_static_scratch_dirty[64] = {};

uaa_status static_scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(UAA_ERR_UNSUPPORTED, "device index %d is above 63", dev);
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
        g_static_scratch_addr[dev] = p;
    }
    *out = g_static_scratch_addr[dev];
    return UAA_OK;
}

}  // namespace

extern "C" uaa_status uaa_decode_attn_static(const uaa_attn_desc* desc, const uaa_step_args* args,
                                             cudaStream_t stream)
{
    UAA_TRY(check_desc(desc));
    if (!args) return fail(UAA_ERR_INVALID_ARGUMENT, "args is NULL");
    const int n_sm = device_sm_count();
    if (n_sm <= 0) return fail(UAA_ERR_CUDA, "no CUDA device: the SM count query failed");
    Plan pl{};
    UAA_TRY(make_plan(desc, args->batch, args->q_len, args->max_seq_len, n_sm, &pl));
    if (pl.total > (size_t)UAA_STATIC_SCRATCH_BYTES)
        return fail(UAA_ERR_INVALID_ARGUMENT,
                    "this step needs %zu bytes of scratch; the built-in scratch of uaa_decode_attn_static "
                    "holds %zu bytes (pass a workspace to uaa_decode_attn instead)",
                    pl.total, (size_t)UAA_STATIC_SCRATCH_BYTES);
    void* scratch = nullptr;
    UAA_TRY(static_scratch_address(&scratch));
    const uaa_workspace ws{scratch, (size_t)UAA_STATIC_SCRATCH_BYTES};
    UAA_TRY(check_args(desc, args, &ws, true));
    if (args->batch == 0) return UAA_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    // Every call starts from a clear status word and arrival counter (the first 8
    // bytes: a launch whose bounded wait gave up may leave the counter short of
    // its wrap). After a call that launched the partial kernel without its
    // combine, the range slots stay claimed: clear the balance state too.
    const size_t clear = g_static_scratch_dirty[dev] ? pl.off_qrot : 2 * sizeof(uint32_t);
    e = cudaMemsetAsync(static_cast<char*>(scratch) + pl.off_status, 0, clear, stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the built-in scratch state");
    g_static_scratch_dirty[dev] = true;
    UAA_TRY(run_step(desc, args, &ws, pl, stream));
    g_static_scratch_dirty[dev] = false;
    return UAA_OK;
}
