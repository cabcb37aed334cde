// append.cu -- step 1 of the decode step: per-head QK RMSNorm, rotary embedding at
// the absolute KV index, and the append of the new k / v rows to the cache.
//
// CTAs of 16 warps per group of tokens of each sequence (one token for a decode
// step, up to 16 of a long chunk), as many as give every warp one of a token's
// Hq + 2 Hkv head rows (a warp walking several rows is a chain of dependent
// loads). A CTA first builds the cos / sin tables of its tokens' positions
// (rope_cos_sin) while each warp loads its first head row; then each warp takes
// whole rows, token after token, loading the next while it processes the current one: q
// rows go to the workspace pre-multiplied by the partial kernel's logit
// prescale, k rows and v rows go to slot seq_lens[b] + t of the cache for token t. vq8 values (and q8 keys, after the rotation) are quantised in fp32
// with IEEE division and round-half-even, the storage rule of the vq8 cache
// (llamay "Models and formats", "The KV cache, in three precisions").
#include "internal.cuh"

namespace uaa {
namespace {

constexpr int kAppendWarps = 16;
constexpr int kAppendMaxTokens = 16;  // tokens of one sequence per CTA at most
constexpr int kAppendAhead = 4;       // head rows in flight per warp

__device__ __forceinline__ void store_kv(void* cache, int dtype, size_t i, float v)
{
    if (dtype == UAA_DTYPE_F32)
        static_cast<float*>(cache)[i] = v;
    else
        static_cast<__nv_bfloat16*>(cache)[i] = __float2bfloat16_rn(v);
}

// vq8 storage of a row of D fp32 values held EPL per lane (vq8_scale, vq8_code).
template <int EPL>
__device__ __forceinline__ void quantize_row(const float (&x)[EPL], int lane, int8_t* codes,
                                             float* scale)
{
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float s = vq8_scale(warp_max(amax));
#pragma unroll
    for (int i = 0; i < EPL; ++i) codes[lane + 32 * i] = vq8_code(x[i], s);
    if (lane == 0) *scale = s;
}

// Row r of token t of sequence b: the q rows (r < Hq), then the k rows, then the v rows.
__device__ __forceinline__ const void* row_source(const AppendParams& p, int b, int t, int r, size_t& at)
{
    const size_t bt = static_cast<size_t>(b) * p.q_len + t;
    if (r < p.Hq) {
        at = (bt * p.Hq + r) * p.D;
        return p.q;
    }
    const int kv = r < p.Hq + p.Hkv ? r - p.Hq : r - p.Hq - p.Hkv;
    at = (bt * p.Hkv + kv) * p.D;
    return r < p.Hq + p.Hkv ? p.k_new : p.v_new;
}

// A key pair whose fp32 rotation lies near a bf16 rounding boundary, queued for
// its fp64 recomputation (key_pair_exact): the pair's cache row (element index),
// position and rotation pair, its raw elements and the row's fp64 norm factor.
struct NearKey {
    size_t slot;
    double inv64;
    int pos;
    short ia, ib, pp;
    float ra, rb;
};
constexpr int kNearCap = 16;  // queued pairs per warp; a full queue is flushed

// T: the io element type (float or __nv_bfloat16); AHEAD: head rows in flight
// per warp (kAppendAhead for token groups, where a warp walks many rows; 1 for
// one token per CTA, so that two CTAs per SM fit without spilling and a short
// step's grid runs in one wave)
template <int D, typename T, int AHEAD>
__global__ void __launch_bounds__(kAppendWarps * 32, 2) append_kernel(const AppendParams p)
{
    constexpr int EPL = D / 32;  // row elements per lane
    constexpr int HALF = D / 2;
    __shared__ float2 cs_all[kAppendMaxTokens][HALF];  // the group's cos / sin tables, one per token
    __shared__ double freq_s[HALF];
    __shared__ float rowbuf[kAppendWarps][D];
    __shared__ NearKey near_q[kAppendWarps][kNearCap];

    grid_dependency_wait();  // the step's inputs and the previous step's reads are complete
    const int n_rows = p.Hq + 2 * p.Hkv;
    const int parts = (n_rows + kAppendWarps - 1) / kAppendWarps;  // CTAs per token group
    const int groups = (p.q_len + p.tokens_per_cta - 1) / p.tokens_per_cta;
    const int bg = blockIdx.x / parts, part = blockIdx.x - bg * parts;
    const int b = bg / groups, grp = bg - b * groups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = part * kAppendWarps + warp;  // this warp's first row
    const int row_step = parts * kAppendWarps;
    const int tok0 = grp * p.tokens_per_cta, tok1 = min(p.q_len, tok0 + p.tokens_per_cta);

    // each warp takes rows row0, row0 + row_step, ... of every token of the group
    // (items k = 0 .. n_items - 1, token-major); the rows of the next kAppendAhead
    // items are in flight while one is processed (the first loads go out before the
    // length's): a row is a few hundred bytes, and one in flight per warp leaves
    // HBM mostly idle
    const int rpw = row0 < n_rows ? (n_rows - 1 - row0) / row_step + 1 : 0;  // rows per token
    const int n_items = rpw * (tok1 - tok0);
    auto load_item = [&](int k, float (&dst)[EPL]) {
        size_t at;
        const void* src = row_source(p, b, tok0 + k / rpw, row0 + (k % rpw) * row_step, at);
#pragma unroll
        for (int i = 0; i < EPL; ++i) dst[i] = load_as_float<T>(src, at + lane + 32 * i);
    };
    float buf[AHEAD][EPL];
#pragma unroll
    for (int u = 0; u < AHEAD; ++u)
        if (u < n_items) load_item(u, buf[u]);

    // the step's tokens take positions L .. L + q_len - 1; a sequence whose tokens do
    // not all fit the cache is not appended (and not advanced)
    const int L = p.seq_lens[b];
    const bool fits = L >= 0 && L + p.q_len <= p.cap;
    if (threadIdx.x == 0 && grp == 0 && part == 0) {
        if (!fits) atomicOr(p.status, UAA_DEVFLAG_CAPACITY);
        else if (L > p.max_len) atomicOr(p.status, UAA_DEVFLAG_LEN_HINT);
    }

    // near-boundary key pairs of this warp: one lane per queued pair recomputes it in
    // fp64 and overwrites the two elements (the fp64 pipe runs whole warps: a queue
    // shares its cost among up to kNearCap pairs)
    int n_near = 0;  // warp-uniform
    auto flush_near = [&]() {
        __syncwarp();
        if (lane < n_near) {
            const NearKey q = near_q[warp][lane];
            const double wa = p.qk_norm ? static_cast<double>(p.k_norm_w[q.ia]) + p.norm_offset : 1.0;
            const double wb = p.qk_norm ? static_cast<double>(p.k_norm_w[q.ib]) + p.norm_offset : 1.0;
            __nv_bfloat16 ha, hb;
            key_pair_exact(q.ra, q.rb, wa, wb, q.inv64,
                           rope_cos_sin64(q.pp, p.half_rot, q.pos, p.inv_freq_over_pi[q.pp], p.mscale64), ha, hb);
            static_cast<__nv_bfloat16*>(p.k_cache)[q.slot + q.ia] = ha;
            static_cast<__nv_bfloat16*>(p.k_cache)[q.slot + q.ib] = hb;
        }
        __syncwarp();
    };

    // the cos / sin tables of every token of the group: one token's by warps 0 ..
    // HALF / 32 - 1 with fixed-offset parameter reads (param_at_lane; a short step
    // is latency-bound), several tokens' by all warps from a shared copy of the
    // frequencies
    if (tok1 - tok0 == 1) {
#pragma unroll
        for (int i0 = 0; i0 < HALF; i0 += 32)
            if (warp == i0 / 32)
                cs_all[0][i0 + lane] = rope_pair_cos_sin(i0 + lane, p.half_rot, fits ? L + tok0 : 0,
                                                         param_at_lane(p.inv_freq_over_pi + i0, lane), p.mscale);
    } else {
        for (int i = threadIdx.x; i < HALF; i += blockDim.x) freq_s[i] = p.inv_freq_over_pi[i];
        __syncthreads();
        for (int i = threadIdx.x; i < (tok1 - tok0) * HALF; i += blockDim.x) {
            const int t = i / HALF, pp = i - t * HALF;
            cs_all[t][pp] = rope_pair_cos_sin(pp, p.half_rot, fits ? L + tok0 + t : 0, freq_s[pp], p.mscale);
        }
    }
    __syncthreads();  // the tables are complete

    // one head row r of token tok, held in x
    auto row_body = [&](int tok, int r, float (&x)[EPL]) {
            const int pos = fits ? L + tok : 0;
            const float2* cs = cs_all[tok - tok0];
            const bool is_q = r < p.Hq;
            const bool is_k = !is_q && r < p.Hq + p.Hkv;
            const int head = is_q ? r : (is_k ? r - p.Hq : r - p.Hq - p.Hkv);
            const size_t in_row = ((static_cast<size_t>(b) * p.q_len + tok) * (is_q ? p.Hq : p.Hkv) + head) * D;

            // the new token's cache row (k and v rows; -1: a paged table entry out of range)
            const long long crow = is_q || !fits ? 0 : cache_row(p.pages, p.Hkv, p.cap, b, head, pos);
            const bool stores = fits && crow >= 0;
            if (!is_q && fits && crow < 0 && lane == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
            const size_t slot = static_cast<size_t>(crow) * D;
            if (!is_q && !is_k) {  // value row: stored as given (or quantised)
                if (!stores) return;
                if (p.kv_dtype == UAA_DTYPE_VQ8 || p.kv_dtype == UAA_DTYPE_Q8) {
                    quantize_row<EPL>(x, lane, static_cast<int8_t*>(p.v_cache) + slot, p.v_scale + crow);
                } else {
#pragma unroll
                    for (int i = 0; i < EPL; ++i) store_kv(p.v_cache, p.kv_dtype, slot + lane + 32 * i, x[i]);
                }
                return;
            }

            if (p.qk_norm) {  // RMSNorm over the head row, before the rotation
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < EPL; ++i) ss += x[i] * x[i];
                ss = warp_sum(ss);
                const float inv = rms_inv(ss, D, p.eps);
                const float* w = is_q ? p.q_norm_w : p.k_norm_w;
#pragma unroll
                for (int i = 0; i < EPL; ++i) x[i] = x[i] * inv * (w[lane + 32 * i] + p.norm_offset);
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) rowbuf[warp][lane + 32 * i] = x[i];
            __syncwarp();

            // keys of a bf16 (or vq8) cache: rounded as their exact values (bf16_near_boundary)
            const bool kbf16 = is_k && stores && p.kv_dtype != UAA_DTYPE_F32 && p.kv_dtype != UAA_DTYPE_Q8;
            bool row_inv_done = false;
            double row_inv64 = 0.0;
            for (int pp = lane; pp < HALF; pp += 32) {
                const int2 e = rope_pair(pp, p.half_rot, D, p.style == UAA_ROPE_NEOX);
                const int ia = e.x, ib = e.y;
                float ya = rowbuf[warp][ia], yb = rowbuf[warp][ib];
                const float a0 = ya, b0 = yb;
                rope_rotate(ya, yb, cs[pp]);
                if (is_q) {
                    float* qp = p.q_prime + in_row;
                    qp[ia] = ya * p.qscale;
                    qp[ib] = yb * p.qscale;
                    if (p.q_rot_out) {
                        p.q_rot_out[in_row + ia] = ya;
                        p.q_rot_out[in_row + ib] = yb;
                    }
                } else if (stores && p.kv_dtype == UAA_DTYPE_Q8) {  // the whole rotated row first: its scale
                    rowbuf[warp][ia] = ya;                            // needs max |k| (pairs are disjoint)
                    rowbuf[warp][ib] = yb;
                } else if (kbf16) {
                    // the fp32 rounding now; a pair near a rounding boundary is queued and
                    // overwritten by its fp64 recomputation when the warp's queue is flushed
                    static_cast<__nv_bfloat16*>(p.k_cache)[slot + ia] = __float2bfloat16_rn(ya);
                    static_cast<__nv_bfloat16*>(p.k_cache)[slot + ib] = __float2bfloat16_rn(yb);
                    const float eb = key_error_bound(a0, b0, cs[pp], p.qk_norm != 0);
                    const bool near = bf16_near_boundary(ya, eb) || bf16_near_boundary(yb, eb);
                    const unsigned mask = __ballot_sync(0xffffffffu, near);
                    if (mask) {
                        size_t at;
                        const void* src = row_source(p, b, tok, r, at);
                        if (p.qk_norm && !row_inv_done) {  // the row's fp64 norm factor, once
                            double raw[EPL];
#pragma unroll
                            for (int i = 0; i < EPL; ++i) raw[i] = load_as_float<T>(src, at + lane + 32 * i);
                            row_inv64 = rms_inv64<EPL>(raw, D, p.eps);
                            row_inv_done = true;
                        }
                        if (n_near + __popc(mask) > kNearCap) {
                            flush_near();
                            n_near = 0;
                        }
                        if (near) {
                            NearKey& q = near_q[warp][n_near + __popc(mask & ((1u << lane) - 1u))];
                            q.slot = slot;
                            q.pos = pos;
                            q.ia = static_cast<short>(ia);
                            q.ib = static_cast<short>(ib);
                            q.pp = static_cast<short>(pp);
                            q.ra = load_as_float<T>(src, at + ia);
                            q.rb = load_as_float<T>(src, at + ib);
                            q.inv64 = p.qk_norm ? row_inv64 : 0.0;
                        }
                        n_near += __popc(mask);
                    }
                } else if (stores) {
                    store_kv(p.k_cache, UAA_DTYPE_F32, slot + ia, ya);
                    store_kv(p.k_cache, UAA_DTYPE_F32, slot + ib, yb);
                }
            }
            __syncwarp();
            if (is_k && stores && p.kv_dtype == UAA_DTYPE_Q8) {  // q8 key: codes and scale of the rotated row
                float y[EPL];
#pragma unroll
                for (int i = 0; i < EPL; ++i) y[i] = rowbuf[warp][lane + 32 * i];
                quantize_row<EPL>(y, lane, static_cast<int8_t*>(p.k_cache) + slot, p.k_scale + crow);
                __syncwarp();  // the row is read before the next one overwrites it
            }
    };
    for (int k0 = 0; k0 < n_items; k0 += AHEAD) {
#pragma unroll
        for (int u = 0; u < AHEAD; ++u) {
            const int k = k0 + u;
            if (k < n_items) {
                float x[EPL];
#pragma unroll
                for (int i = 0; i < EPL; ++i) x[i] = buf[u][i];
                if (k + AHEAD < n_items) load_item(k + AHEAD, buf[u]);
                row_body(tok0 + k / rpw, row0 + (k % rpw) * row_step, x);
            }
        }
    }
    if (n_near) flush_near();
    __syncthreads();
    // every CTA of the grid counts in once it has read its length; the last one
    // advances them all (the counter, the workspace word after the status word,
    // wraps to zero for the next launch)
    __shared__ bool last;
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicInc(p.status + 1, gridDim.x - 1) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const int n = p.seq_lens[i];
        if (n >= 0 && n + p.q_len <= p.cap) p.seq_lens[i] = n + p.q_len;
    }
}

template <int D>
__global__ void __launch_bounds__(256) vq8_quantize_kernel(const void* v, int v_dtype,
                                                           int64_t n_rows, int8_t* codes,
                                                           float* scales)
{
    constexpr int EPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         r < n_rows; r += warps) {
        float x[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = load_elem(v, v_dtype, static_cast<size_t>(r) * D + lane + 32 * i);
        quantize_row<EPL>(x, lane, codes + static_cast<size_t>(r) * D, scales + r);
    }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s)
{
    const int parts = (p.Hq + 2 * p.Hkv + kAppendWarps - 1) / kAppendWarps;  // a warp per head row
    const int groups = (p.q_len + p.tokens_per_cta - 1) / p.tokens_per_cta;
    const long long ctas = static_cast<long long>(p.B) * groups * parts;
    if (ctas > 2147483647LL) return cudaErrorInvalidConfiguration;  // beyond one grid's x extent
    const dim3 grid(static_cast<unsigned>(ctas)), block(kAppendWarps * 32);
    const bool f32 = p.io_dtype == UAA_DTYPE_F32;
    const bool wide = p.tokens_per_cta > 1;
#define UAA_APPEND_LAUNCH(DD)                                                                                     \
    (f32 ? (wide ? launch_dependent(append_kernel<DD, float, kAppendAhead>, grid, block, 0, s, p)                 \
                 : launch_dependent(append_kernel<DD, float, 1>, grid, block, 0, s, p))                           \
         : (wide ? launch_dependent(append_kernel<DD, __nv_bfloat16, kAppendAhead>, grid, block, 0, s, p)         \
                 : launch_dependent(append_kernel<DD, __nv_bfloat16, 1>, grid, block, 0, s, p)))
    switch (p.D) {
    case 64: return UAA_APPEND_LAUNCH(64);
    case 128: return UAA_APPEND_LAUNCH(128);
    case 256: return UAA_APPEND_LAUNCH(256);
    default: return cudaErrorInvalidValue;
    }
#undef UAA_APPEND_LAUNCH
}

cudaError_t launch_vq8_quantize(const void* v, int v_dtype, int64_t n_rows, int D, int8_t* codes,
                                float* scales, cudaStream_t s)
{
    const int64_t blocks64 = (n_rows + 7) / 8;
    const unsigned blocks = static_cast<unsigned>(blocks64 < 65535 * 16 ? blocks64 : 65535 * 16);
    switch (D) {
    case 64: vq8_quantize_kernel<64><<<blocks, 256, 0, s>>>(v, v_dtype, n_rows, codes, scales); break;
    case 128: vq8_quantize_kernel<128><<<blocks, 256, 0, s>>>(v, v_dtype, n_rows, codes, scales); break;
    case 256: vq8_quantize_kernel<256><<<blocks, 256, 0, s>>>(v, v_dtype, n_rows, codes, scales); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace uaa
