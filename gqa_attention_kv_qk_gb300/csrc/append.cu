// append.cu -- step 1 of the decode step: per-head QK RMSNorm, rotary embedding at
// the absolute KV index, and the append of the new k / v rows to the cache.
// q rows go to the workspace pre-multiplied by the partial kernel's logit
// prescale, k rows and v rows go to slot seq_lens[b] + t of the cache for token
// t. vq8 values (and q8 keys, after the rotation) are quantised in fp32 with IEEE
// division and round-half-even, the storage rule of the vq8 cache (llamay "Models
// and formats", "The KV cache, in three precisions"); bf16 keys are rounded as
// their exact values (near a rounding boundary, recomputed in fp64).
//
// Two kernels. One token per sequence (the separate append of fp32 caches, and
// any step whose layout the other does not take): append_kernel, CTAs of 16
// warps per group of tokens of a sequence, as many as give every warp one of a
// token's Hq + 2 Hkv head rows (a warp walking several rows is a chain of
// dependent loads); a CTA first builds the cos / sin tables of its tokens'
// positions (rope_cos_sin) while each warp loads its first head row, then each
// warp takes whole rows, loading the next while it processes the current one.
// Several tokens per sequence (verify steps, prefill chunks): append_staged_kernel
// (below), which streams each stage of tokens through shared memory.
#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"

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

// ---------------------------------------------------------------- chunks: staged rows
// Several tokens per sequence (a verify step or a prefill chunk). The q, k and v
// rows of consecutive tokens of one sequence are three contiguous blocks, so a
// stage of tokens arrives in shared memory as three bulk async copies
// (cp.async.bulk, two stages in flight per CTA), and every thread takes 16
// elements of a head row at a time with 16-byte accesses: a pair-wise rotation
// needs the row's two halves (NeoX) or adjacent elements (interleaved), which a
// row in shared memory gives without shuffles. The rotation angles are reduced
// in 64-bit integer arithmetic (rope_cos_sin_fx: the same remainder, rounded once
// to fp32, as rope_cos_sin, with no fp64 instruction). Near-boundary key pairs go
// to one queue per CTA and are recomputed in fp64 a pair per thread (the fp64
// pipe runs a whole warp per instruction, so a queue per CTA makes far fewer
// passes than a queue per warp). Measured on the 512-token prefill of the
// Llama-3.1-like cache (ncu): 240 us for the row-per-warp kernel (about 32 KB of
// loads in flight per SM, and a warp-wide fp64 pass per warp with a near pair),
// 74 us staged.

constexpr int kStagedThreads = 512;
constexpr int kStagedNearCap = 128;            // queued pairs per CTA (flushed when half full)
constexpr int kStagedInputBytes = 48 * 1024;   // input bytes of one stage, at most (one token at least)

// A queued near-boundary key pair (key_pair_exact): the element index of its cache
// row, its position and rotation pair, the two elements' indices in the row, their
// raw values, and the row's fp64 norm factor (0: no norm).
struct StagedNear {
    size_t slot;
    double inv64;
    int pos;
    short ia, ib, pp, pad;
    float ra, rb;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Elements e .. e + 7 of a head row in shared memory, as fp32 (e a multiple of 8).
template <typename T>
__device__ __forceinline__ void load8(const uint8_t* row, int e, float (&x)[8])
{
    if constexpr (sizeof(T) == 4) {
        const float4 a = *reinterpret_cast<const float4*>(row + 4 * e);
        const float4 c = *reinterpret_cast<const float4*>(row + 4 * e + 16);
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = c.x, x[5] = c.y, x[6] = c.z, x[7] = c.w;
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(row + 2 * e);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <typename T>
__device__ __forceinline__ float elem_at(const uint8_t* row, int e)
{
    if constexpr (sizeof(T) == 4)
        return reinterpret_cast<const float*>(row)[e];
    else
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[e]) << 16);
}

__device__ __forceinline__ void store8_f32(float* dst, const float (&y)[8], float scale)
{
    reinterpret_cast<float4*>(dst)[0] = make_float4(y[0] * scale, y[1] * scale, y[2] * scale, y[3] * scale);
    reinterpret_cast<float4*>(dst)[1] = make_float4(y[4] * scale, y[5] * scale, y[6] * scale, y[7] * scale);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

__device__ __forceinline__ void store8_bf16(void* dst, const float (&y)[8])
{
    *reinterpret_cast<uint4*>(dst) =
        make_uint4(bf16x2_bits(y[0], y[1]), bf16x2_bits(y[2], y[3]), bf16x2_bits(y[4], y[5]), bf16x2_bits(y[6], y[7]));
}

__device__ __forceinline__ void store8_codes(int8_t* dst, const float (&y)[8], float s)
{
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(vq8_code(y[i], s))) << (8 * (i & 3));
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
}

// Sum / maximum over the U lanes that hold one head row (aligned groups of U lanes).
template <int U>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int U>
__device__ __forceinline__ double group_sum64(double v)
{
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int U>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// A queued pair recomputed in fp64 and written over the cache's fp32 rounding.
__device__ __forceinline__ void fix_staged_pair(const AppendParams& p, const StagedNear& q, const double* freq)
{
    const double wa = p.qk_norm ? static_cast<double>(p.k_norm_w[q.ia]) + p.norm_offset : 1.0;
    const double wb = p.qk_norm ? static_cast<double>(p.k_norm_w[q.ib]) + p.norm_offset : 1.0;
    __nv_bfloat16 ha, hb;
    key_pair_exact(q.ra, q.rb, wa, wb, q.inv64, rope_cos_sin64(q.pp, p.half_rot, q.pos, freq[q.pp], p.mscale64), ha,
                   hb);
    static_cast<__nv_bfloat16*>(p.k_cache)[q.slot + q.ia] = ha;
    static_cast<__nv_bfloat16*>(p.k_cache)[q.slot + q.ib] = hb;
}

// A 4-byte asynchronous copy into shared memory (its completion: cp_async_wait_all
// by the issuing thread, then a barrier for the others).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// theta'_p / pi modulo 2 (exact) as a multiple of 2^-63, rounded to nearest: the
// angle pos * theta'_p / pi modulo 2 is then the low 64 bits of pos * g, read as a
// signed multiple of 2^-63 (an error below pos * 2^-64).
__device__ __forceinline__ unsigned long long angle_step(double inv_freq_over_pi)
{
    return __double2ull_rn(ldexp(fmod(inv_freq_over_pi, 2.0), 63));
}

// cos and sin of pos * theta'_p times mscale, as rope_cos_sin computes them: the
// angle in units of pi reduced to [-1, 1) and rounded once to fp32 for sincospif.
// Here the reduction is exact integer arithmetic (no fp64 instruction): the
// product's low 64 bits are the angle modulo 2, and the conversion rounds it to
// nearest.
__device__ __forceinline__ float2 rope_cos_sin_fx(int pos, unsigned long long g, float mscale)
{
    const long long t = static_cast<long long>(static_cast<unsigned long long>(pos) * g);
    float sn, cn;
    sincospif(__ll2float_rn(t) * 0x1p-63f, &sn, &cn);
    return make_float2(cn * mscale, sn * mscale);
}

// Shared memory of the staged kernel with tps tokens per stage.
__host__ __device__ inline size_t staged_stage_bytes(int tps, int Hq, int Hkv, int D, int esz)
{
    return static_cast<size_t>(tps) * (Hq + 2 * Hkv) * D * esz;
}

__host__ __device__ inline size_t staged_smem_bytes(int tps, int Hq, int Hkv, int D, int esz)
{
    return 2 * staged_stage_bytes(tps, Hq, Hkv, D, esz) + static_cast<size_t>(tps) * (D / 2) * sizeof(float2) +
           (D / 2) * (sizeof(double) + sizeof(unsigned long long)) + 2 * D * sizeof(float) +
           kStagedNearCap * sizeof(StagedNear) + 2 * sizeof(uint64_t) + 8 * sizeof(int);
}

// Stages of tokens_per_cta tokens (the last of a sequence may hold fewer); CTA c
// takes stages c, c + gridDim.x, ... Inputs 16-byte aligned; NeoX rotation with
// half_rot a multiple of 8.
template <int D, typename T>
__global__ void __launch_bounds__(kStagedThreads, 2) append_staged_kernel(const AppendParams p)
{
    constexpr int HALF = D / 2;
    constexpr int U = D / 16;  // threads per head row, 16 elements each
    constexpr int ESZ = sizeof(T);
    extern __shared__ __align__(16) uint8_t sm[];
    const int tid = threadIdx.x;
    const int TPS = p.tokens_per_cta;
    const int SPS = (p.q_len + TPS - 1) / TPS;  // stages per sequence
    const int n_stages = p.B * SPS;
    const uint32_t stage_bytes = static_cast<uint32_t>(staged_stage_bytes(TPS, p.Hq, p.Hkv, D, ESZ));
    float2* cs = reinterpret_cast<float2*>(sm + 2 * stage_bytes);       // [TPS][HALF] the stage's (cos, sin)
    double* freq = reinterpret_cast<double*>(cs + TPS * HALF);          // [HALF] theta'_p / pi
    unsigned long long* fstep = reinterpret_cast<unsigned long long*>(freq + HALF);  // [HALF] angle_step
    float* nw = reinterpret_cast<float*>(fstep + HALF);                 // [2][D] q / k norm weights + offset
    StagedNear* nq = reinterpret_cast<StagedNear*>(nw + 2 * D);         // [kStagedNearCap]
    uint64_t* bars = reinterpret_cast<uint64_t*>(nq + kStagedNearCap);  // a full barrier per stage buffer
    // [0] queued pairs, [1] last CTA, [2 + j] the length of the sequence of the stage in
    // buffer j, [4] the next 32-item chunk of the stage to take
    int* ctl = reinterpret_cast<int*>(bars + 2);
    const uint32_t sm_u32 = ptx::smem_u32(sm);
    const bool neox = p.style == UAA_ROPE_NEOX;

    if (tid == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
        ctl[0] = 0;
        ctl[4] = 0;
        ptx::fence_barrier_init();
    }
    grid_dependency_wait();  // the step's inputs and the previous step's reads are complete
    for (int i = tid; i < HALF; i += blockDim.x) {
        const double f = p.inv_freq_over_pi[i];
        freq[i] = f;
        fstep[i] = angle_step(f);
    }
    if (p.qk_norm)
        for (int i = tid; i < 2 * D; i += blockDim.x)
            nw[i] = (i < D ? p.q_norm_w[i] : p.k_norm_w[i - D]) + p.norm_offset;

    // thread 0 issues stage i of this CTA into buffer i & 1, and its sequence's length
    // into ctl[2 + (i & 1)] (an async copy: the thread does not wait for it)
    int issued = 0;
    auto issue = [&](int i) {
        const int st = blockIdx.x + i * gridDim.x;
        if (st >= n_stages) return;
        const int b = st / SPS, t0 = (st - b * SPS) * TPS, nt = min(TPS, p.q_len - t0);
        const size_t tok = static_cast<size_t>(b) * p.q_len + t0;
        const uint32_t qb = static_cast<uint32_t>(nt * p.Hq * D * ESZ), kb = static_cast<uint32_t>(nt * p.Hkv * D * ESZ);
        const uint32_t dst = sm_u32 + (i & 1) * stage_bytes;
        const uint32_t bar = ptx::smem_u32(&bars[i & 1]);
        ptx::mbar_arrive_expect_tx(bar, qb + 2 * kb);
        bulk_load(dst, static_cast<const T*>(p.q) + tok * p.Hq * D, qb, bar);
        bulk_load(dst + qb, static_cast<const T*>(p.k_new) + tok * p.Hkv * D, kb, bar);
        bulk_load(dst + qb + kb, static_cast<const T*>(p.v_new) + tok * p.Hkv * D, kb, bar);
        cp_async_4(ptx::smem_u32(&ctl[2 + (i & 1)]), p.seq_lens + b);
        ptx::cp_async_commit();
        issued = i + 1;
    };
    if (tid == 0) {
        issue(0);
        issue(1);
        ptx::cp_async_wait_all();  // the lengths of the first two stages
    }
    __syncthreads();

    // r / H for head counts H > 1 as __umulhi(r, ceil(2^32 / H)): exact for r < 2^32 / H
    // (here r < 16 H, so for H < 2^14)
    const unsigned div_q = p.Hq > 1 ? 0xFFFFFFFFu / p.Hq + 1u : 0u;
    const unsigned div_kv = p.Hkv > 1 ? 0xFFFFFFFFu / p.Hkv + 1u : 0u;
    int failed_at = -1;
    for (int i = 0;; ++i) {
        const int st = blockIdx.x + i * gridDim.x;
        if (st >= n_stages) break;
        const int b = st / SPS, t0 = (st - b * SPS) * TPS, nt = min(TPS, p.q_len - t0);
        // the stage's tokens take positions L + t0 .. ; a sequence whose tokens do not
        // all fit the cache is not appended (its q rows rotate at position 0)
        const int L = ctl[2 + (i & 1)];
        const bool fits = L >= 0 && L + p.q_len <= p.cap;
        if (tid == 0 && t0 == 0) {
            if (!fits)
                atomicOr(p.status, UAA_DEVFLAG_CAPACITY);
            else if (L > p.max_len)
                atomicOr(p.status, UAA_DEVFLAG_LEN_HINT);
        }
        for (int e = tid; e < nt * HALF; e += blockDim.x) {
            const int t = e / HALF, pp = e - t * HALF;
            cs[e] = pp < p.half_rot ? rope_cos_sin_fx(fits ? L + t0 + t : 0, fstep[pp], p.mscale) : make_float2(1.f, 0.f);
        }
        // one warp waits for the stage's copies; the others wait in the barrier
        const bool landed =
            tid >= 32 || ptx::mbar_wait(ptx::smem_u32(&bars[i & 1]), (i >> 1) & 1, kWaitLimitCycles);
        if (!__syncthreads_and(landed)) {  // also: the table is complete
            if (tid == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
            failed_at = i;
            break;
        }

        const uint8_t* sb = sm + (i & 1) * stage_bytes;
        const int nq_rows = nt * p.Hq, nk_rows = nt * p.Hkv;
        const int n_items = (nq_rows + 2 * nk_rows) * U;  // rows in buffer order: q, then k, then v
        // warps take 32-item chunks from a counter: the chunks holding key items first
        // (the near-boundary checks make them the longest), then the others in order
        const int n_chunks = (n_items + 31) / 32;
        const int kc0 = nq_rows * U / 32, kc1 = ((nq_rows + nk_rows) * U + 31) / 32;
        for (;;) {
            int wi = 0;
            if ((tid & 31) == 0) wi = atomicAdd(&ctl[4], 1);
            wi = __shfl_sync(0xffffffffu, wi, 0);
            if (wi >= n_chunks) break;
            const int chunk = wi < kc1 - kc0 ? kc0 + wi : (wi < kc1 ? wi - (kc1 - kc0) : wi);
            const int it = 32 * chunk + (tid & 31);
            const bool valid = it < n_items;
            const int rr = valid ? it / U : 0, u = it & (U - 1);
            const int kind = rr < nq_rows ? 0 : (rr < nq_rows + nk_rows ? 1 : 2);  // q, k, v
            const int r = kind == 0 ? rr : (kind == 1 ? rr - nq_rows : rr - nq_rows - nk_rows);
            const int H = kind == 0 ? p.Hq : p.Hkv;
            const int tok = H == 1 ? r : static_cast<int>(__umulhi(static_cast<unsigned>(r), kind == 0 ? div_q : div_kv));
            const int head = r - tok * H;
            const int pos = fits ? L + t0 + tok : 0;
            const uint8_t* row = sb + static_cast<size_t>(rr) * D * ESZ;

            // this thread's 16 elements, as two runs of 8 at e0 and e1: a NeoX unit
            // below half_rot pairs element e0 + j with e1 + j (rotation pair 8u + j);
            // otherwise the 16 elements are contiguous (values, interleaved pairs
            // (2pp, 2pp + 1), and NeoX pass-through elements past 2 half_rot)
            const bool neox_rot = neox && kind < 2 && 8 * u < p.half_rot;
            int e0, e1;
            if (neox_rot) {
                e0 = 8 * u;
                e1 = e0 + p.half_rot;
            } else if (neox && kind < 2) {
                e0 = 2 * p.half_rot + 16 * (u - p.half_rot / 8);
                e1 = e0 + 8;
            } else {
                e0 = 16 * u;
                e1 = e0 + 8;
            }
            float x0[8], x1[8];
            load8<T>(row, e0, x0);
            load8<T>(row, e1, x1);

            // RMSNorm over the head row (every lane takes part in the group sum)
            const bool normed = p.qk_norm && kind < 2;
            float inv = 1.f;
            if (p.qk_norm) {
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) ss += x0[j] * x0[j];
#pragma unroll
                for (int j = 0; j < 8; ++j) ss += x1[j] * x1[j];
                ss = group_sum<U>(ss);
                if (normed) {
                    inv = rms_inv(ss, D, p.eps);
                    const float* w = nw + kind * D;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        x0[j] = x0[j] * inv * w[e0 + j];
                        x1[j] = x1[j] * inv * w[e1 + j];
                    }
                }
            }

            // rotation (pass-through elements stay exact)
            const float2* cst = cs + tok * HALF;
            if (kind < 2 && neox) {
                if (neox_rot) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) rope_rotate(x0[j], x1[j], cst[8 * u + j]);
                }
            } else if (kind < 2) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (8 * u + j < p.half_rot) rope_rotate(x0[2 * j], x0[2 * j + 1], cst[8 * u + j]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (8 * u + 4 + j < p.half_rot) rope_rotate(x1[2 * j], x1[2 * j + 1], cst[8 * u + 4 + j]);
            }

            // the new token's cache row (k and v rows; -1: a paged table entry out of range)
            long long crow = -1;
            if (valid && kind > 0 && fits) {
                crow = cache_row(p.pages, p.Hkv, p.cap, b, head, pos);
                if (crow < 0 && u == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
            }
            const bool stores = crow >= 0;

            // row maximum for the int8 codes (q8 keys after the rotation, vq8 / q8 values)
            const bool quant = kind == 1 ? p.kv_dtype == UAA_DTYPE_Q8
                                         : kind == 2 && (p.kv_dtype == UAA_DTYPE_VQ8 || p.kv_dtype == UAA_DTYPE_Q8);
            float amax = 0.f;
            if (__any_sync(0xffffffffu, valid && quant)) {
#pragma unroll
                for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fmaxf(fabsf(x0[j]), fabsf(x1[j])));
                amax = group_max<U>(amax);
            }

            if (valid && kind == 0) {
                const size_t qrow = (static_cast<size_t>(b) * p.q_len + t0 + tok) * p.Hq + head;
                float* qp = p.q_prime + qrow * D;
                store8_f32(qp + e0, x0, p.qscale);
                store8_f32(qp + e1, x1, p.qscale);
                if (p.q_rot_out) {
                    store8_f32(p.q_rot_out + qrow * D + e0, x0, 1.f);
                    store8_f32(p.q_rot_out + qrow * D + e1, x1, 1.f);
                }
            } else if (stores) {
                const size_t slot = static_cast<size_t>(crow) * D;
                if (quant) {
                    const float s = vq8_scale(amax);
                    int8_t* codes = static_cast<int8_t*>(kind == 1 ? p.k_cache : p.v_cache) + slot;
                    store8_codes(codes + e0, x0, s);
                    store8_codes(codes + e1, x1, s);
                    if (u == 0) (kind == 1 ? p.k_scale : p.v_scale)[crow] = s;
                } else if (p.kv_dtype == UAA_DTYPE_F32) {
                    float* c = static_cast<float*>(kind == 1 ? p.k_cache : p.v_cache) + slot;
                    store8_f32(c + e0, x0, 1.f);
                    store8_f32(c + e1, x1, 1.f);
                } else {
                    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(kind == 1 ? p.k_cache : p.v_cache) + slot;
                    store8_bf16(c + e0, x0);
                    store8_bf16(c + e1, x1);
                }
            }

            // keys of a bf16 (or vq8) cache: rounded as their exact values. Pair j of the
            // 8 this thread holds lies near a bf16 rounding boundary (bf16_near_boundary)
            // when the error bound of its fp32 rotation (from the pre-rotation values,
            // recomputed from the staged row) reaches one; an unrotated, unnormalised
            // element is exact.
            unsigned near = 0;
            if (stores && kind == 1 && p.kv_dtype != UAA_DTYPE_F32 && p.kv_dtype != UAA_DTYPE_Q8) {
                float a0[8], a1[8];
                load8<T>(row, e0, a0);
                load8<T>(row, e1, a1);
                if (normed) {
                    const float* w = nw + D;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        a0[j] = a0[j] * inv * w[e0 + j];
                        a1[j] = a1[j] * inv * w[e1 + j];
                    }
                }
                auto check = [&](float pa, float pc, float ya, float yc, int j, int pp, bool rot) {
                    if (!rot && !normed) return;
                    const float2 cj = rot ? cst[pp] : make_float2(1.f, 0.f);
                    const float eb = key_error_bound(pa, pc, cj, normed);
                    if (bf16_near_boundary(ya, eb) || bf16_near_boundary(yc, eb)) near |= 1u << j;
                };
                if (neox) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) check(a0[j], a1[j], x0[j], x1[j], j, 8 * u + j, neox_rot);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        check(a0[2 * j], a0[2 * j + 1], x0[2 * j], x0[2 * j + 1], j, 8 * u + j, 8 * u + j < p.half_rot);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        check(a1[2 * j], a1[2 * j + 1], x1[2 * j], x1[2 * j + 1], 4 + j, 8 * u + 4 + j,
                              8 * u + 4 + j < p.half_rot);
                }
            }

            // near pairs: the row's fp64 norm factor (a group sum), then one queue entry
            // per pair (recomputed here when the queue is full)
            double inv64 = 0.0;
            if (p.qk_norm && __any_sync(0xffffffffu, near != 0u)) {
                double ss = 0.0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const double ra = elem_at<T>(row, e0 + j), rb = elem_at<T>(row, e1 + j);
                    ss = fma(ra, ra, ss);
                    ss = fma(rb, rb, ss);
                }
                ss = group_sum64<U>(ss);
                inv64 = 1.0 / sqrt(ss / static_cast<double>(D) + static_cast<double>(p.eps));
            }
            if (near) {
                const size_t slot = static_cast<size_t>(crow) * D;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    if (!((near >> j) & 1u)) continue;
                    StagedNear q;
                    int ia, ib, pp;
                    if (neox_rot) {
                        ia = e0 + j, ib = e1 + j, pp = 8 * u + j;
                    } else if (neox) {
                        ia = e0 + j, ib = e1 + j, pp = HALF - 1;  // a pass-through pair (pp >= half_rot)
                    } else {
                        ia = (j < 4 ? e0 : e1) + 2 * (j & 3), ib = ia + 1, pp = 8 * u + j;
                    }
                    q.slot = slot;
                    q.inv64 = inv64;
                    q.pos = pos;
                    q.ia = static_cast<short>(ia);
                    q.ib = static_cast<short>(ib);
                    q.pp = static_cast<short>(pp);
                    q.pad = 0;
                    q.ra = elem_at<T>(row, ia);
                    q.rb = elem_at<T>(row, ib);
                    const int at = atomicAdd(&ctl[0], 1);
                    if (at < kStagedNearCap)
                        nq[at] = q;
                    else
                        fix_staged_pair(p, q, freq);  // after this thread's own store of the row
                }
            }
        }
        if (tid == 0) ptx::cp_async_wait_all();  // the next stage's length, issued a stage ago
        __syncthreads();  // the buffer and the table are consumed; queued pairs and the next length are visible
        if (ctl[0] > kStagedNearCap / 2) {  // uniform: read after the barrier
            const int n = min(ctl[0], kStagedNearCap);
            for (int e = tid; e < n; e += blockDim.x) fix_staged_pair(p, nq[e], freq);
            __syncthreads();
            if (tid == 0) ctl[0] = 0;
            __syncthreads();
        }
        if (tid == 0) {
            ctl[4] = 0;  // no warp takes chunks until the next stage's barrier
            issue(i + 2);
        }
    }
    __syncthreads();
    {
        const int n = min(ctl[0], kStagedNearCap);
        for (int e = tid; e < n; e += blockDim.x) fix_staged_pair(p, nq[e], freq);
    }
    if (tid == 0) {
        // no copy into this CTA's shared memory may be in flight at its exit: the
        // length copies, and (bounded) the stages issued after the last one consumed
        ptx::cp_async_wait_all();
        if (failed_at >= 0)
            for (int j = failed_at; j < issued; ++j)
                if (!ptx::mbar_wait(ptx::smem_u32(&bars[j & 1]), (j >> 1) & 1, kWaitLimitCycles)) break;
    }
    __syncthreads();
    // every CTA counts in once its stages are done; the last one advances the lengths
    if (tid == 0) {
        __threadfence();
        ctl[1] = atomicInc(p.status + 1, gridDim.x - 1) == gridDim.x - 1;
    }
    __syncthreads();
    if (!ctl[1]) return;
    __threadfence();
    for (int i = tid; i < p.B; i += blockDim.x) {
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

// The staged kernel for several tokens per sequence, when its layout conditions
// hold; false: use the row-per-warp kernel.
bool launch_staged(const AppendParams& p, cudaStream_t s, cudaError_t& err)
{
    auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (p.q_len < 2 || (p.style == UAA_ROPE_NEOX && p.half_rot % 8 != 0)) return false;
    if (!a16(p.q) || !a16(p.k_new) || !a16(p.v_new) || !a16(p.k_cache) || !a16(p.v_cache) || !a16(p.q_prime) ||
        !a16(p.q_rot_out))
        return false;
    int dev = 0, n_sm = 0, smem_optin = 0, smem_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
        return false;
    const int esz = p.io_dtype == UAA_DTYPE_F32 ? 4 : 2;
    const long long per_token = static_cast<long long>(p.Hq + 2 * p.Hkv) * p.D * esz;
    // tokens per stage: a stage of at most kStagedInputBytes, and small steps spread
    // over the SMs (about two stages per SM before a CTA takes several); among those,
    // the largest whose items fill whole passes of the CTA's threads (a part-filled
    // last pass leaves warps idle at the stage's barrier)
    long long tps = kStagedInputBytes / per_token;
    tps = std::min<long long>(tps, static_cast<long long>(p.B) * p.q_len / (2LL * std::max(n_sm, 1)));
    tps = std::max<long long>(1, std::min<long long>({tps, 16, p.q_len}));
    const long long items_per_token = static_cast<long long>(p.Hq + 2 * p.Hkv) * (p.D / 16);
    for (long long t = tps; t >= 2; --t)
        if (t * items_per_token % kStagedThreads == 0) {
            tps = t;
            break;
        }
    const size_t smem = staged_smem_bytes(static_cast<int>(tps), p.Hq, p.Hkv, p.D, esz);
    if (smem > static_cast<size_t>(smem_optin)) return false;
    AppendParams q = p;
    q.tokens_per_cta = static_cast<int>(tps);
    const long long n_stages = static_cast<long long>(p.B) * ((p.q_len + tps - 1) / tps);
    const long long per_sm = std::max<long long>(1, std::min<long long>(2, smem_sm / static_cast<long long>(smem + 1024)));
    const long long ctas = std::min<long long>(n_stages, per_sm * n_sm);
    const dim3 grid(static_cast<unsigned>(ctas)), block(kStagedThreads);
    const bool f32 = p.io_dtype == UAA_DTYPE_F32;
#define UAA_STAGED_LAUNCH(DD)                                                                                          \
    do {                                                                                                               \
        auto* kern = f32 ? append_staged_kernel<DD, float> : append_staged_kernel<DD, __nv_bfloat16>;                 \
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));        \
        if (err == cudaSuccess) err = launch_dependent(kern, grid, block, smem, s, q);                                 \
    } while (0)
    switch (p.D) {
    case 64: UAA_STAGED_LAUNCH(64); break;
    case 128: UAA_STAGED_LAUNCH(128); break;
    case 256: UAA_STAGED_LAUNCH(256); break;
    default: return false;
    }
#undef UAA_STAGED_LAUNCH
    return true;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s)
{
    cudaError_t staged_err = cudaSuccess;
    if (launch_staged(p, s, staged_err)) return staged_err;
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
