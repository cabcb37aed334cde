// internal.cuh -- kernel parameter blocks, launch declarations and small device
// helpers shared by the kernels of libuaa. Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/uaa.h"

namespace uaa {

constexpr int kTileKeys = 64;        // keys per tile; split boundaries fall on tiles
constexpr int kMaxHeadDim = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at the top SM clock

// ---------------------------------------------------------------- parameters

// Where the cache rows of a step live. Contiguous caches (table null): row
// (b Hkv + g) cap + j holds position j of sequence b, kv head g. Paged caches:
// position j is slot j mod ps of the sequence's logical page j / ps, which
// table[b][j / ps] maps to a physical page of the pool [n_pages][Hkv][ps]:
// row (page Hkv + g) ps + j mod ps (scales: the same row of [n_pages Hkv][ps]).
struct KvPages {
    const int* table;   // [B][per_seq] physical page per logical page, or null
    int shift;          // log2(ps)
    int per_seq;        // row length of the table
    int n_pages;        // pages in the pool
};

struct AppendParams {
    int B, Hq, Hkv, D;
    int q_len;              // tokens per sequence (rows [B][q_len][H][D] of q, k_new, v_new, q_prime)
    int tokens_per_cta;     // consecutive tokens of one sequence a CTA takes
    int cap, max_len;
    int style;              // UAA_ROPE_NEOX / _INTERLEAVED
    int half_rot;           // rotated pairs per head row (rotary_dim / 2)
    int qk_norm;
    float eps;
    float norm_offset;      // added to each RMSNorm weight (0, or 1 for Gemma's stored delta)
    float qscale;           // q_prime = rotated q * qscale (the partial kernel's logit prescale)
    float mscale;           // cos / sin multiplier (YaRN attention factor, else 1)
    double mscale64;        // the same in fp64 (keys recomputed near a bf16 rounding boundary)
    int io_dtype, kv_dtype;
    const void* q;
    const void* k_new;
    const void* v_new;
    const float* q_norm_w;
    const float* k_norm_w;
    void* k_cache;
    void* v_cache;
    float* v_scale;
    float* k_scale;         // q8 caches: the key rows' scales
    KvPages pages;
    int* seq_lens;
    float* q_prime;         // workspace [B][Hq][D]
    float* q_rot_out;       // optional [B][Hq][D]
    unsigned* status;
    double inv_freq_over_pi[kMaxHeadDim / 2];  // theta'_p / pi, fp64
};

// Range-balance state of the tensor-core partial kernel, at a fixed workspace
// offset: header[0] = kBalanceMagic and header[1] = P once the combine has
// written the tables for P slots, header[2] = launch generation (advanced by
// every combine); claim[v] = tag of the launch holding slot v, tag =
// (generation + 1) << 20 | slice (unique per partial launch, so slots are
// never reset); rate[v] = stages per ns of slot v in the last launch (0: none);
// weight[v] = moving average of the rates; cumw[0 .. P] = cumulative integer
// weights (cumw[P] = 0: none yet).
struct BalanceState {
    unsigned* header;
    unsigned long long* claim;
    float* rate;
    float* weight;
    unsigned* cumw;
};
constexpr unsigned kBalanceMagic = 0x42414c31u;

// The partial kernels are persistent and share one stream-K partition. Work is
// the list of ring stages (MG 64-key tiles each) of every unit = (sequence b,
// kv head, head group), units ordered by b then kv head then head group; a
// sequence with visible tiles [t0, t1) has ceil((t1 - t0) / MG) stages per
// unit. With T stages in total and P' = min(launched CTAs, T) ranges, range
// v < P' is stages [start[v], start[v + 1]) (never empty), cut at unit
// boundaries into segments. Uniform ranges: start[v] = floor(v T / P'). The
// tensor-core kernel weights the ranges by each CTA slot's measured speed (see
// Balance below) when T >= the launched CTAs. The kernel that ran writes the
// table start[0 .. P'] to the workspace for the combine. A segment that is a
// whole unit writes the unit's output rows; any other segment writes one
// record (normalised rows + log2-sum-exp) in slot 0 (the range's first
// segment) or 1 (its last), and the combine kernel merges the records of such
// units.
//
// Record index (2 v + slot) of the piece of a cut unit in range v: the piece in
// the first owner vA is that range's first segment (slot 0) only if the unit
// starts where vA starts; every later owner's piece starts its range (slot 0).
//
// Unit owners: the partial kernel writes, for each unit it touches, owners[2 u]
// = (vA + 1) | 2^31 if the first piece is vA's first segment, from the range
// holding the unit's first stage, and owners[2 u + 1] = vB + 1 from the range
// holding its last stage; the combine reads the pair (0: no stages) and clears
// it, so it needs neither the range table nor the stage prefix.
//
// Balance (tensor-core kernel): CTAs run at different speeds on different SMs
// (some groups of SMs stream 7-10 % slower), so equal ranges leave the fast
// CTAs idle at the end. Each CTA claims a range slot tied to its SM (slot
// per_sm * smid + k, k-th CTA on the SM; any free slot if taken), takes the
// range that the slot weights give it, and records its stages per ns. The
// combine that follows blends the rates into the weights (moving average),
// writes the cumulative integer weights for the next launch and frees the
// slots, so a partial launch must be followed by its combine.
struct PartialParams {
    int B, Hq, Hkv, D, G;
    int b_off;              // first sequence of this launch (batches are cut into slices)
    int heads_per_cta;      // query rows per unit (8 * NHT for the tensor-core kernel)
    int head_groups;        // row groups per kv head: ceil(q_len G / heads_per_cta)
    int q_len;              // tokens per sequence: a unit's rows are (token, head) pairs (query_row)
    int attn_window;        // the descriptor's window (0: none), per query row
    int cap, window;        // window: of the partition, attn_window + q_len - 1 (0: none)
    int mg;                 // 64-key tiles per stage
    float softcap_log2e;    // 0: no softcap; else softcap * log2(e)
    const float* q_prime;   // [B][Hq][D] (slice-relative: already offset by b_off)
    void* k_cache;          // whole caches (rows indexed with b_off + b)
    void* v_cache;
    float* v_scale;
    float* k_scale;         // q8 caches: the key rows' scales
    KvPages pages;          // table rows are indexed with b_off + b
    int* seq_lens;          // slice-relative (advanced by the fused kernel only)
    int* prefix;            // [B + 1] stage prefix over sequences, written for the combine
    long long* ranges;      // [P' + 1] range starts, written for the combine
    unsigned* owners;       // [B][units][2] first / last owner of each unit (UnitOwners), for the combine
    // balance state (tensor-core kernel; null: uniform ranges)
    BalanceState bal;
    int slice;              // index of this launch's batch slice (part of the claim tag)
    int uniform;            // uniform ranges whatever the slot weights (reproducible results)
    int per_sm;             // CTAs per SM of the launch
    float* rec_o;           // [2P][heads_per_cta][D]
    float* rec_lse;         // [2P][heads_per_cta]
    const float* sink;      // [Hq] or null
    void* out;              // [B][Hq][D] slice-relative
    int out_dtype;
    unsigned* status;
    // Fused append (steps 1 and 2 in one kernel): seq_lens hold the lengths
    // before the step; a sequence with room (0 <= L < cap) gets its new token at
    // slot L, attends keys up to and including it, and leaves with L + 1.
    int fused;
    int max_len;
    unsigned* arrivals;     // grid arrival counter (zero between launches)
    const void* q;          // [B][Hq][D] io_dtype, slice-relative
    const void* k_new;      // [B][Hkv][D] io_dtype, slice-relative
    const void* v_new;
    int io_dtype, kv_dtype;
    int style, qk_norm;
    int half_rot;           // rotated pairs per head row (rotary_dim / 2)
    float eps, qscale, mscale;
    double mscale64;        // mscale in fp64 (keys recomputed near a bf16 rounding boundary)
    float norm_offset;      // added to each RMSNorm weight
    const float* q_norm_w;
    const float* k_norm_w;
    float* q_rot_out;       // optional [B][Hq][D], slice-relative
    double inv_freq_over_pi[kMaxHeadDim / 2];
};

struct CombineParams {
    int B, Hq, Hkv, D, G;
    int heads_per_cta, head_groups;
    int q_len;
    int window, mg, P;
    int out_dtype;
    const float* sink;      // [Hq] or null
    const int* seq_lens;    // slice-relative
    const int* prefix;      // [B + 1]
    const long long* ranges;  // [P' + 1] range starts of the partial launch
    unsigned* owners;       // [B][units][2] written by the partial launch, cleared here
    BalanceState bal;       // of the tensor-core partial kernel (null pointers otherwise)
    const float* rec_o;
    const float* rec_lse;
    void* out;              // slice-relative
    unsigned* status;
};

// The whole decode step in one launch for fp32 caches and one token per
// sequence (step_f32.cu): a CTA per (sequence, kv head, group of up to 8 query
// heads, key split).
struct StepF32Params {
    int B, Hq, Hkv, D, G;
    int head_groups;        // ceil(G / 8)
    int cap, max_len;
    int window;             // the descriptor's window (0: none)
    int splits;             // key splits per unit: each split_keys keys, the last takes the rest
    int split_keys;
    int style, half_rot, qk_norm;
    float eps, norm_offset, qscale, mscale;
    float softcap_log2e;    // 0: no softcap
    int io_dtype, out_dtype;
    const void* q;          // [B][Hq][D] io_dtype
    const void* k_new;      // [B][Hkv][D]
    const void* v_new;
    const float* q_norm_w;
    const float* k_norm_w;
    const float* sink;      // [Hq] or null
    float* k_cache;
    float* v_cache;
    KvPages pages;
    int* seq_lens;
    void* out;              // [B][Hq][D]
    float* q_rot_out;       // optional [B][Hq][D]
    float* rec_o;           // [B][units][splits][8][D] (splits > 1)
    float* rec_lse;         // [B][units][splits][8]
    unsigned* unit_count;   // [B][units][2]: word 0 counts a unit's finished splits (zero between launches)
    unsigned* arrivals;     // grid arrival counter (zero between launches)
    unsigned* status;
    double inv_freq_over_pi[kMaxHeadDim / 2];
};

// Attention of a long chunk (prefill_umma.cu), after the append: a CTA per
// (sequence, kv head, block of 128 (token, head) rows) streams the keys its rows
// see once and writes their output rows; contiguous bf16 caches, head_dim 64 or
// 128.
struct PrefillParams {
    int B, Hq, Hkv, D, G;
    int q_len;              // tokens per sequence
    int cap;
    int window;             // the descriptor's window per query row (0: none)
    float softcap_log2e;    // 0: no softcap; else softcap * log2(e)
    const float* q_prime;   // [B][q_len][Hq][D], written by the append
    const int* seq_lens;    // lengths after the append
    const float* sink;      // [Hq] or null
    void* out;              // [B][q_len][Hq][D]
    int out_dtype;
    unsigned* status;
};

// ---------------------------------------------------------------- launches
// Each returns the launch error (cudaGetLastError) of its kernel.

cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_partial_simt(const PartialParams& p, int n_ctas, cudaStream_t s);
// Tensor maps of the tensor-core partial kernel: keys, values, value scales and
// key scales with boxes of a whole ring stage (or, for paged pools, of a page
// sub-tile), and the same with boxes of one 64-key tile (contiguous caches,
// for units' last stages that need fewer tiles than a stage holds).
struct PartialMaps {
    CUtensorMap k, v, s, ks;
    CUtensorMap kt, vt, st, kst;
};
cudaError_t launch_partial_tc(const PartialParams& p, const PartialMaps& m, int kv_dtype, int n_head_tiles,
                              int n_ctas, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
// tk, tv: tensor maps of the key and value caches with boxes of kPrefillKeys rows x 64 columns.
cudaError_t launch_prefill_umma(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);
// Query rows per CTA of the prefill kernel, and keys per block (the height of its TMA boxes).
constexpr int kPrefillRows = 128;
constexpr int kPrefillKeys = 128;
cudaError_t launch_step_f32(const StepF32Params& p, cudaStream_t s);
cudaError_t launch_vq8_quantize(const void* v, int v_dtype, int64_t n_rows, int D, int8_t* codes,
                                float* scales, cudaStream_t s);

// Dynamic shared memory the tensor-core partial kernel needs.
size_t partial_tc_smem_bytes(int D, int kv_dtype, int n_head_tiles);
// Keys per ring stage of the tensor-core partial kernel (the TMA box height) for
// n_head_tiles 8-row column tiles per unit.
int partial_tc_keys_per_stage(int D, int kv_dtype, int nht);
// Largest batch slice one partial launch takes (its stage prefix lives in shared memory).
constexpr int kMaxSliceBatch = 1024;

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream finishes; every kernel launched this way runs
// `griddepcontrol.wait` (grid_dependency_wait) before it reads anything an
// earlier launch wrote, so only its launch and set-up overlap.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------- device helpers

// Waits until the previous grid on the stream has completed and its memory is
// visible (a no-op for a kernel launched without programmatic dependence).
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel on the stream (launched with launch_dependent) be
// scheduled before this one completes: its CTAs take SMs as this grid's tail
// frees them and do their set-up; its grid_dependency_wait still waits for this
// grid to complete. The combine and the fp32 one-launch step (a few CTAs) use
// it: triggered from the partial kernel it cost 3 % (combine CTAs parked on SMs
// the partial kernel's tail still used).
__device__ __forceinline__ void allow_dependent_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void store_out(void* out, int dtype, size_t i, float v)
{
    if (dtype == UAA_DTYPE_F32)
        static_cast<float*>(out)[i] = v;
    else
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

// Visible keys of a sequence holding n keys after the append: [lo, n) with a
// window W keeping the last W of them (positions j > pos - W, pos = n - 1).
__host__ __device__ inline void key_range(int n, int window, int& lo, int& hi)
{
    hi = n;
    lo = (window > 0 && n > window) ? n - window : 0;
}

// Ring stages (mg tiles of 64 keys each) covering tiles [lo / 64, ceil(hi / 64)).
__host__ __device__ inline int stages_of(int lo, int hi, int mg)
{
    if (hi <= lo) return 0;
    const int t0 = lo / kTileKeys, t1 = (hi + kTileKeys - 1) / kTileKeys;
    return (t1 - t0 + mg - 1) / mg;
}

__host__ __device__ inline int record_of(int c, int cA, bool first_is_slot0)
{
    return 2 * c + ((c == cA && !first_is_slot0) ? 1 : 0);
}

// Stream-K partition of T stages over P CTAs.
__host__ __device__ inline long long range_start(int c, long long T, int P)
{
    return static_cast<long long>(c) * T / P;
}

// The CTA whose range holds stage x, 0 <= x < T (P <= T): the largest c with
// floor(c T / P) <= x, i.e. ceil((x + 1) P / T) - 1.
__host__ __device__ inline int cta_of(long long x, long long T, int P)
{
    return static_cast<int>(((x + 1) * P + T - 1) / T) - 1;
}

// Visible keys [lo, hi) of sequence b, clamped to the cache (a longer length is
// flagged by the caller).
__device__ __forceinline__ void visible_keys(int n, int window, int cap, int& lo, int& hi)
{
    key_range(n, window, lo, hi);
    if (hi > cap) hi = cap;
}

// Keys that the partial kernel attends for a sequence holding L keys: with the
// fused append the new token (slot L) is included when it fits the cache.
__device__ __forceinline__ void sequence_keys(int L, int window, int cap, bool fused, int& lo, int& hi)
{
    visible_keys(fused && L >= 0 && L < cap ? L + 1 : L, window, cap, lo, hi);
}

// Block-wide prefix[0..B] of units * stages per sequence into shared memory, and
// the lengths themselves into lens[0..B) (warp 0 scans, every thread returns
// after the barrier; nothing reads seq_lens afterwards). Writes the prefix to
// `global_copy` too when it is not null; flags go to `status` when it is not null.
// With `owners` (one CTA of the launch passes it) the owner words of the units
// of a sequence without stages are zeroed: no range writes them, and the
// workspace region may hold other data from a step of another geometry.
__device__ inline void build_stage_prefix(const int* seq_lens, int B, int window, int cap, int mg, int units,
                                          int* prefix, int* lens, int* global_copy, unsigned* status,
                                          bool fused = false, int max_len = 0, unsigned* owners = nullptr)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        if (lane == 0) {
            prefix[0] = 0;
            if (global_copy) global_copy[0] = 0;
        }
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int b = b0 + lane;
            int v = 0;
            if (b < B) {
                const int n = seq_lens[b];
                lens[b] = n;
                if (status && (fused ? (n < 0 || n >= cap) : n > cap)) atomicOr(status, UAA_DEVFLAG_CAPACITY);
                if (status && fused && n >= 0 && n < cap && n > max_len) atomicOr(status, UAA_DEVFLAG_LEN_HINT);
                int lo, hi;
                sequence_keys(n, window, cap, fused, lo, hi);
                v = units * stages_of(lo, hi, mg);
                if (owners && v == 0)
                    for (int u = 0; u < 2 * units; ++u) owners[2 * static_cast<size_t>(b) * units + u] = 0u;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (b < B) {
                prefix[b + 1] = carry + v;
                if (global_copy) global_copy[b + 1] = carry + v;
            }
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
}

// Largest b with prefix[b] <= x (prefix non-decreasing, prefix[0] = 0 <= x < prefix[B]).
__device__ __forceinline__ int find_sequence(const int* prefix, int B, long long x)
{
    int lo = 0, hi = B;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

// One segment of a CTA's stage range.
struct Segment {
    int b;          // slice-relative sequence
    int kvh, hg;    // kv head and head group of the unit
    int st0;        // first stage within the unit
    int n_st;       // stages in the segment
    int stages;     // stages of the whole unit
    int lo, hi;     // visible keys of the sequence
    bool whole;     // the segment is the whole unit
};

__device__ __forceinline__ Segment segment_at(const int* prefix, const int* lens, int B, int window, int cap,
                                              int head_groups, int units, long long pos, long long end,
                                              bool fused = false)
{
    Segment sg;
    sg.b = find_sequence(prefix, B, pos);
    const int per_seq = prefix[sg.b + 1] - prefix[sg.b];
    sg.stages = per_seq / units;
    const int local = static_cast<int>(pos - prefix[sg.b]);
    const int u = local / sg.stages;
    sg.st0 = local - u * sg.stages;
    const long long left = end - pos;
    sg.n_st = left < sg.stages - sg.st0 ? static_cast<int>(left) : sg.stages - sg.st0;
    sg.kvh = u / head_groups;
    sg.hg = u - sg.kvh * head_groups;
    sequence_keys(lens[sg.b], window, cap, fused, sg.lo, sg.hi);
    sg.whole = sg.st0 == 0 && sg.n_st == sg.stages;
    return sg;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float load_elem(const void* base, int dtype, size_t i)
{
    if (dtype == UAA_DTYPE_F32) return static_cast<const float*>(base)[i];
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

// Element i of a row of T (float or __nv_bfloat16) as fp32. Loops over row
// elements take T as a template parameter: a per-element branch on a run-time
// dtype keeps the loads of a loop from issuing back to back.
template <typename T>
__device__ __forceinline__ float load_as_float(const void* base, size_t i)
{
    if constexpr (sizeof(T) == 4)
        return static_cast<const float*>(base)[i];
    else
        return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

// Elements i and i + 1 (i even).
__device__ __forceinline__ float2 load_pair(const void* base, int dtype, size_t i)
{
    if (dtype == UAA_DTYPE_F32) return *reinterpret_cast<const float2*>(static_cast<const float*>(base) + i);
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(base) + i));
}

// ---------------------------------------------------------------- append arithmetic
// One definition each, used by the separate append kernel and by the fused one.

// cos and sin of pos * theta'_p, times mscale. The angle in units of pi,
// t = pos * theta'_p / pi, is formed in fp64 and reduced exactly to
// t - 2 rint(t / 2) in [-1, 1]; the reduced value is rounded to fp32 for
// sincospif (error ~ 2^-24 pi rad at any position).
__device__ __forceinline__ float2 rope_cos_sin(int pos, double inv_freq_over_pi, float mscale)
{
    const double t = static_cast<double>(pos) * inv_freq_over_pi;
    const double r = fma(-2.0, rint(0.5 * t), t);
    float sn, cn;
    sincospif(static_cast<float>(r), &sn, &cn);
    return make_float2(cn * mscale, sn * mscale);
}

// Entry `lane` of 32 consecutive kernel-parameter values (table32 a fixed
// offset into the kernel's parameters). Each read has a fixed offset: a
// per-lane index into kernel parameters would serialise the lanes' reads on the
// constant cache.
__device__ __forceinline__ double param_at_lane(const double* table32, int lane)
{
    double v = 0.0;
#pragma unroll
    for (int i = 0; i < 32; ++i) v = lane == i ? table32[i] : v;
    return v;
}

// (cos, sin) of rotation pair pp of a head whose first half_rot pairs rotate:
// the angle pos * theta'_pp, or (1, 0) for a pair that passes unchanged (the
// dims beyond rotary_dim, which no attention factor scales).
__device__ __forceinline__ float2 rope_pair_cos_sin(int pp, int half_rot, int pos, double inv_freq_over_pi,
                                                    float mscale)
{
    return pp < half_rot ? rope_cos_sin(pos, inv_freq_over_pi, mscale) : make_float2(1.f, 0.f);
}

// Row elements (a, b) of rotation pair pp, 0 <= pp < D/2, in a head of D dims
// whose first 2 half_rot dims rotate. Interleaved: (2pp, 2pp+1) throughout.
// NeoX: (pp, pp + half_rot) for a rotated pair; the pass-through dims
// 2 half_rot .. D-1 are paired as (pp + half_rot, pp + D/2) so that every
// element belongs to exactly one pair (with half_rot = D/2: (pp, pp + D/2)).
__device__ __forceinline__ int2 rope_pair(int pp, int half_rot, int D, bool neox)
{
    if (!neox) return make_int2(2 * pp, 2 * pp + 1);
    return pp < half_rot ? make_int2(pp, pp + half_rot) : make_int2(pp + half_rot, pp + D / 2);
}

// ---------------------------------------------------------------- bf16 keys, rounded as their exact values
// A rotated key element goes to a bf16 cache rounded to nearest-even from its
// exact value (the method's storage precision). The fp32 result y of the
// normalisation and rotation lies within key_error_bound of the exact value;
// where that interval holds no bf16 rounding boundary, RN(y) is the exact
// value's rounding. Otherwise (about one element in 500) the element is
// recomputed in fp64 (rope_cos_sin64, rms_inv64) and rounded from there
// (bf16_from_double).

// Bound on |y - exact| for y = a c - b s computed in fp32 from a, b and c, s
// (sincospif of the exactly reduced angle, cast to fp32, times the multiplier
// mu; |c| + |s| >= mu). The cos / sin error (half an ulp of the angle, one of
// sincospif, the multiplier's rounding: below 2^-21.8 mu) and the rounding of
// the rotation (2^-23 mu) scale with |a| + |b|, not with |y| (they do not
// cancel where the rotation does); an fp32 RMSNorm adds about 12 ulps to a and
// b (2^-20.4). The bound takes 2^-19 (2^-18 after a norm) times (|a| + |b|)
// (|c| + |s|): three to five times the worst case.
__device__ __forceinline__ float key_error_bound(float a, float b, float2 cs, bool normed)
{
    return (normed ? 0x1p-18f : 0x1p-19f) * (fabsf(a) + fabsf(b)) * (fabsf(cs.x) + fabsf(cs.y)) + 0x1p-120f;
}

// Whether bf16 rounding of the exact value may differ from RN(y), |y - exact| <= e:
// a rounding boundary (midpoint between neighbouring bf16 values) lies within e
// of y. Values below 2^-118 always count as near (never met by real keys); inf
// and NaN never.
__device__ __forceinline__ bool bf16_near_boundary(float y, float e)
{
    const uint32_t ab = __float_as_uint(y) & 0x7fffffffu;
    if (ab >= 0x7f800000u) return false;
    const uint32_t rb = (ab + 0x7fffu + ((ab >> 16) & 1u)) & 0xffff0000u;  // RN-even to bf16, as bits of |y|
    const uint32_t E = rb >> 23;                                             // its biased exponent
    if (E < 9) return true;
    const float u = __uint_as_float((E - 7u) << 23);              // bf16 spacing in that binade
    const float h_lo = (rb & 0x007f0000u) ? 0.5f * u : 0.25f * u;  // below a power of two the spacing halves
    const float d = __uint_as_float(ab) - __uint_as_float(rb);     // exact
    return !(e < fminf(0.5f * u - d, h_lo + d));
}

// x rounded to nearest-even bf16 (overflow to infinity): toward zero to fp32 with
// a sticky last bit (round to odd), then to nearest-even.
__device__ __forceinline__ __nv_bfloat16 bf16_from_double(double x)
{
    float f = __double2float_rz(x);
    if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
    return __float2bfloat16_rn(f);
}

// (cos, sin) of the angle pos * theta'_p in fp64, times the multiplier; (1, 0) for a pair that is not rotated.
__device__ __forceinline__ double2 rope_cos_sin64(int pp, int half_rot, int pos, double inv_freq_over_pi,
                                                  double mscale)
{
    if (pp >= half_rot) return make_double2(1.0, 0.0);
    const double t = static_cast<double>(pos) * inv_freq_over_pi;
    const double r = fma(-2.0, rint(0.5 * t), t);
    double sn, cn;
    sincospi(r, &sn, &cn);
    return make_double2(cn * mscale, sn * mscale);
}

// fp64 RMSNorm factor of a head row held EPL elements per lane (every lane of the warp calls it).
template <int EPL>
__device__ __forceinline__ double rms_inv64(const double (&x)[EPL], int D, float eps)
{
    double ss = 0.0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) ss = fma(x[i], x[i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    return 1.0 / sqrt(ss / static_cast<double>(D) + static_cast<double>(eps));
}

// The rotated pair (ra, rb: raw key elements; wa, wb: their norm weights plus
// offset, used when inv64 > 0) in fp64, rounded to bf16.
__device__ __forceinline__ void key_pair_exact(double ra, double rb, double wa, double wb, double inv64, double2 cs,
                                               __nv_bfloat16& ha, __nv_bfloat16& hb)
{
    if (inv64 > 0.0) {
        ra = ra * inv64 * wa;
        rb = rb * inv64 * wb;
    }
    ha = bf16_from_double(ra * cs.x - rb * cs.y);
    hb = bf16_from_double(ra * cs.y + rb * cs.x);
}

// Query row r of a unit of kv head kvh: the rows of a kv head are the (token,
// head) pairs of the step, token-major, so row r is token r / G at query head
// kvh G + r % G. Returns its index in the [B][q_len][Hq] rows of q, q_prime and
// out (with q_len = 1: b Hq + kvh G + r).
__device__ __forceinline__ size_t query_row(int b, int r, int kvh, int G, int Hq, int q_len)
{
    const int t = r / G;
    return (static_cast<size_t>(b) * q_len + t) * Hq + kvh * G + (r - t * G);
}

// Cache row of (sequence b, kv head g, position j) under KvPages, or -1 where
// a paged table entry lies outside [0, n_pages) (the caller flags
// UAA_DEVFLAG_PAGE and neither reads nor writes that row).
__device__ __forceinline__ long long cache_row(const KvPages& pg, int Hkv, int cap, int b, int g, int j)
{
    if (!pg.table) return (static_cast<long long>(b) * Hkv + g) * cap + j;
    const int page = __ldg(pg.table + static_cast<size_t>(b) * pg.per_seq + (j >> pg.shift));
    if (page < 0 || page >= pg.n_pages) return -1;
    return ((static_cast<long long>(page) * Hkv + g) << pg.shift) | (j & ((1 << pg.shift) - 1));
}

// Rotation of pair (a, b) by the angle whose (cos, sin) is cs.
__device__ __forceinline__ void rope_rotate(float& a, float& b, float2 cs)
{
    const float ya = a * cs.x - b * cs.y;
    const float yb = a * cs.y + b * cs.x;
    a = ya;
    b = yb;
}

// RMSNorm factor 1 / sqrt(mean(x^2) + eps) from the row's sum of squares.
__device__ __forceinline__ float rms_inv(float sum_sq, int D, float eps)
{
    return 1.0f / sqrtf(sum_sq / static_cast<float>(D) + eps);
}

// vq8 storage rule of a row with max|v| = amax: s = amax / 127 (IEEE division),
// code = rint(v / s) with ties to even, |code| <= 127; s = 0 gives codes 0.
__device__ __forceinline__ float vq8_scale(float amax) { return __fdiv_rn(amax, 127.0f); }

__device__ __forceinline__ int8_t vq8_code(float v, float s)
{
    if (s == 0.f) return 0;
    const float c = fminf(fmaxf(rintf(__fdiv_rn(v, s)), -127.f), 127.f);
    return static_cast<int8_t>(static_cast<int>(c));
}

// ---------------------------------------------------------------- range slots

__device__ __forceinline__ unsigned long long global_time_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One thread of a tensor-core CTA (while warp 0 scans the lengths): claims a
// range slot v with this launch's tag and returns it with the slot's
// cumulative weights cumw[v], cumw[v + 1] and the total (0 when the tables are
// not for this P). Returns -1 only if every slot carries this launch's tag (a
// partial launch repeated without its combine).
__device__ inline int claim_slot(const PartialParams& p, unsigned& w0, unsigned& w1, unsigned& wP)
{
    const int P = static_cast<int>(gridDim.x);
    const BalanceState& b = p.bal;
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const int v0 = static_cast<int>((static_cast<unsigned long long>(smid) * p.per_sm) % P);
    // one round of independent reads: the header, the first-choice slot and its weights
    const unsigned magic = __ldcg(b.header), hp = __ldcg(b.header + 1), gen = __ldcg(b.header + 2);
    const unsigned c0 = __ldcg(b.cumw + v0), c1 = __ldcg(b.cumw + v0 + 1), cP = __ldcg(b.cumw + P);
    const unsigned long long seen = __ldcg(b.claim + v0);
    const bool tables = magic == kBalanceMagic && hp == static_cast<unsigned>(P);
    const unsigned long long tag = (static_cast<unsigned long long>(gen) + 1ull) << 20 | static_cast<unsigned>(p.slice);
    wP = tables ? cP : 0u;
    if (seen != tag && atomicCAS(b.claim + v0, seen, tag) == seen) {
        w0 = wP ? c0 : 0u;
        w1 = wP ? c1 : 0u;
        return v0;
    }
    for (int k = 1; k < P; ++k) {  // the first choice was taken: the next free slot
        const int v = v0 + k < P ? v0 + k : v0 + k - P;
        const unsigned long long old = __ldcg(b.claim + v);
        if (old != tag && atomicCAS(b.claim + v, old, tag) == old) {
            w0 = wP ? __ldcg(b.cumw + v) : 0u;
            w1 = wP ? __ldcg(b.cumw + v + 1) : 0u;
            return v;
        }
    }
    w0 = w1 = 0;
    return -1;
}

// The range [s, e) of slot v when the launch holds T stages (empty: no work),
// writing start[v] (and start[P'] = T from the last range) for the combine.
// Weighted when every slot has a weight (wP > 0), T >= P and the launch does
// not ask for reproducible results: one stage each, the other T - P shared in
// proportion to the weights; otherwise uniform over P' = min(P, T).
__device__ inline void slot_range(const PartialParams& p, int v, unsigned w0, unsigned w1, unsigned wP, long long T,
                                  long long& s, long long& e)
{
    const int P = static_cast<int>(gridDim.x);
    const int Pp = T < P ? static_cast<int>(T) : P;
    s = e = 0;
    if (v < 0 || v >= Pp) return;
    if (T >= P && wP > 0 && !p.uniform) {
        const long long extra = T - P;
        s = v + extra * w0 / wP;
        e = v + 1 + extra * w1 / wP;
    } else {
        s = range_start(v, T, Pp);
        e = range_start(v + 1, T, Pp);
    }
    p.ranges[v] = s;
    if (v == Pp - 1) p.ranges[Pp] = T;
}

// Warp 0 of one CTA of the combine, after a partial launch of P CTAs: blends
// the slot rates into the weights (moving average; tables written for another
// P start over), writes the cumulative integer weights (each >= 1) for the next
// launch and advances the generation; while any slot has no weight yet the
// next launch uses uniform ranges (cumw[P] = 0).
__device__ inline void rebalance(const BalanceState& b, int P, int lane)
{
    constexpr int kPerLane = 16;  // slots per lane per pass, loaded together
    const bool fresh = !(__ldcg(b.header) == kBalanceMagic && __ldcg(b.header + 1) == static_cast<unsigned>(P));
    float mx = 0.f;
    bool all = true;
    for (int v0 = 0; v0 < P; v0 += 32 * kPerLane) {
        float r[kPerLane], w[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int v = v0 + lane + 32 * i;
            r[i] = v < P ? __ldcg(b.rate + v) : 0.f;
            w[i] = v < P && !fresh ? __ldcg(b.weight + v) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int v = v0 + lane + 32 * i;
            if (v >= P) continue;
            const bool ok = r[i] > 0.f && r[i] < 1e30f;  // a rate this launch measured (every claimed slot writes one)
            const float nw = ok ? (w[i] > 0.f ? 0.75f * w[i] + 0.25f * r[i] : r[i]) : w[i];
            b.weight[v] = nw;
            b.rate[v] = 0.f;
            mx = fmaxf(mx, nw);
            all = all && nw > 0.f;
        }
    }
    mx = warp_max(mx);
    all = __all_sync(0xffffffffu, all) && mx > 0.f;
    unsigned carry = 0;
    if (lane == 0) b.cumw[0] = 0u;
    for (int v0 = 0; v0 < P; v0 += 32) {
        const int v = v0 + lane;
        unsigned x = 0;
        if (v < P && all) x = max(1u, static_cast<unsigned>(65536.f * fminf(b.weight[v] / mx, 1.f)));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (v < P) b.cumw[v + 1] = all ? carry + x : 0u;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
        b.header[0] = kBalanceMagic;
        b.header[1] = static_cast<unsigned>(P);
        b.header[2] = __ldcg(b.header + 2) + 1u;
    }
}

// The range holding stage x: the largest v < n with start[v] <= x (start
// ascending, start[0] = 0 <= x).
__device__ __forceinline__ int range_of(const long long* start, int n, long long x)
{
    int lo = 0, hi = n;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

}  // namespace uaa
