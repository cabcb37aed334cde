// partial_simt.cu -- split-K decode partial on CUDA cores, for fp32 caches.
//
// Persistent over the stream-K partition of internal.cuh (stages of one 64-key
// tile, units of up to 8 query heads). Four warps; the unit's query rows sit in
// registers, D/32 values per lane. Warps take blocks of 16/(D/32) consecutive keys
// round-robin and load a block's rows before using any (a key at a time would
// pay one memory round trip per key); per key the lanes hold D/32 elements of
// the key and value rows, the per-head
// dot products are reduced across the warp, and each warp keeps an online
// softmax (running max, sum, output row) per head in the log2 domain. The four
// warp states are merged in shared memory: a whole unit writes its output rows
// (sink in the denominator), a cut unit writes a record for the combine.
//
// fp32 caches are exact storage; this kernel keeps the arithmetic in fp32
// (the tensor-core kernel serves bf16 and vq8 caches).
#include "internal.cuh"

namespace uaa {
namespace {

constexpr int kSimtWarps = 4;
constexpr int kSimtHeads = 8;

template <int D>
__global__ void __launch_bounds__(kSimtWarps * 32) partial_simt_kernel(const PartialParams p)
{
    constexpr int EPL = D / 32;
    constexpr int KB = 16 / EPL;  // keys per load block: 32 row registers per lane
    __shared__ float red_m[kSimtWarps][kSimtHeads];
    __shared__ float red_l[kSimtWarps][kSimtHeads];
    __shared__ float red_o[kSimtWarps][kSimtHeads][D];
    __shared__ int prefix[kMaxSliceBatch + 1];
    __shared__ int lens[kMaxSliceBatch];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.Hkv * p.head_groups;
    grid_dependency_wait();  // the append's lengths, q rows and cache rows are complete
    build_stage_prefix(p.seq_lens, p.B, p.window, p.cap, 1, units, prefix, lens,
                       blockIdx.x == 0 ? p.prefix : nullptr, blockIdx.x == 0 ? p.status : nullptr, false, 0,
                       blockIdx.x == 0 ? p.owners : nullptr);
    const long long T = prefix[p.B];
    const int P = T < gridDim.x ? static_cast<int>(T) : static_cast<int>(gridDim.x);  // every range non-empty
    const long long s_c = static_cast<int>(blockIdx.x) < P ? range_start(blockIdx.x, T, P) : 0;
    const long long e_c = static_cast<int>(blockIdx.x) < P ? range_start(blockIdx.x + 1, T, P) : 0;
    if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < P) {  // uniform ranges: slot = CTA index
        p.ranges[blockIdx.x] = s_c;
        if (static_cast<int>(blockIdx.x) == P - 1) p.ranges[P] = T;
    }

    for (long long pos = s_c; pos < e_c;) {
        const Segment sg = segment_at(prefix, lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c);
        const int r0 = sg.hg * kSimtHeads;                   // the unit's first query row (query_row)
        const int nh = min(kSimtHeads, p.q_len * p.G - r0);  // its query rows
        // several tokens per sequence: row r (token r / G) sees keys up to its own
        // position, lens[b] - q_len + r / G, and with a window the last attn_window
        int kmax[kSimtHeads], kmin[kSimtHeads];
#pragma unroll
        for (int h = 0; h < kSimtHeads; ++h) {
            kmax[h] = lens[sg.b] - p.q_len + min(r0 + h, p.q_len * p.G - 1) / p.G;
            kmin[h] = p.attn_window > 0 ? kmax[h] - p.attn_window + 1 : 0;
        }
        if (threadIdx.x == 0) {  // this range's part in the unit's owners, for the combine
            unsigned* own = p.owners + 2 * (static_cast<size_t>(sg.b) * units + sg.kvh * p.head_groups + sg.hg);
            if (sg.st0 == 0) own[0] = (blockIdx.x + 1u) | (pos == s_c ? 0x80000000u : 0u);
            if (sg.st0 + sg.n_st == sg.stages) own[1] = blockIdx.x + 1u;
        }
        const int t0 = sg.lo / kTileKeys;
        const int j_beg = max(sg.lo, (t0 + sg.st0) * kTileKeys);
        const int j_end = min(sg.hi, (t0 + sg.st0 + sg.n_st) * kTileKeys);

        float q[kSimtHeads][EPL];
#pragma unroll
        for (int h = 0; h < kSimtHeads; ++h)
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                q[h][i] = h < nh ? p.q_prime[query_row(sg.b, r0 + h, sg.kvh, p.G, p.Hq, p.q_len) * D + lane + 32 * i]
                                 : 0.f;

        float m[kSimtHeads], l[kSimtHeads], o[kSimtHeads][EPL];
#pragma unroll
        for (int h = 0; h < kSimtHeads; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) o[h][i] = 0.f;
        }

        const float* K = static_cast<const float*>(p.k_cache);
        const float* V = static_cast<const float*>(p.v_cache);
        // warp w takes blocks of KB consecutive keys round-robin; a block's rows are
        // all loaded before the first is used (one memory round trip per block)
        for (int jb = j_beg + warp * KB; jb < j_end; jb += kSimtWarps * KB) {
            float kx[KB][EPL], vx[KB][EPL];
#pragma unroll
            for (int u = 0; u < KB; ++u) {
                // the key's cache row (paged: through the block table; -1 reads as zeros)
                const long long row =
                    jb + u < j_end ? cache_row(p.pages, p.Hkv, p.cap, p.b_off + sg.b, sg.kvh, jb + u) : -1;
                if (jb + u < j_end && row < 0 && lane == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    kx[u][i] = row >= 0 ? K[static_cast<size_t>(row) * D + lane + 32 * i] : 0.f;
                    vx[u][i] = row >= 0 ? V[static_cast<size_t>(row) * D + lane + 32 * i] : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < KB; ++u) {
                if (jb + u >= j_end) break;
#pragma unroll
                for (int h = 0; h < kSimtHeads; ++h) {
                    if (h >= nh) break;
                    if (jb + u > kmax[h] || jb + u < kmin[h]) continue;  // beyond the row's own token
                    float dot = 0.f;
#pragma unroll
                    for (int i = 0; i < EPL; ++i) dot = fmaf(q[h][i], kx[u][i], dot);
                    dot = warp_sum(dot);
                    const float sc = p.softcap_log2e > 0.f ? tanhf(dot) * p.softcap_log2e : dot;
                    const float mn = fmaxf(m[h], sc);
                    const float alpha = exp2f(m[h] - mn);
                    const float pj = exp2f(sc - mn);
                    l[h] = l[h] * alpha + pj;
#pragma unroll
                    for (int i = 0; i < EPL; ++i) o[h][i] = fmaf(pj, vx[u][i], o[h][i] * alpha);
                    m[h] = mn;
                }
            }
        }

        __syncthreads();  // the previous segment's merge reads are done
#pragma unroll
        for (int h = 0; h < kSimtHeads; ++h) {
            if (lane == 0) {
                red_m[warp][h] = m[h];
                red_l[warp][h] = l[h];
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) red_o[warp][h][lane + 32 * i] = o[h][i];
        }
        __syncthreads();

        const size_t rec = 2 * static_cast<size_t>(blockIdx.x) + (pos == s_c ? 0 : 1);
        for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
            const int h = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, red_m[w][h]);
            const int hq = sg.kvh * p.G + (r0 + h) % p.G;  // the row's query head
            const float zs = (sg.whole && p.sink) ? p.sink[hq] * kLog2e : -INFINITY;
            if (sg.whole) M = fmaxf(M, zs);
            float L = 0.f, acc = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kSimtWarps; ++w) {
                    const float f = red_m[w][h] == -INFINITY ? 0.f : exp2f(red_m[w][h] - M);
                    L += red_l[w][h] * f;
                    acc += red_o[w][h][d] * f;
                }
            }
            if (sg.whole) {
                const float den = L + (zs == -INFINITY ? 0.f : exp2f(zs - M));
                const float v = den > 0.f ? acc / den : 0.f;
                const size_t oi = query_row(sg.b, r0 + h, sg.kvh, p.G, p.Hq, p.q_len) * D + d;
                if (p.out_dtype == UAA_DTYPE_F32)
                    static_cast<float*>(p.out)[oi] = v;
                else
                    static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(v);
            } else {
                p.rec_o[(rec * kSimtHeads + h) * D + d] = L > 0.f ? acc / L : 0.f;
                if (d == 0) p.rec_lse[rec * kSimtHeads + h] = L > 0.f ? M + log2f(L) : -INFINITY;
            }
        }
        pos += sg.n_st;
    }
}

}  // namespace

cudaError_t launch_partial_simt(const PartialParams& p, int n_ctas, cudaStream_t s)
{
    const dim3 grid(n_ctas), block(kSimtWarps * 32);
    switch (p.D) {
    case 64: return launch_dependent(partial_simt_kernel<64>, grid, block, 0, s, p);
    case 128: return launch_dependent(partial_simt_kernel<128>, grid, block, 0, s, p);
    case 256: return launch_dependent(partial_simt_kernel<256>, grid, block, 0, s, p);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
