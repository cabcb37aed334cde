// partial_simt.cu -- split-K decode partial on CUDA cores, for fp32 caches.
//
// One CTA per (split, kv head x head group, sequence), four warps. The query
// rows of the CTA's heads (at most 8) sit in registers, D/32 values per lane.
// Warps take the split's keys round-robin; per key the lanes hold D/32 elements
// of the key and value rows, the per-head dot products are reduced across the
// warp, and each warp keeps an online softmax (running max, sum, output row)
// per head in the log2 domain. The four warp states are merged in shared
// memory and written as a normalised partial row plus its log2-sum-exp.
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
    __shared__ float red_m[kSimtWarps][kSimtHeads];
    __shared__ float red_l[kSimtWarps][kSimtHeads];
    __shared__ float red_o[kSimtWarps][kSimtHeads][D];

    const int sigma = blockIdx.x;
    const int kvh = blockIdx.y / p.head_groups, hg = blockIdx.y % p.head_groups;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h0 = kvh * p.G + hg * kSimtHeads;
    const int nh = min(kSimtHeads, p.G - hg * kSimtHeads);

    int lo, hi;
    key_range(p.seq_lens[b], p.window, lo, hi);
    if (hi > p.cap) {  // a length past the cache: never read beyond it
        hi = p.cap;
        if (threadIdx.x == 0 && sigma == 0) atomicOr(p.status, UAA_DEVFLAG_CAPACITY);
    }
    const int t0 = lo / kTileKeys, t1 = (hi + kTileKeys - 1) / kTileKeys;
    const int tb = t0 + sigma * p.chunk_tiles;
    if (hi <= lo || tb >= t1) return;
    const int te = min(tb + p.chunk_tiles, t1);
    const int j_beg = max(lo, tb * kTileKeys), j_end = min(hi, te * kTileKeys);

    float q[kSimtHeads][EPL];
#pragma unroll
    for (int h = 0; h < kSimtHeads; ++h)
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            q[h][i] = h < nh ? p.q_prime[(static_cast<size_t>(b) * p.Hq + h0 + h) * D + lane + 32 * i] : 0.f;

    float m[kSimtHeads], l[kSimtHeads], o[kSimtHeads][EPL];
#pragma unroll
    for (int h = 0; h < kSimtHeads; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[h][i] = 0.f;
    }

    const size_t rows0 = (static_cast<size_t>(b) * p.Hkv + kvh) * p.cap;
    const float* K = static_cast<const float*>(p.k_cache) + rows0 * D;
    const float* V = static_cast<const float*>(p.v_cache) + rows0 * D;
    for (int j = j_beg + warp; j < j_end; j += kSimtWarps) {
        float kx[EPL], vx[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            kx[i] = K[static_cast<size_t>(j) * D + lane + 32 * i];
            vx[i] = V[static_cast<size_t>(j) * D + lane + 32 * i];
        }
#pragma unroll
        for (int h = 0; h < kSimtHeads; ++h) {
            if (h >= nh) break;
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) dot = fmaf(q[h][i], kx[i], dot);
            dot = warp_sum(dot);
            const float s = p.softcap_log2e > 0.f ? tanhf(dot) * p.softcap_log2e : dot;
            const float mn = fmaxf(m[h], s);
            const float alpha = exp2f(m[h] - mn);
            const float pj = exp2f(s - mn);
            l[h] = l[h] * alpha + pj;
#pragma unroll
            for (int i = 0; i < EPL; ++i) o[h][i] = fmaf(pj, vx[i], o[h][i] * alpha);
            m[h] = mn;
        }
    }

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

    for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, red_m[w][h]);
        float L = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kSimtWarps; ++w) {
            const float f = red_m[w][h] == -INFINITY ? 0.f : exp2f(red_m[w][h] - M);
            L += red_l[w][h] * f;
            acc += red_o[w][h][d] * f;
        }
        const size_t row = (static_cast<size_t>(b) * p.Hq + h0 + h) * p.S + sigma;
        p.o_part[row * D + d] = L > 0.f ? acc / L : 0.f;
        if (d == 0) p.lse_part[row] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_partial_simt(const PartialParams& p, cudaStream_t s)
{
    const dim3 grid(p.S, p.Hkv * p.head_groups, p.B), block(kSimtWarps * 32);
    switch (p.D) {
    case 64: partial_simt_kernel<64><<<grid, block, 0, s>>>(p); break;
    case 128: partial_simt_kernel<128><<<grid, block, 0, s>>>(p); break;
    case 256: partial_simt_kernel<256><<<grid, block, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace uaa
