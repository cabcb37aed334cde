// combine.cu -- step 3 of the decode step: log-sum-exp merge of the records of
// units that the stream-K partition cut between CTAs, with the per-head sink.
//
// One CTA per unit (sequence, kv head, group of (token, head) query rows: the
// query heads of the kv head for a decode step). A unit that lies inside one
// CTA's range was written by the partial kernel already and is skipped. For a
// cut unit with records (o_c normalised, e_c the log2-sum-exp of the final
// logits) from its owner CTAs, and the sink logit z_h of each head (llamay
// "Models and formats", "Architectures": a per-head sink in the softmax
// denominator):
//   M   = max(max_c e_c, z_h log2 e)
//   out = sum_c o_c 2^(e_c - M) / (sum_c 2^(e_c - M) + 2^(z_h log2 e - M))
// which is the full softmax over every visible key with the sink's mass in the
// denominator only. A sequence with no visible key gets zeros.
//
// Every range is non-empty, so the owners of a cut unit's stages are exactly the
// ranges cA .. cB, which the partial kernel leaves per unit (UnitOwners in
// internal.cuh). The record weights are formed per
// head from one parallel round of loads; every thread then loads all records'
// rows for four output elements before it adds any of them. The CTA has a
// thread per four output elements of a unit (128 to 512 threads), so a unit of
// up to 16 rows of 128 dims is merged in one round of loads: the merge is a
// chain of dependent loads, not a stream of bytes.
#include "internal.cuh"

namespace uaa {
namespace {

constexpr int kCombineMinThreads = 128;
constexpr int kCombineMaxThreads = 512;
constexpr int kMaxHeads = 16;    // heads of one unit
constexpr int kRecBatch = 4;     // records loaded together per output element

__global__ void __launch_bounds__(kCombineMaxThreads) combine_kernel(const CombineParams p)
{
    extern __shared__ float wts[];  // [R][nh]: record log2-sum-exp, then weights
    grid_dependency_wait();         // the partial kernel's records are complete
    allow_dependent_launch();
    if (blockIdx.x == gridDim.x - 1) {     // the extra CTA: the partial kernel's range balance
        if (p.bal.header && threadIdx.x < 32) rebalance(p.bal, p.P, threadIdx.x);
        return;
    }

    const int units = p.Hkv * p.head_groups;
    const int b = blockIdx.x / units, u = blockIdx.x - b * units;
    const int kvh = u / p.head_groups, hg = u - kvh * p.head_groups;
    const int HC = p.heads_per_cta;
    const int r0 = hg * HC;                      // the unit's first query row (query_row)
    const int nh = min(HC, p.q_len * p.G - r0);  // its query rows
    const int D = p.D;
    const int tid = threadIdx.x, nthr = blockDim.x;
    // output element idx (row idx / D, column idx % D) of the unit
    auto out_at = [&](int idx) {
        const int hc = idx / D;
        return query_row(b, r0 + hc, kvh, p.G, p.Hq, p.q_len) * D + (idx - hc * D);
    };
    // the unit's first and last owner, left by the partial kernel (cleared for the next launch)
    unsigned* own = p.owners + 2 * static_cast<size_t>(blockIdx.x);
    const unsigned first = own[0], last = own[1];
    __syncthreads();  // every thread has read the pair
    if (tid == 0) {
        own[0] = 0u;
        own[1] = 0u;
    }
    if (first == 0u || last == 0u) {  // no visible key: zeros
        for (int idx = tid; idx < nh * D; idx += nthr) store_out(p.out, p.out_dtype, out_at(idx), 0.f);
        return;
    }
    const int cA = static_cast<int>(first & 0x7fffffffu) - 1, cB = static_cast<int>(last) - 1;
    if (cA == cB) return;  // a whole unit: the partial kernel wrote it
    if (cA < 0 || cB < cA || cB >= p.P) {  // owner words no range of this launch wrote: not read further
        if (tid == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
        return;
    }
    const bool first_is_slot0 = (first & 0x80000000u) != 0u;
    const int R = cB - cA + 1;  // the unit's records: owners cA .. cB

    for (int i = tid; i < R * nh; i += nthr)
        wts[i] = p.rec_lse[static_cast<size_t>(record_of(cA + i / nh, cA, first_is_slot0)) * HC + (i % nh)];
    __syncthreads();
    for (int hc = tid; hc < nh; hc += nthr) {
        const float z = p.sink ? p.sink[kvh * p.G + (r0 + hc) % p.G] * kLog2e : -INFINITY;
        float M = z;
        for (int r = 0; r < R; ++r) M = fmaxf(M, wts[r * nh + hc]);
        float den = 0.f;
        if (M != -INFINITY) {
            den = p.sink ? exp2f(z - M) : 0.f;
            for (int r = 0; r < R; ++r) {
                const float e = wts[r * nh + hc];
                const float w = e == -INFINITY ? 0.f : exp2f(e - M);
                wts[r * nh + hc] = w;
                den += w;
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        for (int r = 0; r < R; ++r) wts[r * nh + hc] = M == -INFINITY ? 0.f : wts[r * nh + hc] * inv;
    }
    __syncthreads();
    for (int base = tid; base < nh * D; base += 4 * nthr) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r0 = 0; r0 < R; r0 += kRecBatch) {
            float v[kRecBatch][4];
#pragma unroll
            for (int r = 0; r < kRecBatch; ++r)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int idx = base + k * nthr;
                    v[r][k] = 0.f;
                    if (r0 + r < R && idx < nh * D) {
                        const int hc = idx / D, d = idx - hc * D;
                        const int rec = record_of(cA + r0 + r, cA, first_is_slot0);
                        v[r][k] = p.rec_o[(static_cast<size_t>(rec) * HC + hc) * D + d];
                    }
                }
#pragma unroll
            for (int r = 0; r < kRecBatch; ++r)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int idx = base + k * nthr;
                    if (r0 + r < R && idx < nh * D) acc[k] = fmaf(wts[(r0 + r) * nh + idx / D], v[r][k], acc[k]);
                }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int idx = base + k * nthr;
            if (idx < nh * D) store_out(p.out, p.out_dtype, out_at(idx), acc[k]);
        }
    }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s)
{
    // one CTA per unit, and one that rebalances the partial kernel's ranges; a
    // thread per four output elements of a unit's rows, in whole warps
    const long long blocks = static_cast<long long>(p.B) * p.Hkv * p.head_groups + 1;
    if (blocks == 1) return cudaSuccess;
    const int rows = p.heads_per_cta < p.q_len * p.G ? p.heads_per_cta : p.q_len * p.G;
    int threads = (rows * p.D / 4 + 31) / 32 * 32;
    threads = threads < kCombineMinThreads ? kCombineMinThreads : (threads > kCombineMaxThreads ? kCombineMaxThreads : threads);
    // weights for up to every range's record of a unit
    const size_t smem = static_cast<size_t>(p.P) * (p.heads_per_cta < kMaxHeads ? p.heads_per_cta : kMaxHeads) * 4;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), smem, s, p);
}

}  // namespace uaa
