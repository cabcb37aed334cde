// combine.cu -- step 3 of the decode step: log-sum-exp merge of the split-K
// partials and the per-head sink logit.
//
// One thread per output element (b, h, d). With partial rows o_s (normalised)
// and their log2-sum-exp e_s (of the final logits, in log2 units), and the sink
// logit z_h of the head (llamay "Models and formats", "Architectures": a
// per-head sink in the softmax denominator):
//   M   = max(max_s e_s, z_h log2 e)
//   out = sum_s o_s 2^(e_s - M) / (sum_s 2^(e_s - M) + 2^(z_h log2 e - M))
// which is the full softmax over every visible key with the sink's mass in the
// denominator only. A sequence with no visible key and no sink gets zeros.
#include "internal.cuh"

namespace uaa {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p)
{
    const size_t total = static_cast<size_t>(p.B) * p.Hq * p.D;
    for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int d = static_cast<int>(idx % p.D);
        const int h = static_cast<int>((idx / p.D) % p.Hq);
        const int b = static_cast<int>(idx / (static_cast<size_t>(p.D) * p.Hq));
        int lo, hi;
        key_range(p.seq_lens[b], p.window, lo, hi);
        const int ns = splits_needed(lo, hi, p.chunk_tiles);
        float result;
        if (ns > p.S) {  // the max_seq_len bound was broken: not enough split slots
            if (d == 0 && h == 0) atomicOr(p.status, UAA_DEVFLAG_LEN_HINT);
            result = __int_as_float(0x7fc00000);
        } else {
            const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.S;
            const float z = p.sink ? p.sink[h] * kLog2e : -INFINITY;
            float M = z;
            for (int s = 0; s < ns; ++s) M = fmaxf(M, p.lse_part[row + s]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
                den = p.sink ? exp2f(z - M) : 0.f;
                for (int s = 0; s < ns; ++s) {
                    const float e = p.lse_part[row + s];
                    const float w = e == -INFINITY ? 0.f : exp2f(e - M);
                    num = fmaf(w, p.o_part[(row + s) * p.D + d], num);
                    den += w;
                }
            }
            result = den > 0.f ? num / den : 0.f;
        }
        if (p.out_dtype == UAA_DTYPE_F32)
            static_cast<float*>(p.out)[idx] = result;
        else
            static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(result);
    }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s)
{
    const size_t total = static_cast<size_t>(p.B) * p.Hq * p.D;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 8u) blocks = 65535u * 8u;
    combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace uaa
