// step_f32.cu -- the whole decode step in one launch for fp32 caches and one
// token per sequence (uaa_decode_attn's path for the small fp32 steps, whose
// cache sits in L2 and whose three-kernel step is launch-bound).
//
// One CTA (256 threads) per (sequence b, kv head, group of up to 8 query heads,
// key split s): the split count S comes from the length hint, split_keys keys
// each, the last split taking every key that remains, so the keys are covered
// whatever the hint. Each CTA
//   1. reads L = seq_lens[b] and counts in on the grid's arrival counter (the
//      last CTA to count in advances every length that fitted; thread 0 does it
//      while the chunk's rows are being copied);
//   2. forms the q' rows of its heads (RMSNorm, rotation at position L, logit
//      prescale) and, when its keys include the new one (slot L), the new k row
//      (RMSNorm, rotation) and v row, stored into the cache by the head group 0
//      CTA of that split;
//   3. over its keys in chunks (320 keys at head_dim 64, 160 at 128, 80 at 256):
//      the chunk's key and value rows are staged in shared memory by coalesced
//      16-byte asynchronous copies (one round trip); the scores take a warp per
//      eight keys, each lane holding its D/32 dims of every q' row in registers,
//      and sum the lanes' partial dot products with a transposing butterfly
//      (each shuffle step halves the values a lane holds, so 8 keys x NH heads
//      take 8 NH - 2 shuffles); softmax statistics per head (a warp per head);
//      P.V with a thread per four value columns and a group of keys, rescaled
//      across chunks;
//   4. with one split: out = o / (l + sink term); otherwise it writes its record
//      (normalised rows, log2-sum-exp) and the last split of the unit to finish
//      (a per-unit counter, zero between launches) merges the S records in
//      order, the sink in the denominator (llamay "Models and formats",
//      "Architectures"), and writes the output rows.
// The arithmetic is fp32 throughout, like the CUDA-core partial kernel.
#include "internal.cuh"
#include "ptx.cuh"

namespace uaa {
namespace {

constexpr int kStepThreads = 256;
constexpr int kStepWarps = kStepThreads / 32;

// keys of one chunk, whose key and value rows are staged in shared memory
template <int D>
__host__ __device__ constexpr int chunk_keys() { return 20480 / D; }
template <int D>
__host__ __device__ constexpr int ks_stride() { return D + 4; }  // floats per staged row (16 bytes apart in the banks)
template <int D>
constexpr size_t step_dyn_smem() { return 2 * static_cast<size_t>(chunk_keys<D>()) * ks_stride<D>() * 4; }

// One step of the transposing butterfly over the lanes: of the N values a lane
// holds, the half selected by its bit M is kept and summed with the partner's
// (lane ^ M) same half; the other half is sent to the partner.
template <int N, int M>
__device__ __forceinline__ void butterfly_step(float* v, int lane)
{
    const bool up = (lane & M) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
    }
}

// The sums over the 32 lanes of N values (N = 32 or 64): afterwards lane l holds
// the sums of values N/32 l .. N/32 l + N/32 - 1 in v[0 ..].
template <int N>
__device__ __forceinline__ void lane_sums(float (&v)[N], int lane)
{
    static_assert(N == 32 || N == 64, "8 keys x 4 or 8 heads");
    butterfly_step<N, 16>(v, lane);
    butterfly_step<N / 2, 8>(v, lane);
    butterfly_step<N / 4, 4>(v, lane);
    butterfly_step<N / 8, 2>(v, lane);
    butterfly_step<N / 16, 1>(v, lane);
}

template <int D, int NH, typename T>  // NH: query heads per unit (4 or 8); T: io element type
__global__ void __launch_bounds__(kStepThreads) step_f32_kernel(const StepF32Params p)
{
    constexpr int EPL = D / 32;            // row elements per lane
    constexpr int C4 = D / 4;              // float4 columns of a row
    constexpr int KG = kStepThreads / C4;  // key groups of the P.V phase
    constexpr int CK = chunk_keys<D>();
    constexpr int KSTR = ks_stride<D>();
    constexpr int NV = 8 * NH;             // scores of one warp step: 8 keys x NH heads
    static_assert(KG * NH * D >= NH * CK, "the shared buffer holds the scores and the P.V sums");
    __shared__ __align__(16) float qs[NH][D];  // q' rows of the unit's heads
    __shared__ __align__(16) float kn[D];      // the new key row (rotated)
    __shared__ __align__(16) float vn[D];      // the new value row
    __shared__ float2 cs[D / 2];
    __shared__ __align__(16) float buf[KG * NH * D];  // weights [NH][CK], then P.V sums [KG][NH][D]
    __shared__ float m_run[NH], l_run[NH], fac[NH];
    __shared__ bool last;
    extern __shared__ __align__(16) float stage[];  // the chunk's key rows [CK][KSTR], then value rows
    float* ks = stage;
    float* vs = stage + CK * KSTR;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = p.Hkv * p.head_groups;
    const int S = p.splits;
    const int s = blockIdx.x % S;
    const int ug = blockIdx.x / S;  // global unit: b * units + u
    const int b = ug / units, u = ug - b * units;
    const int kvh = u / p.head_groups, hg = u - kvh * p.head_groups;
    const int h0 = kvh * p.G + hg * 8;            // the unit's first query head
    const int nh = min(NH, p.G - hg * 8);         // its heads

    grid_dependency_wait();  // the step's inputs and the previous step's writes are complete
    // the next kernel of the stream (launched as dependent) may take the other SMs and
    // do its set-up now; its own grid_dependency_wait still waits for this grid
    allow_dependent_launch();

    // ---- the length and the keys of this split
    const int L = p.seq_lens[b];  // read by every thread before the CTA counts in (below)
    const bool fits = L >= 0 && L < p.cap;
    int lo, hi;
    visible_keys(fits ? L + 1 : L, p.window, p.cap, lo, hi);
    const int k0 = min(hi, lo + s * p.split_keys);
    const int k1 = s == S - 1 ? hi : min(hi, lo + (s + 1) * p.split_keys);
    const bool has_new = fits && k0 <= L && L < k1;  // the new key is among this split's keys

    // the rows this CTA needs, loaded before anything waits on them
    float x[EPL];
    const bool row_q = warp < nh;
    if (row_q) {
        const size_t at = (static_cast<size_t>(b) * p.Hq + h0 + warp) * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = load_as_float<T>(p.q, at + lane + 32 * i);
    }
    float kx[EPL], vx[EPL];
    if (has_new && warp == kStepWarps - 1) {
        const size_t at = (static_cast<size_t>(b) * p.Hkv + kvh) * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            kx[i] = load_as_float<T>(p.k_new, at + lane + 32 * i);
            vx[i] = load_as_float<T>(p.v_new, at + lane + 32 * i);
        }
    }
    // ---- (cos, sin) of position L, then the q' rows and the new rows
    {
        const int pos = fits ? L : 0;
#pragma unroll
        for (int i0 = 0; i0 < D / 2; i0 += 32)  // warp w takes pairs 32 w .. 32 w + 31
            if (warp == i0 / 32)
                cs[i0 + lane] = rope_pair_cos_sin(i0 + lane, p.half_rot, pos,
                                                  param_at_lane(p.inv_freq_over_pi + i0, lane), p.mscale);
    }
    auto norm_row = [&](float(&r)[EPL], const float* w) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) ss += r[i] * r[i];
        const float inv = rms_inv(warp_sum(ss), D, p.eps);
#pragma unroll
        for (int i = 0; i < EPL; ++i) r[i] = r[i] * inv * (w[lane + 32 * i] + p.norm_offset);
    };
    if (row_q) {
        if (p.qk_norm) norm_row(x, p.q_norm_w);
#pragma unroll
        for (int i = 0; i < EPL; ++i) qs[warp][lane + 32 * i] = x[i];
    } else if (warp < NH) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) qs[warp][lane + 32 * i] = 0.f;  // a missing head scores nothing
    }
    if (has_new && warp == kStepWarps - 1) {
        if (p.qk_norm) norm_row(kx, p.k_norm_w);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            kn[lane + 32 * i] = kx[i];
            vn[lane + 32 * i] = vx[i];
        }
    }
    __syncthreads();  // (cos, sin), the normalised rows; every thread has read its length
    // Thread 0 counts the CTA in; the last CTA of the grid to do so advances every
    // length that fitted.
    auto count_in = [&]() {
        if (u == 0 && s == 0) {
            if (!fits) atomicOr(p.status, UAA_DEVFLAG_CAPACITY);
            else if (L > p.max_len) atomicOr(p.status, UAA_DEVFLAG_LEN_HINT);
        }
        __threadfence();
        if (atomicInc(p.arrivals, gridDim.x - 1) == gridDim.x - 1) {
            __threadfence();
            for (int i = 0; i < p.B; ++i) {
                const int n = p.seq_lens[i];
                if (n >= 0 && n < p.cap) p.seq_lens[i] = n + 1;
            }
        }
    };
    const bool neox = p.style == UAA_ROPE_NEOX;
    for (int idx = tid; idx < (nh + (has_new ? 1 : 0)) * (D / 2); idx += kStepThreads) {
        const int r = idx / (D / 2), pp = idx - r * (D / 2);
        const int2 e = rope_pair(pp, p.half_rot, D, neox);
        float* row = r < nh ? qs[r] : kn;
        float ya = row[e.x], yb = row[e.y];
        rope_rotate(ya, yb, cs[pp]);
        if (r < nh) {
            if (p.q_rot_out && s == 0) {
                const size_t at = (static_cast<size_t>(b) * p.Hq + h0 + r) * D;
                p.q_rot_out[at + e.x] = ya;
                p.q_rot_out[at + e.y] = yb;
            }
            ya *= p.qscale;
            yb *= p.qscale;
        }
        row[e.x] = ya;
        row[e.y] = yb;
    }
    __syncthreads();  // q' rows and the rotated new key
    if (has_new && hg == 0) {  // the new rows into the cache, once per kv head
        const long long crow = cache_row(p.pages, p.Hkv, p.cap, b, kvh, L);
        if (crow < 0) {
            if (tid == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
        } else {
            for (int i = tid; i < D; i += kStepThreads) {
                p.k_cache[static_cast<size_t>(crow) * D + i] = kn[i];
                p.v_cache[static_cast<size_t>(crow) * D + i] = vn[i];
            }
        }
    }
    // this lane's dims of every q' row, for the whole split
    float qr[NH][EPL];
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) qr[h][e] = qs[h][lane + 32 * e];

    // ---- chunks: staged rows, scores, softmax statistics and P.V
    if (tid < NH) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
    }
    const int c = tid % C4, g = tid / C4;  // P.V: float4 column c, key group g
    float o[NH][4];
#pragma unroll
    for (int h = 0; h < NH; ++h) o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;
    const float cap2 = p.softcap_log2e;
    for (int kc = k0; kc < k1; kc += CK) {
        const int nk = min(CK, k1 - kc);  // the chunk: keys kc .. kc + nk - 1
        __syncthreads();  // the previous chunk's rows and weights are used up
        // the chunk's key and value rows into shared memory (a thread per float4 in
        // turn: coalesced 16-byte asynchronous copies); the new key's rows from its
        // staged rows; rows behind an out-of-pool page entry read as zeros
        for (int f = tid; f < nk * C4; f += kStepThreads) {
            const int jj = f / C4, c4 = f - jj * C4, j = kc + jj;
            float* kd = ks + jj * KSTR + 4 * c4;
            float* vd = vs + jj * KSTR + 4 * c4;
            if (has_new && j == L) {
                *reinterpret_cast<float4*>(kd) = reinterpret_cast<const float4*>(kn)[c4];
                *reinterpret_cast<float4*>(vd) = reinterpret_cast<const float4*>(vn)[c4];
            } else {
                const long long row = cache_row(p.pages, p.Hkv, p.cap, b, kvh, j);
                if (row < 0) {
                    if (c4 == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
                    *reinterpret_cast<float4*>(kd) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4*>(vd) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    const size_t at = static_cast<size_t>(row) * D + 4 * c4;
                    ptx::cp_async_16(static_cast<uint32_t>(__cvta_generic_to_shared(kd)), p.k_cache + at);
                    ptx::cp_async_16(static_cast<uint32_t>(__cvta_generic_to_shared(vd)), p.v_cache + at);
                }
            }
        }
        ptx::cp_async_commit();
        if (tid == 0 && kc == k0) count_in();  // while the copies land
        ptx::cp_async_wait_all();
        __syncthreads();  // the chunk's rows

        // scores: a warp per 8 keys; lane partial dot products over its dims, summed
        // over the lanes by the butterfly (lane l ends with scores NV/32 l ..)
        for (int j0 = 8 * warp; j0 < nk; j0 += 8 * kStepWarps) {
            float v[NV];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float kr[EPL];
#pragma unroll
                for (int e = 0; e < EPL; ++e) kr[e] = j0 + r < nk ? ks[(j0 + r) * KSTR + lane + 32 * e] : 0.f;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(qr[h][e], kr[e], acc);
                    v[r * NH + h] = acc;
                }
            }
            lane_sums<NV>(v, lane);
#pragma unroll
            for (int t = 0; t < NV / 32; ++t) {
                const int idx = (NV / 32) * lane + t, r = idx / NH, h = idx - r * NH, jj = j0 + r;
                if (jj < nk) {
                    float sc = v[t];
                    if (cap2 > 0.f) sc = tanhf(sc) * cap2;
                    buf[h * CK + jj] = h < nh ? sc : -INFINITY;
                }
            }
        }
        __syncthreads();  // every score of the chunk
        if (warp < NH) {  // warp h: the chunk's maximum and weights of head h
            float* sh = buf + warp * CK;
            float mx = -INFINITY;
            for (int jj = lane; jj < nk; jj += 32) mx = fmaxf(mx, sh[jj]);
            mx = warp_max(mx);
            const float mo = m_run[warp];
            const float mn = fmaxf(mo, mx);
            const float mu = mn == -INFINITY ? 0.f : mn;
            float sum = 0.f;
            for (int jj = lane; jj < nk; jj += 32) {
                const float w = exp2f(sh[jj] - mu);
                sh[jj] = w;
                sum += w;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float f = mo == -INFINITY ? 0.f : exp2f(mo - mu);
                fac[warp] = f;
                l_run[warp] = l_run[warp] * f + sum;
                m_run[warp] = mn;
            }
        }
        __syncthreads();  // the weights and the rescale factors
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const float f = fac[h];
            o[h][0] *= f;
            o[h][1] *= f;
            o[h][2] *= f;
            o[h][3] *= f;
        }
        // P.V: a thread per float4 column and key group, rows and weights from shared memory
        for (int jj = g; jj < nk; jj += KG) {
            const float4 vv = *reinterpret_cast<const float4*>(vs + jj * KSTR + 4 * c);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float w = buf[h * CK + jj];
                o[h][0] = fmaf(w, vv.x, o[h][0]);
                o[h][1] = fmaf(w, vv.y, o[h][1]);
                o[h][2] = fmaf(w, vv.z, o[h][2]);
                o[h][3] = fmaf(w, vv.w, o[h][3]);
            }
        }
    }
    if (tid == 0 && k0 >= k1) count_in();  // a split without keys
    __syncthreads();  // the last chunk's weights are used up: the buffer takes the P.V sums
#pragma unroll
    for (int h = 0; h < NH; ++h)
        reinterpret_cast<float4*>(buf + (g * NH + h) * D)[c] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    __syncthreads();

    // ---- this split's rows (summed over the key groups): the output, or a record
    constexpr int HR = 8;  // record rows per unit (the workspace's records hold 8 heads)
    const size_t rec = static_cast<size_t>(ug) * S + s;
    for (int idx = tid; idx < nh * D; idx += kStepThreads) {
        const int h = idx / D, d = idx - h * D;
        float acc = 0.f;
#pragma unroll
        for (int gg = 0; gg < KG; ++gg) acc += buf[(gg * NH + h) * D + d];
        const float M = m_run[h], Ls = l_run[h];
        if (S == 1) {
            const float z = p.sink ? p.sink[h0 + h] * kLog2e : -INFINITY;
            const float Mx = fmaxf(M, z);
            float val = 0.f;
            if (Mx != -INFINITY) {
                const float fm = M == -INFINITY ? 0.f : exp2f(M - Mx);
                const float den = Ls * fm + (z == -INFINITY ? 0.f : exp2f(z - Mx));
                val = den > 0.f ? acc * fm / den : 0.f;
            }
            store_out(p.out, p.out_dtype, (static_cast<size_t>(b) * p.Hq + h0 + h) * D + d, val);
        } else {
            p.rec_o[(rec * HR + h) * D + d] = Ls > 0.f ? acc / Ls : 0.f;
            if (d == 0) p.rec_lse[rec * HR + h] = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
        }
    }
    if (S == 1) return;

    // ---- the last split of the unit to finish merges the unit's records in order
    __threadfence();  // this thread's record rows, before the CTA counts in
    __syncthreads();
    if (tid == 0) {
        unsigned* cnt = p.unit_count + 2 * static_cast<size_t>(ug);
        last = atomicAdd(cnt, 1u) == static_cast<unsigned>(S - 1);
        if (last) *cnt = 0u;  // ready for the next launch
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int idx = tid; idx < nh * D; idx += kStepThreads) {
        const int h = idx / D, d = idx - h * D;
        const float z = p.sink ? p.sink[h0 + h] * kLog2e : -INFINITY;
        float M = z;
        for (int ss = 0; ss < S; ++ss) M = fmaxf(M, __ldcg(p.rec_lse + (static_cast<size_t>(ug) * S + ss) * HR + h));
        float den = 0.f, acc = 0.f;
        if (M != -INFINITY) {
            den = z == -INFINITY ? 0.f : exp2f(z - M);
            for (int ss = 0; ss < S; ++ss) {
                const size_t r = static_cast<size_t>(ug) * S + ss;
                const float e = __ldcg(p.rec_lse + r * HR + h);
                const float w = e == -INFINITY ? 0.f : exp2f(e - M);
                den += w;
                acc = fmaf(w, __ldcg(p.rec_o + (r * HR + h) * D + d), acc);
            }
        }
        store_out(p.out, p.out_dtype, (static_cast<size_t>(b) * p.Hq + h0 + h) * D + d, den > 0.f ? acc / den : 0.f);
    }
}

template <int D, int NH, typename T>
cudaError_t launch_step(const StepF32Params& p, dim3 grid, cudaStream_t s)
{
    auto kern = step_f32_kernel<D, NH, T>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(step_dyn_smem<D>()));
        if (e != cudaSuccess) return e;
        if (dev < 31) configured_device_mask |= 1 << dev;
    }
    return launch_dependent(kern, grid, dim3(kStepThreads), step_dyn_smem<D>(), s, p);
}

template <int D, typename T>
cudaError_t launch_heads(const StepF32Params& p, dim3 grid, cudaStream_t s)
{
    // four query heads per kv head or fewer: every unit has at most 4 heads
    return p.G <= 4 ? launch_step<D, 4, T>(p, grid, s) : launch_step<D, 8, T>(p, grid, s);
}

}  // namespace

cudaError_t launch_step_f32(const StepF32Params& p, cudaStream_t s)
{
    const long long ctas = static_cast<long long>(p.B) * p.Hkv * p.head_groups * p.splits;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 2147483647LL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(ctas));
    const bool f32 = p.io_dtype == UAA_DTYPE_F32;
    switch (p.D) {
    case 64: return f32 ? launch_heads<64, float>(p, grid, s) : launch_heads<64, __nv_bfloat16>(p, grid, s);
    case 128: return f32 ? launch_heads<128, float>(p, grid, s) : launch_heads<128, __nv_bfloat16>(p, grid, s);
    case 256: return f32 ? launch_heads<256, float>(p, grid, s) : launch_heads<256, __nv_bfloat16>(p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
