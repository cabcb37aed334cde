// partial_tc.cu -- split-K decode partial for bf16 and vq8 caches: a persistent,
// warp-specialised kernel with TMA tile loads into a shared-memory ring and
// tensor-core contractions.
//
// Work: the stream-K partition of internal.cuh. P = (SMs x resident CTAs) CTAs
// each take one contiguous range of ring stages across all units (sequence,
// kv head, head group); every query head of the unit's group (up to 8 * NHT) is
// served from the same K/V stage, so each key row leaves HBM once.
//
// Warp roles (160 threads):
//   warp 4 (producer): one lane walks the CTA's segments and streams their
//     stages, TK = 64 MG keys each, with 2-D TMA loads (cp.async.bulk.tensor)
//     into a ring of kStages stages, straight across segment boundaries. Key and
//     bf16 value boxes are TK rows x 128 bytes with the 128-byte swizzle; vq8
//     code boxes are TK rows x min(D, 128) bytes with the 64- or 128-byte
//     swizzle; vq8 scales are one TK-float box. Full / empty mbarriers pass
//     stages between the producer and the consumers.
//   warps 0-3 (consumers): warp w owns keys 16 MG w .. 16 MG (w+1) - 1 of every
//     stage, as MG groups of 16 keys that share one softmax round (MG = 2 for
//     head_dim 64, else 1).
//     S^T (16 keys x 8 heads) = K (16 x D) . Q'^T (D x 8) with mma.m16n8k16
//     (keys on M, heads on N: no padding of M). The fp32 q' rows are split into
//     bf16 hi + lo parts, two MMAs each, so the logits keep ~16 significant bits.
//     Online softmax (log2 domain) runs on the fp32 accumulators. P is split into
//     hi + lo parts and moved with movmatrix into the B operand of
//     O^T (D x 8) += V^T (D x 16 keys) . P^T (16 keys x 8 heads).
//       bf16 values: V^T fragments come from ldmatrix.trans on the bf16 stage.
//       vq8 values: ldmatrix.trans runs on the int8 stage itself (a b16 element
//       is then a pair of adjacent codes), one byte permute and one fp16
//       subtract per pair widen the codes exactly, and the PV product runs in
//       fp16. The per-key scale is folded into P; to keep P * scale inside
//       [0, 1] it is divided by the warp's running maximum scale r, and O is
//       kept in units of r (a new maximum rescales O as a new logit maximum does).
//   At the end of a segment the four warp states are merged through the
//   shared memory of the segment's last stage (held back from the producer
//   until the merge is done). A whole unit writes its output rows, with the
//   sink logit in the denominator; a cut unit writes a record for the combine.
//
// Every wait is bounded (kWaitLimitCycles); a wait that gives up sets
// UAA_DEVFLAG_TIMEOUT and the CTA unwinds without further waits.
#include <cuda_fp16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace uaa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// MG: 16-key groups each consumer warp takes per stage (2 for head_dim 64, where a
// key costs few bytes and the per-stage softmax work is shared by 32 keys).
template <int D>
struct KeyGroups {
    static constexpr int kMG = D == 64 ? 2 : 1;
};

template <int D, bool VQ8>
struct Shape {
    static constexpr int kMG = KeyGroups<D>::kMG;
    static constexpr int kTK = kTileKeys * kMG;             // keys per stage
    static constexpr int kBoxBytes = kTK * 128;             // kTK rows x 128 bytes
    static constexpr int kKBoxes = D / 64;                  // 128-byte column boxes of a bf16 row
    static constexpr int kVBoxes = VQ8 ? (D > 128 ? D / 128 : 1) : D / 64;
    static constexpr int kKBytes = kTK * D * 2;
    static constexpr int kVBytes = VQ8 ? kTK * D : kTK * D * 2;
    static constexpr int kSBytes = VQ8 ? kTK * 4 : 0;
    static constexpr int kStageBytes = round_up(kKBytes + kVBytes + kSBytes, 1024);
    static constexpr int kTxBytes = kKBytes + kVBytes + kSBytes;
    static constexpr int kBudget = D == 256 ? 196608 : 104448;
    static constexpr int kStagesRaw = kBudget / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kPrefixBytes = round_up((kMaxSliceBatch + 1) * 4, 16);
    static constexpr int kSmemBytes = 1024 + kRingBytes + 16 * kStages + kPrefixBytes;
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a bf16 stage: boxes of
// TK rows x 128 bytes, chunk index XOR (row mod 8) inside each 128-byte row.
template <int TK>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * (TK * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// The same for an int8 code stage of D-byte rows: D = 64 uses the 64-byte swizzle
// (chunk XOR ((row / 2) mod 4)), D = 128 and 256 the 128-byte one per 128-byte box.
template <int D, int TK>
__device__ __forceinline__ uint32_t code_off(int row, int chunk)
{
    if (D == 64) return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
    return static_cast<uint32_t>((chunk >> 3) * (TK * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// x ~= hi + lo with hi = bf16(x), lo = bf16(x - hi), for two values.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16(x0, x1);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16(x0 - h0, x1 - h1);
}

// The same split into fp16 hi + lo parts (values in [0, 1]).
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b)
{
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// A register from ldmatrix.trans on int8 rows holds codes (key k, value d),
// (k, d+1), (k+1, d), (k+1, d+1) in bytes 0-3. Returns the fp16 pairs
// [(k, d), (k+1, d)] and [(k, d+1), (k+1, d+1)], exactly: byte c + 128 goes into
// the mantissa of 1024 (fp16 0x6400) and 1152 (0x6480) is subtracted.
__device__ __forceinline__ void widen_code_pairs(uint32_t r, uint32_t& d_even, uint32_t& d_odd)
{
    const uint32_t u = r ^ 0x80808080u;
    d_even = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4240), 0x64806480u);
    d_odd = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4341), 0x64806480u);
}

__device__ __forceinline__ bool key_ok(int k, int lo, int hi) { return k >= lo && k < hi; }

template <int D, bool VQ8, int NHT>
__global__ void __launch_bounds__(kThreads, (D == 256 ? 1 : 2))
partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_s, const PartialParams p)
{
    using SH = Shape<D, VQ8>;
    constexpr int MG = SH::kMG;     // 16-key groups per warp per stage
    constexpr int TK = SH::kTK;     // keys per stage
    constexpr int KS = D / 16;      // k-steps of QK, m-tiles of PV
    constexpr int HC = 8 * NHT;     // head columns of a unit
    // merge scratch (inside one stage): all of D at once if it fits, else halves
    constexpr int RC = (kConsumerWarps * HC * (D + 4) + 2 * kConsumerWarps * HC) * 4 <= SH::kStageBytes ? D : D / 2;
    static_assert((kConsumerWarps * HC * (RC + 4) + 2 * kConsumerWarps * HC) * 4 <= SH::kStageBytes,
                  "merge scratch must fit in one stage");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bar_full = base + SH::kRingBytes;
    const uint32_t bar_empty = bar_full + 8 * SH::kStages;
    int* prefix = reinterpret_cast<int*>(base_ptr + SH::kRingBytes + 16 * SH::kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.Hkv * p.head_groups;
    if (threadIdx.x == 0) {  // shared-memory set-up overlaps the previous kernel's tail
        for (int s = 0; s < SH::kStages; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32 * kConsumerWarps) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        if (VQ8) ptx::prefetch_tensormap(&tm_s);
    }
    grid_dependency_wait();  // the append's lengths, q rows and cache rows are complete
    build_stage_prefix(p.seq_lens, p.B, p.window, p.cap, MG, units, prefix, blockIdx.x == 0 ? p.prefix : nullptr,
                       p.status);  // ends with __syncthreads
    const long long T = prefix[p.B];
    const int P = T < gridDim.x ? static_cast<int>(T) : static_cast<int>(gridDim.x);  // every range non-empty
    if (static_cast<int>(blockIdx.x) >= P) return;  // uniform over the CTA: no stages
    const long long s_c = range_start(blockIdx.x, T, P), e_c = range_start(blockIdx.x + 1, T, P);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int it = 0;  // stages issued
            for (long long pos = s_c; pos < e_c && ok;) {
                const Segment sg = segment_at(prefix, p.seq_lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c);
                const int head_row = (p.b_off + sg.b) * p.Hkv + sg.kvh;
                const int row0 = head_row * p.cap;
                const int t0 = sg.lo / kTileKeys;
                for (int k = 0; k < sg.n_st; ++k, ++it) {
                    const int s = it % SH::kStages;
                    if (it >= SH::kStages &&
                        !ptx::mbar_wait(bar_empty + 8 * s, ((it / SH::kStages) & 1) ^ 1, kWaitLimitCycles)) {
                        atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + s * SH::kStageBytes;
                    const uint32_t bar = bar_full + 8 * s;
                    ptx::mbar_arrive_expect_tx(bar, SH::kTxBytes);
                    const int key = (t0 + MG * (sg.st0 + k)) * kTileKeys;
                    const int y = row0 + key;
#pragma unroll
                    for (int c = 0; c < SH::kKBoxes; ++c)
                        ptx::tma_load_2d(st + c * SH::kBoxBytes, &tm_k, c * 64, y, bar);
                    if (VQ8) {
#pragma unroll
                        for (int c = 0; c < SH::kVBoxes; ++c)
                            ptx::tma_load_2d(st + SH::kKBytes + c * SH::kBoxBytes, &tm_v, c * 128, y, bar);
                        ptx::tma_load_2d(st + SH::kKBytes + SH::kVBytes, &tm_s, key, head_row, bar);
                    } else {
#pragma unroll
                        for (int c = 0; c < SH::kVBoxes; ++c)
                            ptx::tma_load_2d(st + SH::kKBytes + c * SH::kBoxBytes, &tm_v, c * 64, y, bar);
                    }
                }
                pos += sg.n_st;
            }
            // Copies in flight land before the CTA may exit (bounded).
            const int first = it > SH::kStages ? it - SH::kStages : 0;
            for (int i = first; i < it && ok; ++i)
                ok = ptx::mbar_wait(bar_full + 8 * (i % SH::kStages), (i / SH::kStages) & 1, kWaitLimitCycles);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int key_w = 16 * MG * warp;  // this warp's first key in a stage
    const float cap2 = p.softcap_log2e;
    // ldmatrix lane roles: matrix q = lane / 8, row r = lane % 8 of that matrix.
    const int lq = lane >> 3, lr = lane & 7;
    bool failed = false;
    int it = 0;  // stages consumed

    for (long long pos = s_c; pos < e_c;) {
        const Segment sg = segment_at(prefix, p.seq_lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c);
        const int lo = sg.lo, hi = sg.hi;
        const int t0 = lo / kTileKeys;
        const int h0 = sg.kvh * p.G + sg.hg * HC;
        const int nh = min(HC, p.G - sg.hg * HC);

        uint32_t qhi[NHT][KS][2], qlo[NHT][KS][2];
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) {
            const int head = nt * 8 + g;
            const float* qrow = p.q_prime + (static_cast<size_t>(sg.b) * p.Hq + h0 + head) * D;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                float2 x01 = make_float2(0.f, 0.f), x89 = make_float2(0.f, 0.f);
                if (head < nh) {
                    x01 = *reinterpret_cast<const float2*>(qrow + 16 * kk + 2 * t);
                    x89 = *reinterpret_cast<const float2*>(qrow + 16 * kk + 2 * t + 8);
                }
                split_bf16(x01.x, x01.y, qhi[nt][kk][0], qlo[nt][kk][0]);
                split_bf16(x89.x, x89.y, qhi[nt][kk][1], qlo[nt][kk][1]);
            }
        }

        float m[NHT][2], l[NHT][2], o[NHT][KS][4];
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) o[nt][mi][0] = o[nt][mi][1] = o[nt][mi][2] = o[nt][mi][3] = 0.f;
        }
        float r_scale = 0.f;  // vq8: the warp's running maximum value scale (O is kept in units of it)

        for (int k = 0; k < sg.n_st; ++k, ++it) {
            const int s = it % SH::kStages;
            if (!failed && !ptx::mbar_wait(bar_full + 8 * s, (it / SH::kStages) & 1, kWaitLimitCycles)) {
                failed = true;
                if (lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
            }
            const int kbase = (t0 + MG * (sg.st0 + k)) * kTileKeys + key_w;  // this warp's first key
            if (!failed && kbase < hi && kbase + 16 * MG > lo) {
                const bool whole = kbase >= lo && kbase + 16 * MG <= hi;
                const uint32_t st = base + s * SH::kStageBytes;

                // S^T = K . Q'^T (keys x heads), one accumulator per 16-key group
                float sacc[MG][NHT][4];
#pragma unroll
                for (int mg = 0; mg < MG; ++mg)
#pragma unroll
                    for (int nt = 0; nt < NHT; ++nt)
                        sacc[mg][nt][0] = sacc[mg][nt][1] = sacc[mg][nt][2] = sacc[mg][nt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
                        uint32_t a[4];
                        ptx::ldsm_x4(a, st + tile_off<TK>(key_w + 16 * mg + lr + 8 * (lq & 1), 2 * kk + (lq >> 1)));
#pragma unroll
                        for (int nt = 0; nt < NHT; ++nt) {
                            ptx::mma_bf16(sacc[mg][nt], a, qhi[nt][kk][0], qhi[nt][kk][1]);
                            ptx::mma_bf16(sacc[mg][nt], a, qlo[nt][kk][0], qlo[nt][kk][1]);
                        }
                    }
                }

                // this thread holds keys 16 mg + g and 16 mg + g + 8, heads 2t and 2t + 1
                bool vg[MG], vg8[MG];
#pragma unroll
                for (int mg = 0; mg < MG; ++mg) {
                    vg[mg] = whole || key_ok(kbase + 16 * mg + g, lo, hi);
                    vg8[mg] = whole || key_ok(kbase + 16 * mg + g + 8, lo, hi);
                }
                float w_g[MG], w_g8[MG], r_ratio = 1.f;
                if (VQ8) {  // per-key scale relative to the running maximum; masked keys get 0
                    const float* scl = reinterpret_cast<const float*>(base_ptr + s * SH::kStageBytes + SH::kKBytes +
                                                                      SH::kVBytes);
                    float smax = 0.f;
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
                        w_g[mg] = vg[mg] ? scl[key_w + 16 * mg + g] : 0.f;
                        w_g8[mg] = vg8[mg] ? scl[key_w + 16 * mg + g + 8] : 0.f;
                        smax = fmaxf(smax, fmaxf(w_g[mg], w_g8[mg]));
                    }
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
                    const float r_new = fmaxf(r_scale, smax);
                    const float inv = r_new > 0.f ? ptx::rcp(r_new) : 0.f;
                    r_ratio = r_new > 0.f ? r_scale * inv : 1.f;
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
                        w_g[mg] *= inv;
                        w_g8[mg] *= inv;
                    }
                    r_scale = r_new;
                }

                float x[MG][NHT][4], f[NHT][2];
                bool rescale = false;
#pragma unroll
                for (int nt = 0; nt < NHT; ++nt) {
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = sacc[mg][nt][e];
                            if (cap2 > 0.f) v = tanhf(v) * cap2;
                            if (!((e < 2) ? vg[mg] : vg8[mg])) v = -INFINITY;
                            x[mg][nt][e] = v;
                        }
                        mx0 = fmaxf(mx0, fmaxf(x[mg][nt][0], x[mg][nt][2]));
                        mx1 = fmaxf(mx1, fmaxf(x[mg][nt][1], x[mg][nt][3]));
                    }
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
                    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
                    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float al0 = ptx::ex2(m[nt][0] - mu0), al1 = ptx::ex2(m[nt][1] - mu1);
                    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
                        x[mg][nt][0] = ptx::ex2(x[mg][nt][0] - mu0);
                        x[mg][nt][1] = ptx::ex2(x[mg][nt][1] - mu1);
                        x[mg][nt][2] = ptx::ex2(x[mg][nt][2] - mu0);
                        x[mg][nt][3] = ptx::ex2(x[mg][nt][3] - mu1);
                        ls0 += x[mg][nt][0] + x[mg][nt][2];
                        ls1 += x[mg][nt][1] + x[mg][nt][3];
                    }
                    l[nt][0] = l[nt][0] * al0 + ls0;
                    l[nt][1] = l[nt][1] * al1 + ls1;
                    m[nt][0] = mn0;
                    m[nt][1] = mn1;
                    f[nt][0] = al0 * r_ratio;
                    f[nt][1] = al1 * r_ratio;
                    rescale |= f[nt][0] != 1.f || f[nt][1] != 1.f;
                }
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
                        for (int mi = 0; mi < KS; ++mi) {
                            o[nt][mi][0] *= f[nt][0];
                            o[nt][mi][1] *= f[nt][1];
                            o[nt][mi][2] *= f[nt][0];
                            o[nt][mi][3] *= f[nt][1];
                        }
                }

#pragma unroll
                for (int mg = 0; mg < MG; ++mg) {
                    uint32_t bph[NHT][2], bpl[NHT][2];
#pragma unroll
                    for (int nt = 0; nt < NHT; ++nt) {
                        uint32_t h01, l01, h23, l23;
                        if (VQ8) {
                            split_f16(x[mg][nt][0] * w_g[mg], x[mg][nt][1] * w_g[mg], h01, l01);     // key g
                            split_f16(x[mg][nt][2] * w_g8[mg], x[mg][nt][3] * w_g8[mg], h23, l23);   // key g+8
                        } else {
                            split_bf16(x[mg][nt][0], x[mg][nt][1], h01, l01);
                            split_bf16(x[mg][nt][2], x[mg][nt][3], h23, l23);
                        }
                        bph[nt][0] = ptx::movmatrix_trans(h01);
                        bph[nt][1] = ptx::movmatrix_trans(h23);
                        bpl[nt][0] = ptx::movmatrix_trans(l01);
                        bpl[nt][1] = ptx::movmatrix_trans(l23);
                    }
                    const int krow = key_w + 16 * mg;  // this group's first row in the stage
                    if (VQ8) {
                        // O^T += V^T . P^T straight from the int8 stage: one ldmatrix.x4.trans covers
                        // 16 keys x 32 values = m-tiles 2j (values 32j .. 32j+15) and 2j+1; in m-tile
                        // mi row g holds value 16 mi + 2g and row g + 8 holds 16 mi + 2g + 1.
                        const uint32_t vst = st + SH::kKBytes;
#pragma unroll
                        for (int j = 0; j < D / 32; ++j) {
                            uint32_t r[4];
                            ptx::ldsm_x4_trans(r, vst + code_off<D, TK>(krow + lr + 8 * (lq >> 1), 2 * j + (lq & 1)));
                            uint32_t a[4], c[4];
                            widen_code_pairs(r[0], a[0], a[1]);  // keys 2t, 2t+1; values 32j + 2g, +1
                            widen_code_pairs(r[2], a[2], a[3]);  // keys 2t+8, 2t+9
                            widen_code_pairs(r[1], c[0], c[1]);  // values 32j + 16 + 2g, +1
                            widen_code_pairs(r[3], c[2], c[3]);
#pragma unroll
                            for (int nt = 0; nt < NHT; ++nt) {
                                ptx::mma_f16(o[nt][2 * j], a, bph[nt][0], bph[nt][1]);
                                ptx::mma_f16(o[nt][2 * j], a, bpl[nt][0], bpl[nt][1]);
                                ptx::mma_f16(o[nt][2 * j + 1], c, bph[nt][0], bph[nt][1]);
                                ptx::mma_f16(o[nt][2 * j + 1], c, bpl[nt][0], bpl[nt][1]);
                            }
                        }
                    } else {
                        // key-validity masks for V^T fragments: registers 0,1 hold keys 2t, 2t+1;
                        // registers 2,3 hold keys 2t+8, 2t+9 (lower half = lower key)
                        uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
                        if (!whole) {
                            const int kq = kbase + 16 * mg + 2 * t;
                            m01 = (key_ok(kq, lo, hi) ? 0x0000ffffu : 0u) | (key_ok(kq + 1, lo, hi) ? 0xffff0000u : 0u);
                            m89 = (key_ok(kq + 8, lo, hi) ? 0x0000ffffu : 0u) |
                                  (key_ok(kq + 9, lo, hi) ? 0xffff0000u : 0u);
                        }
#pragma unroll
                        for (int mi = 0; mi < KS; ++mi) {
                            uint32_t a[4];
                            ptx::ldsm_x4_trans(a, st + SH::kKBytes +
                                                      tile_off<TK>(krow + lr + 8 * (lq >> 1), 2 * mi + (lq & 1)));
                            a[0] &= m01;
                            a[1] &= m01;
                            a[2] &= m89;
                            a[3] &= m89;
#pragma unroll
                            for (int nt = 0; nt < NHT; ++nt) {
                                ptx::mma_bf16(o[nt][mi], a, bph[nt][0], bph[nt][1]);
                                ptx::mma_bf16(o[nt][mi], a, bpl[nt][0], bpl[nt][1]);
                            }
                        }
                    }
                }
            }
            if (k + 1 < sg.n_st) {  // the segment's last stage is held for the merge scratch
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
            }
        }

        // ------------------------------------------------------------ merge
#pragma unroll
        for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], off);

        const int s_last = (it - 1) % SH::kStages;
        float* red_m = reinterpret_cast<float*>(base_ptr + s_last * SH::kStageBytes);
        float* red_l = red_m + kConsumerWarps * HC;
        float* red_o = red_l + kConsumerWarps * HC;
        const float o_unit = VQ8 ? r_scale : 1.f;
        const size_t rec = 2 * static_cast<size_t>(blockIdx.x) + (pos == s_c ? 0 : 1);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += RC) {
            ptx::named_barrier_sync(1, kConsumerWarps * 32);  // stage (or previous round) no longer read
            if (g == 0 && c0 == 0) {
#pragma unroll
                for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        red_m[warp * HC + nt * 8 + 2 * t + j] = m[nt][j];
                        red_l[warp * HC + nt * 8 + 2 * t + j] = l[nt][j];
                    }
            }
#pragma unroll
            for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
                for (int mi = 0; mi < KS; ++mi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int hc = nt * 8 + 2 * t + (e & 1);
                        const int d = VQ8 ? 16 * mi + 2 * g + (e >> 1) : 16 * mi + g + 8 * (e >> 1);
                        if (d >= c0 && d < c0 + RC) red_o[(warp * HC + hc) * (RC + 4) + d - c0] = o[nt][mi][e] * o_unit;
                    }
            ptx::named_barrier_sync(1, kConsumerWarps * 32);
            for (int idx = threadIdx.x; idx < nh * RC; idx += kConsumerWarps * 32) {
                const int hc = idx / RC, dc = idx - hc * RC;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * HC + hc]);
                const float zs = (sg.whole && p.sink) ? p.sink[h0 + hc] * kLog2e : -INFINITY;
                if (sg.whole) M = fmaxf(M, zs);  // the sink joins the denominator of a whole unit
                float L = 0.f, acc = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        const float mw = red_m[w * HC + hc];
                        const float fw = mw == -INFINITY ? 0.f : exp2f(mw - M);
                        L += red_l[w * HC + hc] * fw;
                        acc += red_o[(w * HC + hc) * (RC + 4) + dc] * fw;
                    }
                }
                if (sg.whole) {
                    const float den = L + (zs == -INFINITY ? 0.f : exp2f(zs - M));
                    const float v = den > 0.f ? acc / den : 0.f;
                    const size_t oi = (static_cast<size_t>(sg.b) * p.Hq + h0 + hc) * D + c0 + dc;
                    if (p.out_dtype == UAA_DTYPE_F32)
                        static_cast<float*>(p.out)[oi] = v;
                    else
                        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(v);
                } else {
                    p.rec_o[(rec * HC + hc) * D + c0 + dc] = L > 0.f ? acc / L : 0.f;
                    if (c0 + dc == 0) p.rec_lse[rec * HC + hc] = L > 0.f ? M + log2f(L) : -INFINITY;
                }
            }
        }
        // the stage held for the scratch goes back to the producer (after the generic
        // accesses are ordered before the TMA writes that will refill it)
        ptx::named_barrier_sync(1, kConsumerWarps * 32);
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s_last);
        pos += sg.n_st;
    }
}

template <int D, bool VQ8, int NHT>
cudaError_t launch_one(const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& ts, int n_ctas, cudaStream_t s)
{
    using SH = Shape<D, VQ8>;
    auto kern = partial_tc_kernel<D, VQ8, NHT>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 31) configured_device_mask |= 1 << dev;
    }
    return launch_dependent(kern, dim3(n_ctas), dim3(kThreads), SH::kSmemBytes, s, tk, tv, ts, p);
}

}  // namespace

int partial_tc_keys_per_stage(int D) { return D == 64 ? KeyGroups<64>::kMG * kTileKeys : kTileKeys; }

size_t partial_tc_smem_bytes(int D, int kv_dtype, int n_head_tiles)
{
    (void)n_head_tiles;
    const bool vq8 = kv_dtype == UAA_DTYPE_VQ8;
    switch (D) {
    case 64: return vq8 ? Shape<64, true>::kSmemBytes : Shape<64, false>::kSmemBytes;
    case 128: return vq8 ? Shape<128, true>::kSmemBytes : Shape<128, false>::kSmemBytes;
    case 256: return vq8 ? Shape<256, true>::kSmemBytes : Shape<256, false>::kSmemBytes;
    default: return 0;
    }
}

cudaError_t launch_partial_tc(const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& ts, int kv_dtype, int n_head_tiles, int n_ctas, cudaStream_t s)
{
    const bool vq8 = kv_dtype == UAA_DTYPE_VQ8;
    if (n_head_tiles == 2) {
        switch (p.D) {
        case 64: return vq8 ? launch_one<64, true, 2>(p, tk, tv, ts, n_ctas, s) : launch_one<64, false, 2>(p, tk, tv, ts, n_ctas, s);
        case 128: return vq8 ? launch_one<128, true, 2>(p, tk, tv, ts, n_ctas, s) : launch_one<128, false, 2>(p, tk, tv, ts, n_ctas, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.D) {
    case 64: return vq8 ? launch_one<64, true, 1>(p, tk, tv, ts, n_ctas, s) : launch_one<64, false, 1>(p, tk, tv, ts, n_ctas, s);
    case 128: return vq8 ? launch_one<128, true, 1>(p, tk, tv, ts, n_ctas, s) : launch_one<128, false, 1>(p, tk, tv, ts, n_ctas, s);
    case 256: return vq8 ? launch_one<256, true, 1>(p, tk, tv, ts, n_ctas, s) : launch_one<256, false, 1>(p, tk, tv, ts, n_ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
