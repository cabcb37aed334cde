// partial_tc.cu -- split-K decode partial for bf16 and vq8 caches: TMA tile
// loads into a shared-memory ring, bf16 tensor-core contractions.
//
// Work unit: one CTA per (split, kv head x head group, sequence). Every query
// head of the kv head's group (up to 8 * NHT per CTA) is served from the same
// K/V tiles, so each tile leaves HBM once per CTA.
//
// Warp roles (160 threads):
//   warp 4 (producer): one lane streams the split's 64-key tiles with 2-D TMA
//     loads (cp.async.bulk.tensor) into a ring of kStages stages; K and bf16 V
//     boxes are 64 rows x 128 bytes with the 128-byte swizzle, vq8 codes are
//     one 64 x D-byte box, vq8 scales one 64-float box. Full / empty mbarriers
//     hand stages back and forth.
//   warps 0-3 (consumers): warp w owns keys 16w .. 16w+15 of every tile.
//     S^T (16 keys x 8 heads) = K_tile (16 x D) . Q'^T (D x 8) with mma.m16n8k16
//     (keys on M, heads on N, no padding of M). The fp32 q' rows are split into
//     bf16 hi + lo parts, two MMAs each, so the logits keep ~16 significant bits.
//     Online softmax (log2 domain) runs on the fp32 accumulators; P is split
//     into bf16 hi + lo, transposed in registers with movmatrix into the B
//     operand of O^T (D x 8) += V^T (D x 16 keys) . P^T (16 keys x 8 heads),
//     V^T fragments come from ldmatrix.trans. vq8 codes are widened to bf16
//     (exact) in a per-warp staging area; the per-key scale is folded into P.
//   At the end the four warp states are merged through shared memory and the
//   CTA writes one normalised partial row and its log2-sum-exp per head.
//
// Every wait is bounded (kWaitLimitCycles); a wait that gives up sets
// UAA_DEVFLAG_TIMEOUT and the CTA unwinds without further waits.
#include "internal.cuh"
#include "ptx.cuh"

namespace uaa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBoxBytes = kTileKeys * 128;  // 64 rows x 128 bytes

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, bool VQ8>
struct Shape {
    static constexpr int kBoxes = D / 64;                   // 128-byte column boxes of a bf16 row
    static constexpr int kKBytes = kTileKeys * D * 2;
    static constexpr int kVBytes = VQ8 ? kTileKeys * D : kTileKeys * D * 2;
    static constexpr int kSBytes = VQ8 ? kTileKeys * 4 : 0;
    static constexpr int kStageBytes = round_up(kKBytes + kVBytes + kSBytes, 1024);
    static constexpr int kTxBytes = kKBytes + kVBytes + kSBytes;
    static constexpr int kStagingWarpBytes = VQ8 ? 16 * D * 2 : 0;  // bf16 copy of 16 rows
    static constexpr int kStagingBytes = kConsumerWarps * kStagingWarpBytes;
    static constexpr int kBudget = (D == 256 ? 196608 : 98304) - kStagingBytes;
    static constexpr int kStagesRaw = kBudget / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kStagingBytes + 16 * kStages;
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a ring tile: boxes of
// 64 rows x 128 bytes, chunk index XOR (row mod 8) inside each 128-byte row.
__device__ __forceinline__ uint32_t tile_off(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Same swizzle for a warp's 16-row staging copy.
__device__ __forceinline__ uint32_t staging_off(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
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

// Four int8 codes -> two bf16x2 words, exactly: byte c + 128 is placed in the
// mantissa of 2^23 (fp32), 2^23 + 128 is subtracted, and the upper halves of
// the two fp32 results (integers of magnitude <= 128) are the bf16 values.
__device__ __forceinline__ void widen_codes(uint32_t w, uint32_t& p01, uint32_t& p23)
{
    const uint32_t u = w ^ 0x80808080u;
    const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - 8388736.0f;
    const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - 8388736.0f;
    const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - 8388736.0f;
    const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - 8388736.0f;
    p01 = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
    p23 = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

template <int D, bool VQ8, int NHT>
__global__ void __launch_bounds__(kThreads, (D == 256 ? 1 : 2))
partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_s, const PartialParams p)
{
    using SH = Shape<D, VQ8>;
    constexpr int KS = D / 16;     // k-steps of QK, m-tiles of PV
    constexpr int HC = 8 * NHT;    // head columns of the CTA
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t staging = base + SH::kRingBytes;
    const uint32_t bar_full = staging + SH::kStagingBytes;
    const uint32_t bar_empty = bar_full + 8 * SH::kStages;

    const int sigma = blockIdx.x;
    const int kvh = blockIdx.y / p.head_groups, hg = blockIdx.y % p.head_groups;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int lo, hi;
    key_range(p.seq_lens[b], p.window, lo, hi);
    if (hi > p.cap) {  // a length past the cache: never read beyond it
        hi = p.cap;
        if (threadIdx.x == 0 && sigma == 0) atomicOr(p.status, UAA_DEVFLAG_CAPACITY);
    }
    const int t0 = lo / kTileKeys, t1 = (hi + kTileKeys - 1) / kTileKeys;
    const int tb = t0 + sigma * p.chunk_tiles;
    if (hi <= lo || tb >= t1) return;  // uniform over the CTA: this split has no keys
    const int n_tiles = min(tb + p.chunk_tiles, t1) - tb;
    const int h0 = kvh * p.G + hg * HC;
    const int nh = min(HC, p.G - hg * HC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SH::kStages; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        ptx::fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tensormap(&tm_k);
            ptx::prefetch_tensormap(&tm_v);
            if (VQ8) ptx::prefetch_tensormap(&tm_s);
            const int head_row = b * p.Hkv + kvh;
            const int row0 = head_row * p.cap;
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int s = i % SH::kStages;
                if (i >= SH::kStages &&
                    !ptx::mbar_wait(bar_empty + 8 * s, ((i / SH::kStages) & 1) ^ 1, kWaitLimitCycles)) {
                    atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                    ok = false;
                    break;
                }
                const uint32_t st = base + s * SH::kStageBytes;
                const uint32_t bar = bar_full + 8 * s;
                ptx::mbar_arrive_expect_tx(bar, SH::kTxBytes);
                const int key = (tb + i) * kTileKeys;
                const int y = row0 + key;
#pragma unroll
                for (int c = 0; c < SH::kBoxes; ++c) ptx::tma_load_2d(st + c * kBoxBytes, &tm_k, c * 64, y, bar);
                if (VQ8) {
                    ptx::tma_load_2d(st + SH::kKBytes, &tm_v, 0, y, bar);
                    ptx::tma_load_2d(st + SH::kKBytes + SH::kVBytes, &tm_s, key, head_row, bar);
                } else {
#pragma unroll
                    for (int c = 0; c < SH::kBoxes; ++c)
                        ptx::tma_load_2d(st + SH::kKBytes + c * kBoxBytes, &tm_v, c * 64, y, bar);
                }
            }
            // Copies in flight land before the CTA may exit (bounded).
            const int first = n_tiles > SH::kStages ? n_tiles - SH::kStages : 0;
            for (int i = first; i < n_tiles && ok; ++i)
                ok = ptx::mbar_wait(bar_full + 8 * (i % SH::kStages), (i / SH::kStages) & 1, kWaitLimitCycles);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t qhi[NHT][KS][2], qlo[NHT][KS][2];
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt) {
        const int head = nt * 8 + g;
        const float* qrow = p.q_prime + (static_cast<size_t>(b) * p.Hq + h0 + head) * D;
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

    const int key_w = 16 * warp;
    const float cap2 = p.softcap_log2e;
    const uint32_t my_staging = staging + warp * SH::kStagingWarpBytes;
    // ldmatrix lane roles: matrix q = lane / 8, row r = lane % 8 of that matrix.
    const int lq = lane >> 3, lr = lane & 7;
    bool failed = false;

    for (int i = 0; i < n_tiles; ++i) {
        const int s = i % SH::kStages;
        if (!failed && !ptx::mbar_wait(bar_full + 8 * s, (i / SH::kStages) & 1, kWaitLimitCycles)) {
            failed = true;
            if (lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
        }
        const int key0 = (tb + i) * kTileKeys + key_w;  // absolute slot of this warp's first key
        if (!failed && key0 < hi && key0 + 16 > lo) {
            const bool whole = key0 >= lo && key0 + 16 <= hi;
            const uint32_t st = base + s * SH::kStageBytes;

            // S^T = K . Q'^T (keys x heads)
            float sacc[NHT][4];
#pragma unroll
            for (int nt = 0; nt < NHT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a[4];
                ptx::ldsm_x4(a, st + tile_off(key_w + lr + 8 * (lq & 1), 2 * kk + (lq >> 1)));
#pragma unroll
                for (int nt = 0; nt < NHT; ++nt) {
                    ptx::mma_bf16(sacc[nt], a, qhi[nt][kk][0], qhi[nt][kk][1]);
                    ptx::mma_bf16(sacc[nt], a, qlo[nt][kk][0], qlo[nt][kk][1]);
                }
            }

            // online softmax; this thread holds keys g, g+8 and heads 2t, 2t+1
            bool vg = true, vg8 = true;
            if (!whole) {
                vg = key0 + g >= lo && key0 + g < hi;
                vg8 = key0 + g + 8 >= lo && key0 + g + 8 < hi;
            }
            float sc_g = 1.f, sc_g8 = 1.f;
            if (VQ8) {
                const float* scl = reinterpret_cast<const float*>(base_ptr + s * SH::kStageBytes + SH::kKBytes + SH::kVBytes);
                sc_g = scl[key_w + g];
                sc_g8 = scl[key_w + g + 8];
            }
            uint32_t bph[NHT][2], bpl[NHT][2];
#pragma unroll
            for (int nt = 0; nt < NHT; ++nt) {
                float x0 = sacc[nt][0], x1 = sacc[nt][1], x2 = sacc[nt][2], x3 = sacc[nt][3];
                if (cap2 > 0.f) {
                    x0 = tanhf(x0) * cap2;
                    x1 = tanhf(x1) * cap2;
                    x2 = tanhf(x2) * cap2;
                    x3 = tanhf(x3) * cap2;
                }
                if (!vg) x0 = x1 = -INFINITY;
                if (!vg8) x2 = x3 = -INFINITY;
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
                const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
                const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
                const float al0 = exp2f(m[nt][0] - mu0), al1 = exp2f(m[nt][1] - mu1);
                float p0 = exp2f(x0 - mu0), p1 = exp2f(x1 - mu1);
                float p2 = exp2f(x2 - mu0), p3 = exp2f(x3 - mu1);
                l[nt][0] = l[nt][0] * al0 + p0 + p2;
                l[nt][1] = l[nt][1] * al1 + p1 + p3;
                m[nt][0] = mn0;
                m[nt][1] = mn1;
#pragma unroll
                for (int mi = 0; mi < KS; ++mi) {
                    o[nt][mi][0] *= al0;
                    o[nt][mi][1] *= al1;
                    o[nt][mi][2] *= al0;
                    o[nt][mi][3] *= al1;
                }
                if (VQ8) {  // fold the per-key scale into P; masked keys may hold any bits
                    p0 = vg ? p0 * sc_g : 0.f;
                    p1 = vg ? p1 * sc_g : 0.f;
                    p2 = vg8 ? p2 * sc_g8 : 0.f;
                    p3 = vg8 ? p3 * sc_g8 : 0.f;
                }
                uint32_t h01, l01, h23, l23;
                split_bf16(p0, p1, h01, l01);  // key g, heads 2t, 2t+1
                split_bf16(p2, p3, h23, l23);  // key g+8
                bph[nt][0] = ptx::movmatrix_trans(h01);
                bph[nt][1] = ptx::movmatrix_trans(h23);
                bpl[nt][0] = ptx::movmatrix_trans(l01);
                bpl[nt][1] = ptx::movmatrix_trans(l23);
            }

            if (VQ8) {
                // widen this warp's 16 rows of codes into the bf16 staging copy
                const int r = lane >> 1, half = lane & 1;
                const uint8_t* src = base_ptr + s * SH::kStageBytes + SH::kKBytes +
                                     static_cast<size_t>(key_w + r) * D + half * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(src + 16 * c);
                    uint4 lo4, hi4;
                    widen_codes(w.x, lo4.x, lo4.y);
                    widen_codes(w.y, lo4.z, lo4.w);
                    widen_codes(w.z, hi4.x, hi4.y);
                    widen_codes(w.w, hi4.z, hi4.w);
                    const int oc = half * (D / 16) + 2 * c;
                    uint8_t* stg = base_ptr + (my_staging - base);
                    *reinterpret_cast<uint4*>(stg + staging_off(r, oc)) = lo4;
                    *reinterpret_cast<uint4*>(stg + staging_off(r, oc + 1)) = hi4;
                }
                __syncwarp();
            }

            // key-validity masks for V^T fragments: registers 0,1 hold keys 2t, 2t+1;
            // registers 2,3 hold keys 2t+8, 2t+9 (lower half = lower key)
            uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
            if (!VQ8 && !whole) {
                const int k = key0 + 2 * t;
                m01 = ((k >= lo && k < hi) ? 0x0000ffffu : 0u) | ((k + 1 >= lo && k + 1 < hi) ? 0xffff0000u : 0u);
                m89 = ((k + 8 >= lo && k + 8 < hi) ? 0x0000ffffu : 0u) |
                      ((k + 9 >= lo && k + 9 < hi) ? 0xffff0000u : 0u);
            }

            // O^T += V^T . P^T
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) {
                uint32_t a[4];
                const int row = lr + 8 * (lq >> 1);
                const int chunk = 2 * mi + (lq & 1);
                if (VQ8)
                    ptx::ldsm_x4_trans(a, my_staging + staging_off(row, chunk));
                else
                    ptx::ldsm_x4_trans(a, st + SH::kKBytes + tile_off(key_w + row, chunk));
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
            if (VQ8) __syncwarp();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
    }

    // ---------------------------------------------------------------- merge
#pragma unroll
    for (int nt = 0; nt < NHT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], off);

    ptx::named_barrier_sync(1, kConsumerWarps * 32);  // the ring is no longer read
    constexpr int OS = D + 4;
    float* red_m = reinterpret_cast<float*>(base_ptr);
    float* red_l = red_m + kConsumerWarps * HC;
    float* red_o = red_l + kConsumerWarps * HC;
    if (g == 0) {
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
            for (int k = 0; k < 4; ++k) {
                const int hc = nt * 8 + 2 * t + (k & 1);
                const int d = 16 * mi + g + 8 * (k >> 1);
                red_o[(warp * HC + hc) * OS + d] = o[nt][mi][k];
            }
    ptx::named_barrier_sync(1, kConsumerWarps * 32);

    for (int idx = threadIdx.x; idx < nh * D; idx += kConsumerWarps * 32) {
        const int hc = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * HC + hc]);
        float L = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = red_m[w * HC + hc];
                const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
                L += red_l[w * HC + hc] * f;
                acc += red_o[(w * HC + hc) * OS + d] * f;
            }
        }
        const size_t row = (static_cast<size_t>(b) * p.Hq + h0 + hc) * p.S + sigma;
        p.o_part[row * D + d] = L > 0.f ? acc / L : 0.f;
        if (d == 0) p.lse_part[row] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
}

template <int D, bool VQ8, int NHT>
cudaError_t launch_one(const PartialParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& ts, cudaStream_t s)
{
    using SH = Shape<D, VQ8>;
    auto kern = partial_tc_kernel<D, VQ8, NHT>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 31 && !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device_mask |= 1 << dev;
    }
    const dim3 grid(p.S, p.Hkv * p.head_groups, p.B);
    kern<<<grid, kThreads, SH::kSmemBytes, s>>>(tk, tv, ts, p);
    return cudaGetLastError();
}

}  // namespace

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
                              const CUtensorMap& ts, int kv_dtype, int n_head_tiles, cudaStream_t s)
{
    const bool vq8 = kv_dtype == UAA_DTYPE_VQ8;
    if (n_head_tiles == 2) {
        switch (p.D) {
        case 64: return vq8 ? launch_one<64, true, 2>(p, tk, tv, ts, s) : launch_one<64, false, 2>(p, tk, tv, ts, s);
        case 128: return vq8 ? launch_one<128, true, 2>(p, tk, tv, ts, s) : launch_one<128, false, 2>(p, tk, tv, ts, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.D) {
    case 64: return vq8 ? launch_one<64, true, 1>(p, tk, tv, ts, s) : launch_one<64, false, 1>(p, tk, tv, ts, s);
    case 128: return vq8 ? launch_one<128, true, 1>(p, tk, tv, ts, s) : launch_one<128, false, 1>(p, tk, tv, ts, s);
    case 256: return vq8 ? launch_one<256, true, 1>(p, tk, tv, ts, s) : launch_one<256, false, 1>(p, tk, tv, ts, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
