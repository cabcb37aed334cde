// prefill_tc.cu -- attention of a long chunk of tokens (a prefill chunk) over a
// bf16 cache, tiled over the queries: step 2 for steps of many tokens per
// sequence, after the separate append has written the chunk's rows and q'.
//
// The (token, head) rows of one kv head (token-major: row r is token r / G,
// query head r % G of the group, as in query_row) are cut into blocks of 128.
// One CTA per (sequence, kv head, row block) streams the keys its rows see (the
// cache and the chunk's tokens up to the block's last one, within the window)
// once, 64 keys per ring stage, and writes the block's output rows itself: no
// records, no combine. Each K/V tile is read from L2 once per row block,
// instead of once per 16 rows as in the decode kernel's units; the row blocks
// of one kv head are neighbours in the grid, so they read the same tiles at
// about the same time and HBM delivers each tile about once.
//
// Warps (256 threads, one CTA per SM, two warps per SM sub-partition so that a
// thread may hold up to 255 registers): each of the 8 warps owns 16 query rows;
// thread 0 also streams the key and value tiles of the CTA's key blocks with
// 2-D TMA loads (64 rows x 128 bytes per box, the 128-byte swizzle) into a ring
// of stages with full / empty mbarriers, refilling the slot of the stage
// consumed two iterations earlier (so it seldom waits on a slower warp).
// Queries sit on M of mma.m16n8k16:
//   S (16 rows x 64 keys) = Q' (16 x D) . K^T: the q' rows (fp32, already
//     rotated and prescaled by the append) split into bf16 hi + lo parts held
//     as A fragments for the whole CTA; K^T fragments by ldmatrix from the
//     stage (a key row is a B column);
//   online softmax per row in the log2 domain (the four lanes of a row group
//     reduce with two shuffles), causal and window masks per row on the blocks
//     that need them;
//   O (16 x D) += P (16 x 64) . V: the S accumulators are the A fragments of P
//     directly (hi + lo bf16 parts); V fragments by ldmatrix.trans.
// At the end each row is divided by its sum (with the sink logit in the
// denominator when the descriptor has sinks) and stored.
#include "internal.cuh"
#include "ptx.cuh"

namespace uaa {
namespace {

constexpr int kPfRows = kPrefillRows;  // query rows per CTA
constexpr int kPfConsumers = kPfRows / 16;  // warps of 16 rows
constexpr int kPfThreads = kPfConsumers * 32;
constexpr int kPfKeys = 64;          // keys per ring stage

template <int D>
struct PfShape {
    static constexpr int kBoxes = D / 64;                    // 64-column boxes of a row
    static constexpr int kHalf = kPfKeys * D * 2;            // one tile (keys or values) of a stage
    static constexpr int kStageBytes = 2 * kHalf;
    static constexpr int kStages = D == 128 ? 5 : 8;         // 160 / 128 KB of ring, one CTA per SM
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 16 * kStages;
};

// Byte offset of 16-byte chunk `chunk` (8 dims) of row `row` in a tile of 64 rows
// whose 64-column boxes are stored one after the other with the 128-byte swizzle.
__device__ __forceinline__ uint32_t pf_off(int row, int chunk)
{
    return static_cast<uint32_t>((chunk >> 3) * (kPfKeys * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t pf_pack(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// x ~= hi + lo for two values: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void pf_split(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = pf_pack(x0, x1);
    lo = pf_pack(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const PrefillParams p)
{
    using SH = PfShape<D>;
    constexpr int NS = SH::kStages;
    constexpr int KS = D / 16;  // k-steps of Q.K^T
    constexpr int NO = D / 8;   // 8-column tiles of O
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bar_full = base + NS * SH::kStageBytes;
    const uint32_t bar_empty = bar_full + 8 * NS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rb = (p.q_len * p.G + kPfRows - 1) / kPfRows;
    const int rb = blockIdx.x % n_rb;
    const int bk = blockIdx.x / n_rb;  // b * Hkv + kvh
    const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
    const int rows = p.q_len * p.G;    // query rows of the kv head

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, kPfConsumers);
        }
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    grid_dependency_wait();  // the append's rows, q' and lengths are complete
    __syncthreads();         // the barriers are initialised

    // The chunk's tokens sit at L .. L + q_len - 1 (the append advanced the length
    // past them); a sequence the append could not take keeps its length and is skipped.
    const int L_after = p.seq_lens[b];
    const int L = L_after - p.q_len;
    const bool valid = L >= 0 && L_after <= p.cap;
    const int r_first = rb * kPfRows, r_last = min(rows, r_first + kPfRows) - 1;
    const int hi = valid ? L + r_last / p.G + 1 : 0;  // keys the block sees: [lo, hi)
    const int lo = valid && p.window > 0 ? max(0, L + r_first / p.G + 1 - p.window) : 0;
    const int kb0 = lo / kPfKeys;
    const int n_st = (hi + kPfKeys - 1) / kPfKeys - kb0;  // ring stages (64-key blocks)

    // the loads of stage i into slot i % NS (thread 0); false: the slot never came free
    const int row0 = (b * p.Hkv + kvh) * p.cap + kb0 * kPfKeys;
    int issued = 0;
    auto issue = [&](int i) -> bool {
        const int s = i % NS;
        if (i >= NS && !ptx::mbar_wait(bar_empty + 8 * s, ((i / NS) - 1) & 1, kWaitLimitCycles)) {
            atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
            return false;
        }
        const uint32_t st = base + s * SH::kStageBytes;
        const uint32_t bar = bar_full + 8 * s;
        ptx::mbar_arrive_expect_tx(bar, SH::kStageBytes);
#pragma unroll
        for (int c = 0; c < SH::kBoxes; ++c) {
            // plain loads: the other row blocks of this kv head read the same tiles from L2
            ptx::tma_load_2d(st + c * (kPfKeys * 128), &tm_k, c * 64, row0 + i * kPfKeys, bar);
            ptx::tma_load_2d(st + SH::kHalf + c * (kPfKeys * 128), &tm_v, c * 64, row0 + i * kPfKeys, bar);
        }
        issued = i + 1;
        return true;
    };
    bool loading = threadIdx.x == 0;
    if (loading)
        for (int i = 0; i < min(NS, n_st) && loading; ++i) loading = issue(i);

    // -------------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int lq = lane >> 3, lr = lane & 7;  // ldmatrix: matrix lq, row lr
    // this thread's rows: rA = 16 warp + g and rB = rA + 8 of the block
    const int RA = r_first + 16 * warp + g, RB = RA + 8;
    const bool okA = valid && RA < rows, okB = valid && RB < rows;
    const int kmaxA = L + RA / p.G, kmaxB = L + RB / p.G;  // the last key each row sees
    const int kminA = p.window > 0 ? kmaxA - p.window + 1 : INT_MIN;
    const int kminB = p.window > 0 ? kmaxB - p.window + 1 : INT_MIN;

    // q' rows as A fragments (hi + lo), k-step kk: dims 16 kk + 2t (+1) and + 8
    uint32_t qh[KS][4], ql[KS][4];
    {
        const float* qa = p.q_prime + (okA ? query_row(b, RA, kvh, p.G, p.Hq, p.q_len) : 0) * D;
        const float* qb = p.q_prime + (okB ? query_row(b, RB, kvh, p.G, p.Hq, p.q_len) : 0) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const float2 a0 = okA ? *reinterpret_cast<const float2*>(qa + 16 * kk + 2 * t) : make_float2(0.f, 0.f);
            const float2 a1 = okB ? *reinterpret_cast<const float2*>(qb + 16 * kk + 2 * t) : make_float2(0.f, 0.f);
            const float2 a2 = okA ? *reinterpret_cast<const float2*>(qa + 16 * kk + 2 * t + 8) : make_float2(0.f, 0.f);
            const float2 a3 = okB ? *reinterpret_cast<const float2*>(qb + 16 * kk + 2 * t + 8) : make_float2(0.f, 0.f);
            pf_split(a0.x, a0.y, qh[kk][0], ql[kk][0]);
            pf_split(a1.x, a1.y, qh[kk][1], ql[kk][1]);
            pf_split(a2.x, a2.y, qh[kk][2], ql[kk][2]);
            pf_split(a3.x, a3.y, qh[kk][3], ql[kk][3]);
        }
    }
    float o[NO][4];
#pragma unroll
    for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const float cap2 = p.softcap_log2e;
    bool failed = false;

    for (int it = 0; it < n_st; ++it) {
        const int s = it % NS;
        if (loading && it >= 2 && it - 2 + NS < n_st) loading = issue(it - 2 + NS);
        __syncwarp();
        if (!failed && !ptx::mbar_wait(bar_full + 8 * s, (it / NS) & 1, kWaitLimitCycles)) {
            failed = true;
            if (lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
        }
        const int key0 = (kb0 + it) * kPfKeys;
        // the warp's rows see every key of the block, or some need masks
        const int wlo = r_first + 16 * warp, whi = min(rows - 1, wlo + 15);
        const bool warp_live = valid && wlo < rows && key0 <= L + whi / p.G &&
                               (p.window <= 0 || key0 + kPfKeys - 1 >= L + wlo / p.G - p.window + 1);
        if (!failed && warp_live) {
            const uint32_t sk = base + s * SH::kStageBytes, sv = sk + SH::kHalf;
            const bool full = key0 + kPfKeys - 1 <= L + wlo / p.G &&
                              (p.window <= 0 || key0 >= L + whi / p.G - p.window + 1) && wlo + 15 < rows;
            float sacc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    uint32_t r[4];  // keys 16 jp .. 16 jp + 15, dims 16 kk .. 16 kk + 15
                    ptx::ldsm_x4(r, sk + pf_off(16 * jp + 8 * (lq >> 1) + lr, 2 * kk + (lq & 1)));
                    ptx::mma_bf16(sacc[2 * jp], qh[kk], r[0], r[1]);
                    ptx::mma_bf16(sacc[2 * jp], ql[kk], r[0], r[1]);
                    ptx::mma_bf16(sacc[2 * jp + 1], qh[kk], r[2], r[3]);
                    ptx::mma_bf16(sacc[2 * jp + 1], ql[kk], r[2], r[3]);
                }
            // softcap, masks, the rows' new maxima
            float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = sacc[j][e];
                    if (cap2 > 0.f) v = tanhf(v) * cap2;
                    if (!full) {
                        const int key = key0 + 8 * j + 2 * t + (e & 1);
                        const bool rowA = e < 2;
                        const bool ok = rowA ? (okA && key <= kmaxA && key >= kminA)
                                             : (okB && key <= kmaxB && key >= kminB);
                        if (!ok) v = -INFINITY;
                    }
                    sacc[j][e] = v;
                    if (e < 2) xA = fmaxf(xA, v);
                    else xB = fmaxf(xB, v);
                }
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
            const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
            const float uA = nA == -INFINITY ? 0.f : nA, uB = nB == -INFINITY ? 0.f : nB;
            const float fA = ptx::ex2(mA - uA), fB = ptx::ex2(mB - uB);
            mA = nA;
            mB = nB;
            float sA = 0.f, sB = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sacc[j][0] = ptx::ex2(sacc[j][0] - uA);
                sacc[j][1] = ptx::ex2(sacc[j][1] - uA);
                sacc[j][2] = ptx::ex2(sacc[j][2] - uB);
                sacc[j][3] = ptx::ex2(sacc[j][3] - uB);
                sA += sacc[j][0] + sacc[j][1];
                sB += sacc[j][2] + sacc[j][3];
            }
            lA = lA * fA + sA;
            lB = lB * fB + sB;
#pragma unroll
            for (int n = 0; n < NO; ++n) {
                o[n][0] *= fA;
                o[n][1] *= fA;
                o[n][2] *= fB;
                o[n][3] *= fB;
            }
            // O += P . V, 16 keys per k-step; P's A fragments straight from the accumulators
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                uint32_t ph[4], pl[4];
                pf_split(sacc[2 * k2][0], sacc[2 * k2][1], ph[0], pl[0]);
                pf_split(sacc[2 * k2][2], sacc[2 * k2][3], ph[1], pl[1]);
                pf_split(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1], ph[2], pl[2]);
                pf_split(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3], ph[3], pl[3]);
#pragma unroll
                for (int np = 0; np < NO / 2; ++np) {
                    uint32_t r[4];  // keys 16 k2 .. + 15, dims 16 np .. + 15
                    ptx::ldsm_x4_trans(r, sv + pf_off(16 * k2 + 8 * (lq & 1) + lr, 2 * np + (lq >> 1)));
                    ptx::mma_bf16(o[2 * np], ph, r[0], r[1]);
                    ptx::mma_bf16(o[2 * np], pl, r[0], r[1]);
                    ptx::mma_bf16(o[2 * np + 1], ph, r[2], r[3]);
                    ptx::mma_bf16(o[2 * np + 1], pl, r[2], r[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
    }

    // every issued copy lands before the CTA may exit (a no-op unless a wait failed)
    if (threadIdx.x == 0)
        for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
            if (!ptx::mbar_wait(bar_full + 8 * (i % NS), (i / NS) & 1, kWaitLimitCycles)) {
                atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                break;
            }

    // ---------------------------------------------------------------- the rows
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    // a sequence the append could not take gets zero rows
    auto finish = [&](int R, float m, float l, int e0) {
        if (R >= rows) return;
        const int hq = kvh * p.G + R % p.G;
        const float z = p.sink ? p.sink[hq] * kLog2e : -INFINITY;
        const float M = fmaxf(m, z);
        float scale = 0.f;
        if (M != -INFINITY) {
            const float fm = m == -INFINITY ? 0.f : ptx::ex2(m - M);
            const float den = l * fm + (z == -INFINITY ? 0.f : ptx::ex2(z - M));
            scale = den > 0.f ? fm / den : 0.f;
        }
        const size_t row = query_row(b, R, kvh, p.G, p.Hq, p.q_len) * D;
#pragma unroll
        for (int n = 0; n < NO; ++n) {
            const int d = 8 * n + 2 * t;
            if (p.out_dtype == UAA_DTYPE_F32) {
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + row + d) =
                    make_float2(o[n][e0] * scale, o[n][e0 + 1] * scale);
            } else {
                *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out) + row + d) =
                    __floats2bfloat162_rn(o[n][e0] * scale, o[n][e0 + 1] * scale);
            }
        }
    };
    finish(RA, mA, lA, 0);
    finish(RB, mB, lB, 2);
}

template <int D>
cudaError_t launch_pf(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s)
{
    using SH = PfShape<D>;
    auto kern = prefill_tc_kernel<D>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 31) configured_device_mask |= 1 << dev;
    }
    const long long n_rb = (static_cast<long long>(p.q_len) * p.G + kPfRows - 1) / kPfRows;
    const long long ctas = static_cast<long long>(p.B) * p.Hkv * n_rb;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 2147483647LL) return cudaErrorInvalidConfiguration;
    return launch_dependent(kern, dim3(static_cast<unsigned>(ctas)), dim3(kPfThreads), SH::kSmemBytes, s, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s)
{
    switch (p.D) {
    case 64: return launch_pf<64>(p, tk, tv, s);
    case 128: return launch_pf<128>(p, tk, tv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
