// prefill_umma.cu -- attention of a long chunk of tokens (a prefill chunk) over
// a contiguous bf16 cache on the 5th-generation tensor cores (tcgen05): step 2
// for steps of many tokens per sequence, after the separate append has written
// the chunk's rows and q'.
//
// The (token, head) rows of one kv head (token-major: row r is token r / G,
// query head r % G of the group, as in query_row) are cut into blocks of 128.
// One CTA per (sequence, kv head, row block) streams the keys its rows see (the
// cache and the chunk's tokens up to the block's last one, within the window)
// once, 128 keys per block, and writes the block's output rows itself: no
// records, no combine. The row blocks of one kv head are neighbours in the
// grid, so they read the same tiles at about the same time and HBM delivers
// each tile about once.
//
// Per 128-key block j, with M = 128 rows and N = 128 on the tensor core (the
// shape it runs at full rate; N = 64 takes half again as long per flop):
//   S_j (128 x 128, fp32 in TMEM) = Q' . K_j^T, Q' = the q' rows (fp32, rotated
//     and prescaled by the append) as bf16 hi + lo parts in TMEM (the MMA's A
//     operand; two MMAs per k-step, back to back on the same K chunk), K_j as
//     the TMA wrote it (keys x dims, 128-byte swizzle), so an S MMA reads only
//     K from shared memory;
//   softmax: four threads own row r (TMEM lane r), one per 32-key quarter: they
//     read S_j, apply softcap and the causal / window masks, and keep a
//     running maximum m that they raise only when a logit exceeds it by more
//     than 2^8 (exp2(s - m) <= 256 otherwise; the final division cancels m),
//     rescaling the O row in TMEM then; P_j = exp2(S_j - m) goes back to TMEM
//     as bf16 hi + lo parts (by truncation: 2^-14 relative);
//   O (128 x D, fp32 in TMEM) += P_j . V_j, P_j the MMA's A operand in TMEM,
//     V_j as the TMA wrote it (keys x dims: N-contiguous).
// The MMA warp issues S_{j+1} as soon as the softmax has read S_j into
// registers (one S buffer), and P_j . V_j once P_j is written, so the tensor
// core works while the softmax takes block j; P (one buffer) is written once
// P_{j-1} . V_{j-1} has completed. Keys and values have rings of their own (a
// key tile is free once its S is done, a value tile once its P . V is).
//
// Warps (576 threads, one CTA per SM): warp 0 issues the TMA loads (lane 0 the
// keys, lane 1 the values; full / empty mbarriers, the MMA's commits free the
// slots); warp 1 allocates TMEM and its lane 0 issues every MMA; warps 2-17
// stage the q' rows and run the softmax and the epilogue, four warps per row
// (one per quarter of a block's keys and of O's columns), which exchange row
// maxima and sums through shared memory. Every wait is bounded: a wait that
// gives up sets UAA_DEVFLAG_TIMEOUT, the thread stops waiting from then on, and
// the CTA still drains its copies and MMAs and frees its TMEM before it exits.
#include "internal.cuh"
#include "ptx.cuh"

namespace uaa {
namespace {

constexpr int kUmRows = kPrefillRows;  // query rows per CTA (M of the MMAs)
constexpr int kUmKeys = kPrefillKeys;  // keys per block (N of S, K of P . V)
constexpr int kUmSplit = 4;            // softmax warps per 32-row quarter (threads per row)
constexpr int kUmSoftmax = 4 * 32 * kUmSplit;  // softmax threads
constexpr int kUmThreads = 64 + kUmSoftmax;    // TMA warp, MMA warp, softmax warps
// TMEM columns: S at 0; P at 128 (bf16 hi in the first 64 columns, lo in the
// next 64); O at 256 (D columns); Q' at 384 (bf16 hi in D / 2 columns, lo in
// the next D / 2)
constexpr uint32_t kUmTmemCols = 512;
constexpr uint32_t kUmPCol = 128;
constexpr uint32_t kUmOCol = 256;
constexpr uint32_t kUmQCol = 384;

template <int D>
struct UmShape {
    static constexpr int kBoxes = D / 64;                  // 64-dim boxes of a row
    static constexpr int kTile = kUmKeys * D * 2;          // the keys (or values) of a block
    static constexpr int kKSlots = D == 128 ? 3 : 6;
    static constexpr int kVSlots = D == 128 ? 3 : 6;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKSlots * kTile;
    static constexpr int kOffBar = kOffV + kVSlots * kTile;  // barriers and the TMEM address: 512 bytes
    static constexpr int kOffXch = kOffBar + 512;             // the row exchange: [kUmSplit][128] floats
    static constexpr int kSmemBytes = 1024 + kOffXch + kUmSplit * 4 * kUmRows;
    static_assert(16 * (kKSlots + kVSlots) + 64 <= 512, "barrier area");
};

__device__ __forceinline__ uint32_t um_pack(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// (x0, x1) ~= hi + lo: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void um_split(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = um_pack(x0, x1);
    lo = um_pack(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

// (x0, x1) ~= hi + lo by truncation: hi = the upper 16 bits of x (a bf16), lo =
// the upper 16 bits of x - hi (exact in fp32); |x - hi - lo| < 2^-14 |x|. Integer
// and fp32-add work only, where um_split's conversions share the pipe that
// computes the exponentials.
__device__ __forceinline__ void um_split_trunc(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    const uint32_t h0 = __float_as_uint(x0) & 0xffff0000u, h1 = __float_as_uint(x1) & 0xffff0000u;
    hi = __byte_perm(h0, h1, 0x7632);
    lo = __byte_perm(__float_as_uint(x0 - __uint_as_float(h0)), __float_as_uint(x1 - __uint_as_float(h1)), 0x7632);
}

template <int D>
__global__ void __launch_bounds__(kUmThreads, 1)
prefill_umma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const PrefillParams p)
{
    using SH = UmShape<D>;
    constexpr int NK = SH::kKSlots, NV = SH::kVSlots;
    constexpr int KS = D / 16;       // k-steps of Q'.K^T
    constexpr int KH = kUmKeys / kUmSplit;  // keys per softmax thread and block
    constexpr int CW = D / kUmSplit;        // O columns per softmax thread
    constexpr uint32_t kIdS = ptx::umma_idesc_bf16(kUmRows, kUmKeys, false, false);
    constexpr uint32_t kIdO = ptx::umma_idesc_bf16(kUmRows, D, false, true);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t kring = base + SH::kOffK, vring = base + SH::kOffV;
    const uint32_t bars = base + SH::kOffBar;
    const uint32_t bar_kfull = bars, bar_kempty = bars + 8 * NK;
    const uint32_t bar_vfull = bars + 16 * NK, bar_vempty = bar_vfull + 8 * NV;
    const uint32_t bar_q = bar_vempty + 8 * NV;  // q' rows in TMEM (one arrival per softmax thread)
    const uint32_t bar_s = bar_q + 8;            // S_j in TMEM (MMA commit)
    const uint32_t bar_sfree = bar_s + 8;        // S_j read (one arrival per softmax thread)
    const uint32_t bar_p = bar_sfree + 8;        // P_j in TMEM (one arrival per softmax thread)
    const uint32_t bar_pv = bar_p + 8;           // P_j . V_j done (MMA commit)
    const uint32_t bar_drain = bar_pv + 8;       // every MMA done (MMA commit)
    const uint32_t tmem_slot = bar_drain + 8;
    uint32_t* tmem_slot_ptr = reinterpret_cast<uint32_t*>(smem_raw + (tmem_slot - raw));
    float* xch = reinterpret_cast<float*>(smem_raw + (base + SH::kOffXch - raw));  // [kUmSplit][128]: row maxima / sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = p.q_len * p.G;  // query rows of the kv head
    const int n_rb = (rows + kUmRows - 1) / kUmRows;
    const int rb = blockIdx.x % n_rb;
    const int bk = blockIdx.x / n_rb;  // b * Hkv + kvh
    const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NK; ++s) {
            ptx::mbar_init(bar_kfull + 8 * s, 1);
            ptx::mbar_init(bar_kempty + 8 * s, 1);
        }
        for (int s = 0; s < NV; ++s) {
            ptx::mbar_init(bar_vfull + 8 * s, 1);
            ptx::mbar_init(bar_vempty + 8 * s, 1);
        }
        ptx::mbar_init(bar_q, kUmSoftmax);
        ptx::mbar_init(bar_s, 1);
        ptx::mbar_init(bar_sfree, kUmSoftmax);
        ptx::mbar_init(bar_p, kUmSoftmax);
        ptx::mbar_init(bar_pv, 1);
        ptx::mbar_init(bar_drain, 1);
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kUmTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    grid_dependency_wait();  // the append's rows, q' and lengths are complete
    __syncthreads();         // barriers initialised, TMEM allocated
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot_ptr;
    const uint32_t t_o = tmem + kUmOCol;

    // The chunk's tokens sit at L .. L + q_len - 1 (the append advanced the length
    // past them); a sequence the append could not take keeps its length and gets zero rows.
    const int L_after = p.seq_lens[b];
    const int L = L_after - p.q_len;
    const bool valid = L >= 0 && L_after <= p.cap;
    const int r_first = rb * kUmRows, r_last = min(rows, r_first + kUmRows) - 1;
    const int hi = valid ? L + r_last / p.G + 1 : 0;  // keys the block sees: [lo, hi)
    const int lo = valid && p.window > 0 ? max(0, L + r_first / p.G + 1 - p.window) : 0;
    const int kb0 = lo / kUmKeys;
    const int n_st = (hi + kUmKeys - 1) / kUmKeys - kb0;  // key blocks

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producers
        // lane 0: key tiles into the key ring; lane 1: value tiles into the value ring
        if (lane < 2 && n_st > 0) {
            const bool is_v = lane == 1;
            const int NSL = is_v ? NV : NK;
            const uint32_t ring = is_v ? vring : kring;
            const uint32_t full = is_v ? bar_vfull : bar_kfull, empty = is_v ? bar_vempty : bar_kempty;
            const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
            const int row0 = (b * p.Hkv + kvh) * p.cap + kb0 * kUmKeys;
            int issued = 0;
            for (int i = 0; i < n_st; ++i) {
                const int s = i % NSL;
                if (i >= NSL && !ptx::mbar_wait(empty + 8 * s, ((i / NSL) - 1) & 1, kWaitLimitCycles)) {
                    atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                    break;
                }
                const uint32_t st = ring + s * SH::kTile, bar = full + 8 * s;
                ptx::mbar_arrive_expect_tx(bar, SH::kTile);
#pragma unroll
                for (int c = 0; c < SH::kBoxes; ++c)  // plain loads: the other row blocks read the same tiles from L2
                    ptx::tma_load_2d(st + c * (kUmKeys * 128), tm, c * 64, row0 + i * kUmKeys, bar);
                issued = i + 1;
            }
            // every issued copy lands before the CTA may exit
            for (int i = issued > NSL ? issued - NSL : 0; i < issued; ++i)
                if (!ptx::mbar_wait(full + 8 * (i % NSL), (i / NSL) & 1, kWaitLimitCycles)) {
                    atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                    break;
                }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0 && n_st > 0) {
            bool ok = ptx::mbar_wait(bar_q, 0, kWaitLimitCycles);
            ptx::tc_fence_after();
            // S_j = Q'hi . K_j^T + Q'lo . K_j^T; Q' from TMEM (8 columns per 16 dims), K_j
            // from the ring (hi and lo of one k-step back to back: the tensor core takes
            // a B chunk twice in a row faster than two different ones)
            auto issue_s = [&](int j) {
                const int s = j % NK;
                ok = ok && ptx::mbar_wait(bar_kfull + 8 * s, (j / NK) & 1, kWaitLimitCycles);
                if (!ok) return;
                ptx::tc_fence_after();
                const uint32_t kt = kring + s * SH::kTile;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk)
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint32_t koff = (kk >> 2) * (kUmKeys * 128) + (kk & 3) * 32;
                        ptx::umma_bf16_ts(tmem, tmem + kUmQCol + part * (D / 2) + kk * 8,
                                          ptx::umma_desc(kt + koff, 16, 1024), kIdS, part | kk);
                    }
                ptx::umma_commit(bar_s);
                ptx::umma_commit(bar_kempty + 8 * s);  // the key tile may be refilled
            };
            issue_s(0);
            for (int j = 0; j < n_st && ok; ++j) {
                if (j + 1 < n_st) {  // the S buffer is free once the softmax has read S_j
                    ok = ptx::mbar_wait(bar_sfree, j & 1, kWaitLimitCycles);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_s(j + 1);
                    if (!ok) break;
                }
                const int sv = j % NV;
                ok = ptx::mbar_wait(bar_p, j & 1, kWaitLimitCycles) &&
                     ptx::mbar_wait(bar_vfull + 8 * sv, (j / NV) & 1, kWaitLimitCycles);
                if (!ok) break;
                ptx::tc_fence_after();
                // O += P_j hi . V_j + P_j lo . V_j; P_j from TMEM (8 columns per 16 keys),
                // V_j: keys x dims, dims contiguous
                const uint32_t vt = vring + sv * SH::kTile;
#pragma unroll
                for (int k2 = 0; k2 < kUmKeys / 16; ++k2)
#pragma unroll
                    for (int part = 0; part < 2; ++part)
                        ptx::umma_bf16_ts(t_o, tmem + kUmPCol + part * (kUmKeys / 2) + k2 * 8,
                                          ptx::umma_desc(vt + k2 * 2048, kUmKeys * 128, 1024), kIdO,
                                          (j > 0 || part > 0 || k2 > 0) ? 1u : 0u);
                ptx::umma_commit(bar_pv);
                ptx::umma_commit(bar_vempty + 8 * sv);  // the value tile may be refilled
            }
            if (!ok) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
            // every MMA issued has completed before TMEM is freed
            ptx::umma_commit(bar_drain);
            if (!ptx::mbar_wait(bar_drain, 0, kWaitLimitCycles)) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- softmax + epilogue
        // Warp w (2 <= w < 2 + 4 kUmSplit) takes rows 32 (w % 4) .. + 31 (its TMEM
        // lanes) and key quarter h = (w - 2) / 4 of each block (32 columns of S),
        // so kUmSplit warps share every SM sub-partition's softmax work. The warps
        // of a row quarter exchange row maxima through shared memory and a named
        // barrier, and their partial sums at the end.
        const int h = (warp - 2) >> 2;           // key quarter of a block, and quarter of O's columns
        const int quad = warp & 3;
        const int r = 32 * quad + lane;          // this thread's row and TMEM lane
        const int tid = 32 * (warp - 2) + lane;  // 0 .. kUmSoftmax - 1
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quad) << 16;
        const int quad_bar = 1 + quad;           // named barrier of the row quarter's warps
        const int R = r_first + r;
        const bool row_ok = valid && R < rows;
        const int kmax = L + R / p.G;  // the last key the row sees
        const int kmin = p.window > 0 ? kmax - p.window + 1 : INT_MIN;
        {
            // q' row (this thread: dims CW h .. CW h + CW - 1) as bf16 hi / lo pairs into
            // TMEM, 8 columns (16 dims) at a time (zeros for a missing row)
            const float* q = p.q_prime + (row_ok ? query_row(b, R, kvh, p.G, p.Hq, p.q_len) : 0) * D;
#pragma unroll 1
            for (int c = 0; c < CW / 16; ++c) {
                const int d0 = CW * h + 16 * c;
                uint32_t hh[8], ll[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row_ok) v = *reinterpret_cast<const float4*>(q + d0 + 4 * e);
                    um_split(v.x, v.y, hh[2 * e], ll[2 * e]);
                    um_split(v.z, v.w, hh[2 * e + 1], ll[2 * e + 1]);
                }
                ptx::tmem_st8(tmem + lane_addr + kUmQCol + d0 / 2, hh);
                ptx::tmem_st8(tmem + lane_addr + kUmQCol + D / 2 + d0 / 2, ll);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_q);
        }
        const float cap2 = p.softcap_log2e;
        float m = -INFINITY;  // the running maximum the P values are taken against (the same in both warps)
        float l = 0.f;        // this half's sum of P (relative to m)
        bool ok = true;
        // (tcgen05.ld / st are warp-wide: the branches around them are warp-uniform)
        for (int j = 0; j < n_st; ++j) {
            ok = __all_sync(0xffffffffu, ok && ptx::mbar_wait(bar_s, j & 1, kWaitLimitCycles));
            ptx::tc_fence_after();
            static_assert(KH == 32, "one 32-column TMEM load per thread and block");
            float x[KH];
            {
                uint32_t u[32];
                if (ok) {
                    ptx::tmem_ld32(tmem + lane_addr + KH * h, u);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(u[i]);
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_sfree);  // the S buffer may be overwritten

            const int key0 = (kb0 + j) * kUmKeys + KH * h;  // this thread's first key
            if (cap2 > 0.f) {
#pragma unroll
                for (int i = 0; i < KH; ++i) x[i] = tanhf(x[i]) * cap2;
            }
            if (!(row_ok && key0 + KH - 1 <= kmax && key0 >= kmin)) {  // some keys masked
                const int i_lo = !row_ok ? KH : (p.window > 0 ? kmin - key0 : 0), i_hi = row_ok ? kmax - key0 : -1;
#pragma unroll
                for (int i = 0; i < KH; ++i)
                    if (i < i_lo || i > i_hi) x[i] = -INFINITY;
            }
            float mh;
            {
                float t8[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    t8[a] = x[a];
#pragma unroll
                    for (int i = a + 8; i < KH; i += 8) t8[a] = fmaxf(t8[a], x[i]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) t8[a] = fmaxf(t8[a], t8[a + 4]);
                mh = fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3]));
            }
            // the row's maximum over its quarters (the second barrier: all have read
            // before any writes again)
            xch[h * kUmRows + r] = mh;
            ptx::named_barrier_sync(quad_bar, 32 * kUmSplit);
            float mx = mh;
#pragma unroll
            for (int o = 1; o < kUmSplit; ++o) mx = fmaxf(mx, xch[((h + o) % kUmSplit) * kUmRows + r]);
            ptx::named_barrier_sync(quad_bar, 32 * kUmSplit);

            // raise the reference maximum where a logit exceeds it by more than 2^8
            const bool raise = mx > m + 8.f;
            const float f = raise ? ptx::ex2(m - mx) : 1.f;  // 0 while m = -inf
            const bool rescale = j > 0 && __any_sync(0xffffffffu, raise && m != -INFINITY);
            if (raise) {
                l *= f;
                m = mx;
            }
            const float mu = m == -INFINITY ? 0.f : m;
            {
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < KH; ++i) {
                    x[i] = ptx::ex2(x[i] - mu);
                    s4[i & 3] += x[i];
                }
                l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
            // value rows of keys at or past the sequence's end (unused slots, or another
            // head's rows) may hold anything, NaN included: zero them once they have
            // landed, as P is 0 there
            const int v_keep = L_after - (kb0 + j) * kUmKeys;
            if (v_keep < kUmKeys) {
                const int sv = j % NV;
                ok = __all_sync(0xffffffffu,
                                ok && ptx::mbar_wait(bar_vfull + 8 * sv, (j / NV) & 1, kWaitLimitCycles));
                const uint32_t vt = vring + sv * SH::kTile;
                const int first = max(v_keep, 0), n_chunks = (kUmKeys - first) * SH::kBoxes * 8;
                for (int i = tid; i < n_chunks && ok; i += kUmSoftmax) {
                    const int row = first + i / (SH::kBoxes * 8), rem = i % (SH::kBoxes * 8);
                    ptx::st_shared_v4(vt + (rem >> 3) * (kUmKeys * 128) + row * 128 + (rem & 7) * 16, 0u, 0u, 0u, 0u);
                }
                ptx::fence_proxy_async();  // visible to the tensor core
            }
            // P and O are free once P_{j-1} . V_{j-1} has completed: then the rows' O
            // halves are rescaled (where the maximum rose) and P_j is written
            if (j >= 1)
                ok = __all_sync(0xffffffffu, ok && ptx::mbar_wait(bar_pv, (j - 1) & 1, kWaitLimitCycles));
            ptx::tc_fence_after();
            if (ok && rescale) {  // this thread's CW columns of the O row
#pragma unroll 1
                for (int c = 0; c < CW / 16; ++c) {
                    uint32_t u[16];
                    ptx::tmem_ld16(t_o + lane_addr + CW * h + 16 * c, u);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * f);
                    ptx::tmem_st16(t_o + lane_addr + CW * h + 16 * c, u);
                }
            }
            // P_j (this thread: keys 32 h .. + 31 of its row) as bf16 hi / lo pairs
            if (ok) {
                uint32_t hh[16], lw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) um_split_trunc(x[2 * e], x[2 * e + 1], hh[e], lw[e]);
                const uint32_t tp = tmem + lane_addr + kUmPCol + (KH / 2) * h;
                ptx::tmem_st16(tp, hh);
                ptx::tmem_st16(tp + kUmKeys / 2, lw);
                ptx::tmem_wait_st();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_p);
        }
        if (!ok && lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);

        // ------------------------------------------------------------ the rows
        // the row's sum over its quarters
        xch[h * kUmRows + r] = l;
        ptx::named_barrier_sync(quad_bar, 32 * kUmSplit);
#pragma unroll
        for (int o = 1; o < kUmSplit; ++o) l += xch[((h + o) % kUmSplit) * kUmRows + r];
        // O is complete once the last P . V has (commits complete in order)
        if (n_st > 0) {
            ok = __all_sync(0xffffffffu, ok && ptx::mbar_wait(bar_pv, (n_st - 1) & 1, kWaitLimitCycles));
            ptx::tc_fence_after();
        }
        {
            const int hq = kvh * p.G + R % p.G;
            const float z = p.sink ? p.sink[hq] * kLog2e : -INFINITY;
            const float M = fmaxf(m, z);
            float scale = 0.f;
            if (M != -INFINITY) {
                const float fm = m == -INFINITY ? 0.f : ptx::ex2(m - M);
                const float den = l * fm + (z == -INFINITY ? 0.f : ptx::ex2(z - M));
                scale = den > 0.f ? fm / den : 0.f;
            }
            if (!ok || n_st == 0) scale = 0.f;
            const size_t row = query_row(b, R, kvh, p.G, p.Hq, p.q_len) * D;
#pragma unroll 1
            for (int c = 0; c < CW / 16; ++c) {  // this thread's CW columns, 16 at a time
                const int col = CW * h + 16 * c;
                uint32_t u[16];
                if (ok && n_st > 0) {
                    ptx::tmem_ld16(t_o + lane_addr + col, u);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) u[i] = 0u;
                }
                if (R >= rows) continue;
                if (p.out_dtype == UAA_DTYPE_F32) {
                    float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        o[i] = make_float4(__uint_as_float(u[4 * i]) * scale, __uint_as_float(u[4 * i + 1]) * scale,
                                           __uint_as_float(u[4 * i + 2]) * scale,
                                           __uint_as_float(u[4 * i + 3]) * scale);
                } else {
                    uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row + col);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        o[i] = make_uint4(um_pack(__uint_as_float(u[8 * i]) * scale, __uint_as_float(u[8 * i + 1]) * scale),
                                          um_pack(__uint_as_float(u[8 * i + 2]) * scale, __uint_as_float(u[8 * i + 3]) * scale),
                                          um_pack(__uint_as_float(u[8 * i + 4]) * scale, __uint_as_float(u[8 * i + 5]) * scale),
                                          um_pack(__uint_as_float(u[8 * i + 6]) * scale, __uint_as_float(u[8 * i + 7]) * scale));
                }
            }
        }
    }

    // TMEM is freed by the warp that allocated it, after every reader and the MMAs are done
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kUmTmemCols);
    }
}

template <int D>
cudaError_t launch_um(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s)
{
    using SH = UmShape<D>;
    static_assert(SH::kSmemBytes <= 232448, "shared memory of the prefill kernel");
    auto kern = prefill_umma_kernel<D>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 31) configured_device_mask |= 1 << dev;
    }
    const long long n_rb = (static_cast<long long>(p.q_len) * p.G + kUmRows - 1) / kUmRows;
    const long long ctas = static_cast<long long>(p.B) * p.Hkv * n_rb;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 2147483647LL) return cudaErrorInvalidConfiguration;
    return launch_dependent(kern, dim3(static_cast<unsigned>(ctas)), dim3(kUmThreads), SH::kSmemBytes, s, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill_umma(const PrefillParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s)
{
    switch (p.D) {
    case 64: return launch_um<64>(p, tk, tv, s);
    case 128: return launch_um<128>(p, tk, tv, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace uaa
