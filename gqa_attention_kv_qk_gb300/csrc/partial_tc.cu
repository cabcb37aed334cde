// partial_tc.cu -- split-K decode partial for bf16, vq8 and q8 caches: a persistent,
// warp-specialised kernel with TMA tile loads into a shared-memory ring and
// tensor-core contractions.
//
// Work: the stream-K partition of internal.cuh. P = (SMs x resident CTAs) CTAs
// each take one contiguous range of ring stages across all units (sequence,
// kv head, head group); every query head of the unit's group (up to 8 * NHT) is
// served from the same K/V stage, so each key row leaves HBM once.
//
// With PartialParams.fused the same kernel also performs the append of the
// step (steps 1 and 2 in one launch); otherwise it reads the q' rows that the
// separate append left in the workspace.
//
// Warp roles (192 threads):
//   warp 5 (prep): walks the same segments one ahead of the consumers and
//     writes each segment's q' rows, as bf16 hi + lo fragments, into a shared
//     slot: fused, it normalises, rotates and prescales the unit's q rows
//     itself (lane j takes rotation pairs j + 32 i, both pairings lane-local)
//     and, for the segment that ends a unit, forms the new key row (RMSNorm,
//     rotation, bf16) and value row (bf16, or vq8 codes + scale) into one of
//     two staging slots and, once per kv head, into the cache; the last CTA to
//     have read the lengths advances seq_lens.
//   warp 4 (producer): one lane walks the CTA's segments and streams their
//     stages, TK = 64 MG keys each, with 2-D TMA loads (cp.async.bulk.tensor)
//     into a ring of kStages stages, straight across segment boundaries. bf16
//     key and value boxes are TK rows x 128 bytes with the 128-byte swizzle;
//     int8 code boxes (vq8 / q8 values, q8 keys) are TK rows x min(D, 128) bytes
//     with the 64- or 128-byte swizzle; scales are one TK-float box per row
//     kind. Full / empty mbarriers pass
//     stages between the producer and the consumers.
//   warps 0-3 (consumers): warp w owns keys 16 MG w .. 16 MG (w+1) - 1 of every
//     stage, as MG groups of 16 keys that share one softmax round (MG = 2 for
//     bf16 and 4 for vq8 at head_dim 64, else 1).
//     S^T (16 keys x 8 heads) = K (16 x D) . Q'^T (D x 8) with mma.m16n8k16
//     (keys on M, heads on N: no padding of M). The fp32 q' rows are split into
//     bf16 hi + lo parts, two MMAs each, so the logits keep ~16 significant bits.
//       q8 keys: ldmatrix (not transposed) on the int8 stage hands each thread
//       four consecutive codes of a key row, widened exactly to fp16; the q'
//       parts are fp16 and laid out in the same dim order, and each key's
//       logit is multiplied by its scale after the contraction.
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
//     The warp that owns the new key's row copies the staged rows over that
//     row of the unit's last stage after it lands (the tile load brought
//     whatever the slot held before the step).
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

// Consumer warps come in key groups of four: warp w takes the keys of group w % 4
// of every stage. With one 8-column tile there are four consumer warps; with two
// there are eight, warp w serving tile w / 4, so no warp holds both tiles'
// state. The producer and the prep warp follow the consumers.
constexpr int kKeyGroups = 4;
__host__ __device__ constexpr int consumer_warps(int nht) { return nht == 2 ? 8 : 4; }
__host__ __device__ constexpr int cta_threads(int nht) { return (consumer_warps(nht) + 2) * 32; }

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Cache kinds of the kernel's KV template argument: bf16 keys and values; vq8
// (bf16 keys, int8 value codes + per-key scale); q8 (int8 codes for both).
constexpr int kKvBf16 = 0, kKvVq8 = 1, kKvQ8 = 2;

// MG: 16-key groups each consumer warp takes per stage: where a key costs few
// bytes the consumers, not HBM, set the pace, and MG independent QK chains per
// warp hide their latency. Head_dim 64: 2 for bf16, 4 for vq8 and q8 (one
// 256-key stage); q8 at head_dims 128 and 256: 2 (a q8 key row is half a bf16
// one: with one group its consumers measured 15 % slower); two column tiles at
// head_dim 128: 2 (each key feeds twice the MMAs; one CTA per SM has room for
// three 128-key stages; 6-16 % faster than one group).
template <int D, int KV, int NHT = 1>
struct KeyGroups {
    static constexpr int kMG = D == 64 ? (KV != kKvBf16 ? 4 : 2) : (KV == kKvQ8 || NHT == 2 ? 2 : 1);
};

// Shared memory, from a 1024-byte aligned base: the ring of kStages stages |
// full / empty barriers per stage | q-full, q-empty barriers and the range | stage prefix |
// lengths | q' fragment slot | two new-row staging slots | rotation tables. The ring takes what the
// per-CTA budget leaves (two CTAs per SM below head_dim 256).
template <int D, int KV, int NHT>
struct Shape {
    static constexpr int kD = D;
    static constexpr bool kVQ8 = KV != kKvBf16;              // int8 value codes + scales
    static constexpr bool kKQ8 = KV == kKvQ8;                // int8 key codes + scales
    static constexpr int kMG = KeyGroups<D, KV, NHT>::kMG;
    static constexpr int kTK = kTileKeys * kMG;             // keys per stage
    static constexpr int kHC = 8 * NHT;                     // query heads of a unit
    static constexpr int kBoxBytes = kTK * 128;             // kTK rows x 128 bytes
    static constexpr int kCodeBoxes = D > 128 ? D / 128 : 1;  // boxes of an int8 code row
    static constexpr int kKBoxes = kKQ8 ? kCodeBoxes : D / 64;
    static constexpr int kVBoxes = kVQ8 ? kCodeBoxes : D / 64;
    static constexpr int kKBytes = kKQ8 ? kTK * D : kTK * D * 2;
    static constexpr int kVBytes = kVQ8 ? kTK * D : kTK * D * 2;
    // bytes per row inside one box: 64 for int8 code rows at head_dim 64, else 128
    static constexpr int kKRow = kKQ8 && D == 64 ? 64 : 128;
    static constexpr int kVRow = kVQ8 && D == 64 ? 64 : 128;
    // a stage: keys | values | value scales (int8 values) | key scales (int8 keys)
    static constexpr int kVScaleOff = kKBytes + kVBytes;
    static constexpr int kKScaleOff = kVScaleOff + (kVQ8 ? kTK * 4 : 0);
    static constexpr int kSBytes = (kVQ8 ? kTK * 4 : 0) + (kKQ8 ? kTK * 4 : 0);
    static constexpr int kStageBytes = round_up(kKBytes + kVBytes + kSBytes, 1024);
    static constexpr int kTxBytes = kKBytes + kVBytes + kSBytes;
    static constexpr int kPrefixBytes = round_up((kMaxSliceBatch + 1) * 4, 16);
    static constexpr int kLensBytes = kMaxSliceBatch * 4;
    // q' of one head: D / 2 dim pairs as (bf16x2 hi, bf16x2 lo), rows padded by 32
    // bytes so the 8 rows a warp reads at once fall in distinct banks
    static constexpr int kFragRow = D * 4 + 32;
    static constexpr int kFragBytes = kHC * kFragRow;
    // a new key row (bf16, or int8 codes) at 0, value row (bf16, or int8 codes) at
    // 2 D, then for int8 values the value scale at 3 D and the key scale at 3 D + 4
    static constexpr int kNewRowBytes = round_up(2 * D + (kVQ8 ? D + 8 : 2 * D), 16);
    // q-full and q-empty barriers, then the CTA's range slot, its weights, start, end, go flag
    static constexpr int kCtlBytes = 64;
    // fused append: theta'_p / pi (fp64) and the (cos, sin) of the current sequence, D / 2 each
    static constexpr int kTabBytes = 8 * D;
    // fused append: new key pairs whose fp64 recomputation is deferred (NearQueue)
    static constexpr int kNearBytes = 512;
    static constexpr int kFixedBytes =
        1024 + kCtlBytes + kPrefixBytes + kLensBytes + kFragBytes + 2 * kNewRowBytes + kTabBytes + kNearBytes;
    // one CTA per SM at head_dim 256 and with two column tiles (eight consumer warps)
    static constexpr int kCtaBudget = D == 256 || NHT == 2 ? 227 * 1024 : 228 * 1024 / 2 - 1024;
    static constexpr int kStagesRaw = (kCtaBudget - kFixedBytes) / (kStageBytes + 16);
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static_assert(kStages >= 2, "a ring of at least two stages");
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kSmemBytes = kFixedBytes + kRingBytes + 16 * kStages;
    static_assert(kSmemBytes <= kCtaBudget, "shared memory budget of one CTA");
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

// The same split into fp16 hi + lo parts (|x| below the fp16 range: the P
// weights in [0, 1], or q' rows for int8 keys).
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

// A register from ldmatrix (not transposed) on int8 key rows holds codes
// (key k, dims d .. d+3) in bytes 0-3. Returns the fp16 pairs [(k, d), (k, d+1)]
// and [(k, d+2), (k, d+3)], exactly, by the same mantissa construction.
__device__ __forceinline__ void widen_code_quad(uint32_t r, uint32_t& d01, uint32_t& d23)
{
    const uint32_t u = r ^ 0x80808080u;
    d01 = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4140), 0x64806480u);
    d23 = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4342), 0x64806480u);
}

__device__ __forceinline__ bool key_ok(int k, int lo, int hi) { return k >= lo && k < hi; }

// Once per CTA the prep warp, having issued the reads of its first q rows, lets
// the producer fill the rest of its ring (flag at `go`; the producer issues the
// first stage, then waits for it). Reads issued after the whole first ring
// fill wait behind it in HBM (~30 MB requested at once, 5-8 us); behind one
// stage per CTA they land in ~1.5 us. A flag rather than a barrier: bar.sync
// would wait for the reads to land.
__device__ __forceinline__ void release_producer(uint32_t go, int lane)
{
    if (lane == 0) ptx::flag_set(go, 1u);  // no __syncwarp: it too would wait for the reads
}

// fp16 hi + lo parts of x into element e of a q' fragment row (the operands of
// a q8 cache's int8 keys, which widen to fp16).
__device__ __forceinline__ void store_frag_f16(uint8_t* row, int e, float x)
{
    const __half h = __float2half_rn(x);
    const __half l = __float2half_rn(x - __half2float(h));
    *reinterpret_cast<__half*>(row + (e >> 1) * 8 + (e & 1) * 2) = h;
    *reinterpret_cast<__half*>(row + (e >> 1) * 8 + 4 + (e & 1) * 2) = l;
}

// bf16 hi + lo parts of x into element e of a q' fragment row.
__device__ __forceinline__ void store_frag(uint8_t* row, int e, float x)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    *reinterpret_cast<__nv_bfloat16*>(row + (e >> 1) * 8 + (e & 1) * 2) = h;
    *reinterpret_cast<__nv_bfloat16*>(row + (e >> 1) * 8 + 4 + (e & 1) * 2) = l;
}

// Prep warp, fused append: q' rows of the unit's heads h0 .. h0 + nh - 1 of
// sequence b (RMSNorm, rotation, logit prescale) into the fragment slot; lane
// takes rotation pairs lane + 32 j. When new_seq, (cos, sin) of position pos
// for pair i go to cs[i] first (from theta'_i / pi in freq[i]), while the rows'
// reads are in flight. Rows of missing heads are zero.
// The reads of eight rows go out together; their values are parked in the
// fragment rows (element e as fp32 at byte 4 e, the bytes its hi / lo pair
// takes later) and each head is then finished in a rolled loop: at a launch's
// start this code runs cold, and an unrolled body cost microseconds of
// instruction fetch. F16: fp16 hi / lo parts (for int8 keys), else bf16.
template <int D, int HC, typename T, bool F16>
__device__ void prep_fused_q(const PartialParams& p, int b, int h0, int nh, bool write_rot, bool new_seq, int pos,
                             const double* freq, float2* cs, uint8_t* frag, int row_bytes, uint32_t go, int lane)
{
    constexpr int NP = D / 64;
    int ia[NP], ib[NP];  // the row elements of this lane's pairs
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int2 e = rope_pair(lane + 32 * j, p.half_rot, D, p.style == UAA_ROPE_NEOX);
        ia[j] = e.x;
        ib[j] = e.y;
    }
#pragma unroll 1
    for (int hc0 = 0; hc0 < HC; hc0 += 8) {
        float xa[8][NP], xb[8][NP];
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // all eight rows' loads first
            const size_t qoff = (static_cast<size_t>(b) * p.Hq + h0 + hc0 + i) * D;
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                xa[i][j] = hc0 + i < nh ? load_as_float<T>(p.q, qoff + ia[j]) : 0.f;
                xb[i][j] = hc0 + i < nh ? load_as_float<T>(p.q, qoff + ib[j]) : 0.f;
            }
        }
        if (go && hc0 == 0) release_producer(go, lane);  // the first loads are issued: the key stream may start
        if (new_seq && hc0 == 0) {  // the rows' loads are in flight: (cos, sin) of this sequence's position
#pragma unroll 1
            for (int j = 0; j < NP; ++j)
                cs[lane + 32 * j] = rope_pair_cos_sin(lane + 32 * j, p.half_rot, pos, freq[lane + 32 * j], p.mscale);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float* raw = reinterpret_cast<float*>(frag + (hc0 + i) * row_bytes);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                raw[ia[j]] = xa[i][j];
                raw[ib[j]] = xb[i][j];
            }
        }
        __syncwarp();
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            uint8_t* row = frag + (hc0 + i) * row_bytes;
            const float* raw = reinterpret_cast<const float*>(row);
            const bool hv = hc0 + i < nh;
            float ya[NP], yb[NP];
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                ya[j] = raw[ia[j]];
                yb[j] = raw[ib[j]];
            }
            __syncwarp();  // every lane has its values before any writes fragments over them
            if (p.qk_norm && hv) {
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < NP; ++j) ss += ya[j] * ya[j] + yb[j] * yb[j];
                const float inv = rms_inv(warp_sum(ss), D, p.eps);
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    ya[j] = ya[j] * inv * (p.q_norm_w[ia[j]] + p.norm_offset);
                    yb[j] = yb[j] * inv * (p.q_norm_w[ib[j]] + p.norm_offset);
                }
            }
            const size_t qoff = (static_cast<size_t>(b) * p.Hq + h0 + hc0 + i) * D;
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                if (hv) rope_rotate(ya[j], yb[j], cs[lane + 32 * j]);
                if (write_rot && hv) {
                    p.q_rot_out[qoff + ia[j]] = ya[j];
                    p.q_rot_out[qoff + ib[j]] = yb[j];
                }
                if (F16) {
                    store_frag_f16(row, ia[j], ya[j] * p.qscale);
                    store_frag_f16(row, ib[j], yb[j] * p.qscale);
                } else {
                    store_frag(row, ia[j], ya[j] * p.qscale);
                    store_frag(row, ib[j], yb[j] * p.qscale);
                }
            }
        }
    }
}

// Prep warp, separate append: the workspace's q' rows (already rotated and
// prescaled, fp32) into the fragment slot, eight rows' loads at a time (fp16
// parts for int8 keys when F16).
template <int D, int HC, bool F16>
__device__ __forceinline__ void prep_loaded_q(const PartialParams& p, int b, int kvh, int r0, int nh, uint8_t* frag,
                                              int row_bytes, uint32_t go, int lane)
{
#pragma unroll 1
    for (int hc0 = 0; hc0 < HC; hc0 += 8) {
        float2 x[8][D / 64];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float* qrow =
                p.q_prime + (hc0 + i < nh ? query_row(b, r0 + hc0 + i, kvh, p.G, p.Hq, p.q_len) : 0) * D;
#pragma unroll
            for (int j = 0; j < D / 64; ++j)
                x[i][j] = hc0 + i < nh ? *reinterpret_cast<const float2*>(qrow + 2 * lane + 64 * j)
                                       : make_float2(0.f, 0.f);
        }
        if (go && hc0 == 0) release_producer(go, lane);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                uint32_t h, l;
                if (F16)
                    split_f16(x[i][j].x, x[i][j].y, h, l);
                else
                    split_bf16(x[i][j].x, x[i][j].y, h, l);
                *reinterpret_cast<uint2*>(frag + (hc0 + i) * row_bytes + (lane + 32 * j) * 8) = make_uint2(h, l);
            }
    }
}

// Starts bringing the new k and v rows of (b, kvh) into L2 (their loads follow
// the q rows' processing).
template <int D>
__device__ __forceinline__ void prefetch_new_rows(const PartialParams& p, int b, int kvh, int lane)
{
    const int bytes = D * (p.io_dtype == UAA_DTYPE_F32 ? 4 : 2);
    const size_t off = (static_cast<size_t>(b) * p.Hkv + kvh) * bytes;
    if (lane < 2 * bytes / 128) {
        const int row = lane >= bytes / 128 ? 1 : 0;
        const char* src = static_cast<const char*>(row ? p.v_new : p.k_new) + off + 128 * (lane - row * (bytes / 128));
        ptx::prefetch_l2_keep(src);
    }
}

// Prep warp, fused append: the new key row (RMSNorm, rotation, then bf16, or
// int8 codes and scale for q8) and value row (bf16, or int8 codes and scale) of
// (b, kvh) into a staging slot (key at 0, value at 2 D, value scale at 3 D, key
// scale at 3 D + 4), and into the cache at slot L when `store`.
// New key pairs (fused append) whose fp32 rotation lies near a bf16 rounding
// boundary: the staged row keeps the fp32 rounding (the step's own attention
// uses it, an ulp at most away), and after its last segment the prep warp
// recomputes each queued pair in fp64 and writes it over the cache's copy, so
// that the cache holds the exact value's rounding. A full queue recomputes at once.
struct NearEntry {
    size_t slot;   // the cache row (element index of its first element)
    int src;       // the raw row in k_new (element index), slice-relative
    int pos;       // the token's position
    short ia, ib, pp, pad;
};
struct NearQueue {
    int n;
    int pad[3];
    NearEntry e[20];
};
static_assert(sizeof(NearQueue) <= 512, "the near-key queue's shared memory");

template <int D, typename T>
__device__ void fix_near_keys(const PartialParams& p, NearQueue* q, int lane)
{
    constexpr int EPL = D / 32;
    constexpr int kCap = static_cast<int>(sizeof(q->e) / sizeof(q->e[0]));
    static_assert(kCap <= 32, "one lane per queued pair");
    const int n = q->n;
    // the rows' fp64 norm factors (a whole-warp reduction per distinct row; lane i
    // keeps entry i's), then every pair at once, one per lane
    double inv64 = 0.0;
    if (p.qk_norm) {
        int last_src = -1;
        double last_inv = 0.0;
        for (int i = 0; i < n; ++i) {
            const int src = q->e[i].src;
            if (src != last_src) {
                double raw[EPL];
#pragma unroll
                for (int k = 0; k < EPL; ++k) raw[k] = load_as_float<T>(p.k_new, static_cast<size_t>(src) + lane + 32 * k);
                last_inv = rms_inv64<EPL>(raw, D, p.eps);
                last_src = src;
            }
            if (lane == i) inv64 = last_inv;
        }
    }
    if (lane < n) {
        const NearEntry e = q->e[lane];
        const double wa = p.qk_norm ? static_cast<double>(p.k_norm_w[e.ia]) + p.norm_offset : 1.0;
        const double wb = p.qk_norm ? static_cast<double>(p.k_norm_w[e.ib]) + p.norm_offset : 1.0;
        __nv_bfloat16 ha, hb;
        key_pair_exact(load_as_float<T>(p.k_new, static_cast<size_t>(e.src) + e.ia),
                       load_as_float<T>(p.k_new, static_cast<size_t>(e.src) + e.ib), wa, wb, inv64,
                       rope_cos_sin64(e.pp, p.half_rot, e.pos, p.inv_freq_over_pi[e.pp], p.mscale64), ha, hb);
        __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(p.k_cache) + e.slot;
        kc[e.ia] = ha;
        kc[e.ib] = hb;
    }
    __syncwarp();
    if (lane == 0) q->n = 0;
    __syncwarp();
}

template <int D, int KV, typename T>
__device__ void prep_new_rows(const PartialParams& p, int b, int kvh, int L, const float2* cs, uint8_t* staging,
                              bool store, int lane, NearQueue* nearq)
{
    constexpr bool VQ8 = KV != kKvBf16, KQ8 = KV == kKvQ8;
    constexpr int NP = D / 64;   // rotation pairs per lane
    constexpr int EPL = D / 32;  // values per lane
    const size_t src = (static_cast<size_t>(b) * p.Hkv + kvh) * D;
    const long long crow = cache_row(p.pages, p.Hkv, p.cap, p.b_off + b, kvh, L);
    if (crow < 0) {  // a paged table entry out of range: the rows are staged, not stored
        if (store && lane == 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
        store = false;
    }
    const size_t slot = crow < 0 ? 0 : static_cast<size_t>(crow);
    float ka[NP], kb[NP], v[EPL];
    int ia[NP], ib[NP];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int2 e = rope_pair(lane + 32 * j, p.half_rot, D, p.style == UAA_ROPE_NEOX);
        ia[j] = e.x;
        ib[j] = e.y;
        ka[j] = load_as_float<T>(p.k_new, src + ia[j]);
        kb[j] = load_as_float<T>(p.k_new, src + ib[j]);
        ss += ka[j] * ka[j] + kb[j] * kb[j];
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) v[i] = load_as_float<T>(p.v_new, src + lane + 32 * i);
    if (p.qk_norm) {
        const float inv = rms_inv(warp_sum(ss), D, p.eps);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            ka[j] = ka[j] * inv * (p.k_norm_w[ia[j]] + p.norm_offset);
            kb[j] = kb[j] * inv * (p.k_norm_w[ib[j]] + p.norm_offset);
        }
    }
    float ka0[NP], kb0[NP];  // before the rotation
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        ka0[j] = ka[j];
        kb0[j] = kb[j];
        rope_rotate(ka[j], kb[j], cs[lane + 32 * j]);
    }
    if (KQ8) {  // the rotated row's codes, by the vq8 rule over the whole row
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) amax = fmaxf(amax, fmaxf(fabsf(ka[j]), fabsf(kb[j])));
        const float sc = vq8_scale(warp_max(amax));
        int8_t* ks = reinterpret_cast<int8_t*>(staging);
        int8_t* kc = static_cast<int8_t*>(p.k_cache) + slot * D;
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const int8_t ca = vq8_code(ka[j], sc), cb = vq8_code(kb[j], sc);
            ks[ia[j]] = ca;
            ks[ib[j]] = cb;
            if (store) {
                kc[ia[j]] = ca;
                kc[ib[j]] = cb;
            }
        }
        if (lane == 0) {
            *reinterpret_cast<float*>(staging + 3 * D + 4) = sc;
            if (store) p.k_scale[slot] = sc;
        }
    } else {
        // rounded as the exact values (bf16_near_boundary): the rare pair near a
        // rounding boundary again in fp64
        __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(staging);
        __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(p.k_cache) + slot * D;
        __nv_bfloat16 hka[NP], hkb[NP];
        bool near[NP], any = false;
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            hka[j] = __float2bfloat16_rn(ka[j]);
            hkb[j] = __float2bfloat16_rn(kb[j]);
            const float eb = key_error_bound(ka0[j], kb0[j], cs[lane + 32 * j], p.qk_norm != 0);
            near[j] = bf16_near_boundary(ka[j], eb) || bf16_near_boundary(kb[j], eb);
            any |= near[j];
        }
        // the cache's copy of a near pair is recomputed later (NearQueue); a row that
        // is only staged (not stored) needs nothing more
        if (store && __any_sync(0xffffffffu, any)) {
            int cnt = 0;
#pragma unroll
            for (int j = 0; j < NP; ++j) cnt += near[j] ? 1 : 0;
            int incl = cnt;  // inclusive prefix over the lanes
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            int n0 = nearq->n;
            if (n0 + total > static_cast<int>(sizeof(nearq->e) / sizeof(nearq->e[0]))) {
                fix_near_keys<D, T>(p, nearq, lane);  // full: the queued pairs first
                n0 = 0;
            }
            if (n0 + total <= static_cast<int>(sizeof(nearq->e) / sizeof(nearq->e[0]))) {
                int at = n0 + incl - cnt;
#pragma unroll
                for (int j = 0; j < NP; ++j)
                    if (near[j]) {
                        NearEntry& e = nearq->e[at++];
                        e.slot = slot * D;
                        e.src = static_cast<int>(src);
                        e.pos = L;
                        e.ia = static_cast<short>(ia[j]);
                        e.ib = static_cast<short>(ib[j]);
                        e.pp = static_cast<short>(lane + 32 * j);
                    }
                __syncwarp();
                if (lane == 0) nearq->n = n0 + total;
                __syncwarp();
            }
        }
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const __nv_bfloat16 ha = hka[j], hb = hkb[j];
            ks[ia[j]] = ha;
            ks[ib[j]] = hb;
            if (store) {
                kc[ia[j]] = ha;
                kc[ib[j]] = hb;
            }
        }
    }
    if (VQ8) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const float sc = vq8_scale(warp_max(amax));
        int8_t* vs = reinterpret_cast<int8_t*>(staging + 2 * D);
        int8_t* vc = static_cast<int8_t*>(p.v_cache) + slot * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int8_t code = vq8_code(v[i], sc);
            vs[lane + 32 * i] = code;
            if (store) vc[lane + 32 * i] = code;
        }
        if (lane == 0) {
            *reinterpret_cast<float*>(staging + 3 * D) = sc;
            if (store) p.v_scale[slot] = sc;
        }
    } else {
        __nv_bfloat16* vs = reinterpret_cast<__nv_bfloat16*>(staging + 2 * D);
        __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(p.v_cache) + slot * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v[i]);
            vs[lane + 32 * i] = h;
            if (store) vc[lane + 32 * i] = h;
        }
    }
}

// Fused append, one thread per CTA, after the CTA's lengths are in shared
// memory: counts the CTA in; the last CTA of the grid to do so (every other CTA
// has read seq_lens by then) advances each length whose token fitted. The
// counter wraps to zero on the last arrival, ready for the next launch.
__device__ __noinline__ void count_in_and_advance(const PartialParams& p, const int* lens)
{
    __threadfence();
    if (atomicInc(p.arrivals, gridDim.x - 1) != gridDim.x - 1) return;
    __threadfence();
    for (int b = 0; b < p.B; ++b)
        if (lens[b] >= 0 && lens[b] < p.cap) p.seq_lens[b] = lens[b] + 1;
}

// Producer: the TMA loads of `n` consecutive cache rows starting at row y (key
// and value rows, their scales at (sx, sy) of the scale tensors) into rows r0 ..
// r0 + n - 1 of a stage; n is the tensor maps' box height.
template <class SH>
__device__ __forceinline__ void issue_rows(uint32_t st, int r0, const CUtensorMap* tk, const CUtensorMap* tv,
                                           const CUtensorMap* ts, const CUtensorMap* tks, int y, int sx, int sy,
                                           uint32_t bar, uint64_t policy)
{
#pragma unroll
    for (int c = 0; c < SH::kKBoxes; ++c)
        ptx::tma_load_2d_hint(st + c * SH::kBoxBytes + r0 * SH::kKRow, tk, c * (SH::kKQ8 ? 128 : 64), y, bar, policy);
    if (SH::kKQ8) ptx::tma_load_2d_hint(st + SH::kKScaleOff + 4 * r0, tks, sx, sy, bar, policy);
#pragma unroll
    for (int c = 0; c < SH::kVBoxes; ++c)
        ptx::tma_load_2d_hint(st + SH::kKBytes + c * SH::kBoxBytes + r0 * SH::kVRow, tv, c * (SH::kVQ8 ? 128 : 64),
                              y, bar, policy);
    if (SH::kVQ8) ptx::tma_load_2d_hint(st + SH::kVScaleOff + 4 * r0, ts, sx, sy, bar, policy);
}

// Owner warp of the new key: the staged rows over row r of the loaded stage.
template <class SH>
__device__ __forceinline__ void patch_stage_row(const uint8_t* staging, uint8_t* stage, int r, int lane)
{
    constexpr int D = SH::kD;
    constexpr int TK = SH::kTK;
    if (SH::kKQ8) {
        for (int c = lane; c < D / 16; c += 32)
            *reinterpret_cast<uint4*>(stage + code_off<D, TK>(r, c)) = *reinterpret_cast<const uint4*>(staging + 16 * c);
        if (lane == 0)
            *reinterpret_cast<float*>(stage + SH::kKScaleOff + 4 * r) = *reinterpret_cast<const float*>(staging + 3 * D + 4);
    } else {
        for (int c = lane; c < D / 8; c += 32)
            *reinterpret_cast<uint4*>(stage + tile_off<TK>(r, c)) = *reinterpret_cast<const uint4*>(staging + 16 * c);
    }
    if (SH::kVQ8) {
        for (int c = lane; c < D / 16; c += 32)
            *reinterpret_cast<uint4*>(stage + SH::kKBytes + code_off<D, TK>(r, c)) =
                *reinterpret_cast<const uint4*>(staging + 2 * D + 16 * c);
        if (lane == 0)
            *reinterpret_cast<float*>(stage + SH::kVScaleOff + 4 * r) = *reinterpret_cast<const float*>(staging + 3 * D);
    } else {
        for (int c = lane; c < D / 8; c += 32)
            *reinterpret_cast<uint4*>(stage + SH::kKBytes + tile_off<TK>(r, c)) =
                *reinterpret_cast<const uint4*>(staging + 2 * D + 16 * c);
    }
    __syncwarp();
}

template <int D, int KV, int NHT>
__global__ void __launch_bounds__(cta_threads(NHT), (D == 256 || NHT == 2 ? 1 : 2))
partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_ks,
                  const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
                  const __grid_constant__ CUtensorMap tm_st, const __grid_constant__ CUtensorMap tm_kst,
                  const PartialParams p)
{
    using SH = Shape<D, KV, NHT>;
    constexpr bool VQ8 = SH::kVQ8;  // int8 value codes
    constexpr bool KQ8 = SH::kKQ8;  // int8 key codes
    constexpr int MG = SH::kMG;     // 16-key groups per warp per stage
    constexpr int TK = SH::kTK;     // keys per stage
    constexpr int KS = D / 16;      // k-steps of QK, m-tiles of PV
    constexpr int HC = 8 * NHT;     // head columns of a unit
    constexpr int CW = consumer_warps(NHT);          // consumer warps
    constexpr int NTW = NHT * kKeyGroups / CW;       // 8-column tiles per consumer warp
    constexpr int kProducerWarp = CW, kPrepWarp = CW + 1;
    // merge scratch (inside one stage): all of D at once if it fits, else halves or quarters
    constexpr int kScratchRow = 2 * kKeyGroups * HC * 4;
    constexpr int RC = kKeyGroups * HC * (D + 4) * 4 + kScratchRow <= SH::kStageBytes       ? D
                       : kKeyGroups * HC * (D / 2 + 4) * 4 + kScratchRow <= SH::kStageBytes ? D / 2
                                                                                           : D / 4;
    static_assert(kKeyGroups * HC * (RC + 4) * 4 + kScratchRow <= SH::kStageBytes,
                  "merge scratch must fit in one stage");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t bar_full = base + SH::kRingBytes;
    const uint32_t bar_empty = bar_full + 8 * SH::kStages;
    const uint32_t bar_qfull = bar_empty + 8 * SH::kStages;  // prep warp -> consumers: a segment's q' is ready
    const uint32_t bar_qempty = bar_qfull + 8;               // consumers -> prep warp: the q' slot is free
    // control block: barriers at 0 and 8; slot 16; weights 20-28; range start 32, end 40; go flag 48;
    // staging-ready flags 56, 60
    uint8_t* ctl = base_ptr + SH::kRingBytes + 16 * SH::kStages;
    const uint32_t go = ptx::smem_u32(ctl + 48);  // release_producer's flag (never 0 as an address)
    const uint32_t rows_ready = ptx::smem_u32(ctl + 56);  // [2]: segment + 1 whose new rows staging slot i holds
    int* prefix = reinterpret_cast<int*>(ctl + SH::kCtlBytes);
    int* lens = prefix + SH::kPrefixBytes / 4;
    uint8_t* frag = reinterpret_cast<uint8_t*>(lens) + SH::kLensBytes;
    uint8_t* staging = frag + SH::kFragBytes;  // two slots of kNewRowBytes, by segment parity
    double* freq_s = reinterpret_cast<double*>(staging + 2 * SH::kNewRowBytes);  // [D / 2] theta'_p / pi
    float2* cs_s = reinterpret_cast<float2*>(freq_s + D / 2);                    // [D / 2] (cos, sin)
    NearQueue* nearq = reinterpret_cast<NearQueue*>(cs_s + D / 2);               // deferred key pairs

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.Hkv * p.head_groups;
    if (threadIdx.x == 0) {  // shared-memory set-up overlaps the previous kernel's tail
        for (int s = 0; s < SH::kStages; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, CW);
        }
        ptx::mbar_init(bar_qfull, 1);
        ptx::mbar_init(bar_qempty, CW);
        ptx::flag_set(go, 0u);
        ptx::flag_set(rows_ready, 0u);
        ptx::flag_set(rows_ready + 4, 0u);
        nearq->n = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32 * kProducerWarp) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        if (VQ8) ptx::prefetch_tensormap(&tm_s);
        if (KQ8) ptx::prefetch_tensormap(&tm_ks);
        if (MG > 1 && !p.pages.table) {  // the 64-key maps of units' partial last stages
            ptx::prefetch_tensormap(&tm_kt);
            ptx::prefetch_tensormap(&tm_vt);
            if (VQ8) ptx::prefetch_tensormap(&tm_st);
            if (KQ8) ptx::prefetch_tensormap(&tm_kst);
        }
    }
    grid_dependency_wait();  // the step's inputs (and a separate append's rows) are complete
    if (p.fused && threadIdx.x >= 32 && threadIdx.x < 32 + D / 2)  // the rotation table, while warp 0 scans
        freq_s[threadIdx.x - 32] = p.inv_freq_over_pi[threadIdx.x - 32];
    if (threadIdx.x == 32 * kPrepWarp) {  // the range slot, while warp 0 scans the lengths
        unsigned w0, w1, wP;
        const int v = claim_slot(p, w0, w1, wP);
        if (v < 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);  // slots left claimed by an unfinished launch
        *reinterpret_cast<int*>(ctl + 16) = v;
        *reinterpret_cast<unsigned*>(ctl + 20) = w0;
        *reinterpret_cast<unsigned*>(ctl + 24) = w1;
        *reinterpret_cast<unsigned*>(ctl + 28) = wP;
    }
    build_stage_prefix(p.seq_lens, p.B, p.window, p.cap, MG, units, prefix, lens,
                       blockIdx.x == 0 ? p.prefix : nullptr, blockIdx.x == 0 ? p.status : nullptr, p.fused != 0,
                       p.max_len, blockIdx.x == 0 ? p.owners : nullptr);  // ends with __syncthreads
    unsigned long long t_begin = 0;
    if (threadIdx.x == 0) {
        long long rs, re;
        slot_range(p, *reinterpret_cast<const int*>(ctl + 16), *reinterpret_cast<const unsigned*>(ctl + 20),
                   *reinterpret_cast<const unsigned*>(ctl + 24), *reinterpret_cast<const unsigned*>(ctl + 28),
                   prefix[p.B], rs, re);
        *reinterpret_cast<long long*>(ctl + 32) = rs;
        *reinterpret_cast<long long*>(ctl + 40) = re;
        t_begin = global_time_ns();
    }
    __syncthreads();
    const int slot = *reinterpret_cast<const int*>(ctl + 16);
    const long long s_c = *reinterpret_cast<const long long*>(ctl + 32);
    const long long e_c = *reinterpret_cast<const long long*>(ctl + 40);
    // Fused append: every CTA counts in once its lengths are read (an active CTA's
    // producer does so after its first ring fill, off the consumers' path); the
    // last to count in advances seq_lens once its own work is issued.
    if (e_c <= s_c) {  // uniform over the CTA: no stages
        // a claimed slot always leaves a rate (0: nothing measured), so the combine
        // never reads bytes of another launch geometry as one
        if (threadIdx.x == 0 && slot >= 0) p.bal.rate[slot] = 0.f;
        if (threadIdx.x == 0 && p.fused) count_in_and_advance(p, lens);
        return;
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            bool counted = false;  // fused: this CTA has counted in
            int it = 0;            // stages issued
            const uint64_t stream_policy = ptx::l2_evict_first_policy();  // keys and values are read once
            for (long long pos = s_c; pos < e_c && ok;) {
                const Segment sg = segment_at(prefix, lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c,
                                              p.fused != 0);
                const int head_row = (p.b_off + sg.b) * p.Hkv + sg.kvh;
                const int row0 = p.pages.table ? 0 : head_row * p.cap;  // contiguous caches
                const int t0 = sg.lo / kTileKeys;
                for (int k = 0; k < sg.n_st; ++k, ++it) {
                    const int s = it % SH::kStages;
                    if (it == 1 && !ptx::flag_wait(go, kWaitLimitCycles)) {
                        // the first stage is on its way; the rest of the ring follows the prep
                        // warp's first q reads (release_producer)
                        atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (p.fused && !counted && it == SH::kStages) {  // the ring is full: wait time
                        count_in_and_advance(p, lens);
                        counted = true;
                    }
                    if (it >= SH::kStages &&
                        !ptx::mbar_wait(bar_empty + 8 * s, ((it / SH::kStages) & 1) ^ 1, kWaitLimitCycles)) {
                        atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + s * SH::kStageBytes;
                    const uint32_t bar = bar_full + 8 * s;
                    const int key = (t0 + MG * (sg.st0 + k)) * kTileKeys;
                    // 64-key tiles of this stage up to the unit's last visible key: a unit's
                    // last stage may need fewer than MG (its other rows are masked)
                    const int nt = MG > 1 ? min(MG, (sg.hi - key + kTileKeys - 1) / kTileKeys) : MG;
                    if (!p.pages.table && nt < MG) {
                        ptx::mbar_arrive_expect_tx(bar, nt * (SH::kTxBytes / MG));
                        for (int r0 = 0; r0 < nt * kTileKeys; r0 += kTileKeys)
                            issue_rows<SH>(st, r0, &tm_kt, &tm_vt, &tm_st, &tm_kst, row0 + key + r0, key + r0,
                                           head_row, bar, stream_policy);
                    } else if (!p.pages.table) {
                        ptx::mbar_arrive_expect_tx(bar, SH::kTxBytes);
                        issue_rows<SH>(st, 0, &tm_k, &tm_v, &tm_s, &tm_ks, row0 + key, key, head_row, bar,
                                       stream_policy);
                    } else {
                        ptx::mbar_arrive_expect_tx(bar, SH::kTxBytes);
                        // paged: one load per page-aligned sub-tile; a sub-tile with no visible key
                        // (beyond the unit's end or before its window) is not looked up and reads
                        // as zeros from a negative row (masked by the consumers)
                        const int sub = min(1 << p.pages.shift, kTileKeys);
                        for (int r0 = 0; r0 < TK; r0 += sub) {
                            const int ku = key + r0;
                            long long row = -1;
                            if (ku < sg.hi && ku + sub > sg.lo) {
                                row = cache_row(p.pages, p.Hkv, p.cap, p.b_off + sg.b, sg.kvh, ku);
                                if (row < 0) atomicOr(p.status, UAA_DEVFLAG_PAGE);
                            }
                            const int ps_mask = (1 << p.pages.shift) - 1;
                            issue_rows<SH>(st, r0, &tm_k, &tm_v, &tm_s, &tm_ks, row < 0 ? -sub : static_cast<int>(row),
                                           row < 0 ? 0 : static_cast<int>(row & ps_mask),
                                           row < 0 ? -1 : static_cast<int>(row >> p.pages.shift), bar, stream_policy);
                        }
                    }
                }
                pos += sg.n_st;
            }
            if (p.fused && !counted) count_in_and_advance(p, lens);
            // Every copy this thread issued lands before the CTA may exit, also after a
            // failed wait (then the consumers no longer wait for them): the last kStages
            // issued stages are the only ones not yet consumed, and once the producer
            // stops no barrier starts a new phase, so a phase that completed earlier
            // reads as complete. Bounded: a copy that never lands ends the wait.
            const int first = it > SH::kStages ? it - SH::kStages : 0;
            for (int i = first; i < it; ++i)
                if (!ptx::mbar_wait(bar_full + 8 * (i % SH::kStages), (i / SH::kStages) & 1, kWaitLimitCycles)) {
                    atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                    break;
                }
        }
        return;
    }

    if (warp == kPrepWarp) {
        // ------------------------------------------------------------ prep
        // One segment ahead of the consumers: segment i's q' fragments (and, when
        // the segment ends its unit and the new token fits, the new k / v rows in
        // staging slot i mod 2) are written once the consumers have taken segment
        // i - 1's fragments (which also means segment i - 2 is finished).
        int cs_b = -1;  // the sequence whose (cos, sin) are in cs_s
        int seg = 0;
        for (long long pos = s_c; pos < e_c; ++seg) {
            const Segment sg = segment_at(prefix, lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c,
                                          p.fused != 0);
            if (seg > 0 && !ptx::mbar_wait(bar_qempty, (seg - 1) & 1, kWaitLimitCycles)) {
                if (lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                break;
            }
            const int r0 = sg.hg * HC;                     // the unit's first query row
            const int h0 = sg.kvh * p.G + r0;              // its query head (one token per sequence)
            const int nh = min(HC, p.q_len * p.G - r0);    // its query rows
            if (lane == 0) {  // this range's part in the unit's owners, for the combine
                unsigned* own = p.owners + 2 * (static_cast<size_t>(sg.b) * units + sg.kvh * p.head_groups + sg.hg);
                if (sg.st0 == 0) own[0] = (static_cast<unsigned>(slot) + 1u) | (pos == s_c ? 0x80000000u : 0u);
                if (sg.st0 + sg.n_st == sg.stages) own[1] = static_cast<unsigned>(slot) + 1u;
            }
            if (p.fused) {
                const int L = lens[sg.b];
                const bool fits = L >= 0 && L < p.cap;
                const bool ends = fits && sg.st0 + sg.n_st == sg.stages;
                if (ends) prefetch_new_rows<D>(p, sg.b, sg.kvh, lane);
                const bool rot = p.q_rot_out != nullptr && sg.st0 == 0;
                uint8_t* st_row = staging + (seg & 1) * SH::kNewRowBytes;
                if (p.io_dtype == UAA_DTYPE_F32)
                    prep_fused_q<D, HC, float, KQ8>(p, sg.b, h0, nh, rot, sg.b != cs_b, fits ? L : 0, freq_s, cs_s,
                                                    frag, SH::kFragRow, seg == 0 ? go : 0u, lane);
                else
                    prep_fused_q<D, HC, __nv_bfloat16, KQ8>(p, sg.b, h0, nh, rot, sg.b != cs_b, fits ? L : 0, freq_s,
                                                            cs_s, frag, SH::kFragRow, seg == 0 ? go : 0u, lane);
                cs_b = sg.b;
                // the q' fragments go to the consumers first; the new rows are needed only at
                // the segment's last stage (rows_ready)
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_qfull);
                if (ends) {
                    if (p.io_dtype == UAA_DTYPE_F32)
                        prep_new_rows<D, KV, float>(p, sg.b, sg.kvh, L, cs_s, st_row, sg.hg == 0, lane, nearq);
                    else
                        prep_new_rows<D, KV, __nv_bfloat16>(p, sg.b, sg.kvh, L, cs_s, st_row, sg.hg == 0, lane, nearq);
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence_block();
                        ptx::flag_set(rows_ready + 4 * (seg & 1), static_cast<unsigned>(seg) + 1u);
                    }
                }
                pos += sg.n_st;
                continue;
            } else {
                prep_loaded_q<D, HC, KQ8>(p, sg.b, sg.kvh, r0, nh, frag, SH::kFragRow, seg == 0 ? go : 0u, lane);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_qfull);
            pos += sg.n_st;
        }
        // the deferred key pairs, off the consumers' path: recomputed in fp64 and
        // written over the cache's fp32 rounding
        if (p.fused && KV != kKvQ8) {
            __syncwarp();
            if (p.io_dtype == UAA_DTYPE_F32)
                fix_near_keys<D, float>(p, nearq, lane);
            else
                fix_near_keys<D, __nv_bfloat16>(p, nearq, lane);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int kgrp = CW == kKeyGroups ? warp : warp % kKeyGroups;         // this warp's key group
    const int nt0 = CW == kKeyGroups ? 0 : (warp / kKeyGroups) * NTW;    // and its first 8-column tile
    const int key_w = 16 * MG * kgrp;             // its first key in a stage
    const float cap2 = p.softcap_log2e;
    // ldmatrix lane roles: matrix q = lane / 8, row r = lane % 8 of that matrix.
    const int lq = lane >> 3, lr = lane & 7;
    bool failed = false;
    int it = 0;   // stages consumed
    int seg = 0;  // segments consumed

    for (long long pos = s_c; pos < e_c; ++seg) {
        const Segment sg = segment_at(prefix, lens, p.B, p.window, p.cap, p.head_groups, units, pos, e_c,
                                      p.fused != 0);
        const int lo = sg.lo, hi = sg.hi;
        const int t0 = lo / kTileKeys;
        const int r0 = sg.hg * HC;                   // the unit's first query row (query_row)
        const int nh = min(HC, p.q_len * p.G - r0);  // its query rows
        // several tokens per sequence: row r (token r / G) sees keys up to its own
        // position, lens[b] - q_len + r / G, and with a window the last attn_window
        // of them; this thread's columns 2t, 2t + 1 of each 8-row tile
        const bool causal = p.q_len > 1;
        int kmax[NTW][2], kmin[NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int tok = min(r0 + (nt0 + nt) * 8 + 2 * t + j, p.q_len * p.G - 1) / p.G;
                kmax[nt][j] = lens[sg.b] - p.q_len + tok;
                kmin[nt][j] = p.attn_window > 0 ? kmax[nt][j] - p.attn_window + 1 : INT_MIN;
            }

        // fused append: the new key (slot L) is row new_r of the unit's last stage,
        // which consumer warp new_w owns; -1 when this segment does not end the unit
        const int L = lens[sg.b];
        const bool fits = p.fused && L >= 0 && L < p.cap;
        const int new_r =
            fits && sg.st0 + sg.n_st == sg.stages ? L - (t0 + MG * (sg.stages - 1)) * kTileKeys : -1;
        const int new_w = new_r >= 0 ? new_r / (16 * MG) : -1;

        // this segment's q' fragments from the prep warp: row (nt0 + nt) * 8 + g, as (hi, lo)
        // pairs; k-step kk takes dims 16 kk + 2t (+1) and 16 kk + 2t + 8 (+9) against
        // bf16 keys, and dims 16 kk + 4t .. 16 kk + 4t + 3 against int8 keys (the
        // order in which ldmatrix hands out a code row; the contraction does not care)
        if (!failed && !ptx::mbar_wait(bar_qfull, seg & 1, kWaitLimitCycles)) {
            failed = true;
            if (lane == 0) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
        }
        uint32_t qhi[NTW][KS][2], qlo[NTW][KS][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const uint8_t* row = frag + ((nt0 + nt) * 8 + g) * SH::kFragRow;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                if (KQ8) {
                    const uint4 a = *reinterpret_cast<const uint4*>(row + (8 * kk + 2 * t) * 8);
                    qhi[nt][kk][0] = a.x;
                    qlo[nt][kk][0] = a.y;
                    qhi[nt][kk][1] = a.z;
                    qlo[nt][kk][1] = a.w;
                } else {
                    const uint2 a = *reinterpret_cast<const uint2*>(row + (8 * kk + t) * 8);
                    const uint2 c = *reinterpret_cast<const uint2*>(row + (8 * kk + t + 4) * 8);
                    qhi[nt][kk][0] = a.x;
                    qlo[nt][kk][0] = a.y;
                    qhi[nt][kk][1] = c.x;
                    qlo[nt][kk][1] = c.y;
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_qempty);  // the slot may be refilled

        float m[NTW][2], l[NTW][2], o[NTW][KS][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
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
            if (!failed && kgrp == new_w && k + 1 == sg.n_st) {  // the new key's row, over what the load brought
                bool ready = true;
                if (lane == 0) {
                    ready = ptx::flag_wait_eq(rows_ready + 4 * (seg & 1), static_cast<unsigned>(seg) + 1u,
                                              kWaitLimitCycles);
                    if (!ready) atomicOr(p.status, UAA_DEVFLAG_TIMEOUT);
                    __threadfence_block();
                }
                if (__shfl_sync(0xffffffffu, ready, 0))
                    patch_stage_row<SH>(staging + (seg & 1) * SH::kNewRowBytes, base_ptr + s * SH::kStageBytes, new_r,
                                        lane);
                else
                    failed = true;
            }
            if (!failed && kbase < hi && kbase + 16 * MG > lo) {
                const bool whole = kbase >= lo && kbase + 16 * MG <= hi;
                const uint32_t st = base + s * SH::kStageBytes;

                // S^T = K . Q'^T (keys x heads), one accumulator per 16-key group
                float sacc[MG][NTW][4];
#pragma unroll
                for (int mg = 0; mg < MG; ++mg)
#pragma unroll
                    for (int nt = 0; nt < NTW; ++nt)
                        sacc[mg][nt][0] = sacc[mg][nt][1] = sacc[mg][nt][2] = sacc[mg][nt][3] = 0.f;
                if (KQ8) {
                    // int8 keys: one ldmatrix.x4 covers 16 keys x 32 dims (k-steps 2 kc and
                    // 2 kc + 1); register j holds key g (+8 for odd j), dims 4t .. 4t + 3 of
                    // 16-byte chunk 2 kc + j / 2, widened exactly to fp16 pairs
#pragma unroll
                    for (int kc = 0; kc < KS / 2; ++kc) {
#pragma unroll
                        for (int mg = 0; mg < MG; ++mg) {
                            uint32_t r[4], a0[4], a1[4];
                            ptx::ldsm_x4(r, st + code_off<D, TK>(key_w + 16 * mg + lr + 8 * (lq & 1), 2 * kc + (lq >> 1)));
                            widen_code_quad(r[0], a0[0], a0[2]);
                            widen_code_quad(r[1], a0[1], a0[3]);
                            widen_code_quad(r[2], a1[0], a1[2]);
                            widen_code_quad(r[3], a1[1], a1[3]);
#pragma unroll
                            for (int nt = 0; nt < NTW; ++nt) {
                                ptx::mma_f16(sacc[mg][nt], a0, qhi[nt][2 * kc][0], qhi[nt][2 * kc][1]);
                                ptx::mma_f16(sacc[mg][nt], a0, qlo[nt][2 * kc][0], qlo[nt][2 * kc][1]);
                                ptx::mma_f16(sacc[mg][nt], a1, qhi[nt][2 * kc + 1][0], qhi[nt][2 * kc + 1][1]);
                                ptx::mma_f16(sacc[mg][nt], a1, qlo[nt][2 * kc + 1][0], qlo[nt][2 * kc + 1][1]);
                            }
                        }
                    }
                    // the logit of a code row is its scale times q' . codes
                    const float* ksc = reinterpret_cast<const float*>(base_ptr + s * SH::kStageBytes + SH::kKScaleOff);
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
                        const float k0 = ksc[key_w + 16 * mg + g], k8 = ksc[key_w + 16 * mg + g + 8];
#pragma unroll
                        for (int nt = 0; nt < NTW; ++nt) {
                            sacc[mg][nt][0] *= k0;
                            sacc[mg][nt][1] *= k0;
                            sacc[mg][nt][2] *= k8;
                            sacc[mg][nt][3] *= k8;
                        }
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                        for (int mg = 0; mg < MG; ++mg) {
                            uint32_t a[4];
                            ptx::ldsm_x4(a, st + tile_off<TK>(key_w + 16 * mg + lr + 8 * (lq & 1), 2 * kk + (lq >> 1)));
#pragma unroll
                            for (int nt = 0; nt < NTW; ++nt) {
                                ptx::mma_bf16(sacc[mg][nt], a, qhi[nt][kk][0], qhi[nt][kk][1]);
                                ptx::mma_bf16(sacc[mg][nt], a, qlo[nt][kk][0], qlo[nt][kk][1]);
                            }
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
                    const float* scl = reinterpret_cast<const float*>(base_ptr + s * SH::kStageBytes + SH::kVScaleOff);
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

                float x[MG][NTW][4], f[NTW][2];
                bool rescale = false;
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) {
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int mg = 0; mg < MG; ++mg) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = sacc[mg][nt][e];
                            if (cap2 > 0.f) v = tanhf(v) * cap2;
                            if (!((e < 2) ? vg[mg] : vg8[mg])) v = -INFINITY;
                            if (causal) {
                                const int key = kbase + 16 * mg + g + 8 * (e >> 1);
                                if (key > kmax[nt][e & 1] || key < kmin[nt][e & 1]) v = -INFINITY;
                            }
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
                    for (int nt = 0; nt < NTW; ++nt)
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
                    uint32_t bph[NTW][2], bpl[NTW][2];
#pragma unroll
                    for (int nt = 0; nt < NTW; ++nt) {
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
                            for (int nt = 0; nt < NTW; ++nt) {
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
                            for (int nt = 0; nt < NTW; ++nt) {
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
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], off);

        const int s_last = (it - 1) % SH::kStages;
        float* red_m = reinterpret_cast<float*>(base_ptr + s_last * SH::kStageBytes);
        float* red_l = red_m + kKeyGroups * HC;
        float* red_o = red_l + kKeyGroups * HC;
        const float o_unit = VQ8 ? r_scale : 1.f;
        const size_t rec = 2 * static_cast<size_t>(slot) + (pos == s_c ? 0 : 1);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += RC) {
            ptx::named_barrier_sync(1, CW * 32);  // stage (or previous round) no longer read
            if (g == 0 && c0 == 0) {
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        red_m[kgrp * HC + (nt0 + nt) * 8 + 2 * t + j] = m[nt][j];
                        red_l[kgrp * HC + (nt0 + nt) * 8 + 2 * t + j] = l[nt][j];
                    }
            }
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int mi = 0; mi < KS; ++mi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int hc = (nt0 + nt) * 8 + 2 * t + (e & 1);
                        const int d = VQ8 ? 16 * mi + 2 * g + (e >> 1) : 16 * mi + g + 8 * (e >> 1);
                        if (d >= c0 && d < c0 + RC) red_o[(kgrp * HC + hc) * (RC + 4) + d - c0] = o[nt][mi][e] * o_unit;
                    }
            ptx::named_barrier_sync(1, CW * 32);
            for (int idx = threadIdx.x; idx < nh * RC; idx += CW * 32) {
                const int hc = idx / RC, dc = idx - hc * RC;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kKeyGroups; ++w) M = fmaxf(M, red_m[w * HC + hc]);
                const int hq = sg.kvh * p.G + (r0 + hc) % p.G;  // the row's query head
                const float zs = (sg.whole && p.sink) ? p.sink[hq] * kLog2e : -INFINITY;
                if (sg.whole) M = fmaxf(M, zs);  // the sink joins the denominator of a whole unit
                float L = 0.f, acc = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kKeyGroups; ++w) {
                        const float mw = red_m[w * HC + hc];
                        const float fw = mw == -INFINITY ? 0.f : exp2f(mw - M);
                        L += red_l[w * HC + hc] * fw;
                        acc += red_o[(w * HC + hc) * (RC + 4) + dc] * fw;
                    }
                }
                if (sg.whole) {
                    const float den = L + (zs == -INFINITY ? 0.f : exp2f(zs - M));
                    const float v = den > 0.f ? acc / den : 0.f;
                    const size_t oi = query_row(sg.b, r0 + hc, sg.kvh, p.G, p.Hq, p.q_len) * D + c0 + dc;
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
        ptx::named_barrier_sync(1, CW * 32);
        ptx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s_last);
        pos += sg.n_st;
    }
    if (threadIdx.x == 0) {  // this slot's speed, for the combine's rebalance
        const unsigned long long dt = global_time_ns() - t_begin;
        p.bal.rate[slot] = static_cast<float>(e_c - s_c) / static_cast<float>(dt > 0 ? dt : 1);
    }
}

template <int D, int KV, int NHT>
cudaError_t launch_one(const PartialParams& p, const PartialMaps& m, int n_ctas, cudaStream_t s)
{
    using SH = Shape<D, KV, NHT>;
    auto kern = partial_tc_kernel<D, KV, NHT>;
    static int configured_device_mask = 0;  // bit per device that has the smem attribute set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 31 || !(configured_device_mask & (1 << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SH::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 31) configured_device_mask |= 1 << dev;
    }
    return launch_dependent(kern, dim3(n_ctas), dim3(cta_threads(NHT)), SH::kSmemBytes, s, m.k, m.v, m.s, m.ks, m.kt,
                            m.vt, m.st, m.kst, p);
}

template <int KV>
size_t smem_bytes_kv(int D, int n_head_tiles)
{
    if (n_head_tiles == 2) {
        switch (D) {
        case 64: return Shape<64, KV, 2>::kSmemBytes;
        case 128: return Shape<128, KV, 2>::kSmemBytes;
        default: return 0;
        }
    }
    switch (D) {
    case 64: return Shape<64, KV, 1>::kSmemBytes;
    case 128: return Shape<128, KV, 1>::kSmemBytes;
    case 256: return Shape<256, KV, 1>::kSmemBytes;
    default: return 0;
    }
}

template <int KV>
cudaError_t launch_kv(const PartialParams& p, const PartialMaps& m, int n_head_tiles, int n_ctas, cudaStream_t s)
{
    if (n_head_tiles == 2) {
        switch (p.D) {
        case 64: return launch_one<64, KV, 2>(p, m, n_ctas, s);
        case 128: return launch_one<128, KV, 2>(p, m, n_ctas, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.D) {
    case 64: return launch_one<64, KV, 1>(p, m, n_ctas, s);
    case 128: return launch_one<128, KV, 1>(p, m, n_ctas, s);
    case 256: return launch_one<256, KV, 1>(p, m, n_ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

int kv_kind(int kv_dtype)
{
    return kv_dtype == UAA_DTYPE_Q8 ? kKvQ8 : (kv_dtype == UAA_DTYPE_VQ8 ? kKvVq8 : kKvBf16);
}

template <int KV>
int keys_per_stage_kv(int D, int nht)
{
    switch (D) {
    case 64: return (nht == 2 ? KeyGroups<64, KV, 2>::kMG : KeyGroups<64, KV>::kMG) * kTileKeys;
    case 128: return (nht == 2 ? KeyGroups<128, KV, 2>::kMG : KeyGroups<128, KV>::kMG) * kTileKeys;
    default: return KeyGroups<256, KV>::kMG * kTileKeys;
    }
}

}  // namespace

int partial_tc_keys_per_stage(int D, int kv_dtype, int nht)
{
    switch (kv_kind(kv_dtype)) {
    case kKvQ8: return keys_per_stage_kv<kKvQ8>(D, nht);
    case kKvVq8: return keys_per_stage_kv<kKvVq8>(D, nht);
    default: return keys_per_stage_kv<kKvBf16>(D, nht);
    }
}

size_t partial_tc_smem_bytes(int D, int kv_dtype, int n_head_tiles)
{
    switch (kv_kind(kv_dtype)) {
    case kKvQ8: return smem_bytes_kv<kKvQ8>(D, n_head_tiles);
    case kKvVq8: return smem_bytes_kv<kKvVq8>(D, n_head_tiles);
    default: return smem_bytes_kv<kKvBf16>(D, n_head_tiles);
    }
}

cudaError_t launch_partial_tc(const PartialParams& p, const PartialMaps& m, int kv_dtype, int n_head_tiles,
                              int n_ctas, cudaStream_t s)
{
    switch (kv_kind(kv_dtype)) {
    case kKvQ8: return launch_kv<kKvQ8>(p, m, n_head_tiles, n_ctas, s);
    case kKvVq8: return launch_kv<kKvVq8>(p, m, n_head_tiles, n_ctas, s);
    default: return launch_kv<kKvBf16>(p, m, n_head_tiles, n_ctas, s);
    }
}

}  // namespace uaa
