// internal.cuh -- kernel parameter blocks, launch declarations and small device
// helpers shared by the kernels of libuaa. Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/uaa.h"

namespace uaa {

constexpr int kTileKeys = 64;        // keys per tile; split boundaries fall on tiles
constexpr int kMaxHeadDim = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at the top SM clock

// ---------------------------------------------------------------- parameters

struct AppendParams {
    int B, Hq, Hkv, D;
    int cap, max_len;
    int style;              // UAA_ROPE_NEOX / _INTERLEAVED
    int qk_norm;
    float eps;
    float qscale;           // q_prime = rotated q * qscale (the partial kernel's logit prescale)
    float mscale;           // cos / sin multiplier (YaRN attention factor, else 1)
    int io_dtype, kv_dtype;
    const void* q;
    const void* k_new;
    const void* v_new;
    const float* q_norm_w;
    const float* k_norm_w;
    void* k_cache;
    void* v_cache;
    float* v_scale;
    int* seq_lens;
    float* q_prime;         // workspace [B][Hq][D]
    float* q_rot_out;       // optional [B][Hq][D]
    unsigned* status;
    double inv_freq_over_pi[kMaxHeadDim / 2];  // theta'_p / pi, fp64
};

struct PartialParams {
    int B, Hq, Hkv, D, G;
    int heads_per_cta;      // query heads per CTA
    int head_groups;        // ceil(G / heads_per_cta)
    int cap, window;
    int S, chunk_tiles;
    float softcap_log2e;    // 0: no softcap; else softcap * log2(e)
    const float* q_prime;
    const void* k_cache;
    const void* v_cache;
    const float* v_scale;
    const int* seq_lens;
    float* o_part;          // [B][Hq][S][D]
    float* lse_part;        // [B][Hq][S]
    unsigned* status;
};

struct CombineParams {
    int B, Hq, Hkv, D, G;
    int window, S, chunk_tiles;
    int out_dtype;
    const float* sink;      // [Hq] or null
    const int* seq_lens;
    const float* o_part;
    const float* lse_part;
    void* out;
    unsigned* status;
};

// ---------------------------------------------------------------- launches
// Each returns the launch error (cudaGetLastError) of its kernel.

cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_partial_simt(const PartialParams& p, cudaStream_t s);
cudaError_t launch_partial_tc(const PartialParams& p, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const CUtensorMap& tm_s, int kv_dtype,
                              int n_head_tiles, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_vq8_quantize(const void* v, int v_dtype, int64_t n_rows, int D, int8_t* codes,
                                float* scales, cudaStream_t s);

// Dynamic shared memory the tensor-core partial kernel needs.
size_t partial_tc_smem_bytes(int D, int kv_dtype, int n_head_tiles);
// Keys per ring stage of the tensor-core partial kernel (the TMA box height); its
// splits hold a multiple of keys_per_stage / 64 tiles.
int partial_tc_keys_per_stage(int D);

// ---------------------------------------------------------------- device helpers

// Visible keys of a sequence holding n keys after the append: [lo, n) with a
// window W keeping the last W of them (positions j > pos - W, pos = n - 1).
__host__ __device__ inline void key_range(int n, int window, int& lo, int& hi)
{
    hi = n;
    lo = (window > 0 && n > window) ? n - window : 0;
}

// Splits covering tiles [lo / 64, ceil(hi / 64)) in chunks of chunk_tiles tiles.
__host__ __device__ inline int splits_needed(int lo, int hi, int chunk_tiles)
{
    if (hi <= lo) return 0;
    const int t0 = lo / kTileKeys, t1 = (hi + kTileKeys - 1) / kTileKeys;
    return (t1 - t0 + chunk_tiles - 1) / chunk_tiles;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float load_elem(const void* base, int dtype, size_t i)
{
    if (dtype == UAA_DTYPE_F32) return static_cast<const float*>(base)[i];
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

}  // namespace uaa
