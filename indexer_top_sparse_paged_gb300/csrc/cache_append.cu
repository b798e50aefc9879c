// Cache append: new tokens' latent rows and indexer keys into their paged slots, the step before
// the indexer and the sparse attention ("How the Ascend Computing Platform Achieves Same-Day
// Inference Adaptation ..." §2.2 table: the cache update is fused with the flow that produces the
// new entries; "Day0 Inference Support ... on Huawei Ascend CANN Architecture" §2.2/§3: the
// indexer's keys are quantised on the way in).
//
// One CTA per new token t (sequence b, position pos in the sequence's tail) copies its latent
// row, and in the fp32 / bf16 modes its indexer key, into physical row
// block_table[b][pos / 64] * 64 + pos % 64. With FP8 e4m3 keys (one fp32 scale per 64-token
// block) the first new token of every touched block requantises the whole block: with
// x = code * scale_old (fp32) for the block's earlier tokens and the new keys' values,
// scale = amax / 448 (1 when amax is 0) and every code becomes RNE_e4m3(x / scale), saturating
// at +-448. The new tokens of one block must be consecutive rows (ascending positions). MXFP8
// keys have no block state: each new key's groups of 32 get their own E8M0 scale and codes.
// An FP8 latent cache (DSA_KV_FP8) has no block state either: each new row becomes one record,
// every 128-element tile quantised on its own (one warp per tile), in fp32: scale = amax / 448
// (1 when amax is 0), code = RNE_e4m3(x / scale), saturating ("Day0 Inference Support ... on
// Huawei Ascend CANN Architecture" §3: FP8 block quantisation in the attention stage).
#include "internal.h"

namespace dsa {

constexpr int kAppendThreads = 256;

struct AppendArgs {
    int mode;
    int kv_fp8;  // latent rows stored as FP8 records
    int B, max_blocks, num_blocks;
    int d_I, d;
    int T;
    const void* k_new;
    const void* kv_new;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_seq;
    const int32_t* q_pos;
    void* k_cache;
    void* k_scale;
    void* kv_cache;
    int* err;
};

// Sequence, position and physical cache block of new token t (-1 when invalid).
__device__ __forceinline__ int append_block(const AppendArgs& a, int t, int& b, int& pos) {
    b = a.q_seq ? a.q_seq[t] : t;
    if (b < 0 || b >= a.B) return -1;
    const int L = a.seq_lens[b];
    pos = a.q_pos ? a.q_pos[t] : L - 1;
    if (pos < 0 || pos >= L || pos / kBlock >= a.max_blocks) return -1;
    const int blk = a.block_table[static_cast<int64_t>(b) * a.max_blocks + pos / kBlock];
    return (blk >= 0 && blk < a.num_blocks) ? blk : -1;
}

__device__ __forceinline__ void copy_row(void* dst, const void* src, int bytes) {
    const uint4* s = static_cast<const uint4*>(src);
    uint4* d = static_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < bytes / 16; i += kAppendThreads) d[i] = s[i];
}

__device__ __forceinline__ float e4m3_value(uint8_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);  // exact
    return __half2float(*reinterpret_cast<const __half*>(&h));
}

// One FP8 latent record from a bf16 row of d elements (d % 16 == 0): warp w quantises tiles
// w, w + 8, ...; lane l holds elements 4l .. 4l + 3 of the tile. The padding after the scales is
// zeroed.
__device__ void store_kv_record(uint8_t* rec, const uint16_t* x, int d) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ntiles = (d + 127) / 128;
    for (int j = warp; j < ntiles; j += kAppendThreads / 32) {
        const int e = 128 * j + 4 * lane;
        const bool in = e < d;  // d % 16 == 0: a lane's 4 elements are all in or all out
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (in) {
            const uint2 u = *reinterpret_cast<const uint2*>(x + e);
            v[0] = __uint_as_float(u.x << 16);
            v[1] = __uint_as_float(u.x & 0xFFFF0000u);
            v[2] = __uint_as_float(u.y << 16);
            v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        }
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        if (in) {
            uint32_t c = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                c |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(v[k] / scale, __NV_SATFINITE, __NV_E4M3)) << (8 * k);
            *reinterpret_cast<uint32_t*>(rec + e) = c;
        }
        if (lane == 0) *reinterpret_cast<float*>(rec + d + 4 * j) = scale;
    }
    for (int i = d + 4 * ntiles + static_cast<int>(threadIdx.x); i < DSA_KV_FP8_RECORD_BYTES(d); i += kAppendThreads)
        rec[i] = 0;
}

// New token t's rows into the paged caches (the whole CTA).
__device__ void append_token(const AppendArgs& a, int t) {
    __shared__ float red[kAppendThreads / 32];
    __shared__ int run_end;
    int b, pos;
    const int blk = append_block(a, t, b, pos);
    if (blk < 0) {
        if (threadIdx.x == 0) atomicOr(a.err, (b < 0 || b >= a.B) ? DSA_FAULT_INDEX : DSA_FAULT_BLOCK_TABLE);
        return;
    }
    const int64_t row = static_cast<int64_t>(blk) * kBlock + pos % kBlock;
    const int act = a.mode == DSA_F32 ? 4 : 2;
    if (a.kv_fp8) {
        store_kv_record(static_cast<uint8_t*>(a.kv_cache) + row * DSA_KV_FP8_RECORD_BYTES(a.d),
                        static_cast<const uint16_t*>(a.kv_new) + static_cast<int64_t>(t) * a.d, a.d);
    } else {
        copy_row(static_cast<uint8_t*>(a.kv_cache) + row * a.d * act,
                 static_cast<const uint8_t*>(a.kv_new) + static_cast<int64_t>(t) * a.d * act, a.d * act);
    }
    if (a.mode == DSA_MXFP8) {  // every group of 32 of the new key is quantised on its own
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.k_new) + static_cast<int64_t>(t) * a.d_I);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.k_cache) + row * a.d_I);
        for (int g = threadIdx.x; g < a.d_I / 32; g += kAppendThreads) {
            uint32_t w[16], codes[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = src[4 * g + i];
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
            const int X = mx_encode32(w, codes);
            dst[2 * g] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            dst[2 * g + 1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
            static_cast<uint8_t*>(a.k_scale)[row * (a.d_I / 32) + g] = static_cast<uint8_t>(X + 127);
        }
        return;
    }
    if (a.mode != DSA_BF16_KFP8) {
        copy_row(static_cast<uint8_t*>(a.k_cache) + row * a.d_I * act,
                 static_cast<const uint8_t*>(a.k_new) + static_cast<int64_t>(t) * a.d_I * act, a.d_I * act);
        return;
    }
    // FP8 keys: the first new token of the block requantises it
    const int lb = pos / kBlock;
    if (t > 0) {
        int b0, p0;
        const int prev = append_block(a, t - 1, b0, p0);
        if (prev >= 0 && b0 == b && p0 / kBlock == lb) return;
    }
    // the block's run of new tokens: rows t .. run_end - 1
    if (threadIdx.x == 0) run_end = min(a.T, t + kBlock);  // a block holds at most 64 new tokens
    __syncthreads();
    if (threadIdx.x < kBlock && threadIdx.x > 0) {
        const int u = t + static_cast<int>(threadIdx.x);
        int b2, p2;
        const bool same = u < a.T && append_block(a, u, b2, p2) >= 0 && b2 == b && p2 / kBlock == lb;
        if (!same) atomicMin(&run_end, u);
    }
    __syncthreads();
    const int m = run_end - t;
    const int n_old = pos - lb * kBlock;  // the block's earlier tokens: slots [0, n_old)
    const float old_scale = static_cast<const float*>(a.k_scale)[blk];
    uint8_t* codes = static_cast<uint8_t*>(a.k_cache) + static_cast<int64_t>(blk) * kBlock * a.d_I;
    const uint16_t* knew = static_cast<const uint16_t*>(a.k_new) + static_cast<int64_t>(t) * a.d_I;
    const int n_elem_old = n_old * a.d_I, n_elem_new = m * a.d_I;
    // amax over the earlier tokens (code * old scale) and the new keys
    float amax = 0.0f;
    for (int i = threadIdx.x; i < n_elem_old; i += kAppendThreads) amax = fmaxf(amax, fabsf(e4m3_value(codes[i]) * old_scale));
    for (int i = threadIdx.x; i < n_elem_new; i += kAppendThreads)
        amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(knew[i]) << 16)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kAppendThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    // every code of the block's tokens, re-rounded against the new scale
    for (int i = threadIdx.x; i < n_elem_old; i += kAppendThreads) {
        const float x = e4m3_value(codes[i]) * old_scale;
        codes[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(x / scale, __NV_SATFINITE, __NV_E4M3));
    }
    for (int i = threadIdx.x; i < n_elem_new; i += kAppendThreads) {
        const int u = t + i / a.d_I;  // each new row into its own slot
        const int pu = a.q_pos ? a.q_pos[u] : pos;
        const float x = __uint_as_float(static_cast<uint32_t>(knew[i]) << 16);
        codes[(pu % kBlock) * a.d_I + i % a.d_I] =
            static_cast<uint8_t>(__nv_cvt_float_to_fp8(x / scale, __NV_SATFINITE, __NV_E4M3));
    }
    if (threadIdx.x == 0) static_cast<float*>(a.k_scale)[blk] = scale;
}

__global__ void __launch_bounds__(kAppendThreads) cache_append_kernel(AppendArgs a) { append_token(a, blockIdx.x); }

// Indexer prolog: the cache append of the step's new tokens (CTAs 0 .. T - 1) and, in the same
// launch, the MXFP8 quantisation of the indexer query (the other CTAs, one group of 32 elements per
// thread, written as its exact bf16 values to q_out) -- the two independent preparations the
// indexer needs ("Day0 Inference Support ... on Huawei Ascend CANN Architecture" §2.2, Indexer
// Prolog: Q quantisation runs beside the other preparations instead of after them).
__global__ void __launch_bounds__(kAppendThreads)
    indexer_prolog_kernel(AppendArgs a, const uint16_t* __restrict__ q, uint16_t* __restrict__ q_out, int64_t q_groups) {
    if (static_cast<int>(blockIdx.x) < a.T) {
        append_token(a, blockIdx.x);
        return;
    }
    const int64_t g = static_cast<int64_t>(blockIdx.x - a.T) * kAppendThreads + threadIdx.x;
    if (g < q_groups) mx_quantize_group32(q + g * 32, q_out + g * 32);
}

bool launch_cache_append(const dsa_dims& d, bool kv_fp8, const void* k_new, const void* kv_new,
                         const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                         const int32_t* q_pos, int T, void* k_cache, void* k_scale, void* kv_cache, int* err,
                         cudaStream_t s, int* launches) {
    if (T == 0) return true;
    AppendArgs a{d.mode, kv_fp8 ? 1 : 0, d.B, d.max_blocks, d.num_blocks, d.d_I, d.d, T, k_new, kv_new, block_table,
                 seq_lens, q_seq, q_pos, k_cache, k_scale, kv_cache, err};
    if (!launch_kernel(false, cache_append_kernel, dim3(T), dim3(kAppendThreads), 0, s, a)) return false;
    ++*launches;
    return true;
}

bool launch_indexer_prolog(const dsa_dims& d, bool kv_fp8, const void* k_new, const void* kv_new,
                           const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                           const int32_t* q_pos, int T, void* k_cache, void* k_scale, void* kv_cache, const void* q_I,
                           void* q_out, int64_t q_elements, int* err, cudaStream_t s, int* launches) {
    const int64_t q_groups = q_out ? q_elements / 32 : 0;
    const int64_t q_ctas = (q_groups + kAppendThreads - 1) / kAppendThreads;
    if (T == 0 && q_ctas == 0) return true;
    AppendArgs a{d.mode, kv_fp8 ? 1 : 0, d.B, d.max_blocks, d.num_blocks, d.d_I, d.d, T, k_new, kv_new, block_table,
                 seq_lens, q_seq, q_pos, k_cache, k_scale, kv_cache, err};
    if (!launch_kernel(false, indexer_prolog_kernel, dim3(static_cast<unsigned>(T + q_ctas)), dim3(kAppendThreads), 0, s,
                       a, static_cast<const uint16_t*>(q_I), static_cast<uint16_t*>(q_out), q_groups))
        return false;
    ++*launches;
    return true;
}

}  // namespace dsa
