// Sparse attention on CUDA cores for small head shapes (the fp32 workload: 8 heads of 128). One
// CTA per (query row, head): the selected positions are mapped through the block table once, the
// logits z_i = sm_scale * q . row_i are reduced per warp (each warp reads four whole rows at a time,
// coalesced, so their loads are in flight together), then p = softmax(z) and
// out = sum_i p_i * row_i[0:d_v]: each warp accumulates every 8th row over 4 consecutive columns
// per lane (128 columns per pass, vector loads), and the 8 warps' partial sums are added in shared
// memory ("Day0 Inference Support ... on Huawei Ascend CANN Architecture" §1 and §2.1: the sparse
// attention reads the main KV exactly at the selected indices). With an FP8 latent cache (§3: FP8
// block quantisation in the attention stage) every element read is code * its tile's scale, in
// fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace dsa {

constexpr int kAttnSimtThreads = 256;

__device__ __forceinline__ float act_f(const void* p, int64_t i, bool bf16) {
    return bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16)
                : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ uint16_t to_bf16_rn(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Latent-cache storage: fp32 rows, bf16 rows, or FP8 records (codes, then one fp32 scale per 128).
enum KvKind { kKvF32 = 0, kKvBf16 = 1, kKvFp8 = 2 };

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);  // exact
    return __half2float(*reinterpret_cast<const __half*>(&h));
}

// element e of latent row r
template <int KV>
__device__ __forceinline__ float kv_elem(const AttnArgs& a, int64_t r, int e) {
    if (KV == kKvFp8) {
        const uint8_t* rec = static_cast<const uint8_t*>(a.kv) + r * a.kv_rec;
        return e4m3_to_f32(rec[e]) * *reinterpret_cast<const float*>(rec + a.d + 4 * (e >> 7));
    }
    return act_f(a.kv, r * a.d + e, KV == kKvBf16);
}

// elements c .. c + 3 of latent row r (c % 4 == 0, c + 3 < d: vector loads)
template <int KV>
__device__ __forceinline__ void kv_load4(const AttnArgs& a, int64_t r, int c, float (&v)[4]) {
    if (KV == kKvFp8) {
        const uint8_t* rec = static_cast<const uint8_t*>(a.kv) + r * a.kv_rec;
        const uint32_t codes = *reinterpret_cast<const uint32_t*>(rec + c);
        const float sc = *reinterpret_cast<const float*>(rec + a.d + 4 * (c >> 7));  // one tile: 128 % 4 == 0
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = e4m3_to_f32((codes >> (8 * k)) & 0xFFu) * sc;
    } else if (KV == kKvBf16) {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.kv) + r * a.d + c);
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xFFFF0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
        const float4 f4 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.kv) + r * a.d + c);
        v[0] = f4.x;
        v[1] = f4.y;
        v[2] = f4.z;
        v[3] = f4.w;
    }
}

template <int KV>
__global__ void __launch_bounds__(kAttnSimtThreads) attn_simt_kernel(AttnArgs a) {
    constexpr bool BF16 = KV != kKvF32;  // queries and outputs are bf16 with bf16 or FP8 latent rows
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = a.d, K = a.K;
    float* q_s = reinterpret_cast<float*>(smem);  // [d]
    float* z_s = q_s + d;                          // [K]
    int64_t* row_s = reinterpret_cast<int64_t*>(
        (reinterpret_cast<uintptr_t>(z_s + K) + 7) & ~static_cast<uintptr_t>(7));  // [K] physical rows
    float* part = reinterpret_cast<float*>(row_s + K);                            // [8 warps][128]
    __shared__ float red[kAttnSimtThreads / 32];
    __shared__ float m_s, l_s;

    const int h = blockIdx.x, t = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = a.q_seq ? a.q_seq[t] : t;
    const bool seq_ok = b >= 0 && b < a.B;
    const int L = seq_ok ? a.seq_lens[b] : 0;

    for (int e = tid; e < d; e += kAttnSimtThreads)
        q_s[e] = act_f(a.q, (static_cast<int64_t>(t) * a.H + h) * d + e, BF16);
    griddep_wait();  // idx may come from the previous kernel of this call
    for (int i = tid; i < K; i += kAttnSimtThreads) {
        const int s = a.idx[static_cast<int64_t>(t) * K + i];
        int64_t r = -1;
        if (s != -1) {
            if (s < 0 || s >= L) {
                atomicOr(a.err, DSA_FAULT_INDEX);
            } else {
                const int blk = a.block_table[static_cast<int64_t>(b) * a.max_blocks + (s >> 6)];
                if (blk < 0 || blk >= a.num_blocks) atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
                else r = static_cast<int64_t>(blk) * kBlock + (s & 63);
            }
        }
        row_s[i] = r;
    }
    block_sync();

    // logits: each warp takes four selected rows at a time (rows 4w .. 4w+3 of every 32)
    constexpr int kNW = kAttnSimtThreads / 32;
    for (int i0 = warp * 4; i0 < K; i0 += kNW * 4) {
        int64_t rr[4];
        float dot[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            rr[u] = (i0 + u < K) ? row_s[i0 + u] : -1;
            dot[u] = 0.0f;
        }
        for (int e = lane; e < d; e += 32) {
            const float qe = q_s[e];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (rr[u] >= 0) dot[u] = fmaf(qe, kv_elem<KV>(a, rr[u], e), dot[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot[u] += __shfl_xor_sync(0xFFFFFFFFu, dot[u], o);
            if (lane == 0 && i0 + u < K) z_s[i0 + u] = (rr[u] >= 0) ? dot[u] * a.sm_scale : -INFINITY;
        }
    }
    block_sync();

    float m = -INFINITY;
    for (int i = tid; i < K; i += kAttnSimtThreads) m = fmaxf(m, z_s[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[warp] = m;
    block_sync();
    if (tid == 0) {
        float mm = -INFINITY;
        for (int w = 0; w < kAttnSimtThreads / 32; ++w) mm = fmaxf(mm, red[w]);
        m_s = mm;
    }
    block_sync();
    m = m_s;
    float l = 0.0f;
    for (int i = tid; i < K; i += kAttnSimtThreads) {
        const float p = (z_s[i] == -INFINITY) ? 0.0f : expf(z_s[i] - m);
        z_s[i] = p;
        l += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    block_sync();
    if (lane == 0) red[warp] = l;
    block_sync();
    if (tid == 0) {
        float ll = 0.0f;
        for (int w = 0; w < kAttnSimtThreads / 32; ++w) ll += red[w];
        l_s = ll;
    }
    block_sync();
    l = l_s;
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;

    const int64_t obase = (static_cast<int64_t>(t) * a.H + h) * a.d_v;
    for (int c0 = 0; c0 < a.d_v; c0 += 128) {
        const int c = c0 + lane * 4;  // this lane's 4 columns
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int i = warp; i < K; i += kNW) {
            const int64_t r = row_s[i];
            if (r < 0) continue;  // the same row for the whole warp
            const float p = z_s[i];
            if (c + 3 < a.d_v) {  // d % 4 == 0 (fp32) / d % 8 == 0 (bf16) / records 16-byte aligned
                float v[4];
                kv_load4<KV>(a, r, c, v);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = fmaf(p, v[k], acc[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (c + k < a.d_v) acc[k] = fmaf(p, kv_elem<KV>(a, r, c + k), acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) part[warp * 128 + lane * 4 + k] = acc[k];
        block_sync();
        if (tid < 128 && c0 + tid < a.d_v) {
            float o = 0.0f;
#pragma unroll
            for (int w = 0; w < kNW; ++w) o += part[w * 128 + tid];
            o *= inv;
            if (BF16) static_cast<uint16_t*>(a.out)[obase + c0 + tid] = to_bf16_rn(o);
            else static_cast<float*>(a.out)[obase + c0 + tid] = o;
        }
        block_sync();  // part is rewritten by the next pass
    }
    if (tid == 0 && a.lse) a.lse[static_cast<int64_t>(t) * a.H + h] = (l > 0.0f) ? m + logf(l) : -INFINITY;
}

bool launch_attn_simt(const AttnArgs& a, cudaStream_t s, int* launches) {
    if (a.T == 0) return true;
    const size_t smem = static_cast<size_t>(a.d + a.K) * 4 + 8 + static_cast<size_t>(a.K) * 8 +
                        static_cast<size_t>(kAttnSimtThreads / 32) * 128 * 4;
    dim3 grid(a.H, a.T);
    const bool pdl = a.after_own_kernel != 0;
    auto go = [&](auto kernel) {
        return set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), smem) &&
               launch_kernel(pdl, kernel, grid, dim3(kAttnSimtThreads), smem, s, a);
    };
    const bool ok = a.mode == DSA_F32 ? go(attn_simt_kernel<kKvF32>)
                                      : (a.kv_fp8 ? go(attn_simt_kernel<kKvFp8>) : go(attn_simt_kernel<kKvBf16>));
    if (!ok) return false;
    ++*launches;
    return true;
}

}  // namespace dsa
