// Indexer + streaming Top-K on CUDA cores, for small indexer shapes (the fp32 workload: 4 heads of
// 64) and any storage mode. Each CTA walks its segments of 128-key tiles: the tile's two paged
// blocks are fetched through the block table with 16-byte coalesced loads, widened to fp32 in
// shared memory, scored per key by one thread
//     S = sum_j w_j * max(0, scale_blk * (q_I[j] . k))
// and offered to the CTA's Top-K buffer; no score leaves the chip. ("Day0 Inference Support ...
// on Huawei Ascend CANN Architecture" §2.1: scoring, head-weight weighting and Top-K fused in one
// operator that reads the paged cache directly.) MXFP8 keys: every 16 codes are widened and
// multiplied by their 32-element group's E8M0 scale (exact in fp32); q_I arrives MX-quantised.
#include "internal.h"

#include <type_traits>

namespace dsa {

constexpr int kSimtThreads = 128;

template <typename T>
struct Widen;
template <>
struct Widen<float> {
    static constexpr int kPer16B = 4;
    __device__ static void unpack(const uint4& v, float* out) {
        out[0] = __uint_as_float(v.x);
        out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z);
        out[3] = __uint_as_float(v.w);
    }
};
struct Bf16Tag {};
template <>
struct Widen<Bf16Tag> {
    static constexpr int kPer16B = 8;
    __device__ static void unpack(const uint4& v, float* out) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
struct E4m3Tag {};
// OCP e4m3: sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0 is subnormal (m * 2^-9).
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
    const uint32_t s = (c & 0x80u) << 24;
    const uint32_t e = (c >> 3) & 0xFu;
    const uint32_t m = c & 7u;
    float mag;
    if (e == 0) mag = static_cast<float>(m) * 0.001953125f;  // m * 2^-9, exact
    else mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return __uint_as_float(__float_as_uint(mag) | s);
}
template <>
struct Widen<E4m3Tag> {
    static constexpr int kPer16B = 16;
    __device__ static void unpack(const uint4& v, float* out) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) out[4 * i + b] = e4m3_to_float((w[i] >> (8 * b)) & 0xFFu);
    }
};

struct MxTag {};  // e4m3 codes with one E8M0 scale byte per 32 elements of a key
template <>
struct Widen<MxTag> : Widen<E4m3Tag> {};

template <typename QT>
__device__ __forceinline__ float load_act(const void* p, int64_t i);
template <>
__device__ __forceinline__ float load_act<float>(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
}
template <>
__device__ __forceinline__ float load_act<Bf16Tag>(const void* p, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
}

// KT: key storage (float / Bf16Tag / E4m3Tag); QT: query storage (float / Bf16Tag).
template <typename KT, typename QT>
__global__ void __launch_bounds__(kSimtThreads) indexer_simt_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int H_I = a.H_I, d_I = a.d_I;
    const int kstride = d_I + 1;
    const uint32_t cap = static_cast<uint32_t>(2 * a.K + kSimtThreads);
    float* q_s = reinterpret_cast<float*>(smem);                        // [H_I][d_I]
    float* w_s = q_s + H_I * d_I;                                        // [H_I]
    float* k_s = w_s + H_I;                                              // [128][d_I + 1]
    float* scale_s = k_s + kTileKeys * kstride;                          // [2] per block of the tile
    uint64_t* buf = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(scale_s + 2) + 15) & ~static_cast<uintptr_t>(15));  // [cap]
    __shared__ uint32_t hist[kSimtThreads / 32 * 256];
    __shared__ TopkCtl ctl;
    __shared__ int blk_s[2];

    const int tid = threadIdx.x;
    TopkGroup<kSimtThreads, 33> topk{buf, hist, &ctl, cap, static_cast<uint32_t>(a.K), static_cast<uint32_t>(tid), 1};
    constexpr int per = Widen<KT>::kPer16B;
    const int units_per_row = d_I / per;
    constexpr size_t key_bytes = 16 / per;

    griddep_launch_dependents();
    griddep_wait();  // the work plan (tile prefix) is written
    SegmentIter it;
    it.init(a.tile_prefix, a.T, blockIdx.x, a.G);
    Segment seg;
    while (it.next(seg)) {
        const int t = seg.row;
        const int b = row_seq(a, t);
        const int n = row_len(a, t);
        for (int i = tid; i < H_I * d_I; i += kSimtThreads)
            q_s[i] = load_act<QT>(a.q_I, static_cast<int64_t>(t) * H_I * d_I + i);
        for (int i = tid; i < H_I; i += kSimtThreads) w_s[i] = a.w[static_cast<int64_t>(t) * H_I + i];
        topk.reset();  // includes a barrier: q_s / w_s visible
        for (int j = seg.tile0; j < seg.tile1; ++j) {
            if (tid < 2) {
                const int lb = 2 * j + tid;
                int blk = -1;
                if (lb * kBlock < n) blk = phys_block(a, b, lb);
                blk_s[tid] = blk;
                scale_s[tid] = (std::is_same<KT, E4m3Tag>::value && blk >= 0) ? static_cast<const float*>(a.k_I_scale)[blk]
                                                                                : 1.0f;
            }
            topk.sync();
            for (int u = tid; u < kTileKeys * units_per_row; u += kSimtThreads) {
                const int r = u / units_per_row, c = u % units_per_row;
                const int s = j * kTileKeys + r;
                const int blk = blk_s[r >> 6];
                float vals[per];
                if (s < n && blk >= 0) {
                    const uint8_t* src = static_cast<const uint8_t*>(a.k_I) +
                                         ((static_cast<int64_t>(blk) * kBlock + (r & 63)) * d_I) * key_bytes +
                                         static_cast<int64_t>(c) * 16;
                    Widen<KT>::unpack(*reinterpret_cast<const uint4*>(src), vals);
                    if constexpr (std::is_same<KT, MxTag>::value) {  // 16 codes lie in group c / 2 of the key
                        const float f = e8m0_value(static_cast<const uint8_t*>(a.k_I_scale)
                                                       [(static_cast<int64_t>(blk) * kBlock + (r & 63)) * (d_I / 32) + (c >> 1)]);
#pragma unroll
                        for (int e = 0; e < per; ++e) vals[e] *= f;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < per; ++e) vals[e] = 0.0f;
                }
#pragma unroll
                for (int e = 0; e < per; ++e) k_s[r * kstride + c * per + e] = vals[e];
            }
            topk.sync();
            const int r = tid;
            const int s = j * kTileKeys + r;
            const bool valid = (s < n) && (blk_s[r >> 6] >= 0);
            float score = 0.0f;
            if (valid) {
                const float sc = scale_s[r >> 6];
                const float* kr = k_s + r * kstride;
                for (int h = 0; h < H_I; ++h) {
                    const float* qh = q_s + h * d_I;
                    float dot = 0.0f;
                    for (int e = 0; e < d_I; ++e) dot = fmaf(qh[e], kr[e], dot);
                    score = fmaf(w_s[h], fmaxf(dot * sc, 0.0f), score);
                }
            }
            topk.push(make_key(score, static_cast<uint32_t>(s)), valid);
        }
        const int64_t slot = static_cast<int64_t>(blockIdx.x) + t;
        topk.flush(a.slots + slot * a.K, a.slot_count + slot, a.slot_est + slot);
        topk.sync();
    }
}

static size_t simt_smem_bytes(const IndexerArgs& a) {
    const size_t f = static_cast<size_t>(a.H_I) * a.d_I + a.H_I + static_cast<size_t>(kTileKeys) * (a.d_I + 1) + 2;
    return ((f * 4 + 15) & ~static_cast<size_t>(15)) + static_cast<size_t>(2 * a.K + kSimtThreads) * 8;
}

template <typename KT, typename QT>
static bool launch_typed(const IndexerArgs& a, cudaStream_t s, int* launches) {
    const size_t smem = simt_smem_bytes(a);
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(indexer_simt_kernel<KT, QT>), smem)) return false;
    if (!launch_kernel(true, indexer_simt_kernel<KT, QT>, dim3(a.G), dim3(kSimtThreads), smem, s, a)) return false;
    ++*launches;
    return true;
}

bool launch_indexer_simt(const IndexerArgs& a, cudaStream_t s, int* launches) {
    switch (a.mode) {
        case DSA_F32: return launch_typed<float, float>(a, s, launches);
        case DSA_BF16: return launch_typed<Bf16Tag, Bf16Tag>(a, s, launches);
        case DSA_BF16_KFP8: return launch_typed<E4m3Tag, Bf16Tag>(a, s, launches);
        case DSA_MXFP8: return launch_typed<MxTag, Bf16Tag>(a, s, launches);
        default: return false;
    }
}

size_t indexer_simt_smem(const IndexerArgs& a) { return simt_smem_bytes(a); }

}  // namespace dsa
