// Work plan and Top-K merge.
//
// plan:  tile_prefix[t] = number of 128-key tiles of all query rows before row t (one CTA).
// merge: one CTA per query row gathers the candidate lists that the indexer CTAs left for the
//        row's segments (each already cut to at most K keys, in position order), selects the K
//        largest keys with an MSB-first radix select, and writes their positions in ascending
//        order, then -1 up to K ("Engineering Path for Day-0 Adaptation ..." §3.1: Top-K
//        filtering over large candidate sets is split to match the hardware's thread
//        organisation; "Adapting GPU Software Stacks ..." §3.1: the index format is aligned
//        with the attention that consumes it, so no reordering is needed there).
#include "internal.h"

namespace dsa {

constexpr int kPlanThreads = 1024;
constexpr int kMergeThreads = 1024;
constexpr int kMergeSmemKeys = 24576;  // 192 KB of staged candidates
constexpr int kMaxSpans = kMaxIndexerCtas + 1;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(IndexerArgs a) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < a.T; base += kPlanThreads) {
        const int t = base + tid;
        const int n = (t < a.T) ? row_len(a, t) : 0;
        const int tiles = (n + kTileKeys - 1) / kTileKeys;
        int x = tiles;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += v;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int y = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, y, o);
                if (lane >= o) y += v;
            }
            warp_sums[lane] = y;  // inclusive over warps
        }
        __syncthreads();
        const int excl = carry + (warp ? warp_sums[warp - 1] : 0) + x - tiles;
        if (t < a.T) a.tile_prefix[t] = excl;
        __syncthreads();
        if (tid == kPlanThreads - 1) carry = excl + tiles;
        __syncthreads();
    }
    if (tid == 0) a.tile_prefix[a.T] = carry;
}

// Stable compaction of one span of keys into positions: writes key_pos of every key >= thr.
__device__ __forceinline__ uint32_t emit_span(const uint64_t* span, uint32_t cnt, uint64_t thr, int32_t* out,
                                              uint32_t out_n, uint32_t* warp_cnt, bool take_all, uint32_t limit) {
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    for (uint32_t base = 0; base < cnt; base += kMergeThreads) {
        const uint32_t i = base + tid;
        const uint64_t k = (i < cnt) ? span[i] : 0ull;
        const bool p = (i < cnt) && (take_all || k >= thr);
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, p);
        if (lane == 0) warp_cnt[warp] = __popc(ballot);
        __syncthreads();
        uint32_t off = 0, total = 0;
#pragma unroll
        for (uint32_t w = 0; w < kMergeThreads / 32; ++w) {
            const uint32_t c = warp_cnt[w];
            off += (w < warp) ? c : 0u;
            total += c;
        }
        const uint32_t o = out_n + off + __popc(ballot & ((1u << lane) - 1u));
        if (p && o < limit) out[o] = key_pos(k);
        __syncthreads();
        out_n += total;
    }
    return out_n;
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t merge_smem[];
    uint64_t* stage = reinterpret_cast<uint64_t*>(merge_smem);
    __shared__ const uint64_t* span_ptr[kMaxSpans];
    __shared__ uint32_t span_cnt[kMaxSpans];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_cnt[32];
    __shared__ uint32_t ctl_digit, ctl_above, ctl_bucket;
    __shared__ int n_spans;
    __shared__ uint32_t n_total;

    const int t = blockIdx.x;
    const uint32_t tid = threadIdx.x, lane = tid & 31u;
    const uint32_t K = static_cast<uint32_t>(a.K);
    int32_t* out = a.idx + static_cast<int64_t>(t) * a.K;
    const int64_t p0 = a.tile_prefix[t], p1 = a.tile_prefix[t + 1], total = a.tile_prefix[a.T];

    if (p0 == p1) {
        for (uint32_t i = tid; i < K; i += kMergeThreads) out[i] = -1;
        return;
    }
    if (tid == 0) {
        const int64_t G = a.G;
        int64_t c = (p0 * G) / total;
        if (c > G - 1) c = G - 1;
        while (c + 1 < G && tile_begin(c + 1, total, G) <= p0) ++c;
        while (c > 0 && tile_begin(c, total, G) > p0) --c;
        int ns = 0;
        uint32_t n = 0;
        for (; c < G && tile_begin(c, total, G) < p1; ++c) {
            if (tile_begin(c + 1, total, G) == tile_begin(c, total, G)) continue;  // empty CTA range
            const int64_t slot = c + t;
            const uint32_t cnt = static_cast<uint32_t>(a.slot_count[slot]);
            if (ns < kMaxSpans && cnt > 0) {
                span_ptr[ns] = a.slots + slot * a.K;
                span_cnt[ns] = cnt;
                ++ns;
                n += cnt;
            }
        }
        n_spans = ns;
        n_total = n;
    }
    __syncthreads();
    int ns = n_spans;
    const uint32_t n = n_total;

    if (n <= K) {
        uint32_t out_n = 0;
        for (int s = 0; s < ns; ++s) out_n = emit_span(span_ptr[s], span_cnt[s], 0ull, out, out_n, warp_cnt, true, K);
        for (uint32_t i = out_n + tid; i < K; i += kMergeThreads) out[i] = -1;
        return;
    }

    // stage into shared memory when the candidates fit (one read of global memory)
    if (n <= static_cast<uint32_t>(kMergeSmemKeys)) {
        uint32_t off = 0;
        for (int s = 0; s < ns; ++s) {
            const uint64_t* src = span_ptr[s];
            for (uint32_t i = tid; i < span_cnt[s]; i += kMergeThreads) stage[off + i] = src[i];
            off += span_cnt[s];
        }
        __syncthreads();
        if (tid == 0) {
            span_ptr[0] = stage;
            span_cnt[0] = n;
            n_spans = 1;
        }
        __syncthreads();
        ns = 1;
    }

    // MSB-first radix select of the K-th largest key over the spans
    uint64_t prefix = 0;
    uint32_t rem = K;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (uint32_t i = tid; i < 256; i += kMergeThreads) hist[i] = 0;
        __syncthreads();
        for (int s = 0; s < ns; ++s) {
            const uint64_t* sp = span_ptr[s];
            const uint32_t cnt = span_cnt[s];
            for (uint32_t i = tid; i < cnt; i += kMergeThreads) {
                const uint64_t k = sp[i];
                const bool match = (shift == 56) || ((k >> (shift + 8)) == (prefix >> (shift + 8)));
                if (match) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (tid < 32) {
            uint32_t s = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) s += hist[lane * 8 + b];
            uint32_t S = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, S, o);
                if (lane + o < 32) S += v;
            }
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, S >= rem);
            const int L = 31 - __clz(mask);
            if (static_cast<int>(lane) == L) {
                uint32_t running = S - s;
                for (int b = 7; b >= 0; --b) {
                    const uint32_t h = hist[lane * 8 + b];
                    if (running + h >= rem) {
                        ctl_digit = lane * 8 + b;
                        ctl_above = running;
                        ctl_bucket = h;
                        break;
                    }
                    running += h;
                }
            }
        }
        __syncthreads();
        rem -= ctl_above;
        prefix |= static_cast<uint64_t>(ctl_digit) << shift;
        const bool done = (ctl_bucket == rem);
        __syncthreads();
        if (done) break;
    }
    uint32_t out_n = 0;
    for (int s = 0; s < ns; ++s) out_n = emit_span(span_ptr[s], span_cnt[s], prefix, out, out_n, warp_cnt, false, K);
    for (uint32_t i = out_n + tid; i < K; i += kMergeThreads) out[i] = -1;
}

bool launch_plan(const IndexerArgs& a, cudaStream_t s, int* launches) {
    plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_merge(const IndexerArgs& a, cudaStream_t s, int* launches) {
    if (a.T == 0) return true;
    const size_t smem = static_cast<size_t>(kMergeSmemKeys) * sizeof(uint64_t);
    if (cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return false;
    topk_merge_kernel<<<a.T, kMergeThreads, smem, s>>>(a);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace dsa
