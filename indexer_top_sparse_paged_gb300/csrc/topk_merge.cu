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
constexpr int kMergeSmemKeys = 16384;  // candidates held in registers (16 per thread)
constexpr int kMergeHistBytes = kMergeThreads / 32 * 256 * 4;  // one 256-bin histogram per warp
constexpr int kMergeSmemBytes = kMergeHistBytes + kMergeSmemKeys * 8;  // + the row's candidates
constexpr int kMaxSpans = kMaxIndexerCtas + 1;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(IndexerArgs a) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    griddep_launch_dependents();  // the indexer may start its prologue
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    block_sync();
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
        block_sync();
        if (warp == 0) {
            int y = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, y, o);
                if (lane >= o) y += v;
            }
            warp_sums[lane] = y;  // inclusive over warps
        }
        block_sync();
        const int excl = carry + (warp ? warp_sums[warp - 1] : 0) + x - tiles;
        if (t < a.T) a.tile_prefix[t] = excl;
        block_sync();
        if (tid == kPlanThreads - 1) carry = excl + tiles;
        block_sync();
    }
    if (tid == 0) a.tile_prefix[a.T] = carry;
}

constexpr int kPer = kMergeSmemKeys / kMergeThreads;  // candidates per thread held in registers
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t merge_smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(merge_smem);  // [32 warps][256]
    __shared__ const uint64_t* span_ptr[kMaxSpans];
    __shared__ uint32_t span_off[kMaxSpans + 1];
    __shared__ uint32_t warp_tot[32];
    __shared__ TopkCtl ctl;
    __shared__ int n_spans;
    __shared__ uint32_t n_total;

    griddep_launch_dependents();
    griddep_wait();  // the indexer's candidate lists are complete
    const int t = blockIdx.x;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t K = static_cast<uint32_t>(a.K);
    int32_t* out = a.idx + static_cast<int64_t>(t) * a.K;
    const int64_t p0 = a.tile_prefix[t], p1 = a.tile_prefix[t + 1], total = a.tile_prefix[a.T];

    if (p0 == p1) {
        for (uint32_t i = tid; i < K; i += kMergeThreads) out[i] = -1;
        return;
    }
    // 1. the segments of row t: CTAs whose tile range meets [p0, p1), 32 at a time by warp 0
    if (tid < 32) {
        const int64_t G = a.G;
        int64_t cf = 0;
        if (tid == 0) {
            cf = (p0 * G) / total;
            if (cf > G - 1) cf = G - 1;
            while (cf + 1 < G && tile_begin(cf + 1, total, G) <= p0) ++cf;
            while (cf > 0 && tile_begin(cf, total, G) > p0) --cf;
        }
        cf = __shfl_sync(0xFFFFFFFFu, cf, 0);
        int ns = 0;
        uint32_t n = 0;
        for (int64_t base = cf;; base += 32) {
            const int64_t c = base + tid;
            const bool in = c < G && tile_begin(c, total, G) < p1;
            const bool seg = in && tile_begin(c + 1, total, G) > tile_begin(c, total, G);
            const uint32_t cnt = seg ? static_cast<uint32_t>(a.slot_count[c + t]) : 0u;
            const bool keep = cnt > 0;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
            uint32_t x = cnt;  // inclusive scan of the counts of this group of 32
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (tid >= static_cast<uint32_t>(o)) x += y;
            }
            const int pos = ns + __popc(bal & ((1u << tid) - 1u));
            if (keep && pos < kMaxSpans) {
                span_ptr[pos] = a.slots + (c + t) * a.K;
                span_off[pos] = n + x - cnt;
            }
            ns += __popc(bal);
            n += __shfl_sync(0xFFFFFFFFu, x, 31);
            if (!__any_sync(0xFFFFFFFFu, in)) break;
        }
        if (tid == 0) {
            if (ns > kMaxSpans) ns = kMaxSpans;
            n_spans = ns;
            span_off[ns] = n;
            n_total = n;
        }
    }
    block_sync();
    const int ns = n_spans;
    const uint32_t n = n_total;

    const uint32_t per = (n + kMergeThreads - 1) / kMergeThreads;

    if (per > static_cast<uint32_t>(kPer)) {
        // Long rows (more candidates than the registers hold): radix select streaming the lists
        // from global memory, then emit them list by list.
        __shared__ uint32_t span_cnt[kMaxSpans];
        for (int q = tid; q < ns; q += kMergeThreads) span_cnt[q] = span_off[q + 1] - span_off[q];
        block_sync();
        const uint64_t thr = radix_threshold<kMergeThreads>(span_ptr, span_cnt, ns, K, hist, &ctl, tid, 1);
        uint32_t out_n = 0;
        for (int q = 0; q < ns; ++q) {
            const uint64_t* sp = span_ptr[q];
            for (uint32_t base = 0; base < span_cnt[q]; base += kMergeThreads) {
                const uint32_t i = base + tid;
                const uint64_t k = (i < span_cnt[q]) ? sp[i] : 0ull;
                const bool p = i < span_cnt[q] && k >= thr;
                uint32_t tot;
                const uint32_t o = out_n + group_excl_scan<kMergeThreads>(p ? 1u : 0u, warp_tot, tid, 1, tot);
                if (p && o < K) out[o] = key_pos(k);
                out_n += tot;
            }
        }
        for (uint32_t i = out_n + tid; i < K; i += kMergeThreads) out[i] = -1;
        return;
    }

    // 2. load: the lists are copied into shared memory in order (coalesced, every load in flight
    //    at once), then thread tid takes the contiguous candidates [c0, c1) into registers
    uint64_t* cand = reinterpret_cast<uint64_t*>(merge_smem + kMergeHistBytes);
    for (int q = 0; q < ns; ++q) {
        const uint64_t* sp = span_ptr[q];
        const uint32_t o = span_off[q], m = span_off[q + 1] - o;
        for (uint32_t i = tid; i < m; i += kMergeThreads) cand[o + i] = __ldcg(sp + i);
    }
    block_sync();
    const uint32_t c0 = min(n, tid * per), c1 = min(n, c0 + per);
    const uint32_t cnt = c1 - c0;
    uint64_t keys[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) keys[j] = (static_cast<uint32_t>(j) < cnt) ? cand[c0 + j] : 0ull;

    // 3. threshold: exactly K keys are >= thr (thr = 0 keeps every candidate when n <= K)
    uint64_t thr = 0ull;
    if (n > K) thr = reg_radix_threshold<kMergeThreads, kPer>(keys, cnt, K, hist, &ctl, tid, 1);

    // 4. emit the positions of the kept keys in candidate order (= ascending position)
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) mine += (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) ? 1u : 0u;
    uint32_t kept;
    uint32_t o = group_excl_scan<kMergeThreads>(mine, warp_tot, tid, 1, kept);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) {
            if (o < K) out[o] = key_pos(keys[j]);
            ++o;
        }
    }
    for (uint32_t i = kept + tid; i < K; i += kMergeThreads) out[i] = -1;
}

bool launch_plan(const IndexerArgs& a, cudaStream_t s, int* launches) {
    plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_merge(const IndexerArgs& a, cudaStream_t s, int* launches) {
    if (a.T == 0) return true;
    const size_t smem = kMergeSmemBytes;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(topk_merge_kernel), smem)) return false;
    if (!launch_kernel(true, topk_merge_kernel, dim3(a.T), dim3(kMergeThreads), smem, s, a)) return false;
    ++*launches;
    return true;
}

}  // namespace dsa
