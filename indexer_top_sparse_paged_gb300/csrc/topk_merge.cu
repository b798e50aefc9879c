// Work plan and Top-K merge.
//
// plan:  which groups of 4 prefill rows run on the score GEMM, tile_prefix[t] = number of 128-key
//        tiles of the decode-path rows before row t, the merge groups of every decode-path row,
//        and the tile prefix of the GEMM groups (one CTA).
// merge: the candidate lists that the indexer CTAs left for a row's segments (each already cut
//        to at most K keys, in position order) are reduced by a tree with fan-in 8. A merge
//        CTA selects the K largest keys of up to 8 lists with an MSB-first radix select over
//        keys held in registers. A group that covers the whole row writes its positions in
//        ascending order, then -1 up to K; any other group writes its keys back over its first
//        list, and the last of 8 sibling groups to finish (a counter per parent group) goes on
//        to merge the parent's lists, up to the row's root. Lists of long segments were
//        filtered by a sample estimate of the row's K-th key; the root checks that at least K
//        candidates reach every estimate used and otherwise selects the row again from all of
//        its keys (rescore_row) ("Engineering Path for Day-0
//        Adaptation ..." §3.1: Top-K filtering over large candidate sets is split to match the
//        hardware's thread organisation; "Adapting GPU Software Stacks ..." §3.1: the index
//        format is aligned with the attention that consumes it, so no reordering is needed).
#include "internal.h"

namespace dsa {

constexpr int kPlanThreads = 1024;
constexpr int kMergeThreads = 512;
constexpr int kMergeSmemKeys = 16384;  // candidates held in registers (32 per thread)
constexpr int kMergeHistBytes = kMergeThreads / 32 * 256 * 4;  // one 256-bin histogram per warp
constexpr int kRescoreHeads = 64, kRescoreDim = 128;            // the tensor-core indexer's shape
constexpr int kRescoreBytes = kRescoreHeads * kRescoreDim * 2 + kRescoreHeads * 4;  // a row's q_I (bf16) and w
// per-warp histograms + the row's candidates + the recovery path's query and head weights
constexpr int kMergeSmemBytes = kMergeHistBytes + kMergeSmemKeys * 8 + kRescoreBytes;

// Exclusive scan of v over the block (kPlanThreads threads, in thread order), plus the total.
__device__ __forceinline__ int plan_scan(int v, int* warp_sums, int& total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int x = v;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    block_sync();
    if (warp == 0) {
        int y = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xFFFFFFFFu, y, o);
            if (lane >= o) y += z;
        }
        warp_sums[lane] = y;  // inclusive over warps
    }
    block_sync();
    const int excl = (warp ? warp_sums[warp - 1] : 0) + x - v;
    total = warp_sums[31];
    block_sync();  // warp_sums is rewritten by the next call
    return excl;
}

// Merge groups of row t: lists come from the CTAs c_first..c_last that own the row's tiles
// [p0, p1), kMergeFanIn consecutive CTA indices per group (a row without tiles has one group).
__device__ __forceinline__ int merge_groups(int64_t p0, int64_t p1, int64_t total, int64_t G) {
    if (p1 <= p0) return 1;  // one group writes the row's -1s
    const int64_t n = tile_owner(p1 - 1, total, G) - tile_owner(p0, total, G) + 1;
    return static_cast<int>((n + kMergeFanIn - 1) / kMergeFanIn);
}

// Does group g (rows 4g..4g+3) run on the prefill score GEMM? All four rows belong to one
// valid sequence.
__device__ __forceinline__ bool group_on_gemm(const IndexerArgs& a, int g) {
    if (g >= a.NG) return false;
    const int b = a.q_seq[4 * g];
    if (b < 0 || b >= a.B) return false;
    return a.q_seq[4 * g + 1] == b && a.q_seq[4 * g + 2] == b && a.q_seq[4 * g + 3] == b;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(IndexerArgs a) {
    __shared__ int warp_sums[32];
    griddep_launch_dependents();  // the indexer may start its prologue
    const int tid = threadIdx.x;
    // 1. GEMM groups; tiles per row of the decode path (GEMM rows have none) -> tile_prefix
    int carry = 0;
    for (int base = 0; base < a.T; base += kPlanThreads) {
        const int t = base + tid;
        int tiles = 0;
        if (t < a.T) {
            const bool gemm = group_on_gemm(a, t >> 2);
            if ((t & 3) == 0 && (t >> 2) < a.NG) a.gemm_flag[t >> 2] = gemm ? 1 : 0;
            if (!gemm) tiles = (row_len(a, t) + kTileKeys - 1) / kTileKeys;
        }
        int sum;
        const int excl = plan_scan(tiles, warp_sums, sum);
        if (t < a.T) a.tile_prefix[t] = carry + excl;
        carry += sum;
    }
    if (tid == 0) a.tile_prefix[a.T] = carry;
    block_sync();
    // 2. merge groups per row (none for GEMM rows) -> group_prefix; their counters start at zero
    const int64_t total = carry;
    int gcarry = 0;
    for (int base = 0; base < a.T; base += kPlanThreads) {
        const int t = base + tid;
        const int g = (t < a.T && !gemm_row(a, t)) ? merge_groups(a.tile_prefix[t], a.tile_prefix[t + 1], total, a.G) : 0;
        int sum;
        const int excl = plan_scan(g, warp_sums, sum);
        if (t < a.T) {
            a.group_prefix[t] = gcarry + excl;
            const int GB = merge_group_bound(a.T, a.G);
            for (int l = 0; l < kMergeLevels - 1; ++l)
                for (int i = 0; i < g; ++i) a.merge_count[l * GB + gcarry + excl + i] = 0;
        }
        gcarry += sum;
    }
    if (tid == 0) a.group_prefix[a.T] = gcarry;
    // 3. tiles of the GEMM groups (their longest causal prefix) -> gemm_tile_prefix
    int tcarry = 0;
    for (int base = 0; base < a.NG; base += kPlanThreads) {
        const int g = base + tid;
        int tiles = 0;
        if (g < a.NG && a.gemm_flag[g]) {
            int n = 0;
            for (int q = 0; q < 4; ++q) n = max(n, row_len(a, 4 * g + q));
            tiles = (n + kTileKeys - 1) / kTileKeys;
        }
        int sum;
        const int excl = plan_scan(tiles, warp_sums, sum);
        if (g < a.NG) a.gemm_tile_prefix[g] = tcarry + excl;
        tcarry += sum;
    }
    if (tid == 0 && a.NG > 0) a.gemm_tile_prefix[a.NG] = tcarry;
}

constexpr int kPer = kMergeSmemKeys / kMergeThreads;  // candidates per thread held in registers
static_assert(kMergeFanIn * 2048 <= kMergeSmemKeys, "a merge group must fit the registers");

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The exact Top-K of row t, every causal key rescored on the CUDA cores and streamed through an
// exact selection: the recovery path of a row whose sample estimates turned away keys of its Top-K
// (TopkGroup::estimate). Only rows of the tensor-core decode indexer take estimates, so the keys
// are 64 heads x 128 wide, bf16, FP8 e4m3 with a block scale or MXFP8 (q_I then holds the
// quantised query, as the indexer used it). Writes idx row `out`: ascending positions, then -1.
__device__ __noinline__ void rescore_row(const IndexerArgs& a, int t, int32_t* out, uint64_t* cand, uint32_t* hist,
                                         TopkCtl* ctl, uint8_t* scratch, uint32_t tid) {
    constexpr int H = kRescoreHeads, D = kRescoreDim;
    uint32_t* q_s = reinterpret_cast<uint32_t*>(scratch);  // [H][D / 2] bf16 pairs
    float* w_s = reinterpret_cast<float*>(scratch + H * D * 2);
    const uint32_t* q = static_cast<const uint32_t*>(a.q_I) + static_cast<int64_t>(t) * H * (D / 2);
    for (uint32_t i = tid; i < H * D / 2; i += kMergeThreads) q_s[i] = q[i];
    if (tid < static_cast<uint32_t>(H)) w_s[tid] = a.w[static_cast<int64_t>(t) * H + tid];
    TopkGroup<kMergeThreads, kPer> g{cand, hist, ctl, static_cast<uint32_t>(kMergeSmemKeys), static_cast<uint32_t>(a.K),
                                     tid, 1};
    g.reset();  // a group barrier: q_s and w_s are visible
    const int b = row_seq(a, t);
    const int n = row_len(a, t);
    const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    for (int base = 0; base < n; base += kMergeThreads) {
        const int s = base + static_cast<int>(tid);
        int blk = -1;
        if (s < n) {
            blk = bt[s >> 6];
            if (blk < 0 || blk >= a.num_blocks) {
                atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
                blk = -1;
            }
        }
        float score = 0.0f;
        if (blk >= 0) {
            const int64_t row = static_cast<int64_t>(blk) * kBlock + (s & 63);
            uint32_t kp[D / 2];  // the key as bf16 pairs (exact for every storage)
            float sc = 1.0f;
            if (a.mode == DSA_BF16) {
                const uint4* src = static_cast<const uint4*>(a.k_I) + row * (D * 2 / 16);
#pragma unroll
                for (int c = 0; c < D * 2 / 16; ++c) {
                    const uint4 v = src[c];
                    kp[4 * c] = v.x;
                    kp[4 * c + 1] = v.y;
                    kp[4 * c + 2] = v.z;
                    kp[4 * c + 3] = v.w;
                }
            } else {
                const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.k_I) + row * D);
                uint32_t mx = 0;
                if (a.mode == DSA_MXFP8) mx = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(a.k_I_scale) + row * (D / 32));
                else sc = static_cast<const float*>(a.k_I_scale)[blk];
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint4 lo, hi;
                    if (a.mode == DSA_MXFP8) e4m3x16_to_bf16_scaled(src[c], e8m0_value((mx >> (8 * (c >> 1))) & 0xFFu), lo, hi);
                    else e4m3x16_to_bf16(src[c], lo, hi);
                    kp[8 * c] = lo.x;
                    kp[8 * c + 1] = lo.y;
                    kp[8 * c + 2] = lo.z;
                    kp[8 * c + 3] = lo.w;
                    kp[8 * c + 4] = hi.x;
                    kp[8 * c + 5] = hi.y;
                    kp[8 * c + 6] = hi.z;
                    kp[8 * c + 7] = hi.w;
                }
            }
#pragma unroll 1
            for (int j = 0; j < H; ++j) {
                const uint32_t* qj = q_s + j * (D / 2);
                float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
                for (int i = 0; i < D / 2; ++i) {
                    const uint32_t qw = qj[i];
                    d0 = fmaf(bf16_lo(qw), bf16_lo(kp[i]), d0);
                    d1 = fmaf(bf16_hi(qw), bf16_hi(kp[i]), d1);
                }
                score = fmaf(w_s[j], fmaxf((d0 + d1) * sc, 0.0f), score);
            }
        }
        g.push(make_key(score, static_cast<uint32_t>(s)), blk >= 0);
    }
    const uint32_t kept = g.select_to(cand);  // the K largest, in position order
    g.sync();
    for (uint32_t i = tid; i < static_cast<uint32_t>(a.K); i += kMergeThreads) out[i] = (i < kept) ? key_pos(cand[i]) : -1;
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t merge_smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(merge_smem);  // [16 warps][256]
    uint64_t* cand = reinterpret_cast<uint64_t*>(merge_smem + kMergeHistBytes);
    uint8_t* rescore_scratch = merge_smem + kMergeHistBytes + kMergeSmemKeys * 8;
    __shared__ const uint64_t* span_ptr[kMergeFanIn];
    __shared__ uint32_t span_off[kMergeFanIn + 1];
    __shared__ unsigned long long group_est;  // the largest sample estimate any of the group's lists used
    __shared__ uint32_t warp_tot[32];
    __shared__ TopkCtl ctl;
    __shared__ int row_found;
    __shared__ int is_last;

    griddep_launch_dependents();
    griddep_wait();  // the indexer's candidate lists and the plan are complete
    const uint32_t tid = threadIdx.x, lane = tid & 31u;
    const int b = blockIdx.x;
    if (b >= a.group_prefix[a.T]) return;  // the grid is an upper bound on the groups
    // row t with group_prefix[t] <= b < group_prefix[t + 1], one row per thread (one round trip
    // to memory for up to kMergeThreads rows, where a binary search would chain several)
    if (tid == 0) row_found = -1;
    block_sync();
    for (int base = 0; base < a.T; base += kMergeThreads) {
        const int r = base + static_cast<int>(tid);
        if (r < a.T && a.group_prefix[r] <= b && b < a.group_prefix[r + 1]) row_found = r;
        block_sync();
        if (row_found >= 0) break;
    }
    const int t = row_found;
    if (t < 0) return;
    const uint32_t K = static_cast<uint32_t>(a.K);
    int32_t* out = a.idx + static_cast<int64_t>(t) * a.K;
    const int64_t p0 = a.tile_prefix[t], p1 = a.tile_prefix[t + 1], total = a.tile_prefix[a.T];
    if (p0 == p1) {
        for (uint32_t i = tid; i < K; i += kMergeThreads) out[i] = -1;
        return;
    }
    const int64_t G = a.G;
    const int64_t c_first = tile_owner(p0, total, G);
    const int gp_t = a.group_prefix[t];
    const int GB = merge_group_bound(a.T, a.G);

    // Level 0 lists: the slots c_first + i of the CTAs that own the row's tiles (a CTA with an
    // empty tile range left none). A group of level L >= 1 covers lists 8g..8g+7 of level L - 1;
    // list i of level L - 1 lives in slot c_first + i * 8^(L-1) (its first CTA's slot).
    int g = b - gp_t;
    int64_t nprev = tile_owner(p1 - 1, total, G) - c_first + 1;
    int64_t stride = 1;  // 8^(L-1)
    for (int level = 1;; ++level) {
        const int64_t ncur = (nprev + kMergeFanIn - 1) / kMergeFanIn;
        // 1. the group's lists (warp 0)
        if (tid < 32) {
            const int64_t i = static_cast<int64_t>(g) * kMergeFanIn + lane;
            const int64_t c = c_first + i * stride;
            bool has = lane < static_cast<uint32_t>(kMergeFanIn) && i < nprev;
            if (has && level == 1) has = tile_begin(c + 1, total, G) > tile_begin(c, total, G);
            const uint32_t cnt = has ? static_cast<uint32_t>(__ldcg(a.slot_count + c + t)) : 0u;
            unsigned long long est = has ? static_cast<unsigned long long>(__ldcg(a.slot_est + c + t)) : 0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, est, o);
                est = other > est ? other : est;
            }
            if (lane == 0) group_est = est;
            const bool keep = cnt > 0;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
            uint32_t x = cnt;  // inclusive scan of the counts
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= static_cast<uint32_t>(o)) x += y;
            }
            const int pos = __popc(bal & ((1u << lane) - 1u));
            if (keep) {
                span_ptr[pos] = a.slots + (c + t) * a.K;
                span_off[pos] = x - cnt;
            }
            if (lane == 31) {
                const int ns = __popc(bal);
                for (int q = ns; q <= kMergeFanIn; ++q) span_off[q] = x;  // empty tail spans
            }
        }
        block_sync();
        const uint32_t n = span_off[kMergeFanIn];

        // 2. stage the lists in shared memory, in order: a list holds at most K <= 2048 keys, so
        //    every thread issues its (at most) 4 loads per list, all before its first store
        {
            constexpr int kPerList = 2048 / kMergeThreads;
            uint64_t v[kMergeFanIn][kPerList];
#pragma unroll
            for (int q = 0; q < kMergeFanIn; ++q) {
                const uint32_t m = span_off[q + 1] - span_off[q];
                const uint64_t* sp = span_ptr[q];
#pragma unroll
                for (int j = 0; j < kPerList; ++j) {
                    const uint32_t i = static_cast<uint32_t>(j) * kMergeThreads + tid;
                    v[q][j] = (i < m) ? __ldcg(sp + i) : 0ull;
                }
            }
#pragma unroll
            for (int q = 0; q < kMergeFanIn; ++q) {
                const uint32_t o = span_off[q], m = span_off[q + 1] - o;
#pragma unroll
                for (int j = 0; j < kPerList; ++j) {
                    const uint32_t i = static_cast<uint32_t>(j) * kMergeThreads + tid;
                    if (i < m) cand[o + i] = v[q][j];
                }
            }
        }
        block_sync();
        const uint32_t per = (n + kMergeThreads - 1) / kMergeThreads;
        const uint32_t c0 = min(n, tid * per), c1 = min(n, c0 + per);
        const uint32_t cnt = c1 - c0;
        uint64_t keys[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) keys[j] = (static_cast<uint32_t>(j) < cnt) ? cand[c0 + j] : 0ull;

        // 3. at the row's root, the sample estimates are checked: if at least K candidates are >=
        //    every estimate used, no key of the row's Top-K was turned away (then the K largest
        //    candidates are the row's Top-K); otherwise the row is rescored
        const uint64_t est = group_est;
        if (ncur == 1 && est != 0ull) {
            uint32_t above = 0;
#pragma unroll
            for (int j = 0; j < kPer; ++j) above += (static_cast<uint32_t>(j) < cnt && keys[j] >= est) ? 1u : 0u;
            uint32_t total_above;
            group_excl_scan<kMergeThreads>(above, warp_tot, tid, 1, total_above);
            if (total_above < K) {
                rescore_row(a, t, out, cand, hist, &ctl, rescore_scratch, tid);
                return;
            }
        }
        // 4. threshold: exactly K keys are >= thr (thr = 0 keeps every candidate when n <= K)
        uint64_t thr = 0ull;
        if (n > K) thr = reg_radix_threshold<kMergeThreads, kPer>(keys, cnt, K, hist, &ctl, tid, 1);
        if (est > thr) thr = est;  // keys below an estimate the row used never reach its Top-K (see 3.)

        // 5. the kept keys in candidate order (= ascending position), compacted in shared memory
        //    (over the staged candidates: every thread has its keys in registers) and written out
        //    with coalesced stores: the row's positions at the root, else the keys back over the
        //    group's first list
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) mine += (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) ? 1u : 0u;
        uint32_t kept;
        uint32_t o = group_excl_scan<kMergeThreads>(mine, warp_tot, tid, 1, kept);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) cand[o++] = keys[j];
        }
        block_sync();
        if (ncur == 1) {
            for (uint32_t i = tid; i < K; i += kMergeThreads) out[i] = (i < kept) ? key_pos(cand[i]) : -1;
            return;
        }
        // the group's first list slot: written only by its own segment (c, t), or by no segment
        const int64_t cdst = c_first + static_cast<int64_t>(g) * kMergeFanIn * stride;
        uint64_t* dst = a.slots + (cdst + t) * a.K;
        for (uint32_t i = tid; i < kept; i += kMergeThreads) dst[i] = cand[i];
        if (tid == 0) {
            a.slot_count[cdst + t] = static_cast<int32_t>(kept);
            a.slot_est[cdst + t] = est;  // the parent checks the estimates of all the row's lists
        }
        block_sync();
        // 6. the last of the parent's children to finish merges the parent's lists
        const int parent = g / kMergeFanIn;
        const int64_t left = ncur - static_cast<int64_t>(parent) * kMergeFanIn;
        const int children = left < kMergeFanIn ? static_cast<int>(left) : kMergeFanIn;
        if (tid == 0) {
            __threadfence();  // this group's list before the count that publishes it
            int* counter = a.merge_count + (level - 1) * GB + gp_t + static_cast<int64_t>(parent) * kMergeFanIn * stride;
            is_last = atomicAdd(counter, 1) == children - 1;
        }
        block_sync();
        if (!is_last) return;
        __threadfence();  // the siblings' lists are visible to this CTA
        g = parent;
        nprev = ncur;
        stride *= kMergeFanIn;
    }
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
    // one CTA per merge group: at most T + G / 8 groups over all rows (the plan has the exact count)
    const int grid = merge_group_bound(a.T, a.G);
    if (!launch_kernel(true, topk_merge_kernel, dim3(grid), dim3(kMergeThreads), smem, s, a)) return false;
    ++*launches;
    return true;
}

}  // namespace dsa
