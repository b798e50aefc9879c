// Top-K of the prefill rows over their score rows (written by indexer_prefill_kernel): one CTA
// per query row, keys ordered by (score desc, position asc) as everywhere in this library.
//
//  1. A sample of the row (16 evenly spaced runs of 256 consecutive scores) gives an admission
//     threshold: the score ranked about 1.5 K / n of the way down the sample.
//  2. One pass over the row, 8192 scores per round read straight into registers (16 consecutive
//     positions per lane); lane and warp count scans place the admitted keys, so the candidate
//     buffer stays in position order.
//  3. If at least K and at most the buffer's 8192 keys were admitted, the K-th key is found
//     among them by a radix select in registers, and the kept positions are written in
//     ascending order; every key of the true Top-K was admitted, since at least K keys score at
//     or above the threshold. Otherwise (a degenerate row: many equal scores, or a sample far
//     from the rest) the row is selected exactly by radix passes streaming its scores.
// Scores that are NaN mark keys of an invalid cache block: they are never selected.
#include "internal.h"

namespace dsa {

constexpr int kPtThreads = 512;
constexpr int kPtPer = 16;                          // consecutive positions per thread per round
constexpr int kPtRound = kPtThreads * kPtPer;       // 8192 scores staged per round
constexpr int kPtCap = 8192;                        // candidate keys in shared memory
constexpr int kPtKeysPer = kPtCap / kPtThreads;     // 16 keys per thread in the final select
constexpr int kPtSampleRuns = 16, kPtSampleRun = 256;
constexpr int kPtSample = kPtSampleRuns * kPtSampleRun;  // 4096
constexpr int kPtSamplePer = kPtSample / kPtThreads;     // 8
constexpr size_t kPtSmem = static_cast<size_t>(kPtCap) * 8 + kPtThreads / 32 * 256 * 4;

__device__ __forceinline__ bool score_valid(uint32_t bits) { return (bits & 0x7FFFFFFFu) <= 0x7F800000u; }

__device__ __forceinline__ uint64_t score_key(uint32_t bits, uint32_t pos) {
    return make_key(__uint_as_float(bits), pos);
}

struct PtShared {
    uint64_t* cand;   // [kPtCap]
    uint32_t* hist;   // [16][256]
    TopkCtl* ctl;
    uint32_t* warp_tot;
};

// One pass over the row: keeps, in position order, the keys >= thr of valid scores in sh.cand
// (the first kPtCap of them) and returns how many there were. Per round of 8192 positions, warp w
// owns 512 consecutive positions and lane l of it the 16 consecutive positions from 16 l, read
// straight from global memory with 16-byte loads: a lane marks its admitted scores in a bit mask,
// a scan of the lanes' counts and of the warps' counts places every lane's keys, so the candidate
// buffer stays in position order with one barrier per round. The admission test is one fp32
// comparison against the threshold's score (the ordered score bits are monotonic in the score,
// with -0 = +0, and NaN fails every comparison); the position half of the key only decides at
// the threshold's own score, and a 64-bit key is built only for the keys that are kept.
__device__ uint32_t compact_row(const float* srow, int n, uint64_t thr, PtShared& sh, uint32_t tid) {
    constexpr int kWarpSpan = kPtRound / (kPtThreads / 32);  // 512
    constexpr int kLanePer = kWarpSpan / 32;                 // 16
    const uint32_t lane = tid & 31u, warp = tid >> 5;
    const uint32_t thr_hi = static_cast<uint32_t>(thr >> 32), thr_lo = static_cast<uint32_t>(thr);
    // the score whose ordered bits are thr_hi (thr_hi = 0, below every valid score: -inf)
    const float thr_f = thr_hi == 0u ? __uint_as_float(0xFF800000u)
                                     : __uint_as_float((thr_hi & 0x80000000u) ? (thr_hi & 0x7FFFFFFFu) : ~thr_hi);
    const bool score_only = thr_lo <= 1u;  // 1: every valid key (positions never reach 0xFFFFFFFF)
    uint32_t total = 0, parity = 0;
    for (int base = 0; base < n; base += kPtRound, parity ^= 1u) {
        const int p0 = base + static_cast<int>(warp) * kWarpSpan + static_cast<int>(lane) * kLanePer;
        float x[kLanePer];
#pragma unroll
        for (int k = 0; k < kLanePer / 4; ++k) {
            // the row holds max_blocks * 64 scores (a multiple of 4): a 16-byte load that starts
            // before n stays inside it; positions at or past n are masked below
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (p0 + 4 * k < n) v = __ldcs(reinterpret_cast<const float4*>(srow + p0 + 4 * k));
            x[4 * k] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < kLanePer; ++j) {
            const int p = p0 + j;
            const uint32_t lo = 0xFFFFFFFFu - static_cast<uint32_t>(p);
            const bool pass = p < n && (score_only ? (x[j] >= thr_f) : (x[j] > thr_f || (x[j] == thr_f && lo >= thr_lo)));
            mask |= (pass ? 1u : 0u) << j;
        }
        const uint32_t c = static_cast<uint32_t>(__popc(mask));
        uint32_t incl = c;  // inclusive scan of the lanes' counts
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= static_cast<uint32_t>(o)) incl += y;
        }
        // warp totals alternate between two halves of warp_tot: the next round may write its
        // totals while a slower warp still reads this round's
        uint32_t* wt = sh.warp_tot + parity * (kPtThreads / 32);
        if (lane == 31) wt[warp] = incl;
        block_sync();
        uint32_t off = total + incl - c, round_total = 0;
#pragma unroll
        for (uint32_t w = 0; w < kPtThreads / 32; ++w) {
            const uint32_t cw = wt[w];
            off += (w < warp) ? cw : 0u;
            round_total += cw;
        }
#pragma unroll
        for (int j = 0; j < kLanePer; ++j) {
            if ((mask >> j) & 1u) {
                if (off < static_cast<uint32_t>(kPtCap))
                    sh.cand[off] = (static_cast<uint64_t>(ordered_bits(x[j])) << 32) |
                                   (0xFFFFFFFFu - static_cast<uint32_t>(p0 + j));
                ++off;
            }
        }
        total += round_total;
    }
    block_sync();  // the candidates are complete
    return total;
}

// Exact threshold over the whole row streamed from global memory: MSB-first radix select with
// 8-bit digits on the 64-bit keys (slow path for degenerate rows; nvalid > K).
__device__ uint64_t row_radix_threshold(const float* srow, int n, uint32_t K, PtShared& sh, uint32_t tid) {
    constexpr uint32_t NW = kPtThreads / 32;
    const uint32_t lane = tid & 31u, warp = tid >> 5;
    uint32_t* my_hist = sh.hist + warp * 256;
    uint64_t prefix = 0;
    uint32_t rem = K;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (uint32_t i = lane; i < 256; i += 32) my_hist[i] = 0;
        __syncwarp();
        for (int base = 0; base < n; base += kPtThreads * 4) {
            uint32_t bits[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = base + k * kPtThreads + static_cast<int>(tid);
                bits[k] = (i < n) ? __ldcg(reinterpret_cast<const uint32_t*>(srow) + i) : 0x7FC00000u;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = base + k * kPtThreads + static_cast<int>(tid);
                const uint64_t key = score_key(bits[k], static_cast<uint32_t>(i));
                const bool match = i < n && score_valid(bits[k]) &&
                                   (shift == 56 || (key >> (shift + 8)) == (prefix >> (shift + 8)));
                if (match) atomicAdd(&my_hist[static_cast<uint32_t>(key >> shift) & 255u], 1u);
            }
        }
        named_bar_sync(2, kPtThreads);
        for (uint32_t bin = tid; bin < 256; bin += kPtThreads) {
            uint32_t c = sh.hist[bin];
#pragma unroll
            for (uint32_t w = 1; w < NW; ++w) c += sh.hist[w * 256 + bin];
            sh.hist[bin] = c;
        }
        named_bar_sync(2, kPtThreads);
        if (tid < 32) {
            uint32_t c = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) c += sh.hist[lane * 8 + q];
            uint32_t Sx = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, Sx, o);
                if (lane + o < 32) Sx += v;
            }
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, Sx >= rem);
            const int L = 31 - __clz(mask);
            if (static_cast<int>(lane) == L) {
                uint32_t running = Sx - c;
                for (int q = 7; q >= 0; --q) {
                    const uint32_t h = sh.hist[lane * 8 + q];
                    if (running + h >= rem) {
                        sh.ctl->digit = lane * 8 + q;
                        sh.ctl->above = running;
                        sh.ctl->bucket = h;
                        break;
                    }
                    running += h;
                }
            }
        }
        named_bar_sync(2, kPtThreads);
        rem -= sh.ctl->above;
        prefix |= static_cast<uint64_t>(sh.ctl->digit) << shift;
        const bool done = sh.ctl->bucket == rem;
        named_bar_sync(2, kPtThreads);
        if (done) break;
    }
    return prefix;
}

__global__ void __launch_bounds__(kPtThreads, 2) prefill_topk_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t pt_smem[];
    __shared__ TopkCtl ctl;
    __shared__ uint32_t warp_tot[32];
    griddep_launch_dependents();
    griddep_wait();  // the scores (and the plan) are complete
    const int t = blockIdx.x;
    if (!gemm_row(a, t)) return;
    const uint32_t tid = threadIdx.x;
    PtShared sh{reinterpret_cast<uint64_t*>(pt_smem), reinterpret_cast<uint32_t*>(pt_smem + static_cast<size_t>(kPtCap) * 8),
                &ctl, warp_tot};
    const uint32_t K = static_cast<uint32_t>(a.K);
    const int n = row_len(a, t);
    const float* srow = a.scores + static_cast<int64_t>(t) * a.max_blocks * kBlock;
    int32_t* out = a.idx + static_cast<int64_t>(t) * a.K;

    // 1. admission threshold from a sample (rows that fit the buffer whole admit every key)
    uint64_t thr = 1ull;  // every valid key (valid keys are >= 0x007FFFFF << 32)
    if (n > kPtCap) {
        uint64_t skeys[kPtSamplePer];
#pragma unroll
        for (int k = 0; k < kPtSamplePer; ++k) {
            const int i = k * kPtThreads + static_cast<int>(tid);  // sample entry
            const int run = i / kPtSampleRun;
            const int pos = static_cast<int>(static_cast<int64_t>(run) * (n - kPtSampleRun) / (kPtSampleRuns - 1)) +
                            i % kPtSampleRun;
            const uint32_t bits = __ldcg(reinterpret_cast<const uint32_t*>(srow) + pos);
            // invalid scores take the lowest key (0), so they only lower the threshold
            skeys[k] = score_valid(bits) ? score_key(bits, static_cast<uint32_t>(pos)) : 0ull;
        }
        // the sample entry of rank r ~ 1.5 K * (sample / n): about 1.5 K keys of the row above it
        const uint32_t r = max(1u, static_cast<uint32_t>((static_cast<uint64_t>(3 * K / 2) * kPtSample + n - 1) / n));
        const uint64_t st = reg_radix_threshold<kPtThreads, kPtSamplePer>(skeys, kPtSamplePer, r, sh.hist, &ctl, tid, 2);
        thr = (st >> 32) << 32;  // every position with that score or more
        if (thr == 0ull) thr = 1ull;
    }

    // 2. one pass: the admitted keys, in position order
    uint32_t cnt = compact_row(srow, n, thr, sh, tid);
    if (cnt < K && thr > 1ull) {  // the threshold was above the K-th key: admit every valid key
        thr = 1ull;
        cnt = compact_row(srow, n, thr, sh, tid);
    }

    // 3. exact selection among the candidates, or over the streamed row when they overflowed
    uint64_t kth = 1ull;
    if (cnt <= static_cast<uint32_t>(kPtCap)) {
        const uint32_t per = (cnt + kPtThreads - 1) / kPtThreads;
        const uint32_t c0 = min(cnt, tid * per), c1 = min(cnt, c0 + per);
        uint64_t keys[kPtKeysPer];
#pragma unroll
        for (int j = 0; j < kPtKeysPer; ++j) keys[j] = (static_cast<uint32_t>(j) < c1 - c0) ? sh.cand[c0 + j] : 0ull;
        if (cnt > K) kth = reg_radix_threshold<kPtThreads, kPtKeysPer>(keys, c1 - c0, K, sh.hist, &ctl, tid, 2);
        block_sync();
    } else {
        kth = row_radix_threshold(srow, n, K, sh, tid);
        cnt = compact_row(srow, n, kth, sh, tid);  // exactly K keys, in position order
    }
    // 4. positions of the keys >= kth, ascending (candidate order), then -1 up to K
    if (cnt <= static_cast<uint32_t>(kPtCap) && kth > 1ull) {
        // keep the candidates >= kth in order (compaction in place through registers)
        const uint32_t per = (cnt + kPtThreads - 1) / kPtThreads;
        const uint32_t c0 = min(cnt, tid * per), c1 = min(cnt, c0 + per);
        uint64_t keys[kPtKeysPer];
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kPtKeysPer; ++j) {
            keys[j] = (static_cast<uint32_t>(j) < c1 - c0) ? sh.cand[c0 + j] : 0ull;
            mine += (static_cast<uint32_t>(j) < c1 - c0 && keys[j] >= kth) ? 1u : 0u;
        }
        uint32_t kept;
        uint32_t o = group_excl_scan<kPtThreads>(mine, warp_tot, tid, 2, kept);
#pragma unroll
        for (int j = 0; j < kPtKeysPer; ++j)
            if (static_cast<uint32_t>(j) < c1 - c0 && keys[j] >= kth) sh.cand[o++] = keys[j];
        block_sync();
        cnt = kept;
    }
    const uint32_t m = min(cnt, K);
    for (uint32_t i = tid; i < K; i += kPtThreads) out[i] = (i < m) ? key_pos(sh.cand[i]) : -1;
}

bool launch_prefill_topk(const IndexerArgs& a, cudaStream_t s, int* launches) {
    if (a.NG == 0) return true;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(prefill_topk_kernel), kPtSmem)) return false;
    if (!launch_kernel(true, prefill_topk_kernel, dim3(4 * a.NG), dim3(kPtThreads), kPtSmem, s, a)) return false;
    ++*launches;
    return true;
}

}  // namespace dsa
