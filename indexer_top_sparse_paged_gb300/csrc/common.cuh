// Shared device-side building blocks of the indexer kernels:
//  * the 64-bit selection key (score order, then lower position first),
//  * the work plan that cuts all query rows' key tiles into equal contiguous CTA ranges,
//  * the streaming Top-K buffer (threshold filter + radix select) kept in shared memory.
//
// Index selection is scoring followed by Top-K filtering with a discrete index set as output
// ("Engineering Path for Day-0 Adaptation ... on Domestic AI Accelerators" §3.1); its core loop
// must avoid intra-warp divergence and keep intermediate indices on chip ("Adapting GPU Software
// Stacks ..." §3.1). Candidates are compacted with warp ballots and prefix sums (no divergent
// per-thread insertion), and only the per-CTA survivors leave shared memory.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace dsa {

constexpr int kBlock = 64;      // tokens per physical cache block
constexpr int kTileKeys = 128;  // keys per indexer tile (two cache blocks)

// ------------------------------------------------------------------------------------------------
// selection key: larger key = better. High word: the fp32 score mapped to an unsigned integer
// with the same order (-0 mapped onto +0); low word: 0xFFFFFFFF - position, so that among
// equal scores the lower position has the larger key. Keys of distinct positions never tie.
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ordered_bits(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float score, uint32_t pos) {
    return (static_cast<uint64_t>(ordered_bits(score)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - pos);
}

__device__ __forceinline__ int32_t key_pos(uint64_t key) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

// ------------------------------------------------------------------------------------------------
// work plan
//   tile_prefix[t] = sum over rows r < t of ceil(n_r / kTileKeys), n_r = causal prefix length.
//   CTA c of G owns global tiles [tile_begin(c), tile_begin(c+1)), cut at row boundaries into
//   segments; the candidates of segment (c, t) go to slot c + t (unique: along the tile order
//   c + t strictly increases from one segment to the next).
// ------------------------------------------------------------------------------------------------

__host__ __device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t total, int64_t G) {
    return c * total / G;
}

// First row t with tile_prefix[t] <= tile < tile_prefix[t + 1] (tile < total).
__device__ __forceinline__ int row_of_tile(const int32_t* tile_prefix, int T, int64_t tile) {
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tile_prefix[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct Segment {
    int row;        // query row
    int tile0;      // first tile within the row
    int tile1;      // one past the last tile within the row
};

// Iterates the segments of one CTA in order.
struct SegmentIter {
    const int32_t* tile_prefix;
    int T;
    int64_t cur, end;
    int row;

    __device__ void init(const int32_t* tp, int T_, int c, int G) {
        tile_prefix = tp;
        T = T_;
        const int64_t total = tp[T_];
        cur = tile_begin(c, total, G);
        end = tile_begin(c + 1, total, G);
        row = (cur < end) ? row_of_tile(tp, T_, cur) : T_;
    }
    __device__ bool next(Segment& s) {
        while (cur < end && row < T) {
            const int64_t r0 = tile_prefix[row], r1 = tile_prefix[row + 1];
            if (r1 <= cur) { ++row; continue; }
            const int64_t e = r1 < end ? r1 : end;
            s.row = row;
            s.tile0 = static_cast<int>(cur - r0);
            s.tile1 = static_cast<int>(e - r0);
            cur = e;
            ++row;
            return true;
        }
        return false;
    }
};

// ------------------------------------------------------------------------------------------------
// streaming Top-K buffer in shared memory, driven collectively by NT threads (one named barrier)
// ------------------------------------------------------------------------------------------------

struct TopkCtl {
    uint32_t count;
    uint32_t theta_lo, theta_hi;  // admission threshold: keys below it cannot be in the Top-K
    uint32_t digit, above, bucket;
    uint32_t warp_cnt[32];
};

template <int NT>
struct TopkGroup {
    uint64_t* buf;   // [cap]
    uint32_t* hist;  // [256]
    TopkCtl* ctl;
    uint32_t cap;    // >= K + NT
    uint32_t K;
    uint32_t tid;    // 0..NT-1
    uint32_t bar_id;

    __device__ __forceinline__ void sync() const { named_bar_sync(bar_id, NT); }

    __device__ void reset() {
        if (tid == 0) {
            ctl->count = 0;
            ctl->theta_lo = 0;
            ctl->theta_hi = 0;
        }
        sync();
    }

    // Stable compaction of buf[0, count) keeping keys >= thr; returns the kept count (uniform).
    __device__ uint32_t compact(uint32_t count, uint64_t thr) {
        const uint32_t lane = tid & 31u, warp = tid >> 5;
        uint32_t out = 0;
        for (uint32_t base = 0; base < count; base += NT) {
            const uint32_t i = base + tid;
            const uint64_t k = (i < count) ? buf[i] : 0ull;
            const bool p = (i < count) && (k >= thr);
            const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, p);
            if (lane == 0) ctl->warp_cnt[warp] = __popc(ballot);
            sync();
            uint32_t off = 0, total = 0;
#pragma unroll
            for (uint32_t w = 0; w < NT / 32; ++w) {
                const uint32_t c = ctl->warp_cnt[w];
                off += (w < warp) ? c : 0u;
                total += c;
            }
            if (p) buf[out + off + __popc(ballot & ((1u << lane) - 1u))] = k;
            sync();
            out += total;
        }
        return out;
    }

    // Keeps exactly the K largest of buf[0, count) (count > K), in their original order, and
    // raises the admission threshold to the smallest kept key's radix prefix.
    __device__ void select(uint32_t count) {
        uint64_t prefix = 0;
        uint32_t rem = K;
        const uint32_t lane = tid & 31u;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (uint32_t i = tid; i < 256; i += NT) hist[i] = 0;
            sync();
            for (uint32_t i = tid; i < count; i += NT) {
                const uint64_t k = buf[i];
                const bool match = (shift == 56) || ((k >> (shift + 8)) == (prefix >> (shift + 8)));
                if (match) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            sync();
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
                            ctl->digit = lane * 8 + b;
                            ctl->above = running;
                            ctl->bucket = h;
                            break;
                        }
                        running += h;
                    }
                }
            }
            sync();
            const uint32_t dg = ctl->digit;
            rem -= ctl->above;
            prefix |= static_cast<uint64_t>(dg) << shift;
            if (ctl->bucket == rem) break;  // the whole bucket is selected
        }
        const uint32_t kept = compact(count, prefix);
        if (tid == 0) {
            ctl->count = kept;
            ctl->theta_lo = static_cast<uint32_t>(prefix);
            ctl->theta_hi = static_cast<uint32_t>(prefix >> 32);
        }
        sync();
    }

    // Collective: every thread offers at most one key per call.
    __device__ void push(uint64_t key, bool valid) {
        uint32_t count = ctl->count;
        if (count + NT > cap) {
            select(count);
            count = ctl->count;
        }
        const uint64_t theta = (static_cast<uint64_t>(ctl->theta_hi) << 32) | ctl->theta_lo;
        const bool p = valid && key >= theta;
        const uint32_t lane = tid & 31u, warp = tid >> 5;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, p);
        if (lane == 0) ctl->warp_cnt[warp] = __popc(ballot);
        sync();
        uint32_t off = 0, total = 0;
#pragma unroll
        for (uint32_t w = 0; w < NT / 32; ++w) {
            const uint32_t c = ctl->warp_cnt[w];
            off += (w < warp) ? c : 0u;
            total += c;
        }
        if (p) buf[count + off + __popc(ballot & ((1u << lane) - 1u))] = key;
        sync();
        if (tid == 0) ctl->count = count + total;
        sync();
    }

    // Collective: reduces to at most K keys (in position order) and writes them to `out`.
    __device__ void flush(uint64_t* out, int32_t* count_out) {
        uint32_t count = ctl->count;
        if (count > K) {
            select(count);
            count = ctl->count;
        }
        for (uint32_t i = tid; i < count; i += NT) out[i] = buf[i];
        if (tid == 0) *count_out = static_cast<int32_t>(count);
    }
};

// ------------------------------------------------------------------------------------------------
// kernel parameter blocks
// ------------------------------------------------------------------------------------------------

struct IndexerArgs {
    int mode;
    int B, max_blocks, num_blocks;
    int H_I, d_I, K;
    int T;
    const void* q_I;
    const float* w;
    const void* k_I;
    const float* k_I_scale;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_seq;  // may be null: row t is sequence t
    const int32_t* q_pos;  // may be null: decode, pos = seq_len - 1
    int32_t* tile_prefix;  // [T + 1] (workspace)
    int32_t* slot_count;   // [G + T] (workspace)
    uint64_t* slots;       // [G + T][K] (workspace)
    int32_t* idx;          // [T][K] out
    int* err;              // device error word (workspace)
    int G;                 // indexer CTAs
};

__device__ __forceinline__ int row_seq(const IndexerArgs& a, int t) { return a.q_seq ? a.q_seq[t] : t; }

// Causal prefix length of query row t (0 when the row's sequence or position is out of range).
__device__ __forceinline__ int row_len(const IndexerArgs& a, int t) {
    const int b = row_seq(a, t);
    if (b < 0 || b >= a.B) return 0;
    const int L = a.seq_lens[b];
    const int pos = a.q_pos ? a.q_pos[t] : L - 1;
    const int n = pos + 1;
    if (n <= 0) return 0;
    const int cap = min(L, a.max_blocks * kBlock);
    return n < cap ? n : cap;
}

// Physical cache block of logical block `lb` of sequence b; -1 (and the fault bit) if invalid.
__device__ __forceinline__ int phys_block(const IndexerArgs& a, int b, int lb) {
    const int blk = a.block_table[static_cast<int64_t>(b) * a.max_blocks + lb];
    if (blk < 0 || blk >= a.num_blocks) {
        atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
        return -1;
    }
    return blk;
}

}  // namespace dsa
