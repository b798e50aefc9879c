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

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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

// The CTA that owns global tile x (x < total): the largest c with tile_begin(c) <= x.
__host__ __device__ __forceinline__ int64_t tile_owner(int64_t x, int64_t total, int64_t G) {
    return ((x + 1) * G - 1) / total;
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
// Top-K selection: control block, warp-aggregated histograms, radix threshold
// ------------------------------------------------------------------------------------------------

struct TopkCtl {
    uint32_t count;
    uint32_t theta_lo, theta_hi;  // admission threshold: keys below it cannot be in the Top-K
    uint32_t digit, above, bucket;
    unsigned long long diff;      // OR of (key ^ first key): the bits where candidates differ
    uint32_t warp_cnt[32];        // two arrays of 16 per-warp counts (alternating)
};

// Adds 1 to hist[bin] for every active lane of the warp. `hist` is the warp's private histogram,
// so only lanes of one warp can collide on a bin (shared-memory atomics serialise those lanes).
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool active) {
    if (active) atomicAdd(&hist[bin], 1u);
}

// Collective over NT threads (named barrier bar_id): exclusive prefix of v over the threads in
// thread order, and the total. Two barriers; warp_tot is free again when it returns.
template <int NT>
__device__ __forceinline__ uint32_t group_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t tid, uint32_t bar_id,
                                                    uint32_t& total) {
    const uint32_t lane = tid & 31u, warp = tid >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= static_cast<uint32_t>(o)) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    named_bar_sync(bar_id, NT);
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (uint32_t w = 0; w < NT / 32; ++w) {
        const uint32_t c = warp_tot[w];
        before += (w < warp) ? c : 0u;
        total += c;
    }
    named_bar_sync(bar_id, NT);
    return before + x - v;
}

// Collective over NT threads (named barrier bar_id): the threshold thr such that exactly K of the
// keys are >= thr (keys are distinct; more than K in total), over keys held in registers, keys[j]
// valid for j < cnt; thread 0 must hold at least one key. MSB-first radix select with digits of
// up to 8 bits, the first one starting at the highest bit in which two keys differ (bit-aligned,
// so no pass is spent on bits all keys share), stopping as soon as the boundary bucket is taken
// whole. `hist` holds NT/32 private 256-bin histograms (one per warp, so warps never contend on a
// hot bin); they are summed into the first one after every pass.
// With max_passes, the select stops early and returns a threshold that keeps the whole boundary
// bucket: at least K keys (fewer passes, a few keys more than K).
template <int NT, int PER>
__device__ uint64_t reg_radix_threshold(const uint64_t (&keys)[PER], uint32_t cnt, uint32_t K, uint32_t* hist,
                                        TopkCtl* ctl, uint32_t tid, uint32_t bar_id, int max_passes = 64) {
    constexpr uint32_t NW = NT / 32;
    const uint32_t lane = tid & 31u, warp = tid >> 5;
    uint32_t* my_hist = hist + warp * 256;
    if (tid == 0) {  // reference key for the bits every key shares
        ctl->theta_lo = static_cast<uint32_t>(keys[0]);
        ctl->theta_hi = static_cast<uint32_t>(keys[0] >> 32);
        ctl->diff = 0ull;
    }
    named_bar_sync(bar_id, NT);
    const uint64_t ref = (static_cast<uint64_t>(ctl->theta_hi) << 32) | ctl->theta_lo;
    uint64_t d = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (static_cast<uint32_t>(j) < cnt) d |= keys[j] ^ ref;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d |= __shfl_xor_sync(0xFFFFFFFFu, d, o);
    if (lane == 0 && d) atomicOr(&ctl->diff, static_cast<unsigned long long>(d));
    named_bar_sync(bar_id, NT);
    const int hi = 63 - __clzll(static_cast<long long>(ctl->diff | 1ull));
    // digit window [shift, top): bits >= top are fixed (shared by every key, or chosen by earlier passes)
    int top = hi + 1;
    int shift = top > 8 ? top - 8 : 0;
    uint64_t prefix = (top >= 64) ? 0ull : (ref & (~0ull << top));
    uint32_t rem = K;
    for (;;) {
        const uint32_t dmask = (1u << (top - shift)) - 1u;
        for (uint32_t i = lane; i < 256; i += 32) my_hist[i] = 0;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const uint64_t k = keys[j];
            const bool match = static_cast<uint32_t>(j) < cnt && ((top >= 64) || ((k >> top) == (prefix >> top)));
            if (match) atomicAdd(&my_hist[static_cast<uint32_t>(k >> shift) & dmask], 1u);
        }
        named_bar_sync(bar_id, NT);
        for (uint32_t b = tid; b < 256; b += NT) {
            uint32_t c = hist[b];
#pragma unroll
            for (uint32_t w = 1; w < NW; ++w) c += hist[w * 256 + b];
            hist[b] = c;
        }
        named_bar_sync(bar_id, NT);
        if (tid < 32) {
            uint32_t c = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) c += hist[lane * 8 + b];
            uint32_t S = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, S, o);
                if (lane + o < 32) S += v;
            }
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, S >= rem);
            const int L = 31 - __clz(mask);
            if (static_cast<int>(lane) == L) {
                uint32_t running = S - c;
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
        named_bar_sync(bar_id, NT);
        rem -= ctl->above;
        prefix |= static_cast<uint64_t>(ctl->digit) << shift;
        const bool done = ctl->bucket == rem;
        named_bar_sync(bar_id, NT);
        if (done || shift == 0 || --max_passes == 0) break;
        top = shift;
        shift = top > 8 ? top - 8 : 0;
    }
    return prefix;
}

// ------------------------------------------------------------------------------------------------
// streaming Top-K buffer in shared memory, driven collectively by NT threads (one named barrier)
// ------------------------------------------------------------------------------------------------

template <int NT, int PER>
struct TopkGroup {
    uint64_t* buf;   // [cap], cap <= NT * PER
    uint32_t* hist;  // [NT/32][256]
    TopkCtl* ctl;
    uint32_t cap;    // >= K + NT
    uint32_t K;
    uint32_t tid;    // 0..NT-1
    uint32_t bar_id;
    // uniform across the group (every thread computes the same values)
    uint32_t count = 0;
    uint64_t theta = 0;  // admission threshold: keys below it are not admitted
    uint64_t est = 0;    // the largest sample estimate applied to this candidate set (0: none)
    uint32_t parity = 0;

    __device__ __forceinline__ void sync() const { named_bar_sync(bar_id, NT); }

    // Collective. Starts a new candidate set (after the previous flush has been read).
    __device__ void reset() {
        count = 0;
        theta = 0;
        est = 0;
        sync();
    }

    // Collective: raises the admission threshold to the r-th largest key of the buffer (0 < r <
    // count), which holds every valid key offered so far (a sample of the row). Unlike the
    // thresholds of select(), this is an estimate of the row's K-th key, not a bound: whoever
    // merges the row's candidate lists must check that at least K of them are >= every estimate
    // used (then no key of the row's Top-K was turned away) and recompute the row otherwise. The
    // buffer keeps all its keys.
    __device__ void estimate(uint32_t r) {
        sync();  // every push's writes to buf are visible
        const uint32_t n = count;
        const uint32_t per = (n + NT - 1) / NT;
        const uint32_t c0 = min(n, tid * per), c1 = min(n, c0 + per);
        const uint32_t cnt = c1 - c0;
        uint64_t keys[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) keys[j] = (static_cast<uint32_t>(j) < cnt) ? buf[c0 + j] : 0ull;
        const uint64_t e = reg_radix_threshold<NT, PER>(keys, cnt, r, hist, ctl, tid, bar_id);
        if (e > theta) theta = e;
        if (e > est) est = e;
    }

    // Collective: exclusive offset of this thread's predicate among the group and the total.
    // One barrier; the per-warp counts alternate between two arrays so that the next call
    // cannot overwrite counts another thread is still reading.
    __device__ __forceinline__ uint32_t scan(bool p, uint32_t& total) {
        const uint32_t lane = tid & 31u, warp = tid >> 5;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, p);
        uint32_t* wc = ctl->warp_cnt + parity * 16;
        if (lane == 0) wc[warp] = __popc(ballot);
        sync();
        uint32_t off = 0;
        total = 0;
#pragma unroll
        for (uint32_t w = 0; w < NT / 32; ++w) {
            const uint32_t c = wc[w];
            off += (w < warp) ? c : 0u;
            total += c;
        }
        parity ^= 1u;
        return off + __popc(ballot & ((1u << lane) - 1u));
    }

    // Collective: writes the min(count, K) largest keys of buf that are >= the admission threshold,
    // in buffer (= position) order, to dst (shared or global; may be buf itself) and returns how
    // many. Each thread loads its contiguous chunk into registers first, so writing over buf is
    // safe. The keys below the threshold are those of an estimate's sample: dropping them is safe
    // under the merge's estimate check (it counts only keys >= the largest estimate).
    __device__ uint32_t select_to(uint64_t* dst, int max_passes = 64) {
        sync();  // every push's writes to buf are visible
        const uint32_t n = count;
        const uint32_t per = (n + NT - 1) / NT;
        const uint32_t c0 = min(n, tid * per), c1 = min(n, c0 + per);
        const uint32_t cnt = c1 - c0;
        uint64_t keys[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) keys[j] = (static_cast<uint32_t>(j) < cnt) ? buf[c0 + j] : 0ull;
        uint64_t thr = 0ull;
        if (n > K) thr = reg_radix_threshold<NT, PER>(keys, cnt, K, hist, ctl, tid, bar_id, max_passes);
        if (theta > thr) thr = theta;  // keys below the admission threshold (e.g. a sample's) never qualify
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) mine += (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) ? 1u : 0u;
        uint32_t kept;
        uint32_t o = group_excl_scan<NT>(mine, ctl->warp_cnt, tid, bar_id, kept);  // all loads done before
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            if (static_cast<uint32_t>(j) < cnt && keys[j] >= thr) dst[o++] = keys[j];
        }
        theta = thr;
        return kept;
    }

    // Keeps the K largest keys of buf (in order) and raises the admission threshold.
    // (mid-stream: two radix passes bound the threshold tightly enough; the flush is exact). Two
    // passes keep the whole boundary bucket, which can be most of the buffer when many keys share
    // one score (e.g. scores that the ReLU made exactly 0): then the exact selection runs, so the
    // next push always has room.
    __device__ void select() {
        for (int passes = 2;; passes = 64) {  // one call site: the exact retry is rare
            count = select_to(buf, passes);
            if (count + NT <= cap || passes > 2) break;
        }
        sync();
    }

    // Collective: every thread offers at most one key per call.
    __device__ void push(uint64_t key, bool valid) {
        if (count + NT > cap) select();
        const bool p = valid && key >= theta;
        uint32_t total;
        const uint32_t o = scan(p, total);
        if (p) buf[count + o] = key;
        count += total;
    }

    // Collective: writes at most K keys (in position order) to `out`, their number to count_out
    // and the estimate the set was filtered with (0: none) to est_out.
    __device__ void flush(uint64_t* out, int32_t* count_out, uint64_t* est_out) {
        const uint32_t kept = select_to(out);
        if (tid == 0) {
            *count_out = static_cast<int32_t>(kept);
            *est_out = est;
        }
    }
};

// ------------------------------------------------------------------------------------------------
// FP8 e4m3 key tiles -> bf16 tensor-core operands
// ------------------------------------------------------------------------------------------------

// 16 e4m3 codes -> 16 bf16 (two 16-byte groups), exactly: e4m3 -> f16 is exact (every e4m3 value,
// subnormals included, is an f16 normal or zero), and so is f16 -> fp32 -> bf16 for values with
// at most 4 significant bits inside bf16's exponent range.
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4& in, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hlf)) & 0xFFFFu);
            const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
            const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);  // .x = the lower code
            o[2 * i + hlf] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Key row r (0..127) of a staged e4m3 tile: two 64-token blocks of 64 rows x 128 codes, each
// row 128 bytes, 128-byte swizzled as the TMA wrote it (16-byte group c of row rr at c ^ (rr & 7)).
__device__ __forceinline__ void load_e4m3_row(const uint8_t* tile, int r, uint4 (&codes)[8]) {
    const uint8_t* src = tile + (r >> 6) * (64 * 128) + (r & 63) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) codes[c] = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
}

// Writes key row r as bf16 into the tensor core's operand stage: two K halves of [128 rows x 64
// bf16] (16 KB each), rows 128 bytes apart, 128-byte swizzled. Codes 16c..16c+15 go to K half
// c / 4, 16-byte groups 2(c % 4) and 2(c % 4) + 1.
__device__ __forceinline__ void store_bf16_row(uint8_t* stage, int r, const uint4 (&codes)[8]) {
    uint8_t* dst = stage + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 lo, hi;
        e4m3x16_to_bf16(codes[c], lo, hi);
        uint8_t* row = dst + (c >> 2) * (128 * 128);
        const int g = 2 * (c & 3);
        *reinterpret_cast<uint4*>(row + ((g ^ sw) << 4)) = lo;
        *reinterpret_cast<uint4*>(row + (((g + 1) ^ sw) << 4)) = hi;
    }
}

// ------------------------------------------------------------------------------------------------
// MXFP8 (OCP Microscaling Formats: E4M3 elements sharing one E8M0 scale 2^(byte - 127) per 32)
// ------------------------------------------------------------------------------------------------

// 2^(byte - 127) as fp32; byte 0 is the subnormal 2^-127. Byte 255 (NaN in the MX format) is not
// a supported input (it reads as +inf).
__device__ __forceinline__ float e8m0_value(uint32_t byte) { return __uint_as_float(byte ? (byte << 23) : 0x00400000u); }

// Shared exponent of a group whose largest magnitude is amax (finite): X = floor(log2(amax)) - 8,
// at least -127 (so -127 for amax = 0). amax's fp32 exponent field is floor(log2(amax)) + 127
// for normal values; subnormal amax (field 0) lies below 2^-126 and clamps to -127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const int E = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    return max(E - 135, -127);
}

// OCP MX quantisation of 32 bf16 values (16 words of two, the lower element in the low half):
// returns the shared exponent X and writes the codes RNE_e4m3(x * 2^-X), saturating at +-448,
// four per word (element 4i + k in byte k of word i). x * 2^-X is exact in fp32 whenever the
// code can be non-zero.
__device__ __forceinline__ int mx_encode32(const uint32_t (&w)[16], uint32_t (&codes)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    const int X = mx_exponent(amax);                                          // -127 .. 119
    const float down = __uint_as_float(static_cast<uint32_t>(127 - X) << 23);  // 2^-X, a normal float
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t c = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t word = w[2 * i + (k >> 1)];
            const float x = __uint_as_float((k & 1) ? (word & 0xFFFF0000u) : (word << 16));
            c |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(x * down, __NV_SATFINITE, __NV_E4M3)) << (8 * k);
        }
        codes[i] = c;
    }
    return X;
}

// One group of 32 bf16 values (64 bytes at src, 16-byte aligned) -> their MXFP8 values as bf16
// (exact: code * 2^X), at dst: the MX quantisation of a query group for the tensor-core indexer.
__device__ __forceinline__ void mx_quantize_group32(const uint16_t* src, uint16_t* dst) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = s4[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    uint32_t codes[8];
    const int X = mx_encode32(w, codes);
    const float up = e8m0_value(static_cast<uint32_t>(X + 127));  // 2^X
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // element pair 2i, 2i + 1: bytes 2(i % 2), 2(i % 2) + 1 of code word i / 2
        const __nv_fp8x2_storage_t c = static_cast<__nv_fp8x2_storage_t>((codes[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
        const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2));  // .x = the lower code
        const __nv_bfloat162 b = __floats2bfloat162_rn(v.x * up, v.y * up);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// 16 e4m3 codes times the power of two f -> 16 bf16. The fp32 products are exact (at most 4
// significant bits, magnitudes >= 2^-136); so is their bf16 rounding unless a value lies below
// bf16's normal range (an MX exponent under -117).
__device__ __forceinline__ void e4m3x16_to_bf16_scaled(const uint4& in, float f, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hlf)) & 0xFFFFu);
            const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2));
            const __nv_bfloat162 b = __floats2bfloat162_rn(v.x * f, v.y * f);
            o[2 * i + hlf] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// As store_bf16_row for MXFP8 keys of width 128: byte g of `scales` is the E8M0 scale of
// elements 32g..32g+31 (codes group c holds elements 16c..16c+15, so it takes byte c / 2).
__device__ __forceinline__ void store_bf16_row_mx(uint8_t* stage, int r, const uint4 (&codes)[8], uint32_t scales) {
    uint8_t* dst = stage + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 lo, hi;
        e4m3x16_to_bf16_scaled(codes[c], e8m0_value((scales >> (8 * (c >> 1))) & 0xFFu), lo, hi);
        uint8_t* row = dst + (c >> 2) * (128 * 128);
        const int g = 2 * (c & 3);
        *reinterpret_cast<uint4*>(row + ((g ^ sw) << 4)) = lo;
        *reinterpret_cast<uint4*>(row + (((g + 1) ^ sw) << 4)) = hi;
    }
}

// ------------------------------------------------------------------------------------------------
// kernel parameter blocks
// ------------------------------------------------------------------------------------------------

// Sample estimate of a row's K-th key (streaming Top-K of the decode indexer): after the first
// kEstTiles tiles of a segment of at least kEstMinTiles tiles, the admission threshold rises to
// the r-th largest of the sampled keys. The sample's count X of keys from the row's Top-K is
// hypergeometric with mean mu = sample * K / n (n = the row's causal keys), and the r-th sample key
// lies above the row's K-th key only if X >= r. r = ceil(mu + 6.5 sqrt(mu) + 6) keeps that
// probability below 4e-11 for every row length (the exact tail, evaluated for rows of 2K to 4M keys
// and samples of 256 to 512 keys) while admitting as few keys as that allows; a fixed multiple of
// mu admits more keys on short rows and fails far more often on rows of 30K to 130K keys, where mu
// is small. No estimate applies when it would admit three quarters of the keys or more. A sample
// of four tiles (512 keys) puts r closer to mu than two tiles do: measured, the batch-32 decode
// indexer call 79 -> 74 us and the 1M-key row 113 -> 102 us (with the flush dropping the sample's
// keys below the estimate).
// Segments shorter than kEstMinTiles end too soon after their sample for the estimate's select to
// pay for itself (measured: batch-32 decode rows split into segments of 8..15 tiles took longer
// with an estimate than without).
constexpr int kEstTiles = 4;
constexpr int kEstMinTiles = 16;

// The rank of the estimate for a sample of `sample` valid keys of a row of n causal keys, or 0
// when no estimate applies.
__device__ __forceinline__ uint32_t estimate_rank(uint32_t sample, int n, int K) {
    if (n <= K) return 0;
    const float mu = static_cast<float>(sample) * static_cast<float>(K) / static_cast<float>(n);
    const uint32_t r = static_cast<uint32_t>(ceilf(mu + 6.5f * sqrtf(mu) + 6.0f));
    return (4 * r < 3 * sample) ? r : 0u;
}

struct IndexerArgs {
    int mode;
    int B, max_blocks, num_blocks;
    int H_I, d_I, K;
    int T;
    const void* q_I;
    const float* w;
    const void* k_I;
    const void* k_I_scale;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_seq;  // may be null: row t is sequence t
    const int32_t* q_pos;  // may be null: decode, pos = seq_len - 1
    int32_t* tile_prefix;  // [T + 1] (workspace)
    int32_t* group_prefix; // [T + 1] merge groups before row t (workspace)
    int32_t* merge_count;  // [3][merge groups] finished children per merge-tree group (workspace)
    int32_t* slot_count;   // [G + T] (workspace)
    uint64_t* slots;       // [G + T][K] (workspace)
    uint64_t* slot_est;    // [G + T] sample estimate each candidate list was filtered with, 0: none (workspace)
    int32_t* idx;          // [T][K] out
    int* err;              // device error word (workspace)
    int G;                 // indexer CTAs
    // prefill: groups of 4 consecutive query rows of one sequence are scored by a GEMM kernel
    int NG;                     // candidate groups (T / 4), 0 when the call has no prefill path
    int32_t* gemm_flag;         // [NG] 1: group g runs on the score GEMM (its rows skip the decode path)
    int32_t* gemm_tile_prefix;  // [NG + 1] 128-key tiles of the GEMM groups before group g
    float* scores;              // [T][max_blocks * 64] fp32 scores of the GEMM rows (NaN: excluded)
    int G2;                     // score GEMM CTAs
    int self_plan;              // 1: the decode indexer computes the work plan itself (no plan kernel)
    int after_quant;            // 1: q_I is the MX-quantised copy written by this call's first kernel
};

// Is query row t scored by the prefill GEMM (written by the plan)?
__device__ __forceinline__ bool gemm_row(const IndexerArgs& a, int t) {
    return (t >> 2) < a.NG && a.gemm_flag[t >> 2] != 0;
}

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
