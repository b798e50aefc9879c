// Decode indexer + streaming Top-K on the 5th-generation tensor cores (tcgen05), for 64 indexer
// heads of width 128 with bf16 keys, or FP8 e4m3 keys with one fp32 scale per 64-token block.
//
// Per 128-key tile (two 64-token cache blocks fetched by TMA through the block table) the tile
// is one M=128 x N=64 x K=128 contraction: A = the tile's keys (one key per row, K-major, 128-byte
// swizzled), B = the query row's 64 heads (K-major), D = 128 x 64 fp32 in tensor memory. Each
// epilogue thread owns one TMEM lane = one key, so the head-weighted ReLU sum
//     S[s] = sum_j w_j * max(0, D[s, j])
// runs in-thread with no shuffles, and the key goes straight into the CTA's Top-K buffer: no
// score tensor is written to global memory ("Day0 Inference Support ... on Huawei Ascend CANN
// Architecture" §2.1: scoring, head-weight weighting and Top-K fused in one operator reading the
// paged cache; "Engineering Path for Day-0 Adaptation ..." §3.1: the scoring reuses a matrix
// multiplication).
//
// Roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer, warps 2..5 =
// scoring (TMEM lane quarter = warp % 4), warps 6..9 = streaming Top-K, fed by a ring of 16 score
// tiles in shared memory. Pipelines: 3 smem stages of 32 KB (96 KB in flight per SM keeps the
// stream at full rate; deeper rings only lengthen HBM's queue), 4 TMEM accumulators of 64
// columns, one query buffer.
//
// FP8 keys (320 threads): the TMA lands the e4m3 codes of a tile (16 KB) in a staging ring of 6
// stages, warps 6..9 (one key row per thread) widen them to bf16 in the swizzled operand layout
// of a 2-stage ring that the MMA reads, and warps 2..5 both score and select (no score ring).
// Every e4m3 value is exactly a bf16 value,
// so the product is still exact-input bf16 x bf16 -> fp32; the block's scale multiplies the
// accumulator in the epilogue, before the ReLU:
//     S[s] = sum_j w_j * max(0, scale_blk * D[s, j]).
//
// MXFP8 keys (OCP Microscaling: one E8M0 scale per 32 elements of a key) take the FP8 pipeline;
// the TMA producer also fetches each block's 256 scale bytes (64 keys x 4) with an untiled bulk
// copy into the same stage, and the converters multiply every code by its group's power of two
// while widening (exact), so no scale is left for the epilogue. q_I arrives already MX-quantised
// (and decoded to bf16, exactly) by this call's first kernel ("Day0 Inference Support ... on
// Huawei Ascend CANN Architecture" §3: MXFP8 dynamic quantisation in the indexing stage).
#include "internal.h"

namespace dsa {
namespace tcidx {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kHalfBytes = kTileKeys * 128;   // [128 keys x 64 bf16] = 16 KB
constexpr int kStageBytes = 2 * kHalfBytes;   // both K halves = 32 KB
constexpr int kQHalfBytes = kHeads * 128;     // [64 heads x 64 bf16] = 8 KB
constexpr int kQBytes = 2 * kQHalfBytes;      // 16 KB
constexpr int kEpiThreads = 128;
constexpr int kAcc = 4;  // score accumulators in TMEM (64 columns each): the MMA runs ahead of a busy epilogue
constexpr int kTmemCols = kAcc * 64;
constexpr uint32_t kIdesc = idesc_f16(128, kHeads, 1u, 0u, 0u);
constexpr int kF8TileBytes = kTileKeys * kDim;  // e4m3 codes of one tile: 16 KB
constexpr int kF8BlockBytes = kBlock * kDim;    // one 64-token block: 8 KB
constexpr int kMxBlockBytes = kBlock * kDim / 32;  // MXFP8 scale bytes of one block: 256
constexpr int kMxTileBytes = 2 * kMxBlockBytes;

constexpr int kRing = 16;  // score tiles between the scoring warps and the Top-K warps (bf16 keys)

// Shape of the pipelines per key storage. bf16 keys: warps 2-5 score, warps 6-9 select (a ring
// of score tiles between them); FP8 keys: warps 6-9 convert, warps 2-5 score and select.
template <bool kFp8>
struct Cfg {
    static constexpr int kThreads = 320;
    // bf16 operand stages (32 KB) the MMA reads. Three, not more: with 152 SMs each keeping that
    // many tiles in flight the stream still runs at full rate, while deeper rings only lengthen
    // HBM's queue, and with it every other load of the kernel (code, tables) that waits behind the
    // stream (measured at batch 32: 5 stages 67.6 us, 4: 64.5, 3: 63.5, 2: 67.6 per call).
    static constexpr int kStages = kFp8 ? 2 : 3;
    static constexpr int kStages8 = kFp8 ? 6 : 1;      // e4m3 staging stages (16 KB) the TMA fills
    static constexpr size_t kOffA = 0;
    static constexpr size_t kOffQ = kOffA + static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kOffF8 = kOffQ + kQBytes;
    static constexpr size_t kOffF8S = kOffF8 + (kFp8 ? static_cast<size_t>(kStages8) * kF8TileBytes : 0);  // MX scales
    static constexpr size_t kOffBuf = kOffF8S + (kFp8 ? static_cast<size_t>(kStages8) * kMxTileBytes : 0);
};

template <bool kFp8>
struct Smem {
    uint64_t full[Cfg<kFp8>::kStages], empty[Cfg<kFp8>::kStages];
    uint64_t full8[Cfg<kFp8>::kStages8], empty8[Cfg<kFp8>::kStages8];
    uint64_t qfull, qempty;
    uint64_t tfull[kAcc], tempty[kAcc];
    uint64_t ring_full[kRing], ring_empty[kRing];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    uint32_t hist[kEpiThreads / 32 * 256];
    TopkCtl ctl;
    uint32_t ring_valid[kRing][kEpiThreads / 32];  // validity bits of a ring tile's keys, per warp
    alignas(16) float w_s[kHeads];                  // FP8 keys: the current row's head weights
};

constexpr int kTopkPer = 33;  // candidate keys per epilogue thread held in registers while selecting
constexpr size_t kSmemLimit = 232448;
__host__ __device__ constexpr uint32_t topk_cap(int K) { return static_cast<uint32_t>(2 * K + kEpiThreads); }

constexpr size_t kPlanBytes = (kSelfPlanRows + 1) * sizeof(int32_t);  // the work plan, when computed in the kernel

template <bool kFp8>
__host__ __device__ constexpr size_t smem_bytes(int K) {
    return 1024 /*alignment slack*/ + Cfg<kFp8>::kOffBuf + static_cast<size_t>(topk_cap(K)) * 8 +
           (kFp8 ? 0 : static_cast<size_t>(kRing) * kTileKeys * 4) + sizeof(Smem<kFp8>) + kPlanBytes + 64;
}

// Exclusive scan of v over the CTA (in thread order) and the total; `sums` holds one int per warp.
template <int NT>
__device__ __forceinline__ int cta_scan(int v, int* sums, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sums[warp] = x;
    block_sync();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int c = sums[w];
        before += (w < warp) ? c : 0;
        total += c;
    }
    block_sync();
    return before + x - v;
}

// The decode work plan computed by every CTA into shared memory (plan[t] = tiles of the rows
// before t); CTA 0 also publishes it with the rows' merge groups and clears the merge counters,
// as the plan kernel would.
template <int NT>
__device__ void self_plan(const IndexerArgs& a, int32_t* plan, int* sums) {
    int carry = 0;
    for (int base = 0; base < a.T; base += NT) {
        const int t = base + static_cast<int>(threadIdx.x);
        const int tiles = t < a.T ? (row_len(a, t) + kTileKeys - 1) / kTileKeys : 0;
        int tot;
        const int excl = cta_scan<NT>(tiles, sums, tot);
        if (t < a.T) plan[t] = carry + excl;
        carry += tot;
    }
    if (threadIdx.x == 0) plan[a.T] = carry;
    block_sync();
    if (blockIdx.x != 0) return;
    const int64_t total = carry, G = a.G;
    const int GB = merge_group_bound(a.T, a.G);
    int gcarry = 0;
    for (int base = 0; base < a.T; base += NT) {
        const int t = base + static_cast<int>(threadIdx.x);
        int g = 0;
        if (t < a.T) {
            const int64_t p0 = plan[t], p1 = plan[t + 1];
            if (p1 <= p0) g = 1;
            else g = static_cast<int>((tile_owner(p1 - 1, total, G) - tile_owner(p0, total, G) + kMergeFanIn) / kMergeFanIn);
        }
        int tot;
        const int excl = cta_scan<NT>(g, sums, tot);
        if (t < a.T) {
            a.tile_prefix[t] = plan[t];
            a.group_prefix[t] = gcarry + excl;
            for (int l = 0; l < kMergeLevels - 1; ++l)
                for (int i = 0; i < g; ++i) a.merge_count[l * GB + gcarry + excl + i] = 0;
        }
        gcarry += tot;
    }
    if (threadIdx.x == 0) {
        a.tile_prefix[a.T] = carry;
        a.group_prefix[a.T] = gcarry;
    }
}
static_assert(topk_cap(2048) <= static_cast<uint32_t>(kEpiThreads * kTopkPer), "candidate buffer exceeds registers");
static_assert(smem_bytes<false>(2048) <= kSmemLimit, "indexer shared memory over the limit");
static_assert(smem_bytes<true>(2048) <= kSmemLimit, "FP8 indexer shared memory over the limit");

template <bool kFp8, bool kMx>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    indexer_tc_kernel(IndexerArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k) {
    static_assert(kFp8 || !kMx, "MXFP8 keys take the FP8 pipeline");
    using C = Cfg<kFp8>;
    constexpr int kStages = C::kStages;
    constexpr int kStages8 = C::kStages8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem + C::kOffA);
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sF8 = smem_u32(smem + C::kOffF8);
    const uint32_t sF8S = smem_u32(smem + C::kOffF8S);
    uint64_t* buf = reinterpret_cast<uint64_t*>(smem + C::kOffBuf);
    float* ring = reinterpret_cast<float*>(smem + C::kOffBuf + static_cast<size_t>(topk_cap(a.K)) * 8);  // [kRing][128]
    Smem<kFp8>& S = *reinterpret_cast<Smem<kFp8>*>(reinterpret_cast<uint8_t*>(ring) +
                                                   (kFp8 ? 0 : static_cast<size_t>(kRing) * kTileKeys * 4));
    int32_t* plan_s = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(&S) + sizeof(Smem<kFp8>));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_flag = &S.abort_flag;
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            // FP8: filled by the four converter warps (one elected arrive each), else by the TMA
            mbar_init(smem_u32(&S.full[i]), kFp8 ? 4 : 1);
            mbar_init(smem_u32(&S.empty[i]), 1);
        }
        if (kFp8) {
            for (int i = 0; i < kStages8; ++i) {
                mbar_init(smem_u32(&S.full8[i]), 1);
                mbar_init(smem_u32(&S.empty8[i]), 4);  // the four converter warps
            }
        }
        mbar_init(smem_u32(&S.qfull), 1);
        mbar_init(smem_u32(&S.qempty), 1);
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_u32(&S.tfull[i]), 1);
            mbar_init(smem_u32(&S.tempty[i]), kEpiThreads / 32);  // one elected arrive per epilogue warp
        }
        if (!kFp8) {
            for (int i = 0; i < kRing; ++i) {
                mbar_init(smem_u32(&S.ring_full[i]), kEpiThreads / 32);   // the four scoring warps
                mbar_init(smem_u32(&S.ring_empty[i]), kEpiThreads / 32);  // the four Top-K warps
            }
        }
        mbar_init(smem_u32(&S.mma_done), 1);
        S.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    block_sync();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    griddep_wait();  // the work plan (tile prefix) is written (or the inputs, when planned here)
    const int32_t* plan = a.tile_prefix;
    if (a.self_plan) {
        __shared__ int scan_sums[C::kThreads / 32];
        self_plan<C::kThreads>(a, plan_s, scan_sums);
        plan = plan_s;
    }

    SegmentIter it;
    it.init(plan, a.T, blockIdx.x, a.G);
    Segment seg;

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer (whole warp)
        // The block-table entries of a segment are read 32 pages at a time by the 32 lanes, one
        // window ahead of use, so no table load sits between two TMA issues.
        uint32_t sg = 0, n_it = 0;
        bool ok = true;
        // Every key is read exactly once: its lines go into L2 marked evict-first, so the 200 MB
        // stream does not push out what is used again (the Top-K's and merge's code, block tables,
        // queries, candidate lists). Measured: without it the first selection of each CTA stalled
        // 12-17 us on instruction fetches while the stream held HBM (batch-32 call 75.5 -> 67.6 us).
        const uint64_t kpol = l2_policy_evict_first();
        while (ok && it.next(seg)) {
            const int t = seg.row;
            const int b = row_seq(a, t);
            const int n = row_len(a, t);
            const int npages = (n + kBlock - 1) / kBlock;
            const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
            auto load_window = [&](int w0) -> int {  // entry of page w0 + lane, -1 if past the row
                const int pg = w0 + lane;
                if (pg >= npages) return -1;
                const int v = bt[pg];
                return v;
            };
            // one query buffer, reloaded once the previous segment's MMAs are done with it. The
            // segment's key tiles do not wait for that: they keep filling the ring while the
            // previous segment drains, and the query is loaded as soon as its buffer is free
            // (probed after every tile, waited for at the end of the segment's tiles).
            bool q_loaded = false;
            auto load_q = [&](bool block) -> bool {  // warp-uniform; false only on a failed wait
                if (q_loaded) return true;
                const uint32_t qe = smem_u32(&S.qempty), par = (sg & 1u) ^ 1u;
                bool ready = __shfl_sync(0xFFFFFFFFu, mbar_test(qe, par) ? 1 : 0, 0) != 0;
                if (!ready && block) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(qe, par, abort_flag, a.err))) return false;
                    ready = true;
                }
                if (ready) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(smem_u32(&S.qfull), kQBytes);
                        tma_load_2d(sQ, &map_q, 0, t * kHeads, smem_u32(&S.qfull));
                        tma_load_2d(sQ + kQHalfBytes, &map_q, 64, t * kHeads, smem_u32(&S.qfull));
                    }
                    q_loaded = true;
                }
                return true;
            };
            load_q(false);
            int w0 = (2 * seg.tile0) & ~31;
            int cur = load_window(w0), nxt = load_window(w0 + 32);
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                if (2 * j >= w0 + 32) {  // advance the window (pages come in pairs: never straddles)
                    w0 += 32;
                    cur = nxt;
                    nxt = load_window(w0 + 32);
                }
                const uint32_t st = n_it % (kFp8 ? kStages8 : kStages), use = n_it / (kFp8 ? kStages8 : kStages);
                const uint32_t ebar = kFp8 ? smem_u32(&S.empty8[st]) : smem_u32(&S.empty[st]);
                // a full ring can only drain once the MMA has this segment's query: load it first
                if (!q_loaded && __shfl_sync(0xFFFFFFFFu, mbar_test(ebar, (use & 1u) ^ 1u) ? 1 : 0, 0) == 0) {
                    ok = load_q(true);
                    if (!ok) break;
                }
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(ebar, (use & 1u) ^ 1u, abort_flag, a.err));
                if (!ok) break;
                int blk[2];
                uint32_t bytes = 0;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int lb = 2 * j + p;
                    const int v = __shfl_sync(0xFFFFFFFFu, cur, lb - w0);
                    const bool inside = lb * kBlock < n;
                    const bool good = v >= 0 && v < a.num_blocks;
                    if (inside && !good && lane == 0) atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
                    blk[p] = (inside && good) ? v : -1;
                    if (blk[p] >= 0) bytes += kFp8 ? kF8BlockBytes + (kMx ? kMxBlockBytes : 0) : 2 * (kBlock * 128);
                }
                if (lane == 0) {
                    const uint32_t fb = kFp8 ? smem_u32(&S.full8[st]) : smem_u32(&S.full[st]);
                    mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        if (blk[p] < 0) continue;
                        if (kFp8) {
                            tma_load_2d_policy(sF8 + st * kF8TileBytes + p * kF8BlockBytes, &map_k, 0, blk[p] * kBlock, fb, kpol);
                            if (kMx)
                                bulk_load_g2s(sF8S + st * kMxTileBytes + p * kMxBlockBytes,
                                              static_cast<const uint8_t*>(a.k_I_scale) +
                                                  static_cast<int64_t>(blk[p]) * kMxBlockBytes,
                                              kMxBlockBytes, fb);
                        } else {
                            const uint32_t dst = sA + st * kStageBytes + p * (kBlock * 128);
                            tma_load_2d_policy(dst, &map_k, 0, blk[p] * kBlock, fb, kpol);
                            tma_load_2d_policy(dst + kHalfBytes, &map_k, 64, blk[p] * kBlock, fb, kpol);
                        }
                    }
                }
                __syncwarp();
                load_q(false);
            }
            if (ok) ok = load_q(true);
            ++sg;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t sg = 0, n_it = 0;
            bool ok = true;
            while (ok && it.next(seg)) {
                ok = mbar_wait(smem_u32(&S.qfull), sg & 1u, abort_flag, a.err);
                if (!ok) break;
                for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                    const uint32_t st = n_it % kStages, use = n_it / kStages;
                    const uint32_t acc = n_it % kAcc, ause = n_it / kAcc;
                    ok = mbar_wait(smem_u32(&S.full[st]), use & 1u, abort_flag, a.err);
                    if (!ok) break;
                    ok = mbar_wait(smem_u32(&S.tempty[acc]), (ause & 1u) ^ 1u, abort_flag, a.err);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + acc * kHeads;
#pragma unroll
                    for (int k = 0; k < kDim / 16; ++k) {
                        const uint32_t half = k >> 2, kk = k & 3;
                        const uint64_t ad = sw128_desc(sA + st * kStageBytes + half * kHalfBytes + kk * 32, 16, 1024);
                        const uint64_t bd = sw128_desc(sQ + half * kQHalfBytes + kk * 32, 16, 1024);
                        mma_ss(d, ad, bd, kIdesc, k > 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&S.empty[st]));
                    tc_commit(smem_u32(&S.tfull[acc]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&S.qempty));
                ++sg;
            }
            // every MMA issued so far must be complete before TMEM is released
            tc_commit(smem_u32(&S.mma_done));
            mbar_wait_drain(smem_u32(&S.mma_done), 0, a.err);
        }
        __syncwarp();  // the whole warp reaches the final CTA barrier together
    } else if (!kFp8 && warp >= 2 && warp < 6) {
        // ------------------------------------------------------------- scoring (bf16 keys)
        // Thread = TMEM lane = key row of the tile: S[s] = sum_j w_j max(0, D[s, j]) into ring
        // slot n_it % kRing with the warp's validity bits; no group barrier, so the tensor
        // memory is drained at the pace of the stream while the Top-K warps select.
        const uint32_t quarter = warp & 3;
        const uint32_t row = quarter * 32 + lane;
        uint32_t n_it = 0;
        bool ok = true;
        while (ok && it.next(seg)) {
            const int t = seg.row;
            const int n = row_len(a, t);
            float wv[kHeads];
            const float4* w4 = reinterpret_cast<const float4*>(a.w + static_cast<int64_t>(t) * kHeads);
#pragma unroll
            for (int i = 0; i < kHeads / 4; ++i) {
                const float4 v = w4[i];
                wv[4 * i] = v.x;
                wv[4 * i + 1] = v.y;
                wv[4 * i + 2] = v.z;
                wv[4 * i + 3] = v.w;
            }
            const int32_t* bt = a.block_table + static_cast<int64_t>(row_seq(a, t)) * a.max_blocks;
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                const uint32_t acc = n_it % kAcc, ause = n_it / kAcc;
                const uint32_t slot = n_it % kRing, ruse = n_it / kRing;
                const int s = j * kTileKeys + static_cast<int>(row);
                const int blk = (s < n) ? bt[s >> 6] : -1;  // issued before the wait: latency hidden
                const bool valid = s < n && blk >= 0 && blk < a.num_blocks;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&S.tfull[acc]), ause & 1u, abort_flag, a.err));
                if (!ok) break;
                tc_fence_after();
                uint32_t v0[32], v1[32];
                const uint32_t taddr = tmem + acc * kHeads + ((quarter * 32) << 16);
                tmem_ld32(taddr, v0);
                tmem_ld32(taddr + 32, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
                // four independent partial sums (heads j mod 4) keep the FMA pipe busy
                float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    p0 = fmaf(wv[h], fmaxf(__uint_as_float(v0[h]), 0.0f), p0);
                    p1 = fmaf(wv[h + 1], fmaxf(__uint_as_float(v0[h + 1]), 0.0f), p1);
                    p2 = fmaf(wv[h + 2], fmaxf(__uint_as_float(v0[h + 2]), 0.0f), p2);
                    p3 = fmaf(wv[h + 3], fmaxf(__uint_as_float(v0[h + 3]), 0.0f), p3);
                }
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    p0 = fmaf(wv[32 + h], fmaxf(__uint_as_float(v1[h]), 0.0f), p0);
                    p1 = fmaf(wv[33 + h], fmaxf(__uint_as_float(v1[h + 1]), 0.0f), p1);
                    p2 = fmaf(wv[34 + h], fmaxf(__uint_as_float(v1[h + 2]), 0.0f), p2);
                    p3 = fmaf(wv[35 + h], fmaxf(__uint_as_float(v1[h + 3]), 0.0f), p3);
                }
                const float score = (p0 + p1) + (p2 + p3);
                const uint32_t vbits = __ballot_sync(0xFFFFFFFFu, valid);
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&S.ring_empty[slot]), (ruse & 1u) ^ 1u, abort_flag, a.err));
                if (!ok) break;
                ring[slot * kTileKeys + row] = score;
                if (lane == 0) S.ring_valid[slot][quarter] = vbits;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.ring_full[slot]));
            }
        }
    } else if (!kFp8 && warp >= 6) {
        // ------------------------------------------------------------- Top-K (bf16 keys)
        // Thread = key row of the tile (TopkGroup index, so stable compaction keeps position
        // order); consumes the ring's score tiles in the plan's order.
        const uint32_t row = static_cast<uint32_t>(warp - 6) * 32 + lane;
        TopkGroup<kEpiThreads, kTopkPer> topk{buf, S.hist, &S.ctl, topk_cap(a.K), static_cast<uint32_t>(a.K), row, 1};
        uint32_t n_it = 0;
        while (it.next(seg)) {
            topk.reset();
            const int n = row_len(a, seg.row);
            const bool sampled = seg.tile1 - seg.tile0 >= kEstMinTiles;
            bool ok = true;
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                const uint32_t slot = n_it % kRing, ruse = n_it / kRing;
                const bool got = mbar_wait(smem_u32(&S.ring_full[slot]), ruse & 1u, abort_flag, a.err);
                if (named_bar_or(1, kEpiThreads, !got)) { ok = false; break; }
                const float score = ring[slot * kTileKeys + row];
                const bool valid = (S.ring_valid[slot][row >> 5] >> (row & 31)) & 1u;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.ring_empty[slot]));
                const int s = j * kTileKeys + static_cast<int>(row);
                topk.push(make_key(score, static_cast<uint32_t>(s)), valid);
                if (sampled && j == seg.tile0 + kEstTiles - 1) {  // the segment's first tiles are the sample
                    const uint32_t r = estimate_rank(topk.count, n, a.K);
                    if (r) topk.estimate(r);
                }
            }
            if (!ok) break;
            const int64_t slot = static_cast<int64_t>(blockIdx.x) + seg.row;
            topk.flush(a.slots + slot * a.K, a.slot_count + slot, a.slot_est + slot);
            topk.sync();
        }
    } else if (kFp8 && warp >= 6) {
        // ------------------------------------------------------------- e4m3 -> bf16 converters
        // Thread r widens key row r of the tile: 8 swizzled 16-byte groups of codes (block r / 64,
        // row r % 64) become 16 swizzled 16-byte groups of bf16 in the two K halves of the operand
        // stage. Rows whose block was not loaded hold stale codes; the epilogue masks their keys.
        const int r = threadIdx.x - 192;
        uint32_t n_it = 0;
        bool ok = true;
        while (ok && it.next(seg)) {
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                const uint32_t s8 = n_it % kStages8, u8 = n_it / kStages8;
                const uint32_t st = n_it % kStages, use = n_it / kStages;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&S.full8[s8]), u8 & 1u, abort_flag, a.err) &&
                                                 mbar_wait(smem_u32(&S.empty[st]), (use & 1u) ^ 1u, abort_flag, a.err));
                if (!ok) break;
                uint4 codes[8];
                load_e4m3_row(smem + C::kOffF8 + s8 * kF8TileBytes, r, codes);
                uint32_t mx = 0;  // the row's four E8M0 bytes
                if (kMx) mx = *reinterpret_cast<const uint32_t*>(smem + C::kOffF8S + s8 * kMxTileBytes + r * 4);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.empty8[s8]));  // codes are in registers
                if (kMx) store_bf16_row_mx(smem + C::kOffA + st * kStageBytes, r, codes, mx);
                else store_bf16_row(smem + C::kOffA + st * kStageBytes, r, codes);
                fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.full[st]));
            }
        }
    } else if (kFp8) {
        // ------------------------------------------------------------- epilogue + Top-K (FP8 keys)
        const uint32_t quarter = warp & 3;             // TMEM lane quarter of this warp
        const uint32_t row = quarter * 32 + lane;      // key within the tile
        // the group's thread index is the key row, so stable compaction keeps position order
        TopkGroup<kEpiThreads, kTopkPer> topk{buf, S.hist, &S.ctl, topk_cap(a.K), static_cast<uint32_t>(a.K), row, 1};
        uint32_t n_it = 0;
        while (it.next(seg)) {
            const int t = seg.row;
            const int n = row_len(a, t);
            // the row's head weights live in shared memory and are read back as broadcasts, so the
            // registers hold the TMEM values and the Top-K candidates without spilling (the end of
            // the previous segment was a group barrier: nobody still reads the old weights)
            if (row < kHeads / 4)
                reinterpret_cast<float4*>(S.w_s)[row] = reinterpret_cast<const float4*>(a.w + static_cast<int64_t>(t) * kHeads)[row];
            topk.reset();  // a group barrier: the weights are visible
            const bool sampled = seg.tile1 - seg.tile0 >= kEstMinTiles;
            const float4* wv4 = reinterpret_cast<const float4*>(S.w_s);
            bool ok = true;
            const int32_t* bt = a.block_table + static_cast<int64_t>(row_seq(a, t)) * a.max_blocks;
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                const uint32_t acc = n_it % kAcc, ause = n_it / kAcc;
                const int s = j * kTileKeys + static_cast<int>(row);
                const int blk = (s < n) ? bt[s >> 6] : -1;  // issued before the wait: latency hidden
                const bool blk_ok = blk >= 0 && blk < a.num_blocks;
                float sc = 1.0f;
                if (kFp8 && !kMx) sc = blk_ok ? static_cast<const float*>(a.k_I_scale)[blk] : 0.0f;
                const bool got = mbar_wait(smem_u32(&S.tfull[acc]), ause & 1u, abort_flag, a.err);
                if (named_bar_or(1, kEpiThreads, !got)) { ok = false; break; }
                tc_fence_after();
                uint32_t v0[32], v1[32];
                const uint32_t taddr = tmem + acc * kHeads + ((quarter * 32) << 16);
                tmem_ld32(taddr, v0);
                tmem_ld32(taddr + 32, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
                // four independent partial sums (heads j mod 4) keep the FMA pipe busy
                float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
                if (!kFp8 || sc >= 0.0f) {
                    // scale >= 0: max(0, scale * x) = scale * max(0, x), applied once to the sum
#pragma unroll
                    for (int h = 0; h < 32; h += 4) {
                        const float4 wa = wv4[h / 4], wb = wv4[8 + h / 4];
                        p0 = fmaf(wa.x, fmaxf(__uint_as_float(v0[h]), 0.0f), p0);
                        p1 = fmaf(wa.y, fmaxf(__uint_as_float(v0[h + 1]), 0.0f), p1);
                        p2 = fmaf(wa.z, fmaxf(__uint_as_float(v0[h + 2]), 0.0f), p2);
                        p3 = fmaf(wa.w, fmaxf(__uint_as_float(v0[h + 3]), 0.0f), p3);
                        p0 = fmaf(wb.x, fmaxf(__uint_as_float(v1[h]), 0.0f), p0);
                        p1 = fmaf(wb.y, fmaxf(__uint_as_float(v1[h + 1]), 0.0f), p1);
                        p2 = fmaf(wb.z, fmaxf(__uint_as_float(v1[h + 2]), 0.0f), p2);
                        p3 = fmaf(wb.w, fmaxf(__uint_as_float(v1[h + 3]), 0.0f), p3);
                    }
                } else {
                    // scale < 0: max(0, scale * x) = scale * min(0, x)
#pragma unroll
                    for (int h = 0; h < 32; h += 4) {
                        const float4 wa = wv4[h / 4], wb = wv4[8 + h / 4];
                        p0 = fmaf(wa.x, fminf(__uint_as_float(v0[h]), 0.0f), p0);
                        p1 = fmaf(wa.y, fminf(__uint_as_float(v0[h + 1]), 0.0f), p1);
                        p2 = fmaf(wa.z, fminf(__uint_as_float(v0[h + 2]), 0.0f), p2);
                        p3 = fmaf(wa.w, fminf(__uint_as_float(v0[h + 3]), 0.0f), p3);
                        p0 = fmaf(wb.x, fminf(__uint_as_float(v1[h]), 0.0f), p0);
                        p1 = fmaf(wb.y, fminf(__uint_as_float(v1[h + 1]), 0.0f), p1);
                        p2 = fmaf(wb.z, fminf(__uint_as_float(v1[h + 2]), 0.0f), p2);
                        p3 = fmaf(wb.w, fminf(__uint_as_float(v1[h + 3]), 0.0f), p3);
                    }
                }
                float score = (p0 + p1) + (p2 + p3);
                if (kFp8 && !kMx) score *= sc;
                // a block whose table entry is invalid was never loaded: its keys do not count
                const bool valid = s < n && blk_ok;
                topk.push(make_key(score, static_cast<uint32_t>(s)), valid);
                if (sampled && j == seg.tile0 + kEstTiles - 1) {  // the segment's first tiles are the sample
                    const uint32_t r = estimate_rank(topk.count, n, a.K);
                    if (r) topk.estimate(r);
                }
            }
            if (!ok) break;
            const int64_t slot = static_cast<int64_t>(blockIdx.x) + t;
            topk.flush(a.slots + slot * a.K, a.slot_count + slot, a.slot_est + slot);
            topk.sync();
        }
    }

    tc_fence_before();
    block_sync();
    if (warp == 1) {
        __syncwarp();  // the issuing lane rejoins its warp: dealloc is a whole-warp (aligned) instruction
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kFp8, bool kMx>
static bool launch(const IndexerArgs& a, cudaStream_t s, int* launches) {
    CUtensorMap map_q, map_k;
    if (!make_tmap_2d(&map_q, a.q_I, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kDim, static_cast<uint64_t>(a.T) * kHeads,
                      kDim * 2, 64, 64))
        return false;
    if (kFp8) {
        if (!make_tmap_2d(&map_k, a.k_I, CU_TENSOR_MAP_DATA_TYPE_UINT8, kDim,
                          static_cast<uint64_t>(a.num_blocks) * kBlock, kDim, kDim, kBlock))
            return false;
    } else {
        if (!make_tmap_2d(&map_k, a.k_I, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kDim,
                          static_cast<uint64_t>(a.num_blocks) * kBlock, kDim * 2, 64, 64))
            return false;
    }
    const size_t smem = smem_bytes<kFp8>(a.K);
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(indexer_tc_kernel<kFp8, kMx>), smem)) return false;
    // the first kernel of the call when it plans itself (and q_I needs no quantisation): it waits
    // for all earlier work on the stream
    if (!launch_kernel(!a.self_plan || a.after_quant, indexer_tc_kernel<kFp8, kMx>, dim3(a.G),
                       dim3(Cfg<kFp8>::kThreads), smem, s, a, map_q, map_k))
        return false;
    ++*launches;
    return true;
}

}  // namespace tcidx

bool launch_indexer_tc(const IndexerArgs& a, cudaStream_t s, int* launches) {
    if (a.mode == DSA_MXFP8) return tcidx::launch<true, true>(a, s, launches);
    return a.mode == DSA_BF16_KFP8 ? tcidx::launch<true, false>(a, s, launches) : tcidx::launch<false, false>(a, s, launches);
}


}  // namespace dsa
