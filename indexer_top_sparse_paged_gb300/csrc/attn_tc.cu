// Sparse MQA attention over gathered latent rows on tcgen05 tensor cores, for 128 query heads and
// 576-wide rows whose first 512 columns are the values ("Day0 Inference Support ... on Huawei
// Ascend CANN Architecture" §1: a sparse flash attention module reads the KV pairs at the Top-K
// positions; §2.1: it reads the main KV exactly at the selected indices).
//
// Work unit: a cluster of two CTAs per (query row t, split of its K selected rows). The pair
// divides the latent dimension: CTA 0 owns columns 0..255, CTA 1 owns columns 256..575, so every
// selected row is gathered from memory exactly once. For every tile of 64 gathered rows each CTA
//   1. gathers only its columns of the 64 rows (the index list, resolved once to physical cache
//      rows, drives 16-byte cp.async row copies by seven warps straight into the
//      128-byte-swizzled layout the tensor core reads; four row stages),
//   2. computes its partial logits S_r[128 heads x 64 rows] = Q[:, cols_r] . R[:, cols_r]^T with
//      tcgen05 (M = 128 heads, N = 64 rows; an MMA of N < 64 would leave the tensor pipe idle),
//   3. the producer warps, as soon as S_r is in tensor memory, round it to fp16(S_r * 2^-8) and
//      store it into the other CTA's shared memory with st.async (completion counted in bytes on
//      the receiver's mbarrier; the sender never waits); the softmax adds the two rounded
//      partials, which both CTAs do with identical operands, so both see the same logits,
//   4. runs the online softmax (two threads per head, one per half of the tile's rows, sharing the
//      running maximum; lazy rescaling of O when a head's running maximum grows by more than
//      2^8) and writes P as bf16 over its S in tensor memory,
//   5. accumulates O_r[128 x 256] += P . V_r with V_r = its 256 value columns (CTA 0: values
//      0..255, CTA 1: values 256..511 -- both inside the columns it already holds).
// With an FP8 latent cache (records of e4m3 codes with one fp32 scale per 128 elements; §3: FP8
// block quantisation in the attention stage) step 1 gathers the codes of the CTA's columns into the
// upper half of the operand stage (cp.async, 16 codes per copy) and converter warps widen them in
// place into bf16, code * tile scale in fp32 rounded to nearest even: the gathered bytes halve, the
// tensor-core work is unchanged.
// Split-K partials (m, l, O) are merged by attn_combine_kernel. Tensor memory holds the O
// accumulator (256 fp32 columns), two S/P buffers and all but the first 64 query columns of the
// CTA (A operand from TMEM); shared memory holds the first query chunk, four row stages, two
// exchange slots and the resolved rows of the split.
//
// Roles (512 threads = 16 warps per CTA): warps 0-3 and 9-12 softmax / epilogue in two groups
// (thread = head = TMEM lane; group 0 takes rows 0..31 of every tile and O columns 0..127, group 1
// rows 32..63 and O columns 128..255), warps 4-7 producers (send the partial logits of their TMEM
// lane quarter; bf16 rows: gather a quarter of each tile), warp 8 TMEM allocator + MMA issuer
// (+ the TMA loads of the query), warps 13-15 fill the operand stages (bf16 rows: cp.async
// gathers of the other three quarters, with L2 prefetches of later tiles' rows in windows of 8
// tiles when rows are split; FP8 records: widen the codes that the producers copied into the
// stage).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace dsa {
namespace tcattn {

constexpr int kHeads = 128;
constexpr int kD = 576;
constexpr int kDV = 512;
constexpr int kDVH = 256;                     // value columns per CTA
constexpr int kRows = 64;                     // gathered rows per tile
constexpr int kStagesMax = 4;                 // bf16 operand stages
constexpr int kChunkBytes = kRows * 128;      // [64 rows x 64 bf16]
constexpr int kQChunkBytes = kHeads * 128;    // [128 heads x 64 bf16]
constexpr int kMaxChunks = 5;                 // row chunks per CTA (CTA 0: 4, CTA 1: 5)
constexpr int kStageBytes = kMaxChunks * kChunkBytes;
constexpr int kRecBytes = DSA_KV_FP8_RECORD_BYTES(kD);  // an FP8 latent record: 576 codes + 5 scales + pad
constexpr int kCodeBytes = kRows * kMaxChunks * 64;     // FP8 codes of a tile: 64 rows x up to 320 = 20 KB
constexpr int kCodeOff = kStageBytes - kCodeBytes;      // ... staged in the upper half of their operand stage
constexpr int kXBytes = kHeads * kRows * 2;   // one partial-logit tile (fp16, prescaled by 2^-8)
constexpr float kXScale = 1.0f / 256.0f;      // partial logits travel as fp16(S_r * 2^-8)
constexpr int kMaxRows = 2048;
constexpr int kThreads = 512;     // 16 warps (the register file holds no more at 128 registers a thread)
constexpr int kWarpFill = 13;     // the operand-stage fillers: warps 13..15
constexpr int kFillThreads = 96;
constexpr int kFillRows = 48;     // bf16 rows: the fillers gather rows 0..47 of a tile, the producers 48..63
constexpr int kProducers = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;  // S/P buffers at 256 and 320; Q chunks 32 apart
constexpr uint32_t kIdescQK = idesc_f16(128, kRows, 1u, 0u, 0u);
constexpr uint32_t kIdescPV = idesc_f16(128, kDVH, 1u, 0u, 1u);

struct Smem {
    uint64_t full[kStagesMax], empty[kStagesMax];
    uint64_t codes_full[kStagesMax];  // FP8 records: a tile's codes have landed in its stage
    uint64_t s_full[2], p_full[2], s_free[2];
    uint64_t qfull, o_full, mma_done;
    uint64_t xfull[2], xempty[2];  // both arrived on by the peer: its partial landed / it consumed ours
    uint64_t s_sent[2];            // the producers have read S out of tensor memory
    uint32_t tmem_base;
    int abort_flag;
};

// Shared memory of one CTA (the same for bf16 rows and FP8 records, whose codes are staged inside
// their own operand stage).
template <bool kKv8>
struct Layout {
    static constexpr int kStages = 4;
    static constexpr size_t kOffQ = 0;
    static constexpr size_t kOffKv = kOffQ + kQChunkBytes;
    static constexpr size_t kOffX = kOffKv + static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kOffValid = kOffX + 2 * kXBytes;                // 1 bit per selected row
    static constexpr size_t kOffPhys = kOffValid + kMaxRows / 8;            // physical row per selected row
    static constexpr size_t kOffRed = kOffPhys + kMaxRows * sizeof(int32_t);  // softmax maxima / row sums
    static constexpr size_t kOffCtl = kOffRed + 4 * kHeads * sizeof(float);
    static constexpr size_t kSmemBytes = 1024 + kOffCtl + sizeof(Smem);
};
static_assert(Layout<false>::kSmemBytes <= 232448, "attention shared memory over the limit");
static_assert(Layout<true>::kSmemBytes <= 232448, "FP8 attention shared memory over the limit");
static_assert(kCodeBytes <= kStageBytes / 2, "FP8 codes fit the upper half of their stage");

__host__ __device__ inline int split_rows(int K, int S) {
    const int per = (K + S - 1) / S;
    return (per + kRows - 1) / kRows * kRows;
}

// Exchange-slot byte offset of head h's 16-byte group g (64 fp16 per head, 8 groups): groups are
// the outer index, so the 32 heads of a warp touch one contiguous 512-byte run per access (no bank
// conflicts on either side).
__device__ __forceinline__ uint32_t xoff(int h, int g) { return static_cast<uint32_t>((g * kHeads + h) * 16); }

// 2^x on the special-function unit (flushes subnormal results to zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool kKv8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads)
    attn_tc_kernel(AttnArgs a, const __grid_constant__ CUtensorMap map_q) {
    constexpr int kNT = kThreads;
    constexpr int kWarpSoftB = 9;  // second softmax group: warps 9..12
    using Lay = Layout<kKv8>;
    constexpr int kStages = Lay::kStages;
    constexpr size_t kOffQ = Lay::kOffQ, kOffKv = Lay::kOffKv, kOffX = Lay::kOffX, kOffValid = Lay::kOffValid;
    constexpr size_t kOffPhys = Lay::kOffPhys, kOffRed = Lay::kOffRed, kOffCtl = Lay::kOffCtl;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sKv = smem_u32(smem + kOffKv);
    const uint32_t sX = smem_u32(smem + kOffX);
    uint32_t* valid_bits = reinterpret_cast<uint32_t*>(smem + kOffValid);
    int32_t* phys_s = reinterpret_cast<int32_t*>(smem + kOffPhys);
    Smem& S = *reinterpret_cast<Smem*>(smem + kOffCtl);
    volatile int* abort_flag = &S.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();
    const uint32_t rank = cluster_ctarank();  // 0: columns 0..255, 1: columns 256..575
    const uint32_t peer = rank ^ 1u;
    const int nchunks = rank ? 5 : 4;         // row chunks of 64 columns this CTA gathers
    const int c0 = rank ? 4 : 0;              // first global chunk
    const int split = blockIdx.x >> 1, t = blockIdx.y;
    const int R = split_rows(a.K, a.S);
    const int r0 = split * R;
    const int r1 = min(a.K, r0 + R);
    const int nrows = max(0, r1 - r0);
    const int ntiles = (nrows + kRows - 1) / kRows;
    const int b = a.q_seq ? a.q_seq[t] : t;
    const bool seq_ok = b >= 0 && b < a.B;
    const int L = seq_ok ? a.seq_lens[b] : 0;
    const int32_t* idx_row = a.idx + static_cast<int64_t>(t) * a.K + r0;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(seq_ok ? b : 0) * a.max_blocks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&S.full[i]), kKv8 ? kFillThreads : kFillThreads + kProducers * 32);  // every filling thread arrives
            mbar_init(smem_u32(&S.empty[i]), 1);
            mbar_init(smem_u32(&S.codes_full[i]), kProducers * 32);  // FP8 records: every producer thread arrives
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&S.s_full[i]), 1);
            mbar_init(smem_u32(&S.p_full[i]), 8);  // one elected arrive per softmax warp
            mbar_init(smem_u32(&S.s_free[i]), 1);
            mbar_init(smem_u32(&S.xfull[i]), 1);   // arrive.expect_tx here + the peer's st.async bytes
            mbar_init(smem_u32(&S.xempty[i]), 8);  // the peer's eight softmax warps
            mbar_init(smem_u32(&S.s_sent[i]), 4);  // this CTA's four producer warps
        }
        mbar_init(smem_u32(&S.qfull), 1);
        mbar_init(smem_u32(&S.o_full), 1);
        mbar_init(smem_u32(&S.mma_done), 1);
        S.abort_flag = 0;
        fence_mbar_init();
        // exchange slots 0 and 1 expect the peer's tiles 0 and 1 (re-armed as tiles are consumed)
        mbar_arrive_expect_tx(smem_u32(&S.xfull[0]), kXBytes);
        mbar_arrive_expect_tx(smem_u32(&S.xfull[1]), kXBytes);
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 8 && lane == 0 && ntiles > 0) {
        // the CTA's query chunks: the first to its own buffer (A operand from shared memory), the
        // rest to the still idle row stages, from where they move to tensor memory below
        mbar_arrive_expect_tx(smem_u32(&S.qfull), static_cast<uint32_t>(nchunks * kQChunkBytes));
        tma_load_2d(sQ, &map_q, c0 * 64, t * kHeads, smem_u32(&S.qfull));
        for (int k = 1; k < nchunks; ++k)
            tma_load_2d(sKv + (k - 1) * kQChunkBytes, &map_q, (c0 + k) * 64, t * kHeads, smem_u32(&S.qfull));
    }
    griddep_wait();  // idx may come from the previous kernel of this call
    // every selected row resolved once to its physical cache row (-1: no position, or a bad entry,
    // whose fault CTA 0 records) plus a validity bit per row for the softmax; all index loads are
    // issued before the dependent block-table loads
    {
        constexpr int kPerThread = (kMaxRows + kNT - 1) / kNT;
        int sv[kPerThread];
#pragma unroll
        for (int q = 0; q < kPerThread; ++q) {
            const int i = (q * (kNT / 32) + warp) * 32 + lane;
            sv[q] = (i < nrows) ? idx_row[i] : -1;
        }
        int blk[kPerThread];
#pragma unroll
        for (int q = 0; q < kPerThread; ++q)
            blk[q] = (sv[q] >= 0 && sv[q] < L && (sv[q] >> 6) < a.max_blocks) ? bt_row[sv[q] >> 6] : -1;
#pragma unroll
        for (int q = 0; q < kPerThread; ++q) {
            const int w0 = (q * (kNT / 32) + warp) * 32;
            if (w0 >= ntiles * kRows) break;  // warp-uniform
            const int i = w0 + lane;
            int32_t p = -1;
            if (i < nrows && sv[q] != -1) {
                if (sv[q] < 0 || sv[q] >= L) {
                    if (rank == 0) atomicOr(a.err, DSA_FAULT_INDEX);
                } else if (blk[q] < 0 || blk[q] >= a.num_blocks) {
                    if (rank == 0) atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
                } else {
                    p = blk[q] * kBlock + (sv[q] & 63);
                }
            }
            phys_s[i] = p;
            const uint32_t word = __ballot_sync(0xFFFFFFFFu, p >= 0);
            if (lane == 0) valid_bits[w0 >> 5] = word;
        }
    }
    if (warp < 4 && ntiles > 0) {
        // query chunks 1.. of head h (row h of the 128-byte-swizzled boxes) -> TMEM lane h, bf16 pairs
        const bool got = mbar_wait(smem_u32(&S.qfull), 0, abort_flag, a.err);
        if (__all_sync(0xFFFFFFFFu, got)) {
            const int h = threadIdx.x;
            for (int k = 0; k + 1 < nchunks; ++k) {
                const uint8_t* row = smem + kOffKv + k * kQChunkBytes + (h >> 3) * 1024 + (h & 7) * 128;
                uint32_t w[32];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + ((g ^ (h & 7)) << 4));
                    w[4 * g] = v.x;
                    w[4 * g + 1] = v.y;
                    w[4 * g + 2] = v.z;
                    w[4 * g + 3] = v.w;
                }
                tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kColQ + k * 32, w);
            }
            tmem_st_wait();
        }
    }
    tc_fence_before();
    block_sync();
    tc_fence_after();

    // L2 prefetch of the valid selected rows i0, i0 + n, ... < i1: this CTA's columns (4 or 5 lines of
    // 128 B; FP8: the record's codes of these columns and its scales), requested ahead so that the
    // gathers find them in L2
    auto prefetch_rows = [&](int i0, int i1, int n) {
        for (int row = i0; row < i1; row += n) {
            const int p = phys_s[row];
            if (p < 0) continue;
            if constexpr (!kKv8) {
                const uint8_t* rp = static_cast<const uint8_t*>(a.kv) + c0 * 128 + static_cast<int64_t>(p) * (kD * 2);
                for (int c = 0; c < nchunks; ++c) asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + c * 128));
            } else {
                const uint8_t* rp = static_cast<const uint8_t*>(a.kv) + static_cast<int64_t>(p) * kRecBytes;
                const int lo = c0 * 64, hi = lo + nchunks * 64;
                for (int o = lo; o < hi; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + o));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + hi - 1));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + kD));
            }
        }
    };
    if (warp >= 4 && warp < 4 + kProducers) {
        // ------------------------------------------------------------- producers: send
        // Producer warp pw (TMEM lane quarter pw; with FP8 records after requesting its share of
        // the selected records into L2; with bf16 rows it also gathers rows 48 + pw, 52 + pw, ... of
        // every tile) for every tile j
        //  send(j):   once S(j) is in tensor memory, reads the partial logits of heads 32pw..32pw+31,
        //             rounds them to fp16(S * 2^-8) and stores them into the peer's exchange slot
        //             j & 1 (distributed shared memory; the peer's softmax frees the slot).
        // A gather waits only for a stage that the tensor pipe frees before the next S, so a partial
        // leaves as soon as its MMA has completed.
        const int pw = warp - 4;
        const int h = pw * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(pw * 32) << 16;
        const uint32_t peer_x = mapa_shared(sX, peer);
        const uint32_t peer_xfull = mapa_shared(smem_u32(&S.xfull[0]), peer);  // [1] at +8
        auto send = [&](int j) -> bool {
            const int sb = j & 1;
            const bool got = mbar_wait(smem_u32(&S.s_full[sb]), (j >> 1) & 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, got)) return false;
            tc_fence_after();
            uint32_t v0[32], v1[32];
            tmem_ld32(tmem + lane_base + kColS + sb * kRows, v0);
            tmem_ld32(tmem + lane_base + kColS + sb * kRows + 32, v1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.s_sent[sb]));  // the softmax may overwrite S(j) with P
            uint32_t hp[32];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const __half2 x0 = __floats2half2_rn(__uint_as_float(v0[2 * e]) * kXScale, __uint_as_float(v0[2 * e + 1]) * kXScale);
                const __half2 x1 = __floats2half2_rn(__uint_as_float(v1[2 * e]) * kXScale, __uint_as_float(v1[2 * e + 1]) * kXScale);
                hp[e] = *reinterpret_cast<const uint32_t*>(&x0);
                hp[16 + e] = *reinterpret_cast<const uint32_t*>(&x1);
            }
            const bool free_ok = mbar_wait_cluster(smem_u32(&S.xempty[sb]), ((j >> 1) & 1) ^ 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, free_ok)) return false;
            const uint32_t dst = peer_x + sb * kXBytes;
#pragma unroll
            for (int g = 0; g < 8; ++g)
                st_async_v4(dst + xoff(h, g), hp[4 * g], hp[4 * g + 1], hp[4 * g + 2], hp[4 * g + 3], peer_xfull + sb * 8);
            return true;
        };
        if constexpr (kKv8) {
            // FP8 records: the producers copy the codes of this CTA's columns of every tile into the
            // upper half of its stage (rows pw, pw + 4, ...: lane q < 16 or 20 copies 16-byte group q
            // of the row, group index row * groups-per-row + q; rows with no position read as
            // zeros), three tiles ahead, in the gaps between sends, as for bf16 rows; the filler
            // warps widen them. L2 prefetches of later tiles' records go out in windows of 12
            // tiles once the first three tiles' copies are queued (when the call splits its rows).
            const int gpr = nchunks * 4;
            const uint8_t* kvb = static_cast<const uint8_t*>(a.kv);
            auto gather_codes = [&](int tile) -> bool {
                const int st = tile % kStages;
                const bool got = mbar_wait(smem_u32(&S.empty[st]), ((tile / kStages) & 1) ^ 1, abort_flag, a.err);
                if (!__all_sync(0xFFFFFFFFu, got)) return false;
                const uint32_t base = sKv + st * kStageBytes + kCodeOff;
#pragma unroll 4
                for (int k = 0; k < kRows / kProducers; ++k) {
                    const int r = kProducers * k + pw;
                    const int p = phys_s[tile * kRows + r];
                    if (lane < gpr)
                        cp_async16(base + (r * gpr + lane) * 16,
                                   p >= 0 ? kvb + static_cast<int64_t>(p) * kRecBytes + c0 * 64 + lane * 16 : kvb,
                                   p >= 0 ? 16u : 0u);
                }
                cp_async_arrive_noinc(smem_u32(&S.codes_full[st]));  // once this thread's copies have landed
                return true;
            };
            int pf_end = min(kStages - 1, ntiles);  // tiles below pf_end are copied or requested
            auto prefetch_window = [&]() {           // the records of the next 12 tiles
                prefetch_rows(pf_end * kRows + pw * 32 + lane, min(nrows, (pf_end + 12) * kRows), kProducers * 32);
                pf_end += 12;
            };
            bool ok = true;
            for (int t0 = 0; ok && t0 < pf_end; ++t0) ok = gather_codes(t0);
            if (a.S == 1) pf_end = ntiles;  // one split per row: no L2 prefetch (as for bf16 rows)
            else prefetch_window();
            for (int j = 0; ok && j < ntiles; ++j) {
                ok = send(j);
                const int tn = j + kStages - 1;
                if (ok && tn < ntiles) {
                    ok = gather_codes(tn);
                    if (pf_end < ntiles && pf_end - tn <= 5) prefetch_window();  // the next window, ahead of its copies
                }
            }
            cp_async_wait<0>();  // nothing of this thread's is still in flight when the CTA exits
        } else {
            // bf16 rows: rows 48..63 of every tile are the producers' (4 per warp), gathered as
            // the fillers gather theirs, in the gaps between sends: gather(t) runs once stage t % 4
            // is free, three tiles ahead, in the order the tensor pipe frees the stages
            const uint8_t* kv = static_cast<const uint8_t*>(a.kv) + c0 * 128;
            const int c = lane >> 3, g = lane & 7;  // chunk and 16-byte group this lane copies
            auto gather = [&](int tile) -> bool {
                const int st = tile % kStages;
                const bool got = mbar_wait(smem_u32(&S.empty[st]), ((tile / kStages) & 1) ^ 1, abort_flag, a.err);
                if (!__all_sync(0xFFFFFFFFu, got)) return false;
                const uint32_t base = sKv + st * kStageBytes;
#pragma unroll
                for (int k = 0; k < kRows / 4 / kProducers; ++k) {
                    const int r = kFillRows + kProducers * k + pw;
                    const int p = phys_s[tile * kRows + r];
                    const uint8_t* src = p >= 0 ? kv + static_cast<int64_t>(p) * (kD * 2) : kv;
                    const uint32_t nb = p >= 0 ? 16u : 0u;  // 0: zero-fill
                    const uint32_t rowoff = static_cast<uint32_t>(r * 128);
                    cp_async16(base + c * kChunkBytes + rowoff + ((g ^ (r & 7)) << 4), src + (p >= 0 ? c * 128 + g * 16 : 0), nb);
                    if (nchunks == 5 && lane < 8)
                        cp_async16(base + 4 * kChunkBytes + rowoff + ((lane ^ (r & 7)) << 4),
                                   src + (p >= 0 ? 4 * 128 + lane * 16 : 0), nb);
                }
                cp_async_arrive_noinc(smem_u32(&S.full[st]));  // once this thread's copies have landed
                return true;
            };
            bool ok = true;
            for (int t0 = 0; ok && t0 < kStages - 1 && t0 < ntiles; ++t0) ok = gather(t0);
            for (int j = 0; ok && j < ntiles; ++j) {
                ok = send(j);
                if (ok && j + kStages - 1 < ntiles) ok = gather(j + kStages - 1);
            }
            cp_async_wait<0>();  // nothing of this thread's is still in flight when the CTA exits
        }
    } else if (!kKv8 && warp >= kWarpFill) {
        // ------------------------------------------------------------- bf16 row gathers
        // Filler warp fw copies rows fw, fw + 3, ... < 48 of tile t once stage t % 4 is free: 16-byte
        // cp.async per lane (lane = chunk lane / 8, 16-byte group lane % 8; CTA 1's fifth chunk
        // from lanes 0..7) into the 128-byte-swizzled layout, from the physical cache rows
        // resolved up front; rows with no position read as zeros. The fillers run up to four
        // tiles ahead of the tensor core. When the call splits its rows (S > 1: few rows, each
        // CTA's rows its own) they also request rows into L2 ahead of their copies, in windows of 8
        // tiles: tiles 4..11 once the first four tiles are issued (the stages start free; issued
        // earlier, those requests would queue ahead of the first tiles' copies), then window k
        // (tiles 4 + 8k ..) five tiles before its first copy. Per-tile requests a few tiles ahead
        // leave the copies waiting on HBM; windows of 12 tiles queued more than the copies needed
        // (52.2 -> 50.1 us at batch 32 with 8). With one split per row (T >= 76 on 152 SMs: prefill chunks, whose rows share most
        // of their selected cache rows with other CTAs') no prefetch: measured, it cost 16% in a
        // 2048-row chunk over one 131K-token context and 6% in a 2 x 4096-row prefill.
        const int fw = warp - kWarpFill;
        const uint8_t* kv = static_cast<const uint8_t*>(a.kv) + c0 * 128;
        const int c = lane >> 3, g = lane & 7;  // chunk and 16-byte group this lane copies
        const int last_free = min(kStages, ntiles) - 1;
        for (int tile = 0; tile < ntiles; ++tile) {
            const int st = tile % kStages;
            const bool got = mbar_wait(smem_u32(&S.empty[st]), ((tile / kStages) & 1) ^ 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            const uint32_t base = sKv + st * kStageBytes;
#pragma unroll 2
            for (int r = fw; r < kFillRows; r += kFillThreads / 32) {
                const int p = phys_s[tile * kRows + r];
                const uint8_t* src = p >= 0 ? kv + static_cast<int64_t>(p) * (kD * 2) : kv;
                const uint32_t nb = p >= 0 ? 16u : 0u;  // 0: zero-fill
                const uint32_t rowoff = static_cast<uint32_t>(r * 128);
                cp_async16(base + c * kChunkBytes + rowoff + ((g ^ (r & 7)) << 4), src + (p >= 0 ? c * 128 + g * 16 : 0), nb);
                if (nchunks == 5 && lane < 8)
                    cp_async16(base + 4 * kChunkBytes + rowoff + ((lane ^ (r & 7)) << 4),
                               src + (p >= 0 ? 4 * 128 + lane * 16 : 0), nb);
            }
            cp_async_arrive_noinc(smem_u32(&S.full[st]));  // once this thread's copies have landed
            if (a.S > 1 && (tile == last_free || (tile > last_free && (tile + 1) % 8 == 0))) {  // the next window
                const int w0 = tile == last_free ? kStages : tile + 5;
                prefetch_rows(w0 * kRows + fw * 32 + lane, min(nrows, (w0 + 8) * kRows), kFillThreads);
            }
        }
        cp_async_wait<0>();  // nothing of this thread's is still in flight when the CTA exits
    } else if (kKv8 && warp >= kWarpFill) {
        // ------------------------------------------------------------- FP8 converters
        // convert(t): once tile t's codes have landed in the upper half of its stage (the producers
        // copy them), every thread loads the 16-code groups it converts, the converters meet at a
        // named barrier (the stage is then overwritten in place), and each widens its groups, times
        // their tile scale, into the 128-byte-swizzled bf16 layout (code * scale in fp32, bf16
        // RNE). Each group's scale is loaded one tile ahead. Every converter takes every barrier,
        // so a wait that gives up only stops the work.
        constexpr int kPT = kFillThreads;
        constexpr int kGPT = (kCodeBytes / 16 + kPT - 1) / kPT;  // 16-code groups per thread and tile (<= 14)
        const int gpr = nchunks * 4;                               // groups per row of this CTA: 16 or 20
        const int ngroups = kRows * gpr;
        const int pt = (warp - kWarpFill) * 32 + lane;
        const uint8_t* kvb = static_cast<const uint8_t*>(a.kv);
        bool dead = false;
        auto load_scales = [&](int tile, float (&sc)[kGPT]) {
#pragma unroll
            for (int k = 0; k < kGPT; ++k) {
                const int gi = pt + k * kPT;
                sc[k] = 0.0f;
                if (gi < ngroups) {
                    const int r = gi / gpr, q = gi - r * gpr;
                    const int p = phys_s[tile * kRows + r];
                    if (p >= 0)
                        sc[k] = __ldg(reinterpret_cast<const float*>(kvb + static_cast<int64_t>(p) * kRecBytes + kD) +
                                      ((c0 * 64 + q * 16) >> 7));
                }
            }
        };
        auto convert = [&](int tile, const float (&sc)[kGPT]) {
            const int st = tile % kStages;
            const bool got = mbar_wait(smem_u32(&S.codes_full[st]), (tile / kStages) & 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, got)) dead = true;
            uint8_t* stage = smem + kOffKv + st * kStageBytes;
            uint4 codes[kGPT];
#pragma unroll
            for (int k = 0; k < kGPT; ++k) {
                const int gi = pt + k * kPT;
                codes[k] = (!dead && gi < ngroups) ? *reinterpret_cast<const uint4*>(stage + kCodeOff + gi * 16)
                                                   : make_uint4(0u, 0u, 0u, 0u);
            }
            dead = named_bar_or(5, kFillThreads, dead);  // every code is in registers: the stage may be overwritten
            if (dead) return;
#pragma unroll
            for (int k = 0; k < kGPT; ++k) {
                const int gi = pt + k * kPT;
                if (gi < ngroups) {
                    const int r = gi / gpr, q = gi - r * gpr;
                    uint4 lo, hi;
                    e4m3x16_to_bf16_scaled(codes[k], sc[k], lo, hi);
                    uint8_t* row = stage + (q >> 2) * kChunkBytes + r * 128;  // chunk q / 4
                    const int g2 = 2 * (q & 3);
                    *reinterpret_cast<uint4*>(row + ((g2 ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(row + (((g2 + 1) ^ (r & 7)) << 4)) = hi;
                }
            }
            fence_proxy_async_smem();  // generic-proxy stores -> visible to the tensor core
            mbar_arrive(smem_u32(&S.full[st]));
        };
        // two tiles per iteration, so that each tile's scales sit in a statically named array
        float sc0[kGPT], sc1[kGPT];
        if (ntiles > 0) load_scales(0, sc0);
        for (int t = 0; t < ntiles; t += 2) {
            if (t + 1 < ntiles) load_scales(t + 1, sc1);
            convert(t, sc0);
            if (t + 1 < ntiles) {
                if (t + 2 < ntiles) load_scales(t + 2, sc0);
                convert(t + 1, sc1);
            }
        }
        cp_async_wait<0>();  // nothing of this thread's is still in flight when the CTA exits
    } else if (warp == 8) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0 && ntiles > 0) {
            bool ok = mbar_wait(smem_u32(&S.qfull), 0, abort_flag, a.err);
            const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
            const uint64_t dkv0 = sw128_desc(sKv, 16, 1024);
            const uint64_t dv0 = sw128_desc(sKv, kChunkBytes, 1024);  // V: MN-major, atoms 8 KB apart
            auto qk = [&](int i) -> bool {
                const int st = i % kStages;
                if (!mbar_wait(smem_u32(&S.full[st]), (i / kStages) & 1, abort_flag, a.err)) return false;
                fence_proxy_async_smem();  // rows written by cp.async -> visible to the tensor core
                tc_fence_after();
                const uint32_t d = tmem + kColS + (i & 1) * kRows;
                const uint64_t kvb = dkv0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // first chunk: query from shared memory
                    const uint64_t ad = dq0 + static_cast<uint64_t>((kk * 32) >> 4);
                    const uint64_t bd = kvb + static_cast<uint64_t>((kk * 32) >> 4);
                    mma_ss(d, ad, bd, kIdescQK, kk != 0 ? 1u : 0u);
                }
                for (int cc = 1; cc < nchunks; ++cc) {  // the rest: query from tensor memory
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = kvb + static_cast<uint64_t>((cc * kChunkBytes + kk * 32) >> 4);
                        mma_ts(d, tmem + kColQ + (cc - 1) * 32 + kk * 8, bd, kIdescQK, 1u);
                    }
                }
                tc_commit(smem_u32(&S.s_full[i & 1]));
                return true;
            };
            if (ok) ok = qk(0);
            if (ok && ntiles > 1) ok = qk(1);
            for (int i = 0; ok && i < ntiles; ++i) {
                ok = mbar_wait(smem_u32(&S.p_full[i & 1]), (i >> 1) & 1, abort_flag, a.err);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vb = dv0 + static_cast<uint64_t>(((i % kStages) * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk) {
                    const uint64_t vd = vb + static_cast<uint64_t>((kk * 16 * 128) >> 4);
                    mma_ts(tmem + kColO, tmem + kColS + (i & 1) * kRows + kk * 8, vd, kIdescPV,
                           (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(smem_u32(&S.empty[i % kStages]));
                tc_commit(smem_u32(&S.s_free[i & 1]));
                if (i + 2 < ntiles) ok = qk(i + 2);  // same S buffer: the pipe runs PV(i) first
            }
            if (ok) tc_commit(smem_u32(&S.o_full));
            tc_commit(smem_u32(&S.mma_done));
            mbar_wait_drain(smem_u32(&S.mma_done), 0, a.err);
        }
    } else if (warp < 4 || (warp >= kWarpSoftB && warp < kWarpSoftB + 4)) {
        // ------------------------------------------------------------- softmax + epilogue
        // Two warps per TMEM lane quarter: group 0 (warps 0-3) takes rows 0..31 of every tile and
        // O columns 0..127 of the CTA, group 1 (warps 10-13) rows 32..63 and O columns 128..255.
        // The two threads of a head agree on the running maximum through shared memory, so both
        // scale by the same reference; each keeps its own part of the row sum l.
        const int grp = warp < 4 ? 0 : 1;
        const int quarter = warp & 3;                 // TMEM lanes this warp can access
        const int h = quarter * 32 + lane;            // head = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const float scale2 = a.sm_scale * 1.4426950408889634f / kXScale;  // exchanged units -> log2 units
        const uint32_t peer_xempty = mapa_shared(smem_u32(&S.xempty[0]), peer);  // [1] at +8
        float* red = reinterpret_cast<float*>(smem + kOffRed);  // [2 tiles][2 groups][128 heads]
        float m_ref = -INFINITY, l = 0.0f;
        bool dead = false;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i & 1;
            const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&S.s_full[sb]), (i >> 1) & 1, abort_flag, a.err) &&
                                                         mbar_wait_cluster(smem_u32(&S.xfull[sb]), (i >> 1) & 1, abort_flag, a.err));
            float z[32];
            float mloc = -INFINITY;
            if (got) {
                tc_fence_after();
                // this CTA's partial, rounded exactly as the producers sent it, plus the peer's;
                // both in units of 2^8 (the scale is folded into scale2)
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColS + sb * kRows + grp * 32, v);
                tmem_ld_wait();
                const uint8_t* theirs = smem + kOffX + sb * kXBytes;
                const uint32_t vm = valid_bits[2 * i + grp];  // rows without a position take no weight
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 w = *reinterpret_cast<const uint4*>(theirs + xoff(h, 4 * grp + g));
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = 8 * g + 2 * q;  // rows grp*32 + r, + 1
                        const float2 a2 = __half22float2(
                            __floats2half2_rn(__uint_as_float(v[r]) * kXScale, __uint_as_float(v[r + 1]) * kXScale));
                        const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&ws[q]));
                        z[r] = ((vm >> r) & 1u) ? a2.x + b2.x : -INFINITY;
                        z[r + 1] = ((vm >> (r + 1)) & 1u) ? a2.y + b2.y : -INFINITY;
                    }
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int j = 0; j < 32; ++j) mx[j & 3] = fmaxf(mx[j & 3], z[j]);
                mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            }
            red[(sb * 2 + grp) * kHeads + h] = mloc;
            if (named_bar_or(3, 256, dead || !got)) {  // also publishes red (double-buffered by tile)
                dead = true;
                break;
            }
            // scale2 > 0 and rounding is monotone, so max(z) * scale2 is the max of the scaled logits
            const float mt = fmaxf(red[(sb * 2) * kHeads + h], red[(sb * 2 + 1) * kHeads + h]) * scale2;
            const bool need = mt > m_ref + 8.0f;
            if (__any_sync(0xFFFFFFFFu, need)) {  // the partner warp sees the same heads: same decision
                const float m_new = need ? mt : m_ref;
                if (i > 0) {
                    const bool freed = mbar_wait(smem_u32(&S.s_free[(i - 1) & 1]), ((i - 1) >> 1) & 1, abort_flag, a.err);
                    if (__any_sync(0xFFFFFFFFu, !freed)) dead = true;
                    if (!dead) {
                        tc_fence_after();
                        const float alpha = (m_new == m_ref) ? 1.0f : exp2f(m_ref - m_new);
#pragma unroll 1
                        for (int cc = 0; cc < kDVH / 64; ++cc) {  // this group's half of O
                            const uint32_t col = kColO + grp * (kDVH / 2) + cc * 32;
                            uint32_t v[32];
                            tmem_ld32(tmem + lane_base + col, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            tmem_st32(tmem + lane_base + col, v);
                        }
                        tmem_st_wait();
                        l *= alpha;
                    }
                }
                m_ref = m_new;
            }
            // p = 2^(z * scale2 - m_ref), rounded to bf16 in pairs; l sums the rounded values that
            // the P.V product uses (masked rows: 2^-inf = 0)
            uint32_t packed[16];
            float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const float neg_m = (m_ref == -INFINITY) ? 0.0f : -m_ref;  // no valid row yet: all p = 0
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float p0 = ex2_approx(fmaf(z[j], scale2, neg_m));
                const float p1 = ex2_approx(fmaf(z[j + 1], scale2, neg_m));
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // .x (low half) = p0
                const uint32_t u = *reinterpret_cast<const uint32_t*>(&pb);
                packed[j / 2] = u;
                ls[(j >> 1) & 3] += __uint_as_float(u << 16) + __uint_as_float(u & 0xFFFF0000u);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // P (bf16 pairs) over S columns grp*16 .. +16, once the producers have read S
            const bool read_ok = mbar_wait(smem_u32(&S.s_sent[sb]), (i >> 1) & 1, abort_flag, a.err);
            if (__any_sync(0xFFFFFFFFu, !read_ok)) dead = true;
            if (!dead) {
                tmem_st16(tmem + lane_base + kColS + sb * kRows + grp * 16, packed);
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&S.p_full[sb]));
                // the peer may refill this exchange slot: every value read from it has been consumed
                mbar_arrive_remote_relaxed(peer_xempty + sb * 8);
            }
            // the slot now expects the peer's tile i + 2 (its phase for tile i is complete)
            if (threadIdx.x == 0 && i + 2 < ntiles) mbar_arrive_expect_tx(smem_u32(&S.xfull[sb]), kXBytes);
        }
        if (ntiles > 0) {  // every softmax thread takes this barrier, dead or not
            const bool got = dead ? false : mbar_wait(smem_u32(&S.o_full), 0, abort_flag, a.err);
            dead = named_bar_or(3, 256, dead || !got);
        }
        // the full row sum: both groups' parts
        red[grp * kHeads + h] = l;
        named_bar_sync(3, 256);
        l = red[h] + red[kHeads + h];
        const bool have_o = ntiles > 0 && !dead;
        if (have_o) tc_fence_after();
        // O rows leave through a per-warp 32 x 32 transpose in the (now idle) row stages, so that
        // every store of a warp covers whole 128-byte runs of head rows
        float* tile = reinterpret_cast<float*>(smem + kOffKv) + (grp * 4 + quarter) * (32 * 33);
        const int h0 = quarter * 32;
        const bool zero = !(have_o && l > 0.0f);  // the row is written as zeros
        const int col0 = rank * kDVH + grp * (kDVH / 2);
        auto stage_chunk = [&](int cc) {  // O[h0 + lane][col0 + cc*32 .. +32) -> tile[lane][.]
            uint32_t v[32];
            if (have_o) {
                tmem_ld32(tmem + lane_base + kColO + grp * (kDVH / 2) + cc * 32, v);
                tmem_ld_wait();
            }
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 32; ++e) tile[lane * 33 + e] = zero ? 0.0f : __uint_as_float(v[e]);
            __syncwarp();
        };
        const int tq = lane & 7;  // after the transpose: lane covers columns 4tq..4tq+3 of heads (lane >> 3) + 4j
        if (a.S == 1) {
            const float inv = zero ? 0.0f : 1.0f / l;
            float invk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) invk[j] = __shfl_sync(0xFFFFFFFFu, inv, (lane >> 3) + 4 * j);
#pragma unroll 1
            for (int cc = 0; cc < kDVH / 64; ++cc) {
                stage_chunk(cc);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = (lane >> 3) + 4 * j;
                    const float* tr = tile + k * 33 + 4 * tq;
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(tr[0] * invk[j], tr[1] * invk[j]);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(tr[2] * invk[j], tr[3] * invk[j]);
                    uint16_t* out = static_cast<uint16_t*>(a.out) + (static_cast<int64_t>(t) * kHeads + h0 + k) * kDV +
                                    col0 + cc * 32 + 4 * tq;
                    *reinterpret_cast<uint2*>(out) =
                        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                }
            }
            if (rank == 0 && grp == 0 && a.lse)
                a.lse[static_cast<int64_t>(t) * kHeads + h] =
                    (l > 0.0f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
            // split-K: this CTA's partial (O half, m, l) to the workspace; attn_combine_kernel merges
#pragma unroll 1
            for (int cc = 0; cc < kDVH / 64; ++cc) {
                stage_chunk(cc);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = (lane >> 3) + 4 * j;
                    const float* tr = tile + k * 33 + 4 * tq;
                    float* po = a.part_o + ((static_cast<int64_t>(t) * a.S + split) * kHeads + h0 + k) * kDV + col0 +
                                cc * 32 + 4 * tq;
                    *reinterpret_cast<float4*>(po) = make_float4(tr[0], tr[1], tr[2], tr[3]);
                }
            }
            if (grp == 0) {
                const int64_t mlrow = ((static_cast<int64_t>(t) * a.S + split) * 2 + rank) * kHeads + h;
                a.part_ml[mlrow * 2] = (l > 0.0f && !zero) ? m_ref : -INFINITY;
                a.part_ml[mlrow * 2 + 1] = zero ? 0.0f : l;
            }
        }
    }

    tc_fence_before();
    cluster_sync_all();  // no remote access to this CTA's shared memory may follow its exit
    if (warp == 8) {
        __syncwarp();  // the issuing lane rejoins its warp: dealloc is a whole-warp (aligned) instruction
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// out[t][h][:] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over the splits of row t.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
    griddep_wait();  // the partials of every split are written
    const int h = blockIdx.x, t = blockIdx.y;
    const int c = threadIdx.x * 4;
    float M = -INFINITY;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, a.part_ml[((static_cast<int64_t>(t) * a.S + s) * 2 * kHeads + h) * 2]);
    float wsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int s = 0; s < a.S; ++s) {
            const int64_t prow = (static_cast<int64_t>(t) * a.S + s) * kHeads + h;
            const int64_t mlrow = (static_cast<int64_t>(t) * a.S + s) * 2 * kHeads + h;  // CTA 0's (m, l)
            const float ms = a.part_ml[mlrow * 2];
            if (ms == -INFINITY) continue;
            const float f = exp2f(ms - M);
            wsum += f * a.part_ml[mlrow * 2 + 1];
            const float4 o = *reinterpret_cast<const float4*>(a.part_o + prow * kDV + c);
            acc.x = fmaf(f, o.x, acc.x);
            acc.y = fmaf(f, o.y, acc.y);
            acc.z = fmaf(f, o.z, acc.z);
            acc.w = fmaf(f, o.w, acc.w);
        }
    }
    const float inv = (wsum > 0.0f) ? 1.0f / wsum : 0.0f;
    uint16_t* out = static_cast<uint16_t*>(a.out) + (static_cast<int64_t>(t) * kHeads + h) * kDV + c;
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.x * inv))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y * inv))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.z * inv))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w * inv))) << 16);
    *reinterpret_cast<uint2*>(out) = make_uint2(lo, hi);
    if (threadIdx.x == 0 && a.lse)
        a.lse[static_cast<int64_t>(t) * kHeads + h] = (wsum > 0.0f) ? (M + log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace tcattn

template <bool kKv8>
static bool launch_attn_tc_typed(const AttnArgs& a, const CUtensorMap& map_q, cudaStream_t s) {
    const size_t smem = tcattn::Layout<kKv8>::kSmemBytes;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(tcattn::attn_tc_kernel<kKv8>), smem)) return false;
    return launch_kernel(a.after_own_kernel != 0, tcattn::attn_tc_kernel<kKv8>, dim3(2 * a.S, a.T),
                         dim3(tcattn::kThreads), smem, s, a, map_q);
}

bool launch_attn_tc(const AttnArgs& a, cudaStream_t s, int* launches) {
    if (a.T == 0) return true;
    CUtensorMap map_q;
    if (!make_tmap_2d(&map_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tcattn::kD,
                      static_cast<uint64_t>(a.T) * tcattn::kHeads, tcattn::kD * 2, 64, 128))
        return false;
    if (!(a.kv_fp8 ? launch_attn_tc_typed<true>(a, map_q, s) : launch_attn_tc_typed<false>(a, map_q, s))) return false;
    ++*launches;
    if (a.S > 1) {
        if (!launch_kernel(true, tcattn::attn_combine_kernel, dim3(tcattn::kHeads, a.T), dim3(128), 0, s, a)) return false;
        ++*launches;
    }
    return true;
}

size_t attn_tc_smem() { return tcattn::Layout<false>::kSmemBytes; }

}  // namespace dsa
