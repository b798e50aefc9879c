// Sparse MQA attention over gathered latent rows on tcgen05 tensor cores, for 128 query heads and
// 576-wide rows whose first 512 columns are the values ("Day0 Inference Support ... on Huawei
// Ascend CANN Architecture" §1: a sparse flash attention module reads the KV pairs at the Top-K
// positions; §2.1: it reads the main KV exactly at the selected indices).
//
// Work unit: a cluster of two CTAs per (query row t, split of its K selected rows). The pair
// divides the latent dimension: CTA 0 owns columns 0..255, CTA 1 owns columns 256..575. For every
// tile of 64 gathered rows each CTA
//   1. gathers only its columns of the 64 rows (the index list drives TMA tile::gather4 row
//      gathers into the 128-byte-swizzled layout the tensor core reads),
//   2. computes its partial logits S_r[128 heads x 64 rows] = Q[:, cols_r] . R[:, cols_r]^T with
//      tcgen05 (M = 128 heads, N = 64 rows; an MMA of N < 64 would leave the tensor pipe idle),
//   3. sends S_r to the other CTA through distributed shared memory and adds the one it receives
//      (S_0 + S_1 in both CTAs: fp32 addition commutes, so both see the same logits),
//   4. runs the online softmax (one thread per head, lazy rescaling of O when a head's running
//      maximum grows by more than 2^8) and writes P as bf16 over its S in tensor memory,
//   5. accumulates O_r[128 x 256] += P . V_r with V_r = its 256 value columns (CTA 0: values
//      0..255, CTA 1: values 256..511 -- both inside the columns it already holds).
// No row byte is loaded twice and no product is computed twice. The O accumulator (256 fp32
// columns) plus two S/P buffers fit the 512 tensor-memory columns; CTA 1 keeps the last 64 query
// columns in tensor memory (A operand from TMEM) so that its shared memory holds 3 row stages.
//
// Roles (288 threads per CTA): warps 0-3 softmax / epilogue (thread = head = TMEM lane), warps
// 4-6 gather producers (warp 4 + s owns row stage s), warp 7 idle, warp 8 TMEM allocator + MMA
// issuer (+ the TMA load of the query).
#include <cuda_bf16.h>

#include "internal.h"

namespace dsa {
namespace tcattn {

constexpr int kHeads = 128;
constexpr int kD = 576;
constexpr int kDV = 512;
constexpr int kDVH = 256;              // value columns per CTA
constexpr int kRows = 64;              // gathered rows per tile
constexpr int kStages = 3;
constexpr int kChunkBytes = kRows * 128;      // [64 rows x 64 bf16]
constexpr int kQChunkBytes = kHeads * 128;    // [128 heads x 64 bf16]
constexpr int kQSmemChunks = 4;               // query chunks in shared memory (both CTAs)
constexpr int kMaxChunks = 5;                 // row chunks per CTA (CTA 0: 4, CTA 1: 5)
constexpr int kStageBytes = kMaxChunks * kChunkBytes;
constexpr int kXBytes = kHeads * kRows * 4;   // one partial-logit tile (fp32)
constexpr int kMaxRows = 2048;
constexpr int kThreads = 288;
constexpr int kPrefetchTiles = 9;  // tiles of rows prefetched into L2 ahead of their copy (a multiple of kStages)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;  // S/P buffers at 256 and 320
constexpr uint32_t kIdescQK = idesc_f16(128, kRows, 1u, 0u, 0u);
constexpr uint32_t kIdescPV = idesc_f16(128, kDVH, 1u, 0u, 1u);

struct Smem {
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], p_full[2], s_free[2];
    uint64_t qfull, o_full, mma_done;
    uint64_t xfull, xempty;  // arrived on by the other CTA of the pair
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kOffQ = 0;
constexpr size_t kOffKv = kOffQ + static_cast<size_t>(kQSmemChunks) * kQChunkBytes;
constexpr size_t kOffX = kOffKv + static_cast<size_t>(kStages) * kStageBytes;
constexpr size_t kOffPhys = kOffX + kXBytes;
constexpr size_t kOffCtl = kOffPhys + kMaxRows * sizeof(int32_t);
constexpr size_t kSmemBytes = 1024 + kOffCtl + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "attention shared memory over the limit");

__host__ __device__ inline int split_rows(int K, int S) {
    const int per = (K + S - 1) / S;
    return (per + kRows - 1) / kRows * kRows;
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Exchange-buffer byte offset of head h's 16-byte group g (64 fp32 per head, 16 groups): groups
// are the outer index, so the 32 heads of a warp write one contiguous 512-byte run per store
// (remote stores travel as whole segments) and read it back without bank conflicts.
__device__ __forceinline__ uint32_t xoff(int h, int g) { return static_cast<uint32_t>((g * kHeads + h) * 16); }

// 2^x on the special-function unit (flushes subnormal results to zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads)
    attn_tc_kernel(AttnArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sKv = smem_u32(smem + kOffKv);
    const uint32_t sX = smem_u32(smem + kOffX);
    int32_t* phys_s = reinterpret_cast<int32_t*>(smem + kOffPhys);
    Smem& S = *reinterpret_cast<Smem*>(smem + kOffCtl);
    volatile int* abort_flag = &S.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&S.full[i]), 1);
            mbar_init(smem_u32(&S.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&S.s_full[i]), 1);
            mbar_init(smem_u32(&S.p_full[i]), 4);  // one elected arrive per softmax warp
            mbar_init(smem_u32(&S.s_free[i]), 1);
        }
        mbar_init(smem_u32(&S.qfull), 1);
        mbar_init(smem_u32(&S.o_full), 1);
        mbar_init(smem_u32(&S.mma_done), 1);
        mbar_init(smem_u32(&S.xfull), 4);   // the peer's four softmax warps
        mbar_init(smem_u32(&S.xempty), 4);
        S.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 8 && lane == 0 && ntiles > 0) {
        mbar_arrive_expect_tx(smem_u32(&S.qfull), kQSmemChunks * kQChunkBytes);
        for (int c = 0; c < kQSmemChunks; ++c)
            tma_load_2d(sQ + c * kQChunkBytes, &map_q, (c0 + c) * 64, t * kHeads, smem_u32(&S.qfull));
    }
    if (rank == 1 && warp < 4 && ntiles > 0) {
        // query columns 512..575 (the fifth chunk of CTA 1) go to tensor memory, packed in pairs
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                           (static_cast<int64_t>(t) * kHeads + threadIdx.x) * kD + 512);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = src[i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kColQ, w);
        tmem_st_wait();
    }
    // resolve every selected position of this split to its physical cache row once
    for (int i = threadIdx.x; i < nrows; i += kThreads) {
        const int s = a.idx[static_cast<int64_t>(t) * a.K + r0 + i];
        int32_t p = -1;
        if (s != -1) {
            if (s < 0 || s >= L) {
                atomicOr(a.err, DSA_FAULT_INDEX);
            } else {
                const int blk = a.block_table[static_cast<int64_t>(b) * a.max_blocks + (s >> 6)];
                if (blk < 0 || blk >= a.num_blocks) atomicOr(a.err, DSA_FAULT_BLOCK_TABLE);
                else p = blk * kBlock + (s & 63);
            }
        }
        phys_s[i] = p;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp >= 4 && warp < 4 + kStages) {
        // ------------------------------------------------------------- gather producers
        // Producer warp w owns stage w and fills tiles w, w + 3, ...: successive fills of a stage
        // come from one warp, so each waits for exactly the previous use's release. The index
        // list drives TMA row gathers: one tile::gather4 per 4 rows x one 64-column chunk, straight
        // into the 128-byte-swizzled layout (rows with no position read as zeros).
        const int pw = warp - 4;
        const uint8_t* kv = static_cast<const uint8_t*>(a.kv);
        auto prefetch_tile = [&](int i) {
            if (i >= ntiles) return;
            for (int rr = lane; rr < kRows; rr += 32) {
                const int row = i * kRows + rr;
                const int p = (row < nrows) ? phys_s[row] : -1;
                if (p >= 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                     kv + static_cast<int64_t>(p) * (kD * 2) + c0 * 128),
                                 "r"(nchunks * 128)
                                 : "memory");
            }
        };
        if (lane == 0) tma_prefetch_desc(&map_kv);
        for (int i = pw; i < kPrefetchTiles; i += kStages) prefetch_tile(i);
        for (int i = pw; i < ntiles; i += kStages) {
            prefetch_tile(i + kPrefetchTiles - (kPrefetchTiles % kStages));
            const int st = pw, use = i / kStages;
            const bool got = mbar_wait(smem_u32(&S.empty[st]), (use & 1) ^ 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            const uint32_t fb = smem_u32(&S.full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(kRows * nchunks * 128));
            __syncwarp();
            const uint32_t base = sKv + st * kStageBytes;
            if (lane < kRows / 4) {  // lane g gathers rows 4g..4g+3 of the tile, all chunks
                int rw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = i * kRows + 4 * lane + j;
                    rw[j] = (row < nrows) ? phys_s[row] : -1;  // -1: outside the tensor -> zeros
                }
                for (int cc = 0; cc < nchunks; ++cc)
                    tma_gather4(base + cc * kChunkBytes + lane * 4 * 128, &map_kv, (c0 + cc) * 64, rw[0], rw[1],
                                rw[2], rw[3], fb);
            }
        }
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
                tc_fence_after();
                const uint32_t d = tmem + kColS + (i & 1) * kRows;
                const uint64_t kvb = dkv0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
#pragma unroll
                for (int c = 0; c < kQSmemChunks; ++c) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = dq0 + static_cast<uint64_t>((c * kQChunkBytes + kk * 32) >> 4);
                        const uint64_t bd = kvb + static_cast<uint64_t>((c * kChunkBytes + kk * 32) >> 4);
                        mma_ss(d, ad, bd, kIdescQK, (c | kk) != 0 ? 1u : 0u);
                    }
                }
                if (nchunks == 5) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = kvb + static_cast<uint64_t>((4 * kChunkBytes + kk * 32) >> 4);
                        mma_ts(d, tmem + kColQ + kk * 8, bd, kIdescQK, 1u);
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
    } else if (warp < 4) {
        // ------------------------------------------------------------- softmax + epilogue
        const int h = threadIdx.x;  // head = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float scale2 = a.sm_scale * 1.4426950408889634f;  // logits in log2 units
        const uint32_t peer_x = mapa_shared(sX, peer);
        const uint32_t peer_xfull = mapa_shared(smem_u32(&S.xfull), peer);
        const uint32_t peer_xempty = mapa_shared(smem_u32(&S.xempty), peer);
        float m_ref = -INFINITY, l = 0.0f;
        bool dead = false;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i & 1;
            bool got = mbar_wait(smem_u32(&S.s_full[sb]), (i >> 1) & 1, abort_flag, a.err);
            if (named_bar_or(2, 128, dead || !got)) { dead = true; break; }
            tc_fence_after();
            uint32_t v0[32], v1[32];
            const uint32_t sa = tmem + lane_base + kColS + sb * kRows;
            tmem_ld32(sa, v0);
            tmem_ld32(sa + 32, v1);
            tmem_ld_wait();
            // send this CTA's partial logits to the peer ...
            got = mbar_wait_cluster(smem_u32(&S.xempty), (i & 1) ^ 1, abort_flag, a.err);
            if (__any_sync(0xFFFFFFFFu, !got)) dead = true;
            if (!dead) {
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    st_cluster_v4(peer_x + xoff(h, g), __uint_as_float(v0[4 * g]), __uint_as_float(v0[4 * g + 1]),
                                  __uint_as_float(v0[4 * g + 2]), __uint_as_float(v0[4 * g + 3]));
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    st_cluster_v4(peer_x + xoff(h, 8 + g), __uint_as_float(v1[4 * g]), __uint_as_float(v1[4 * g + 1]),
                                  __uint_as_float(v1[4 * g + 2]), __uint_as_float(v1[4 * g + 3]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(peer_xfull);
            // ... and add the peer's
            got = mbar_wait_cluster(smem_u32(&S.xfull), i & 1, abort_flag, a.err);
            if (__any_sync(0xFFFFFFFFu, !got)) dead = true;
            float z[kRows];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                z[j] = __uint_as_float(v0[j]);
                z[32 + j] = __uint_as_float(v1[j]);
            }
            if (!dead) {
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    const float4 o = *reinterpret_cast<const float4*>(smem + kOffX + xoff(h, g));
                    z[4 * g] += o.x;
                    z[4 * g + 1] += o.y;
                    z[4 * g + 2] += o.z;
                    z[4 * g + 3] += o.w;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(peer_xempty);  // the peer may refill our buffer
            // rows without a position (past the split's end, or idx -1) take no weight
            const int rlo = i * kRows + lane, rhi = rlo + 32;
            const uint32_t vm0 = __ballot_sync(0xFFFFFFFFu, rlo < nrows && phys_s[rlo] >= 0);
            const uint32_t vm1 = __ballot_sync(0xFFFFFFFFu, rhi < nrows && phys_s[rhi] >= 0);
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const uint32_t vm = j < 32 ? vm0 : vm1;
                z[j] = ((vm >> (j & 31)) & 1u) ? z[j] : -INFINITY;
                mx[j & 3] = fmaxf(mx[j & 3], z[j]);
            }
            // scale2 > 0 and rounding is monotone, so max(z) * scale2 is the max of the scaled logits
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale2;
            const bool need = mt > m_ref + 8.0f;
            if (__any_sync(0xFFFFFFFFu, need)) {
                const float m_new = need ? mt : m_ref;
                if (i > 0) {
                    got = mbar_wait(smem_u32(&S.s_free[(i - 1) & 1]), ((i - 1) >> 1) & 1, abort_flag, a.err);
                    if (__any_sync(0xFFFFFFFFu, !got)) dead = true;
                    if (!dead) {
                        tc_fence_after();
                        const float alpha = (m_new == m_ref) ? 1.0f : exp2f(m_ref - m_new);
#pragma unroll 1
                        for (int cc = 0; cc < kDVH / 32; ++cc) {
                            uint32_t v[32];
                            tmem_ld32(tmem + lane_base + kColO + cc * 32, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                            tmem_st32(tmem + lane_base + kColO + cc * 32, v);
                        }
                        tmem_st_wait();
                        l *= alpha;
                    }
                }
                m_ref = m_new;
            }
            // p = 2^(z * scale2 - m_ref), rounded to bf16 in pairs; l sums the rounded values that
            // the P.V product uses (masked rows: 2^-inf = 0)
            uint32_t packed[kRows / 2];
            float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const float neg_m = (m_ref == -INFINITY) ? 0.0f : -m_ref;  // no valid row yet: all p = 0
#pragma unroll
            for (int j = 0; j < kRows; j += 2) {
                const float p0 = ex2_approx(fmaf(z[j], scale2, neg_m));
                const float p1 = ex2_approx(fmaf(z[j + 1], scale2, neg_m));
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // .x (low half) = p0
                const uint32_t u = *reinterpret_cast<const uint32_t*>(&pb);
                packed[j / 2] = u;
                ls[(j >> 1) & 3] += __uint_as_float(u << 16) + __uint_as_float(u & 0xFFFF0000u);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            if (!dead) {  // P (bf16) over the first 32 columns of this tile's S
                tmem_st32(sa, packed);
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.p_full[sb]));
        }
        if (ntiles > 0) {  // every softmax thread takes this barrier, dead or not
            const bool got = dead ? false : mbar_wait(smem_u32(&S.o_full), 0, abort_flag, a.err);
            dead = named_bar_or(2, 128, dead || !got);
        }
        const bool have_o = ntiles > 0 && !dead;
        if (have_o) tc_fence_after();
        const int64_t prow = (static_cast<int64_t>(t) * a.S + split) * kHeads + h;
        if (a.S == 1) {
            const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
            uint16_t* out =
                static_cast<uint16_t*>(a.out) + (static_cast<int64_t>(t) * kHeads + h) * kDV + rank * kDVH;
#pragma unroll 1
            for (int cc = 0; cc < kDVH / 32; ++cc) {
                uint32_t v[32];
                if (have_o) {
                    tmem_ld32(tmem + lane_base + kColO + cc * 32, v);
                    tmem_ld_wait();
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float o0 = have_o ? __uint_as_float(v[2 * e]) * inv : 0.0f;
                    const float o1 = have_o ? __uint_as_float(v[2 * e + 1]) * inv : 0.0f;
                    w[e] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o0))) |
                           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o1))) << 16);
                }
                uint4* dst = reinterpret_cast<uint4*>(out + cc * 32);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
            if (rank == 0 && a.lse)
                a.lse[static_cast<int64_t>(t) * kHeads + h] =
                    (l > 0.0f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
            float* po = a.part_o + prow * kDV + rank * kDVH;
#pragma unroll 1
            for (int cc = 0; cc < kDVH / 32; ++cc) {
                uint32_t v[32];
                if (have_o) {
                    tmem_ld32(tmem + lane_base + kColO + cc * 32, v);
                    tmem_ld_wait();
                }
                float4* dst = reinterpret_cast<float4*>(po + cc * 32);
                const bool zero = !(have_o && l > 0.0f);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    dst[q] = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                                  : make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            if (rank == 0) {
                a.part_ml[prow * 2] = (l > 0.0f) ? m_ref : -INFINITY;
                a.part_ml[prow * 2 + 1] = l;
            }
        }
    }

    tc_fence_before();
    cluster_sync_all();  // no remote access to this CTA's shared memory may follow its exit
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// out[t][h][:] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over the splits of row t.
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
    const int h = blockIdx.x, t = blockIdx.y;
    const int c = threadIdx.x * 4;
    float M = -INFINITY;
    for (int s = 0; s < a.S; ++s) M = fmaxf(M, a.part_ml[((static_cast<int64_t>(t) * a.S + s) * kHeads + h) * 2]);
    float wsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int s = 0; s < a.S; ++s) {
            const int64_t prow = (static_cast<int64_t>(t) * a.S + s) * kHeads + h;
            const float ms = a.part_ml[prow * 2];
            if (ms == -INFINITY) continue;
            const float f = exp2f(ms - M);
            wsum += f * a.part_ml[prow * 2 + 1];
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

bool launch_attn_tc(const AttnArgs& a, cudaStream_t s, int* launches) {
    if (a.T == 0) return true;
    CUtensorMap map_q;
    if (!make_tmap_2d(&map_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tcattn::kD,
                      static_cast<uint64_t>(a.T) * tcattn::kHeads, tcattn::kD * 2, 64, 128))
        return false;
    CUtensorMap map_kv;  // [num_blocks * 64 rows][576 cols], gathered one row x 64 columns at a time
    if (!make_tmap_2d(&map_kv, a.kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tcattn::kD,
                      static_cast<uint64_t>(a.num_blocks) * kBlock, tcattn::kD * 2, 64, 1))
        return false;
    if (cudaFuncSetAttribute(tcattn::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tcattn::kSmemBytes)) != cudaSuccess)
        return false;
    dim3 grid(2 * a.S, a.T);
    tcattn::attn_tc_kernel<<<grid, tcattn::kThreads, tcattn::kSmemBytes, s>>>(a, map_q, map_kv);
    ++*launches;
    if (cudaGetLastError() != cudaSuccess) return false;
    if (a.S > 1) {
        tcattn::attn_combine_kernel<<<dim3(tcattn::kHeads, a.T), 128, 0, s>>>(a);
        ++*launches;
        if (cudaGetLastError() != cudaSuccess) return false;
    }
    return true;
}

size_t attn_tc_smem() { return tcattn::kSmemBytes; }

}  // namespace dsa
