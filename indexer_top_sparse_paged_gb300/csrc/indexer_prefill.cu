// Prefill indexer scores on the 5th-generation tensor cores (tcgen05): groups of four consecutive
// query rows of one sequence share every key tile of their causal prefix.
//
// Per 128-key tile the group is one M=128 x N=256 x K=128 contraction: A = the tile's keys (two
// 64-token cache blocks fetched by TMA through the block table, one key per row, K-major,
// 128-byte swizzled), B = the 4 rows x 64 heads of the group's queries, D = 128 x 256 fp32 in
// tensor memory (two accumulators). Each epilogue thread owns one key and forms, for each of
// the four rows,
//     S[t, s] = sum_j w[t, j] * max(0, scale_blk * (q_I[t, j] . k_I[s]))
// (scale_blk = 1 for bf16 keys), written as fp32 to a score matrix with coalesced stores; keys
// outside a row's causal prefix are not written, keys of an invalid block are written as NaN
// (excluded). A row's Top-K is then selected by prefill_topk_kernel. At prefill the scoring is a
// dense contraction over the whole prefix ("Engineering Path for Day-0 Adaptation ..." §3.1: the
// scoring reuses a matrix multiplication), so here it runs on the tensor cores at full width
// while the selection streams the scores once.
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer, warps 2..9 = epilogue (two
// warps per TMEM lane quarter = warp % 4, each taking two of the four rows, so the epilogue's
// arithmetic keeps up with the tensor pipe); FP8 keys add warps 10..13, which widen the staged
// e4m3 codes to bf16 operands exactly (as the decode indexer does), once per tile for all rows.
// MXFP8 keys take the FP8 pipeline with each block's E8M0 scale bytes fetched beside its codes and
// applied by the converters (see the decode indexer); q_I arrives MX-quantised.
#include "internal.h"

namespace dsa {
namespace tcpre {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kRowsPerGroup = 4;
constexpr int kN = kRowsPerGroup * kHeads;    // 256
constexpr int kHalfBytes = kTileKeys * 128;   // [128 keys x 64 bf16] = 16 KB
constexpr int kStageBytes = 2 * kHalfBytes;   // 32 KB
constexpr int kQHalfBytes = kN * 128;         // [256 rows x 64 bf16] = 32 KB
constexpr int kQBytes = 2 * kQHalfBytes;      // 64 KB
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kConvWarp0 = 2 + kEpiWarps;  // first converter warp (FP8 keys)
constexpr int kAcc = 2;
constexpr int kTmemCols = kAcc * kN;          // 512
constexpr uint32_t kIdesc = idesc_f16(128, kN, 1u, 0u, 0u);
constexpr int kF8TileBytes = kTileKeys * kDim;
constexpr int kF8BlockBytes = kBlock * kDim;
constexpr int kMxBlockBytes = kBlock * kDim / 32;  // MXFP8 scale bytes of one block: 256
constexpr int kMxTileBytes = 2 * kMxBlockBytes;

template <bool kFp8>
struct Cfg {
    static constexpr int kThreads = kFp8 ? 32 * (kConvWarp0 + 4) : 32 * kConvWarp0;
    static constexpr int kStages = kFp8 ? 2 : 4;
    static constexpr int kStages8 = kFp8 ? 5 : 1;
    static constexpr size_t kOffQ = 0;
    static constexpr size_t kOffA = kOffQ + kQBytes;
    static constexpr size_t kOffF8 = kOffA + static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kOffF8S = kOffF8 + (kFp8 ? static_cast<size_t>(kStages8) * kF8TileBytes : 0);  // MX scales
    static constexpr size_t kOffW = kOffF8S + (kFp8 ? static_cast<size_t>(kStages8) * kMxTileBytes : 0);
    static constexpr size_t kOffCtl = kOffW + kN * sizeof(float);
};

template <bool kFp8>
struct Smem {
    uint64_t full[Cfg<kFp8>::kStages], empty[Cfg<kFp8>::kStages];
    uint64_t full8[Cfg<kFp8>::kStages8], empty8[Cfg<kFp8>::kStages8];
    uint64_t qfull, qempty;
    uint64_t tfull[kAcc], tempty[kAcc];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

template <bool kFp8>
__host__ __device__ constexpr size_t smem_bytes() {
    return 1024 + Cfg<kFp8>::kOffCtl + sizeof(Smem<kFp8>);
}
static_assert(smem_bytes<false>() <= 232448, "prefill indexer shared memory over the limit");
static_assert(smem_bytes<true>() <= 232448, "FP8 prefill indexer shared memory over the limit");

// Sequence and key count (longest causal prefix of its four rows) of GEMM group g.
__device__ __forceinline__ void group_shape(const IndexerArgs& a, int g, int& b, int& n) {
    b = row_seq(a, kRowsPerGroup * g);
    n = 0;
#pragma unroll
    for (int q = 0; q < kRowsPerGroup; ++q) n = max(n, row_len(a, kRowsPerGroup * g + q));
}

template <bool kFp8, bool kMx>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    indexer_prefill_kernel(IndexerArgs a, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k) {
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
    float* sW = reinterpret_cast<float*>(smem + C::kOffW);
    Smem<kFp8>& S = *reinterpret_cast<Smem<kFp8>*>(smem + C::kOffCtl);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_flag = &S.abort_flag;
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&S.full[i]), kFp8 ? 4 : 1);
            mbar_init(smem_u32(&S.empty[i]), 1);
        }
        if (kFp8) {
            for (int i = 0; i < kStages8; ++i) {
                mbar_init(smem_u32(&S.full8[i]), 1);
                mbar_init(smem_u32(&S.empty8[i]), 4);
            }
        }
        mbar_init(smem_u32(&S.qfull), 1);
        mbar_init(smem_u32(&S.qempty), 1);
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_u32(&S.tfull[i]), 1);
            mbar_init(smem_u32(&S.tempty[i]), kEpiWarps);
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
    griddep_wait();  // the plan (groups, tile prefix) is written

    SegmentIter it;
    it.init(a.gemm_tile_prefix, a.NG, blockIdx.x, a.G2);
    Segment seg;  // seg.row = group

    if (warp == 0) {
        // ------------------------------------------------------------- TMA producer (whole warp)
        uint32_t sg = 0, n_it = 0;
        bool ok = true;
        while (ok && it.next(seg)) {
            const int g = seg.row;
            int b, n;
            group_shape(a, g, b, n);
            const int npages = (n + kBlock - 1) / kBlock;
            const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
            auto load_window = [&](int w0) -> int {
                const int pg = w0 + lane;
                return pg < npages ? bt[pg] : -1;
            };
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&S.qempty), (sg & 1u) ^ 1u, abort_flag, a.err));
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(smem_u32(&S.qfull), kQBytes);
                tma_load_2d(sQ, &map_q, 0, g * kN, smem_u32(&S.qfull));
                tma_load_2d(sQ + kQHalfBytes, &map_q, 64, g * kN, smem_u32(&S.qfull));
            }
            int w0 = (2 * seg.tile0) & ~31;
            int cur = load_window(w0), nxt = load_window(w0 + 32);
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                if (2 * j >= w0 + 32) {
                    w0 += 32;
                    cur = nxt;
                    nxt = load_window(w0 + 32);
                }
                const uint32_t st = n_it % (kFp8 ? kStages8 : kStages), use = n_it / (kFp8 ? kStages8 : kStages);
                const uint32_t ebar = kFp8 ? smem_u32(&S.empty8[st]) : smem_u32(&S.empty[st]);
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
                            tma_load_2d(sF8 + st * kF8TileBytes + p * kF8BlockBytes, &map_k, 0, blk[p] * kBlock, fb);
                            if (kMx)
                                bulk_load_g2s(sF8S + st * kMxTileBytes + p * kMxBlockBytes,
                                              static_cast<const uint8_t*>(a.k_I_scale) +
                                                  static_cast<int64_t>(blk[p]) * kMxBlockBytes,
                                              kMxBlockBytes, fb);
                        } else {
                            const uint32_t dst = sA + st * kStageBytes + p * (kBlock * 128);
                            tma_load_2d(dst, &map_k, 0, blk[p] * kBlock, fb);
                            tma_load_2d(dst + kHalfBytes, &map_k, 64, blk[p] * kBlock, fb);
                        }
                    }
                }
                __syncwarp();
            }
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
                    const uint32_t d = tmem + acc * kN;
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
            tc_commit(smem_u32(&S.mma_done));
            mbar_wait_drain(smem_u32(&S.mma_done), 0, a.err);
        }
        __syncwarp();
    } else if (kFp8 && warp >= kConvWarp0) {
        // ------------------------------------------------------------- e4m3 -> bf16 converters
        const int r = threadIdx.x - 32 * kConvWarp0;
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
                if (lane == 0) mbar_arrive(smem_u32(&S.empty8[s8]));
                if (kMx) store_bf16_row_mx(smem + C::kOffA + st * kStageBytes, r, codes, mx);
                else store_bf16_row(smem + C::kOffA + st * kStageBytes, r, codes);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&S.full[st]));
            }
        }
    } else {
        // ------------------------------------------------------------- epilogue: scores
        const uint32_t quarter = warp & 3;
        const uint32_t row = quarter * 32 + lane;  // key within the tile
        const int etid = threadIdx.x - 64;         // 0..255 over the epilogue warps
        const int q0 = (warp - 2) / 4 * 2;         // this warp's two rows of the group: q0, q0 + 1
        const int64_t lmax = static_cast<int64_t>(a.max_blocks) * kBlock;
        uint32_t n_it = 0;
        while (it.next(seg)) {
            const int g = seg.row;
            int b, n;
            group_shape(a, g, b, n);
            int nq[kRowsPerGroup];
#pragma unroll
            for (int q = 0; q < kRowsPerGroup; ++q) nq[q] = row_len(a, kRowsPerGroup * g + q);
            named_bar_sync(1, kEpiThreads);  // the previous group's weights are no longer read
            for (int i = etid; i < kN; i += kEpiThreads) sW[i] = a.w[static_cast<int64_t>(kRowsPerGroup * g) * kHeads + i];
            named_bar_sync(1, kEpiThreads);
            const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
            float* srow = a.scores + static_cast<int64_t>(kRowsPerGroup * g) * lmax;
            bool ok = true;
            for (int j = seg.tile0; j < seg.tile1; ++j, ++n_it) {
                const uint32_t acc = n_it % kAcc, ause = n_it / kAcc;
                const int s = j * kTileKeys + static_cast<int>(row);
                const int blk = (s < n) ? bt[s >> 6] : -1;
                const bool blk_ok = blk >= 0 && blk < a.num_blocks;
                float sc = 1.0f;
                if (kFp8 && !kMx) sc = blk_ok ? static_cast<const float*>(a.k_I_scale)[blk] : 0.0f;
                const bool got = mbar_wait(smem_u32(&S.tfull[acc]), ause & 1u, abort_flag, a.err);
                if (named_bar_or(1, kEpiThreads, !got)) { ok = false; break; }  // one decision for all epilogue warps
                tc_fence_after();
                const uint32_t taddr = tmem + acc * kN + ((quarter * 32) << 16);
#pragma unroll 1
                for (int q = q0; q < q0 + 2; ++q) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(taddr + q * kHeads, v0);
                    tmem_ld32(taddr + q * kHeads + 32, v1);
                    tmem_ld_wait();
                    if (q == q0 + 1) {  // this warp has read all of its columns of the accumulator
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&S.tempty[acc]));
                    }
                    // two packed fp32x2 accumulators (heads j mod 4): one paired FMA per two heads
                    const float4* w4 = reinterpret_cast<const float4*>(sW + q * kHeads);
                    float2 pa = make_float2(0.0f, 0.0f), pb = make_float2(0.0f, 0.0f);
                    if (!kFp8 || sc >= 0.0f) {
#pragma unroll
                        for (int h = 0; h < 16; ++h) {
                            const float4 wv = w4[h];
                            const uint32_t* v = h < 8 ? v0 + 4 * h : v1 + 4 * (h - 8);
                            pa = __ffma2_rn(make_float2(wv.x, wv.y),
                                            make_float2(fmaxf(__uint_as_float(v[0]), 0.0f), fmaxf(__uint_as_float(v[1]), 0.0f)), pa);
                            pb = __ffma2_rn(make_float2(wv.z, wv.w),
                                            make_float2(fmaxf(__uint_as_float(v[2]), 0.0f), fmaxf(__uint_as_float(v[3]), 0.0f)), pb);
                        }
                    } else {  // scale < 0: max(0, scale * x) = scale * min(0, x)
#pragma unroll
                        for (int h = 0; h < 16; ++h) {
                            const float4 wv = w4[h];
                            const uint32_t* v = h < 8 ? v0 + 4 * h : v1 + 4 * (h - 8);
                            pa = __ffma2_rn(make_float2(wv.x, wv.y),
                                            make_float2(fminf(__uint_as_float(v[0]), 0.0f), fminf(__uint_as_float(v[1]), 0.0f)), pa);
                            pb = __ffma2_rn(make_float2(wv.z, wv.w),
                                            make_float2(fminf(__uint_as_float(v[2]), 0.0f), fminf(__uint_as_float(v[3]), 0.0f)), pb);
                        }
                    }
                    float score = (pa.x + pb.x) + (pa.y + pb.y);
                    if (kFp8 && !kMx) score *= sc;
                    if (s < nq[q]) srow[q * lmax + s] = blk_ok ? score : __uint_as_float(0x7FC00000u);
                }
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    block_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kFp8, bool kMx>
static bool launch(const IndexerArgs& a, cudaStream_t s, int* launches) {
    CUtensorMap map_q, map_k;
    if (!make_tmap_2d(&map_q, a.q_I, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kDim, static_cast<uint64_t>(a.T) * kHeads,
                      kDim * 2, 64, kN))
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
    const size_t smem = smem_bytes<kFp8>();
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(indexer_prefill_kernel<kFp8, kMx>), smem)) return false;
    if (!launch_kernel(true, indexer_prefill_kernel<kFp8, kMx>, dim3(a.G2), dim3(Cfg<kFp8>::kThreads), smem, s, a, map_q,
                       map_k))
        return false;
    ++*launches;
    return true;
}

}  // namespace tcpre

bool launch_indexer_prefill(const IndexerArgs& a, cudaStream_t s, int* launches) {
    if (a.mode == DSA_MXFP8) return tcpre::launch<true, true>(a, s, launches);
    return a.mode == DSA_BF16_KFP8 ? tcpre::launch<true, false>(a, s, launches) : tcpre::launch<false, false>(a, s, launches);
}

}  // namespace dsa
