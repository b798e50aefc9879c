// Sparse MQA attention over gathered latent rows on tcgen05 tensor cores, for 128 query heads and
// 576-wide rows with the first 512 columns as values ("Day0 Inference Support ... on Huawei
// Ascend CANN Architecture" §1: sparse flash attention reads the KV pairs at the Top-K positions;
// §2.1: it reads the main KV exactly at the selected indices).
//
// One CTA = (query row t, value half, split of the K selected rows). With the 128 heads stacked
// as M, every 16-row tile of gathered rows is two dense contractions:
//   S[128 x 16]  = Q[128 x 576] . R^T          (tcgen05, A = Q in smem, B = rows, K-major)
//   O[128 x 256] += P[128 x 16] . R[:, half]    (tcgen05, A = P in TMEM, B = rows, MN-major)
// with an online softmax between them (one thread per head, lazy rescaling of O in TMEM only when
// a head's running maximum grows by more than 2^8). The value columns are split across two CTAs
// because O for all 512 columns would need the whole tensor memory; each CTA computes S itself.
//
// The index list drives the staging: the physical row of every selected position is resolved
// through the block table once per CTA, then 128 producer threads gather each tile's rows with
// 16-byte cp.async into the 128-byte-swizzled layout the MMA reads, arriving on the tile's
// mbarrier when their copies land.
//
// Roles (288 threads): warps 0-3 softmax / epilogue (one head per thread), warps 4-7 producers,
// warp 8 TMEM allocator + MMA issuer (+ the TMA load of Q).
#include <cuda_bf16.h>

#include "internal.h"

namespace dsa {
namespace tcattn {

constexpr int kHeads = 128;
constexpr int kD = 576;
constexpr int kDV = 512;
constexpr int kDVH = 256;
constexpr int kRows = 16;  // gathered rows per tile
constexpr int kChunks = kD / 64;
constexpr int kStages = 4;
constexpr int kQChunkBytes = kHeads * 128;              // [128 heads x 64 bf16]
constexpr int kQBytes = kChunks * kQChunkBytes;         // 144 KB
constexpr int kKvChunkBytes = kRows * 128;              // [16 rows x 64 bf16]
constexpr int kKvStageBytes = kChunks * kKvChunkBytes;  // 18 KB
constexpr int kMaxRows = 2048;
constexpr int kThreads = 288;
constexpr int kNB = 4;          // S / P buffers (tiles the tensor core may run ahead of softmax)
constexpr int kPrefetch = 8;    // tiles of gathered rows prefetched into L2 ahead of their cp.async
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = kColS + kNB * kRows;
constexpr uint32_t kIdescQK = idesc_f16(128, kRows, 1u, 0u, 0u);
constexpr uint32_t kIdescPV = idesc_f16(128, kDVH, 1u, 0u, 1u);

struct Smem {
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[kNB], s_empty[kNB], p_full[kNB], p_empty[kNB];
    uint64_t qfull, o_full, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kOffQ = 0;
constexpr size_t kOffKv = kOffQ + kQBytes;
constexpr size_t kOffPhys = kOffKv + static_cast<size_t>(kStages) * kKvStageBytes;
constexpr size_t kOffCtl = kOffPhys + kMaxRows * sizeof(int32_t);
constexpr size_t kSmemBytes = 1024 + kOffCtl + sizeof(Smem);

__host__ __device__ inline int split_rows(int K, int S) {
    const int per = (K + S - 1) / S;
    return (per + kRows - 1) / kRows * kRows;
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs a, const __grid_constant__ CUtensorMap map_q) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sKv = smem_u32(smem + kOffKv);
    int32_t* phys_s = reinterpret_cast<int32_t*>(smem + kOffPhys);
    Smem& S = *reinterpret_cast<Smem*>(smem + kOffCtl);
    volatile int* abort_flag = &S.abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1, split = blockIdx.x >> 1, t = blockIdx.y;
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
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&S.s_full[i]), 1);
            mbar_init(smem_u32(&S.s_empty[i]), 4);  // one elected arrive per softmax warp
            mbar_init(smem_u32(&S.p_full[i]), 4);
            mbar_init(smem_u32(&S.p_empty[i]), 1);
        }
        mbar_init(smem_u32(&S.qfull), 1);
        mbar_init(smem_u32(&S.o_full), 1);
        mbar_init(smem_u32(&S.mma_done), 1);
        S.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp == 8 && lane == 0 && ntiles > 0) {
        mbar_arrive_expect_tx(smem_u32(&S.qfull), kQBytes);
        for (int c = 0; c < kChunks; ++c)
            tma_load_2d(sQ + c * kQChunkBytes, &map_q, c * 64, t * kHeads, smem_u32(&S.qfull));
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
    __syncthreads();

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------- gather producers
        // Producer warp w fills stage w with tiles w, w + 4, ...: its 32 lanes copy the tile's
        // 16 rows x 72 16-byte units with cp.async, wait for their own copies, and one lane
        // arrives on the stage's barrier. Rows of later tiles are prefetched into L2 first.
        const int pw = warp - 4;
        const uint8_t* kv = static_cast<const uint8_t*>(a.kv);
        auto prefetch_tile = [&](int i) {
            const int row = i * kRows + lane;
            if (lane < kRows && i < ntiles && row < nrows) {
                const int p = phys_s[row];
                if (p >= 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kv + static_cast<int64_t>(p) * (kD * 2)),
                                 "r"(kD * 2)
                                 : "memory");
            }
        };
        prefetch_tile(pw);
        prefetch_tile(pw + kStages);
        for (int i = pw; i < ntiles; i += kStages) {
            prefetch_tile(i + 2 * kStages);
            const int st = pw, use = i / kStages;
            const bool got = mbar_wait(smem_u32(&S.empty[st]), (use & 1) ^ 1, abort_flag, a.err);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            const uint32_t base = sKv + st * kKvStageBytes;
#pragma unroll 4
            for (int e = lane; e < kRows * (kD / 8); e += 32) {
                const int r = e / (kD / 8), u = e % (kD / 8);
                const int c = u >> 3, sub = u & 7;
                const int row = i * kRows + r;
                const int p = (row < nrows) ? phys_s[row] : -1;
                const uint32_t dst = base + c * kKvChunkBytes + r * 128 + ((sub ^ (r & 7)) << 4);
                cp_async16(dst, (p >= 0) ? kv + static_cast<int64_t>(p) * (kD * 2) + u * 16 : kv, (p >= 0) ? 16u : 0u);
            }
            cp_async_wait_all();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.full[st]));
        }
        cp_async_wait_all();
    } else if (warp == 8) {
        // ------------------------------------------------------------- MMA issuer
        // Polls instead of blocking: QK of a tile is issued as soon as its rows have landed and an
        // S buffer is free; PV as soon as softmax has written P. The tensor core thus computes S
        // for the next tiles while softmax works on the current one.
        if (lane == 0 && ntiles > 0) {
            bool ok = mbar_wait(smem_u32(&S.qfull), 0, abort_flag, a.err);
            const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
            const uint64_t dkv0 = sw128_desc(sKv, 16, 1024);
            const uint64_t dv0 = sw128_desc(sKv + (4 * half) * kKvChunkBytes, kKvChunkBytes, 1024);
            int qk = 0, pv = 0;
            long long t_idle = 0;
            while (ok && pv < ntiles) {
                bool did = false;
                if (pv < qk && mbar_test(smem_u32(&S.p_full[pv % kNB]), (pv / kNB) & 1)) {
                    tc_fence_after();
                    const uint64_t vd = dv0 + static_cast<uint64_t>(((pv % kStages) * kKvStageBytes) >> 4);
                    mma_ts(tmem + kColO, tmem + kColP + (pv % kNB) * (kRows / 2), vd, kIdescPV, pv > 0 ? 1u : 0u);
                    tc_commit(smem_u32(&S.empty[pv % kStages]));
                    tc_commit(smem_u32(&S.p_empty[pv % kNB]));
                    ++pv;
                    did = true;
                } else if (qk < ntiles && qk - pv < kNB &&
                           mbar_test(smem_u32(&S.full[qk % kStages]), (qk / kStages) & 1) &&
                           mbar_test(smem_u32(&S.s_empty[qk % kNB]), ((qk / kNB) & 1) ^ 1)) {
                    tc_fence_after();
                    const uint32_t d = tmem + kColS + (qk % kNB) * kRows;
                    const uint64_t kvb = dkv0 + static_cast<uint64_t>(((qk % kStages) * kKvStageBytes) >> 4);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = dq0 + static_cast<uint64_t>((c * kQChunkBytes + kk * 32) >> 4);
                            const uint64_t bd = kvb + static_cast<uint64_t>((c * kKvChunkBytes + kk * 32) >> 4);
                            mma_ss(d, ad, bd, kIdescQK, (c | kk) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(smem_u32(&S.s_full[qk % kNB]));
                    ++qk;
                    did = true;
                }
                if (did) {
                    t_idle = 0;
                } else if (t_idle == 0) {
                    t_idle = clock64();
                } else if (*abort_flag) {
                    ok = false;
                } else if (clock64() - t_idle > kWaitCycles) {
                    *abort_flag = 1;
                    atomicOr(a.err, DSA_FAULT_TIMEOUT);
                    ok = false;
                }
            }
            if (ok) tc_commit(smem_u32(&S.o_full));
            tc_commit(smem_u32(&S.mma_done));
            mbar_wait_drain(smem_u32(&S.mma_done), 0, a.err);
        }
    } else {
        // ------------------------------------------------------------- softmax + epilogue
        const int h = threadIdx.x;  // head = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float scale2 = a.sm_scale * 1.4426950408889634f;  // logits in log2 units
        float m_ref = -INFINITY, l = 0.0f;
        bool dead = false;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i % kNB;
            bool got = mbar_wait(smem_u32(&S.s_full[sb]), (i / kNB) & 1, abort_flag, a.err);
            if (named_bar_or(2, 128, dead || !got)) { dead = true; break; }
            tc_fence_after();
            uint32_t sv[16];
            tmem_ld16(tmem + lane_base + kColS + sb * kRows, sv);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.s_empty[sb]));
            float z[kRows];
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                const int row = i * kRows + j;
                const bool valid = row < nrows && phys_s[row] >= 0;
                z[j] = valid ? __uint_as_float(sv[j]) * scale2 : -INFINITY;
                mt = fmaxf(mt, z[j]);
            }
            const bool need = mt > m_ref + 8.0f;
            if (__any_sync(0xFFFFFFFFu, need)) {
                const float m_new = need ? mt : m_ref;
                if (i > 0) {
                    got = mbar_wait(smem_u32(&S.p_empty[(i - 1) % kNB]), ((i - 1) / kNB) & 1, abort_flag, a.err);
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
            uint32_t packed[kRows / 2];
#pragma unroll
            for (int j = 0; j < kRows; j += 2) {
                const float p0 = (z[j] == -INFINITY) ? 0.0f : exp2f(z[j] - m_ref);
                const float p1 = (z[j + 1] == -INFINITY) ? 0.0f : exp2f(z[j + 1] - m_ref);
                const __nv_bfloat16 b0 = __float2bfloat16_rn(p0), b1 = __float2bfloat16_rn(p1);
                l += __bfloat162float(b0) + __bfloat162float(b1);
                packed[j / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
            }
            if (i >= kNB) {
                got = mbar_wait(smem_u32(&S.p_empty[i % kNB]), ((i - kNB) / kNB) & 1, abort_flag, a.err);
                if (__any_sync(0xFFFFFFFFu, !got)) dead = true;
            }
            if (!dead) {
                tc_fence_after();
                tmem_st8(tmem + lane_base + kColP + (i % kNB) * (kRows / 2), packed);
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&S.p_full[i % kNB]));
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
            uint16_t* out = static_cast<uint16_t*>(a.out) + (static_cast<int64_t>(t) * kHeads + h) * kDV + half * kDVH;
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
            if (half == 0 && a.lse)
                a.lse[static_cast<int64_t>(t) * kHeads + h] =
                    (l > 0.0f) ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
            float* po = a.part_o + prow * kDV + half * kDVH;
#pragma unroll 1
            for (int cc = 0; cc < kDVH / 32; ++cc) {
                uint32_t v[32];
                if (have_o) {
                    tmem_ld32(tmem + lane_base + kColO + cc * 32, v);
                    tmem_ld_wait();
                }
                float4* dst = reinterpret_cast<float4*>(po + cc * 32);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const bool z = !(have_o && l > 0.0f);
                    dst[q] = z ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                             __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                }
            }
            if (half == 0) {
                a.part_ml[prow * 2] = (l > 0.0f) ? m_ref : -INFINITY;
                a.part_ml[prow * 2 + 1] = l;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
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
    if (cudaFuncSetAttribute(tcattn::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tcattn::kSmemBytes)) != cudaSuccess)
        return false;
    dim3 grid(2 * a.S, a.T);
    tcattn::attn_tc_kernel<<<grid, tcattn::kThreads, tcattn::kSmemBytes, s>>>(a, map_q);
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
