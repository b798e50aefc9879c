// Hierarchical (coarse -> fine) index selection ("Engineering Path for Day-0 Adaptation ..."
// §3.1: coarse filtering at block granularity followed by refinement; "How the Ascend Computing
// Platform Achieves Same-Day Inference Adaptation ..." §3.1: the coarse filter reuses summary
// information held in the cache, the fine filter computes only within the candidate blocks).
//
//  summaries  one bf16 key per 64-token block: the mean of the block's valid keys (fp32 sum in
//             token order, fp32 division by the count, round to nearest even), stored per
//             sequence in logical block order, 64 summaries per summary page.
//  coarse     the indexer over the summaries (a dense paged "cache" whose page i of sequence b is
//             row b * pages + i; query row t at block position pos(t) / 64) with Top-K = n_sel.
//  fine       the indexer over the tokens of the chosen blocks: each row gets a virtual sequence
//             whose pages are its chosen blocks in ascending order (so the last one, the only one
//             that can be cut by the causal limit, is last) and whose length ends at pos(t).
//  remap      virtual positions back to logical positions (ascending order is preserved).
#include "internal.h"

namespace dsa {

constexpr int kSumThreads = 128;

// The summary of logical block lb of sequence b (one CTA): the mean of the block's valid keys,
// fp32 sum in token order (never contracted), fp32 division, bf16 round to nearest even.
__device__ void block_summary(int mode, int max_blocks, int num_blocks, int d_I, int sum_rows, const void* k_I,
                              const void* k_scale, const int32_t* block_table, const int32_t* seq_lens, int b, int lb,
                              uint16_t* summaries, int* err) {
    const int L = seq_lens[b];
    if (lb < 0 || lb * kBlock >= L || lb >= max_blocks) return;
    const int blk = block_table[static_cast<int64_t>(b) * max_blocks + lb];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) atomicOr(err, DSA_FAULT_BLOCK_TABLE);
        return;
    }
    const int cnt = min(kBlock, L - lb * kBlock);
    const float sc = mode == DSA_BF16_KFP8 ? static_cast<const float*>(k_scale)[blk] : 1.0f;
    uint16_t* dst = summaries + (static_cast<int64_t>(b) * sum_rows + lb) * d_I;
    for (int d = threadIdx.x; d < d_I; d += kSumThreads) {
        float acc = 0.0f;
        for (int i = 0; i < cnt; ++i) {
            const int64_t e = (static_cast<int64_t>(blk) * kBlock + i) * d_I + d;
            float x;
            if (mode == DSA_F32) x = static_cast<const float*>(k_I)[e];
            else if (mode == DSA_BF16) x = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(k_I)[e]) << 16);
            else {
                const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<const uint8_t*>(k_I)[e], __NV_E4M3);
                const float f = mode == DSA_MXFP8
                                    ? e8m0_value(static_cast<const uint8_t*>(k_scale)[(e / d_I) * (d_I / 32) + d / 32])
                                    : sc;
                x = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(&h)), f);
            }
            acc = __fadd_rn(acc, x);  // in token order, never contracted
        }
        dst[d] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(acc, static_cast<float>(cnt))));
    }
}

// Every valid block: one per CTA (blockIdx.x = lb, blockIdx.y = b).
__global__ void __launch_bounds__(kSumThreads) block_summaries_kernel(int mode, int max_blocks, int num_blocks,
                                                                      int d_I, int sum_rows, const void* k_I,
                                                                      const void* k_scale, const int32_t* block_table,
                                                                      const int32_t* seq_lens, uint16_t* summaries,
                                                                      int* err) {
    block_summary(mode, max_blocks, num_blocks, d_I, sum_rows, k_I, k_scale, block_table, seq_lens, blockIdx.y,
                  blockIdx.x, summaries, err);
}

// The blocks that new tokens touched: the CTA of a block's first new token (rows of one block are
// consecutive) recomputes that block's summary from the updated cache.
__global__ void __launch_bounds__(kSumThreads) summaries_append_kernel(int mode, int B, int max_blocks, int num_blocks,
                                                                       int d_I, int sum_rows, int T, const void* k_I,
                                                                       const void* k_scale, const int32_t* block_table,
                                                                       const int32_t* seq_lens, const int32_t* q_seq,
                                                                       const int32_t* q_pos, uint16_t* summaries, int* err) {
    const int t = blockIdx.x;
    auto where = [&](int r, int& b, int& lb) -> bool {
        b = q_seq ? q_seq[r] : r;
        if (b < 0 || b >= B) return false;
        const int pos = q_pos ? q_pos[r] : seq_lens[b] - 1;
        if (pos < 0) return false;
        lb = pos / kBlock;
        return true;
    };
    int b, lb;
    if (!where(t, b, lb)) return;
    if (t > 0) {
        int b0, lb0;
        if (where(t - 1, b0, lb0) && b0 == b && lb0 == lb) return;
    }
    block_summary(mode, max_blocks, num_blocks, d_I, sum_rows, k_I, k_scale, block_table, seq_lens, b, lb, summaries, err);
}

// coarse paging: page i of sequence b is summary page b * pages + i; block counts and block
// positions of the query rows
__global__ void hier_setup_kernel(int B, int pages, int T, const int32_t* seq_lens, const int32_t* q_seq,
                                  const int32_t* q_pos, int32_t* coarse_table, int32_t* coarse_lens, int32_t* coarse_pos,
                                  int* fine_err) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *fine_err = 0;  // the fine stage's own error word starts clear
    if (i < B * pages) coarse_table[i] = i;
    if (i < B) coarse_lens[i] = (seq_lens[i] + kBlock - 1) / kBlock;
    if (i < T) {
        const int b = q_seq ? q_seq[i] : i;
        const int pos = q_pos ? q_pos[i] : ((b >= 0 && b < B) ? seq_lens[b] - 1 : -1);
        coarse_pos[i] = pos >= 0 ? pos / kBlock : -1;
    }
}

// per row: the chosen blocks (ascending, -1 padded) -> a virtual block table and length
__global__ void hier_virtualize_kernel(int B, int max_blocks, int n_sel, int T, const int32_t* block_table,
                                       const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos,
                                       const int32_t* bidx, int32_t* vtable, int32_t* vlen, int32_t* blocks_out) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int b = q_seq ? q_seq[t] : t;
    const bool ok = b >= 0 && b < B;
    const int pos = ok ? (q_pos ? q_pos[t] : seq_lens[b] - 1) : -1;
    int cnt = 0, last = -1;
    for (int i = 0; i < n_sel; ++i) {
        const int lb = ok ? bidx[static_cast<int64_t>(t) * n_sel + i] : -1;
        if (blocks_out) blocks_out[static_cast<int64_t>(t) * n_sel + i] = lb;
        vtable[static_cast<int64_t>(t) * n_sel + i] =
            (lb >= 0 && lb < max_blocks) ? block_table[static_cast<int64_t>(b) * max_blocks + lb] : -1;
        if (lb >= 0) {
            ++cnt;
            last = lb;
        }
    }
    int len = 0;
    if (cnt > 0 && pos >= 0) len = kBlock * (cnt - 1) + (last == pos / kBlock ? pos % kBlock + 1 : kBlock);
    vlen[t] = len;
}

// virtual positions -> logical positions; the fine stage's fault bits join the call's
__global__ void hier_remap_kernel(int T, int n_sel, int K, const int32_t* bidx, const int32_t* vidx, int32_t* idx,
                                  int* fine_err, int* err) {
    const int t = blockIdx.y;
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (t == 0 && k == 0 && *fine_err) {
        atomicOr(err, *fine_err);
        *fine_err = 0;
    }
    if (k >= K) return;
    const int v = vidx[static_cast<int64_t>(t) * K + k];
    idx[static_cast<int64_t>(t) * K + k] =
        v < 0 ? -1 : bidx[static_cast<int64_t>(t) * n_sel + v / kBlock] * kBlock + v % kBlock;
}

bool launch_block_summaries(const dsa_dims& d, const void* k_I, const void* k_scale, const int32_t* block_table,
                            const int32_t* seq_lens, uint16_t* summaries, int* err, cudaStream_t s, int* launches) {
    const int sum_rows = (d.max_blocks + kBlock - 1) / kBlock * kBlock;
    block_summaries_kernel<<<dim3(d.max_blocks, d.B), kSumThreads, 0, s>>>(d.mode, d.max_blocks, d.num_blocks, d.d_I,
                                                                           sum_rows, k_I, k_scale, block_table,
                                                                           seq_lens, summaries, err);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_summaries_append(const dsa_dims& d, const void* k_I, const void* k_scale, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, int T,
                             uint16_t* summaries, int* err, cudaStream_t s, int* launches) {
    if (T == 0) return true;
    const int sum_rows = (d.max_blocks + kBlock - 1) / kBlock * kBlock;
    summaries_append_kernel<<<T, kSumThreads, 0, s>>>(d.mode, d.B, d.max_blocks, d.num_blocks, d.d_I, sum_rows, T, k_I,
                                                      k_scale, block_table, seq_lens, q_seq, q_pos, summaries, err);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_hier_setup(int B, int pages, int T, const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos,
                       int32_t* coarse_table, int32_t* coarse_lens, int32_t* coarse_pos, int* fine_err, cudaStream_t s,
                       int* launches) {
    const int n = max(B * pages, max(B, T));
    hier_setup_kernel<<<(n + 255) / 256, 256, 0, s>>>(B, pages, T, seq_lens, q_seq, q_pos, coarse_table, coarse_lens,
                                                      coarse_pos, fine_err);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_hier_virtualize(int B, int max_blocks, int n_sel, int T, const int32_t* block_table,
                            const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, const int32_t* bidx,
                            int32_t* vtable, int32_t* vlen, int32_t* blocks_out, cudaStream_t s, int* launches) {
    hier_virtualize_kernel<<<(T + 127) / 128, 128, 0, s>>>(B, max_blocks, n_sel, T, block_table, seq_lens, q_seq,
                                                           q_pos, bidx, vtable, vlen, blocks_out);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

bool launch_hier_remap(int T, int n_sel, int K, const int32_t* bidx, const int32_t* vidx, int32_t* idx, int* fine_err,
                       int* err, cudaStream_t s, int* launches) {
    hier_remap_kernel<<<dim3((K + 255) / 256, T), 256, 0, s>>>(T, n_sel, K, bidx, vidx, idx, fine_err, err);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace dsa
