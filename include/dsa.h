/*
 * dsa.h -- C ABI of the GB300 (sm_103a) index-selection sparse attention library (libdsa.so).
 *
 * The operation (one query row t of sequence b = q_seq[t] at absolute position pos = q_pos[t]):
 *
 *   paged fetch   logical position s of sequence b is physical cache row
 *                 block_table[b][s / 64] * 64 + s % 64
 *                 ("Engineering Path for Day-0 Adaptation ... on Domestic AI Accelerators" §3.2:
 *                 fixed-size blocks, an index maps to block number and in-block offset)
 *   indexer       S[t,s] = sum_j w[t,j] * max(0, q_I[t,j,:] . k_I[s,:])   for s in [0, pos]
 *                 with k_I[s,:] = e4m3 code * block scale for FP8 indexer keys
 *                 ("Day0 Inference Support ... on Huawei Ascend CANN Architecture" §2.1: relevance
 *                 scoring, head-weight weighting and Top-K selection fused over the paged cache; §3:
 *                 FP8 quantized indexer data; formula fixed by the problem statement)
 *   Top-K         the K largest S[t,s], ties to the lower s; fewer than K positions -> all of them
 *                 ("Engineering Path ..." §3.1: index selection is scoring plus Top-K filtering and
 *                 yields a discrete index set)
 *   attention     z_i = sm_scale * q[t,h,:] . row_i ; out[t,h,:] = sum_i softmax(z)_i * row_i[0:d_v]
 *                 over the rows row_i = kv_cache[phys(idx[t][i])] of one shared latent cache
 *                 ("Day0 Inference Support ..." §1: a sparse flash attention module reads the KV
 *                 pairs at the selected positions; V is the first d_v columns of the same row)
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller, row-major and densely packed
 *    in the shapes given below. Inputs are only read; idx / out / lse / ws are written.
 *  - The library allocates, frees and synchronises nothing (except dsa_read_error, which says so).
 *    All work is enqueued on `stream` (NULL = the legacy default stream) in launch order.
 *  - A return value other than DSA_OK means nothing was launched, except DSA_ERR_LAUNCH, which
 *    means a launch failed part way (the stream then holds a partial result).
 *  - Faults the host cannot see (a block-table entry outside [0, num_blocks), an idx entry outside
 *    [0, seq_len) other than -1, a pipeline wait that timed out) set bits of an error word in the
 *    workspace; the offending rows are skipped (read as zeros) and dsa_read_error reports them.
 *  - The workspace `ws` (>= dsa_workspace_size bytes, 256-byte aligned) is scratch owned by one
 *    call at a time: calls that share a workspace must be ordered on one stream.
 *  - No shared mutable state besides a per-thread launch counter: calls on different streams with
 *    distinct workspaces may run concurrently.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* identical to cudaStream_t */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null pointer, inconsistent sizes, misaligned pointer */
    DSA_ERR_UNSUPPORTED = 2, /* shape or mode outside the compiled set (see dsa_dims) */
    DSA_ERR_WORKSPACE = 3,   /* ws == NULL or ws_bytes < dsa_workspace_size(...) */
    DSA_ERR_LAUNCH = 4,      /* a CUDA launch or tensor-map encode failed */
    DSA_ERR_DEVICE = 5,      /* dsa_read_error found a device-side fault bit (see DSA_FAULT_*) */
    DSA_ERR_TIMEOUT = 6,     /* dsa_read_error found a pipeline wait that gave up */
    DSA_ERR_TOO_LARGE = 7    /* dsa_indexer_topk_noalloc: the call needs more than its static scratch */
} dsa_status;

/* bits of the device error word */
#define DSA_FAULT_BLOCK_TABLE 0x1 /* block_table entry outside [0, num_blocks) */
#define DSA_FAULT_INDEX 0x2       /* idx entry outside [0, seq_len) and not -1 */
#define DSA_FAULT_TIMEOUT 0x4     /* a bounded wait inside a kernel expired */

typedef enum {
    DSA_F32 = 0,       /* q_I, k_I, q, kv, out: fp32 */
    DSA_BF16 = 1,      /* q_I, k_I, q, kv, out: bf16 */
    DSA_BF16_KFP8 = 2, /* as DSA_BF16, but k_I is OCP e4m3 with one fp32 scale per 64-token block */
    DSA_MXFP8 = 3      /* as DSA_BF16, but the indexer runs in MXFP8 (OCP Microscaling, E4M3 elements):
                        * k_I is e4m3 codes with one E8M0 scale byte per 32 elements of a key, and
                        * q_I (bf16) is quantised the same way inside the call ("Day0 Inference
                        * Support ... on Huawei Ascend CANN Architecture" §3: MXFP8 dynamic
                        * quantisation in the indexing stage) */
} dsa_mode;

/*
 * Flag OR-ed into dsa_dims.mode (with DSA_BF16, DSA_BF16_KFP8 or DSA_MXFP8): the latent cache
 * kv_cache holds FP8 records instead of bf16 rows ("Day0 Inference Support ... on Huawei Ascend CANN
 * Architecture" §3: FP8 block quantisation in the attention stage, an independent block of 128
 * elements per token and head). A record is the d e4m3 codes of the row, then ceil(d / 128) fp32
 * scales (tile j covers elements 128j .. 128j + 127, the last tile the remaining d mod 128), then
 * zero bytes up to DSA_KV_FP8_RECORD_BYTES(d), a multiple of 16; element e of the row is
 * code[e] * scale[e / 128]. The attention dequantises every element to bf16 (code * scale in fp32,
 * rounded to nearest even) before its tensor-core products; q, out and lse keep their types.
 * dsa_cache_append quantises each new latent row tile by tile, in fp32: scale = amax / 448 (1 when
 * amax is 0), code = RNE_e4m3(x / scale), saturating at +-448. The indexer ignores the flag.
 * Requires d % 16 == 0.
 */
#define DSA_KV_FP8 0x10
#define DSA_KV_FP8_RECORD_BYTES(d) ((((d) + 4 * (((d) + 127) / 128)) + 15) / 16 * 16)

/*
 * Problem dimensions.
 *   block_size must be 64 (tokens per physical cache block).
 *   DSA_F32:              H_I <= 64, d_I <= 256, d_I % 4 == 0, H <= 128, d <= 1024, d % 4 == 0, d_v <= d
 *   DSA_BF16 / _KFP8 / DSA_MXFP8: indexer (H_I, d_I) == (64, 128) [tensor cores] or H_I <= 64, d_I <= 256,
 *                         d_I % 8 == 0 (DSA_MXFP8: d_I % 32 == 0);
 *                         attention (H, d, d_v) == (128, 576, 512) [tensor cores] or H <= 128, d <= 1024,
 *                         d % 8 == 0, d_v <= d, d_v % 8 == 0
 *   1 <= K <= 2048.
 */
typedef struct {
    int32_t mode;       /* dsa_mode, optionally | DSA_KV_FP8 | DSA_Q_MX_READY */
    int32_t B;          /* number of sequences (rows of block_table, entries of seq_lens) */
    int32_t max_blocks; /* block_table row length */
    int32_t num_blocks; /* physical blocks in k_I_cache and kv_cache */
    int32_t block_size; /* 64 */
    int32_t H_I, d_I;   /* indexer heads, indexer head dim */
    int32_t H, d, d_v;  /* attention heads, latent row width, value width (V = row[0:d_v]) */
    int32_t K;          /* Top-K */
} dsa_dims;

/* Clears the error word of a freshly allocated workspace (enqueued on `stream`). Call once after
 * allocating `ws`; dsa_read_error clears it again after each read. */
dsa_status dsa_workspace_init(void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Bytes of workspace needed by any of the calls below for T query rows with these dims on the
 * current device. T > B means some sequence has several query rows (prefill): on the tensor-core
 * indexer shapes this includes the prefill score matrix, T * max_blocks * 64 fp32 values.
 * Returns 0 for invalid dims. */
size_t dsa_workspace_size(const dsa_dims* dims, int32_t T);

/*
 * Indexer + Top-K ("lightning indexer": scores -> top_k_indices).
 *   q_I        [T][H_I][d_I]        fp32 or bf16 (per mode)
 *   w          [T][H_I]             fp32 head weights (any sign)
 *   k_I_cache  [num_blocks][64][d_I] fp32 / bf16 / e4m3 codes (per mode)
 *   k_I_scale  DSA_BF16_KFP8: [num_blocks] fp32 per-block scale; DSA_MXFP8: [num_blocks][64][d_I / 32]
 *              uint8 E8M0 scales (value 2^(byte - 127); byte 255, NaN in the MX format, is not a
 *              supported input), 16-byte aligned; ignored in the other modes
 *   (DSA_MXFP8: each group of 32 elements of every q_I head row is quantised to E4M3 with shared
 *   exponent X = floor(log2(amax)) - 8, at least -127, codes RNE(x * 2^-X) saturating at +-448,
 *   and scored with the values code * 2^X; keys score with code * 2^(byte - 127).)
 *   block_table[B][max_blocks]      int32 physical block ids (entries past a sequence's end unread)
 *   seq_lens   [B]                  int32 cached positions per sequence, new tokens included
 *   q_seq      [T]                  int32 sequence of each query row; NULL means row t is sequence t (T == B)
 *   q_pos      [T]                  int32 absolute position of each query row (< seq_len of its
 *                                   sequence); NULL means decode: q_pos[t] = seq_lens[q_seq[t]] - 1
 *   idx        [T][K]               int32 out: the selected logical positions of each row in
 *                                   ascending order, then -1 for the slots past min(K, pos + 1)
 * Decode-shaped calls (each sequence has at most one query row) stream the keys once with the
 * Top-K fused (no score tensor leaves the chip). In calls with more rows than sequences on the
 * tensor-core indexer shapes (H_I, d_I) == (64, 128), every group of four consecutive rows
 * (4g..4g+3) of one sequence is scored on the tensor cores as one contraction over the group's
 * causal prefix into an fp32 score matrix in the workspace, then each row's Top-K is selected from
 * its scores; the other rows take the decode kernels. The result is the same either way.
 * ("Day0 Inference Support ... on Huawei Ascend CANN Architecture" §2.1: the lightning indexer
 * maps the quantised query, head weights and paged key cache to Top-K indices; "Engineering Path
 * for Day-0 Adaptation ..." §3.1: index selection is scoring followed by Top-K filtering.)
 */
dsa_status dsa_indexer_topk(const dsa_dims* dims, const void* q_I, const float* w, const void* k_I_cache,
                            const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_seq, const int32_t* q_pos, int32_t T, int32_t* idx, void* ws,
                            size_t ws_bytes, dsa_stream_t stream);

/*
 * Sparse attention over the positions idx selects ("sparse flash attention").
 *   q          [T][H][d]            fp32 or bf16
 *   kv_cache   [num_blocks][64][d]  fp32 or bf16 shared latent rows (K = row, V = row[0:d_v]);
 *                                   with DSA_KV_FP8: [num_blocks][64][DSA_KV_FP8_RECORD_BYTES(d)] FP8
 *                                   records (see DSA_KV_FP8)
 *   idx        [T][K]               int32 logical positions, -1 = empty slot (any order)
 *   sm_scale   softmax scale (usually 1/sqrt(d))
 *   out        [T][H][d_v]          fp32 (DSA_F32) or bf16 out
 *   lse        [T][H]               fp32 natural-log sum of exp of the logits, or NULL; rows with no
 *                                   valid index give out = 0 and lse = -inf
 */
dsa_status dsa_sparse_attn(const dsa_dims* dims, const void* q, const void* kv_cache, const int32_t* block_table,
                           const int32_t* seq_lens, const int32_t* q_seq, const int32_t* idx, int32_t T,
                           float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream);

/*
 * Fused decode step: one query row per sequence (T = B, q_seq = NULL, q_pos = NULL), the indexer +
 * Top-K followed by sparse attention on one stream. idx may be NULL (the indices then live in the
 * workspace only). Arguments as in dsa_indexer_topk / dsa_sparse_attn.
 */
dsa_status dsa_decode(const dsa_dims* dims, const void* q_I, const float* w, const void* k_I_cache,
                      const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens, const void* q,
                      const void* kv_cache, float sm_scale, int32_t* idx, void* out, float* lse, void* ws,
                      size_t ws_bytes, dsa_stream_t stream);

/*
 * Cache append: writes new tokens' indexer keys and latent rows into their paged slots (the step
 * before dsa_indexer_topk / dsa_sparse_attn; "How the Ascend Computing Platform Achieves Same-Day
 * Inference Adaptation ..." §2.2: the cache update is fused with the flow producing the entries;
 * "Day0 Inference Support ... on Huawei Ascend CANN Architecture" §3: the indexer's keys are
 * quantised on the way in).
 *   k_I_new    [T][d_I]   fp32 (DSA_F32) or bf16 (the other modes; DSA_BF16_KFP8 and DSA_MXFP8: the
 *                         values to quantise)
 *   kv_new     [T][d]     fp32 or bf16 latent rows (with DSA_KV_FP8: bf16, quantised into FP8 records)
 *   seq_lens   [B]        cached positions per sequence AFTER the append (new tokens included)
 *   q_seq, q_pos [T]      sequence and position of each new token, as in dsa_indexer_topk (NULL: one
 *                         token per sequence at position seq_lens - 1)
 *   k_I_cache, k_I_scale, kv_cache   updated in place (k_I_scale only for DSA_BF16_KFP8 / DSA_MXFP8)
 *   ws         any workspace of this library (only its error word is used), ws_bytes >= 256
 * The new tokens of a sequence are its tail (positions seq_len - n .. seq_len - 1), given as
 * consecutive rows in ascending position. fp32 / bf16 keys and all latent rows are copied. FP8
 * keys: every block that receives new tokens is requantised as a whole: with x = code * scale
 * (fp32) for its earlier tokens and the new keys' values, the block's scale becomes amax / 448
 * (1 when amax is 0) and each code RNE_e4m3(x / scale), saturating at +-448, all in fp32.
 * MXFP8 keys: each new key's groups of 32 are quantised on their own (as q_I is in the indexer),
 * writing its codes and its d_I / 32 scale bytes; no other row changes. Rows
 * with an invalid sequence, position or block-table entry are skipped and reported through the
 * error word (DSA_FAULT_INDEX / DSA_FAULT_BLOCK_TABLE). Requires (d * elem) and (d_I * elem) to be
 * multiples of 16 bytes.
 */
dsa_status dsa_cache_append(const dsa_dims* dims, const void* k_I_new, const void* kv_new,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                            const int32_t* q_pos, int32_t T, void* k_I_cache, void* k_I_scale, void* kv_cache,
                            void* ws, size_t ws_bytes, dsa_stream_t stream);

/*
 * Indexer prolog: one launch that prepares the indexer's inputs for a step ("Day0 Inference Support
 * ... on Huawei Ascend CANN Architecture" §2.2, Indexer Prolog: the query quantisation runs beside
 * the other preparations instead of after them):
 *  - the cache append of T_new new tokens, exactly as dsa_cache_append with the same arguments;
 *  - with q_I_mx not NULL (DSA_MXFP8 only): the MXFP8 quantisation of the indexer query q_I
 *    [T_q][H_I][d_I] (bf16), written to q_I_mx [T_q][H_I][d_I] as the exact bf16 values of its MX
 *    elements (code * 2^X; the same rounding dsa_indexer_topk applies).
 * Pass q_I_mx as q_I to dsa_indexer_topk / dsa_decode with DSA_Q_MX_READY in dims.mode: they then
 * skip their own quantisation of the query (one launch fewer); the indices are the same, since
 * quantising MX values again returns them unchanged. ws as for dsa_cache_append (only its error
 * word is used). Either part may be empty (T_new = 0, or q_I_mx = NULL).
 */
#define DSA_Q_MX_READY 0x20
dsa_status dsa_indexer_prolog(const dsa_dims* dims, const void* k_I_new, const void* kv_new,
                              const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                              const int32_t* q_pos, int32_t T_new, void* k_I_cache, void* k_I_scale, void* kv_cache,
                              const void* q_I, int32_t T_q, void* q_I_mx, void* ws, size_t ws_bytes,
                              dsa_stream_t stream);

/*
 * Hierarchical (coarse -> fine) index selection ("Engineering Path for Day-0 Adaptation ..." §3.1:
 * coarse filtering at block granularity followed by refinement; "How the Ascend Computing
 * Platform Achieves Same-Day Inference Adaptation ..." §3.1: the coarse filter reuses summary
 * information held in the cache, the fine filter computes only within the candidate blocks).
 * A variant of dsa_indexer_topk that reads one summary key per 64-token block plus the keys of
 * n_sel chosen blocks per row instead of every key; its result is the method's own, not the
 * exact Top-K (they agree when n_sel covers every block).
 *
 * dsa_block_summaries: summaries [B][pages * 64][d_I] bf16, pages = ceil(max_blocks / 64): row
 *   b * pages * 64 + lb of every valid logical block lb of sequence b (lb < ceil(seq_len / 64))
 *   receives the mean of the block's valid keys -- fp32 sum in token order of the keys' values
 *   (FP8: code * block scale in fp32; MXFP8: code * 2^(byte - 127)), fp32 division by the count,
 *   bf16 round to nearest even.
 *   Other rows are not written. Any workspace with ws_bytes >= 256 (only its error word is used).
 * dsa_indexer_topk_hier: arguments as dsa_indexer_topk (bf16 modes only; DSA_F32 gives
 *   DSA_ERR_UNSUPPORTED), plus the summaries and n_sel (1..2048):
 *   1. coarse: the n_sel blocks with the largest indexer score of their summary (the indexer
 *      formula with the summary as the key and the bf16 q_I as given, also in DSA_MXFP8; ties to
 *      the lower block) among the blocks
 *      0 .. pos(t) / 64 of the row's sequence;
 *   2. fine: the K largest indexer scores (ties to the lower position) among the tokens of the
 *      chosen blocks with s <= pos(t).
 *   idx [T][K] ascending positions then -1; blocks_out [T][n_sel] (optional) the chosen logical
 *   blocks ascending then -1. ws of at least dsa_hier_workspace_size(dims, T, n_sel) bytes,
 *   initialised with dsa_workspace_init.
 */
size_t dsa_hier_workspace_size(const dsa_dims* dims, int32_t T, int32_t n_sel);
/* After dsa_cache_append of the same T new tokens (same q_seq / q_pos convention, seq_lens after
 * the append): recomputes the summaries of the blocks those tokens touched, exactly as
 * dsa_block_summaries would (the other blocks' summaries are unchanged by an append). */
dsa_status dsa_block_summaries_append(const dsa_dims* dims, const void* k_I_cache, const void* k_I_scale,
                                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                                      const int32_t* q_pos, int32_t T, uint16_t* summaries, void* ws, size_t ws_bytes,
                                      dsa_stream_t stream);
dsa_status dsa_block_summaries(const dsa_dims* dims, const void* k_I_cache, const void* k_I_scale,
                               const int32_t* block_table, const int32_t* seq_lens, uint16_t* summaries, void* ws,
                               size_t ws_bytes, dsa_stream_t stream);
dsa_status dsa_indexer_topk_hier(const dsa_dims* dims, const void* q_I, const float* w, const void* k_I_cache,
                                 const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* q_seq, const int32_t* q_pos, int32_t T, const uint16_t* summaries,
                                 int32_t n_sel, int32_t* idx, int32_t* blocks_out, void* ws, size_t ws_bytes,
                                 dsa_stream_t stream);

/*
 * Indexer + Top-K that allocates nothing and takes no workspace: the same computation as
 * dsa_indexer_topk (arguments as there) on its decode-path kernels for every row, with the scratch
 * in one statically sized device buffer inside libdsa.so (DSA_NOALLOC_SCRATCH_BYTES per device).
 *
 * The method's pages have no counterpart of this call: it serves callers that cannot allocate
 * device memory or hand over a workspace -- code running inside another framework's caching
 * allocator or memory pool that forbids raw allocations, plugins whose host owns all device
 * memory, and launch sequences that must not change the device's memory map between calls.
 *
 *   fault_word  optional DEVICE int32 (may be NULL) that receives this call's DSA_FAULT_* bits,
 *               copied on `stream` after the kernels; bad rows are skipped as in dsa_indexer_topk.
 *
 * The first call on each device (with that device current) resolves the device address of the
 * static buffer (cudaGetSymbolAddress); make that first call before any stream capture. Every
 * call then clears the buffer's error word on `stream` and launches the same kernels as
 * dsa_indexer_topk. All calls on one device share the one buffer: calls that overlap in time
 * (different streams or threads without ordering between them) race and give wrong indices;
 * order them on one stream.
 * Returns DSA_ERR_TOO_LARGE, launching nothing, when the indexer's scratch (error word, work plan
 * and candidate lists: about (indexer CTAs + T) * K * 8 bytes, plus T * H_I * d_I * 2 bytes for
 * the quantised query in DSA_MXFP8) exceeds DSA_NOALLOC_SCRATCH_BYTES (for K = 2048: T <= 870
 * rows with the 64 x 128 bf16 indexer on 152 SMs). This size check comes before the pointer checks,
 * so a call with null buffers tells whether T rows fit without launching anything.
 * T = 0 launches nothing and leaves the static scratch alone (only *fault_word is cleared);
 * DSA_ERR_LAUNCH when the set-up or a launch fails.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (16u << 20)
dsa_status dsa_indexer_topk_noalloc(const dsa_dims* dims, const void* q_I, const float* w, const void* k_I_cache,
                                    const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                                    const int32_t* q_seq, const int32_t* q_pos, int32_t T, int32_t* idx,
                                    int32_t* fault_word, dsa_stream_t stream);

/* Synchronises `stream`, copies the device error word of `ws` to *fault_bits (may be NULL) and
 * clears it. Returns DSA_OK when no bit was set, DSA_ERR_TIMEOUT when DSA_FAULT_TIMEOUT was set,
 * DSA_ERR_DEVICE for any other bit, DSA_ERR_LAUNCH if the copy failed. */
dsa_status dsa_read_error(void* ws, int32_t* fault_bits, dsa_stream_t stream);

/* Self-test of the failure path every pipeline wait of this library takes: launches one CTA whose
 * bounded wait on an mbarrier that nothing completes gives up after its limit (about one second),
 * sets DSA_FAULT_TIMEOUT in the error word of `ws` (any workspace, ws_bytes >= 256) and returns;
 * dsa_read_error then reports DSA_ERR_TIMEOUT and the context stays usable. */
dsa_status dsa_selftest_wait_timeout(void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Number of kernels the last successful call on this thread launched (0 before any call). */
int32_t dsa_last_launch_count(void);

/* Static string for a status code. */
const char* dsa_status_string(dsa_status status);

/* ABI version (major * 100 + minor). */
int32_t dsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
