// Host-side internals shared by the translation units of libdsa.so: the workspace layout and
// the per-kernel launchers. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dsa.h"
#include "common.cuh"

namespace dsa {

constexpr int kMaxSplits = 32;   // split-K pieces per attention row
constexpr int kMaxIndexerCtas = 1024;
constexpr int kMergeFanIn = 8;   // candidate lists one merge CTA selects from (<= 8 x 2048 keys)
constexpr int kMergeLevels = 4;  // 8^4 >= kMaxIndexerCtas lists per row
constexpr int kSelfPlanRows = 512;  // decode calls up to this many rows plan inside the indexer kernel

// Upper bound on the merge groups of a call (one merge CTA each): sum over rows of
// ceil(lists / 8) <= T + G / 8, since the rows' lists number at most G + T.
__host__ __device__ inline int merge_group_bound(int T, int G) { return T + (G + kMergeFanIn - 1) / kMergeFanIn + 1; }

// Byte offsets of the workspace regions for one call shape.
struct WsLayout {
    size_t err;          // int32 error word (+ padding to 256 B)
    size_t tile_prefix;  // int32 [T + 1]
    size_t group_prefix; // int32 [T + 1] merge groups before each row
    size_t merge_count;  // int32 [3][T + G/8 + 1] finished children of the merge tree's groups (levels 2..4)
    size_t slot_count;   // int32 [G + T]
    size_t slots;        // uint64 [G + T][K]
    size_t slot_est;     // uint64 [G + T] the sample estimate each list was filtered with
    size_t q_mx;         // bf16 [T][H_I][d_I] the MX-quantised q_I (DSA_MXFP8 only)
    size_t idx;          // int32 [T][K] (dsa_decode without a caller idx)
    size_t part_o;       // fp32 [T][S][H][d_v]
    size_t part_ml;      // fp32 [T][S][2 CTAs][H][2] (m, l)
    size_t gemm_flag;    // int32 [NG] prefill groups on the score GEMM (prefill path only)
    size_t gemm_tile_prefix;  // int32 [NG + 1]
    size_t scores;       // fp32 [T][max_blocks * 64] (prefill path only)
    size_t total;
    int G;               // indexer CTAs
    int S;               // attention splits
    int NG;              // candidate prefill groups (T / 4), 0 without the prefill path
};

int device_sm_count();
int indexer_ctas(const dsa_dims& d);
int attn_splits(const dsa_dims& d, int T);
// The prefill path (score GEMM + per-row Top-K for groups of 4 rows of one sequence) is taken
// by calls with more query rows than sequences, on the tensor-core indexer shapes.
bool prefill_path(const dsa_dims& d, int T);
WsLayout ws_layout(const dsa_dims& d, int T, bool allow_prefill = true);

bool indexer_uses_tc(const dsa_dims& d);
bool attn_uses_tc(const dsa_dims& d);

// Encodes a 2-D row-major tensor map (inner extent `cols` elements, `rows` rows, row pitch
// `pitch_bytes`) with a box of box_cols x box_rows and 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

// Raises a kernel's dynamic shared memory limit once per device (cached).
bool set_max_dynamic_smem(const void* func, size_t bytes);

// Launches `kernel`; with `pdl` the launch may overlap the tail of the previous kernel on the
// stream (programmatic dependent launch), so the kernel must call griddep_wait() before it reads
// anything that kernel writes. Only kernels that follow another kernel of the same call use it:
// the first kernel of a call always waits for all earlier work on the stream.
template <typename... KArgs, typename... Args>
inline bool launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess;
}

// ---- launchers (return false if a launch failed; each adds its launches to *launches) ----------

bool launch_plan(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_merge(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_indexer_simt(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_indexer_tc(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_indexer_prefill(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_prefill_topk(const IndexerArgs& a, cudaStream_t s, int* launches);
// MXFP8 q_I: `elements` bf16 values (a multiple of 32) -> their MXFP8 values as bf16, into `out`
bool launch_mx_quantize_q(const void* q_I, void* out, int64_t elements, cudaStream_t s, int* launches);

struct AttnArgs {
    int mode;
    int B, max_blocks, num_blocks;
    int H, d, d_v, K;
    int T;
    float sm_scale;
    const void* q;
    const void* kv;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* q_seq;
    const int32_t* idx;
    void* out;
    float* lse;
    float* part_o;
    float* part_ml;
    int S;
    int* err;
    int after_own_kernel;  // 1: launched right after this library's kernel (dsa_decode) -> PDL
    int kv_fp8;            // 1: kv holds FP8 records of kv_rec bytes (DSA_KV_FP8)
    int kv_rec;            // bytes per latent row (record) in the cache
};

bool launch_attn_simt(const AttnArgs& a, cudaStream_t s, int* launches);
bool launch_block_summaries(const dsa_dims& d, const void* k_I, const void* k_scale, const int32_t* block_table,
                            const int32_t* seq_lens, uint16_t* summaries, int* err, cudaStream_t s, int* launches);
bool launch_summaries_append(const dsa_dims& d, const void* k_I, const void* k_scale, const int32_t* block_table,
                             const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, int T,
                             uint16_t* summaries, int* err, cudaStream_t s, int* launches);
bool launch_hier_setup(int B, int pages, int T, const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos,
                       int32_t* coarse_table, int32_t* coarse_lens, int32_t* coarse_pos, int* fine_err, cudaStream_t s,
                       int* launches);
bool launch_hier_virtualize(int B, int max_blocks, int n_sel, int T, const int32_t* block_table,
                            const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, const int32_t* bidx,
                            int32_t* vtable, int32_t* vlen, int32_t* blocks_out, cudaStream_t s, int* launches);
bool launch_hier_remap(int T, int n_sel, int K, const int32_t* bidx, const int32_t* vidx, int32_t* idx, int* fine_err,
                       int* err, cudaStream_t s, int* launches);
bool launch_cache_append(const dsa_dims& d, bool kv_fp8, const void* k_new, const void* kv_new,
                         const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                         const int32_t* q_pos, int T, void* k_cache, void* k_scale, void* kv_cache, int* err,
                         cudaStream_t s, int* launches);
bool launch_indexer_prolog(const dsa_dims& d, bool kv_fp8, const void* k_new, const void* kv_new,
                           const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                           const int32_t* q_pos, int T, void* k_cache, void* k_scale, void* kv_cache, const void* q_I,
                           void* q_out, int64_t q_elements, int* err, cudaStream_t s, int* launches);
bool launch_attn_tc(const AttnArgs& a, cudaStream_t s, int* launches);
bool launch_wait_timeout(int* err, cudaStream_t s, int* launches);

}  // namespace dsa
