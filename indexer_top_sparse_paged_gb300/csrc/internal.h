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

// Byte offsets of the workspace regions for one call shape.
struct WsLayout {
    size_t err;          // int32 error word (+ padding to 256 B)
    size_t tile_prefix;  // int32 [T + 1]
    size_t slot_count;   // int32 [G + T]
    size_t slots;        // uint64 [G + T][K]
    size_t idx;          // int32 [T][K] (dsa_decode without a caller idx)
    size_t part_o;       // fp32 [T][S][H][d_v]
    size_t part_ml;      // fp32 [T][S][2 CTAs][H][2] (m, l)
    size_t scores;       // fp32 [T][max_blocks * 64] (prefill only)
    size_t total;
    int G;               // indexer CTAs
    int S;               // attention splits
};

int device_sm_count();
int indexer_ctas(const dsa_dims& d);
int attn_splits(const dsa_dims& d, int T);
WsLayout ws_layout(const dsa_dims& d, int T);

bool indexer_uses_tc(const dsa_dims& d);
bool attn_uses_tc(const dsa_dims& d);

// Encodes a 2-D row-major tensor map (inner extent `cols` elements, `rows` rows, row pitch
// `pitch_bytes`) with a box of box_cols x box_rows and 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows);

// ---- launchers (return false if a launch failed; each adds its launches to *launches) ----------

bool launch_plan(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_merge(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_indexer_simt(const IndexerArgs& a, cudaStream_t s, int* launches);
bool launch_indexer_tc(const IndexerArgs& a, cudaStream_t s, int* launches);

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
};

bool launch_attn_simt(const AttnArgs& a, cudaStream_t s, int* launches);
bool launch_attn_tc(const AttnArgs& a, cudaStream_t s, int* launches);

}  // namespace dsa
