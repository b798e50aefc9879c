// Host side of the C ABI (include/dsa.h): argument checks, workspace layout, kernel selection and
// launch order. Nothing here allocates, frees or synchronises (dsa_read_error excepted).
//
// Kernel selection follows the shape of the call ("Adapting GPU Software Stacks ..." §3.3:
// separate implementations per path, chosen at run time from batch size and sequence length):
// tensor-core kernels for the 64x128 indexer and the 128-head x 576 latent attention, CUDA-core
// kernels for small shapes (the fp32 workload).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace dsa {

static thread_local int g_last_launches = 0;

constexpr int kMaxDevices = 64;

int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < kMaxDevices && (n = cache[dev].load(std::memory_order_relaxed)) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool set_max_dynamic_smem(const void* func, size_t bytes) {
    struct Entry {
        int dev;
        const void* func;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : done)
        if (e.dev == dev && e.func == func && e.bytes >= bytes) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
        return false;
    done.push_back({dev, func, bytes});
    return true;
}

bool indexer_uses_tc(const dsa_dims& d) {
    return (d.mode == DSA_BF16 || d.mode == DSA_BF16_KFP8 || d.mode == DSA_MXFP8) && d.H_I == 64 && d.d_I == 128;
}

bool attn_uses_tc(const dsa_dims& d) {
    return (d.mode == DSA_BF16 || d.mode == DSA_BF16_KFP8 || d.mode == DSA_MXFP8) && d.H == 128 && d.d == 576 &&
           d.d_v == 512;
}

int indexer_ctas(const dsa_dims& d) {
    const int sms = device_sm_count();
    const int G = indexer_uses_tc(d) ? sms : 2 * sms;
    return G < kMaxIndexerCtas ? G : kMaxIndexerCtas;
}

int attn_splits(const dsa_dims& d, int T) {
    if (!attn_uses_tc(d) || T <= 0) return 1;
    const int sms = device_sm_count();
    int S = sms / (2 * T);
    int smax = d.K / 64;
    if (smax > kMaxSplits) smax = kMaxSplits;
    if (S > smax) S = smax;
    return S < 1 ? 1 : S;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool prefill_path(const dsa_dims& d, int T) { return indexer_uses_tc(d) && T >= 4 && T > d.B; }

WsLayout ws_layout(const dsa_dims& d, int T, bool allow_prefill) {
    WsLayout w{};
    w.G = indexer_ctas(d);
    w.S = attn_splits(d, T);
    w.NG = (allow_prefill && prefill_path(d, T)) ? T / 4 : 0;
    size_t off = 0;
    w.err = off;
    off += 256;
    w.tile_prefix = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(T) + 1));
    w.group_prefix = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(T) + 1));
    w.merge_count = off;
    off = align256(off + sizeof(int32_t) * (kMergeLevels - 1) * static_cast<size_t>(merge_group_bound(T, w.G)));
    w.slot_count = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(w.G) + T));
    w.slots = off;
    off = align256(off + sizeof(uint64_t) * (static_cast<size_t>(w.G) + T) * d.K);
    w.slot_est = off;
    off = align256(off + sizeof(uint64_t) * (static_cast<size_t>(w.G) + T));
    w.q_mx = off;
    if (d.mode == DSA_MXFP8) off = align256(off + sizeof(uint16_t) * static_cast<size_t>(T) * d.H_I * d.d_I);
    w.idx = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T) * d.K);
    w.part_o = off;
    if (w.S > 1) off = align256(off + sizeof(float) * static_cast<size_t>(T) * w.S * d.H * d.d_v);
    w.part_ml = off;
    if (w.S > 1) off = align256(off + sizeof(float) * static_cast<size_t>(T) * w.S * 2 * d.H * 2);
    w.gemm_flag = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(w.NG));
    w.gemm_tile_prefix = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(w.NG) + 1));
    w.scores = off;
    if (w.NG > 0) off = align256(off + sizeof(float) * static_cast<size_t>(T) * d.max_blocks * kBlock);
    w.total = off;
    return w;
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

static EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiled fn = encode_fn();
    if (!fn || rows == 0) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------------------------
// argument checks
// ------------------------------------------------------------------------------------------------

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The public mode may carry DSA_KV_FP8 (the latent cache's storage); every kernel below takes the
// indexer-key mode alone, and the attention and the cache append get the flag on its own.
static dsa_status split_mode(const dsa_dims* in, dsa_dims* out, bool* kv8) {
    if (!in) return DSA_ERR_INVALID_ARG;
    *out = *in;
    *kv8 = (in->mode & DSA_KV_FP8) != 0;
    out->mode = in->mode & ~(DSA_KV_FP8 | DSA_Q_MX_READY);
    if (*kv8 && (out->mode == DSA_F32 || in->d % 16)) return DSA_ERR_UNSUPPORTED;
    if ((in->mode & DSA_Q_MX_READY) && out->mode != DSA_MXFP8) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// DSA_Q_MX_READY: q_I already holds the MXFP8 values (dsa_indexer_prolog wrote them).
static bool q_mx_ready(const dsa_dims* in) { return (in->mode & DSA_Q_MX_READY) != 0; }

static dsa_status check_common(const dsa_dims* d) {
    if (!d) return DSA_ERR_INVALID_ARG;
    if (d->mode < DSA_F32 || d->mode > DSA_MXFP8) return DSA_ERR_UNSUPPORTED;
    if (d->block_size != kBlock) return DSA_ERR_UNSUPPORTED;
    if (d->B <= 0 || d->max_blocks <= 0 || d->num_blocks <= 0) return DSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(d->num_blocks) * kBlock >= (1ll << 31)) return DSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(d->max_blocks) * kBlock >= (1ll << 31)) return DSA_ERR_UNSUPPORTED;
    if (d->K <= 0 || d->K > 2048) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

static dsa_status check_indexer_dims(const dsa_dims* d) {
    dsa_status st = check_common(d);
    if (st != DSA_OK) return st;
    if (d->H_I <= 0 || d->d_I <= 0) return DSA_ERR_INVALID_ARG;
    if (indexer_uses_tc(*d)) return DSA_OK;
    if (d->H_I > 64 || d->d_I > 256) return DSA_ERR_UNSUPPORTED;
    const int unit = d->mode == DSA_F32 ? 4 : (d->mode == DSA_BF16 ? 8 : (d->mode == DSA_MXFP8 ? 32 : 16));
    if (d->d_I % unit) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// The key scales a mode needs: fp32 per block (FP8 keys) or E8M0 bytes, 16-byte aligned (MXFP8,
// fetched with bulk copies).
static bool scale_ok(const dsa_dims* d, const void* k_I_scale) {
    if (d->mode == DSA_BF16_KFP8) return k_I_scale != nullptr;
    if (d->mode == DSA_MXFP8) return k_I_scale != nullptr && aligned16(k_I_scale);
    return true;
}

static dsa_status check_attn_dims(const dsa_dims* d) {
    dsa_status st = check_common(d);
    if (st != DSA_OK) return st;
    if (d->H <= 0 || d->d <= 0 || d->d_v <= 0 || d->d_v > d->d) return DSA_ERR_INVALID_ARG;
    if (attn_uses_tc(*d)) return DSA_OK;
    if (d->H > 128 || d->d > 1024) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

static dsa_status check_ws(const dsa_dims* d, int T, void* ws, size_t ws_bytes) {
    if (!ws) return DSA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return DSA_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(*d, T).total) return DSA_ERR_WORKSPACE;
    return DSA_OK;
}

static dsa_status run_indexer(const dsa_dims* d, const void* q_I, const float* w, const void* k_I_cache,
                              const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* q_seq, const int32_t* q_pos, int32_t T, int32_t* idx, void* ws,
                              cudaStream_t stream, int* launches, bool allow_prefill = true, bool q_ready = false) {
    const WsLayout L = ws_layout(*d, T, allow_prefill);
    uint8_t* base = static_cast<uint8_t*>(ws);
    IndexerArgs a{};
    a.mode = d->mode;
    a.B = d->B;
    a.max_blocks = d->max_blocks;
    a.num_blocks = d->num_blocks;
    a.H_I = d->H_I;
    a.d_I = d->d_I;
    a.K = d->K;
    a.T = T;
    a.q_I = q_I;
    a.w = w;
    a.k_I = k_I_cache;
    a.k_I_scale = k_I_scale;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.q_seq = q_seq;
    a.q_pos = q_pos;
    a.tile_prefix = reinterpret_cast<int32_t*>(base + L.tile_prefix);
    a.group_prefix = reinterpret_cast<int32_t*>(base + L.group_prefix);
    a.merge_count = reinterpret_cast<int32_t*>(base + L.merge_count);
    a.slot_count = reinterpret_cast<int32_t*>(base + L.slot_count);
    a.slots = reinterpret_cast<uint64_t*>(base + L.slots);
    a.slot_est = reinterpret_cast<uint64_t*>(base + L.slot_est);
    a.idx = idx;
    a.err = reinterpret_cast<int*>(base + L.err);
    a.G = L.G;
    a.NG = q_seq ? L.NG : 0;
    a.gemm_flag = reinterpret_cast<int32_t*>(base + L.gemm_flag);
    a.gemm_tile_prefix = reinterpret_cast<int32_t*>(base + L.gemm_tile_prefix);
    a.scores = reinterpret_cast<float*>(base + L.scores);
    a.G2 = device_sm_count();
    if (d->mode == DSA_MXFP8 && !q_ready) {  // the quantised query first; the indexer kernels read it as bf16
        void* q_mx = base + L.q_mx;
        if (!launch_mx_quantize_q(q_I, q_mx, static_cast<int64_t>(T) * d->H_I * d->d_I, stream, launches))
            return DSA_ERR_LAUNCH;
        a.q_I = q_mx;
        a.after_quant = 1;
    }
    // decode calls on the tensor-core indexer plan inside its kernel (no plan kernel, no gap)
    a.self_plan = (a.NG == 0 && indexer_uses_tc(*d) && T <= kSelfPlanRows) ? 1 : 0;
    if (!a.self_plan && !launch_plan(a, stream, launches)) return DSA_ERR_LAUNCH;
    if (a.NG > 0 && !launch_indexer_prefill(a, stream, launches)) return DSA_ERR_LAUNCH;
    const bool ok = indexer_uses_tc(*d) ? launch_indexer_tc(a, stream, launches) : launch_indexer_simt(a, stream, launches);
    if (!ok) return DSA_ERR_LAUNCH;
    if (!launch_merge(a, stream, launches)) return DSA_ERR_LAUNCH;
    if (a.NG > 0 && !launch_prefill_topk(a, stream, launches)) return DSA_ERR_LAUNCH;
    return DSA_OK;
}

static dsa_status run_attn(const dsa_dims* d, bool kv8, const void* q, const void* kv_cache,
                           const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                           const int32_t* idx, int32_t T, float sm_scale, void* out, float* lse, void* ws,
                           cudaStream_t stream, int* launches, bool after_own_kernel) {
    const WsLayout L = ws_layout(*d, T);
    uint8_t* base = static_cast<uint8_t*>(ws);
    AttnArgs a{};
    a.mode = d->mode;
    a.B = d->B;
    a.max_blocks = d->max_blocks;
    a.num_blocks = d->num_blocks;
    a.H = d->H;
    a.d = d->d;
    a.d_v = d->d_v;
    a.K = d->K;
    a.T = T;
    a.sm_scale = sm_scale;
    a.q = q;
    a.kv = kv_cache;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.q_seq = q_seq;
    a.idx = idx;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float*>(base + L.part_o);
    a.part_ml = reinterpret_cast<float*>(base + L.part_ml);
    a.S = L.S;
    a.err = reinterpret_cast<int*>(base + L.err);
    a.after_own_kernel = after_own_kernel ? 1 : 0;
    a.kv_fp8 = kv8 ? 1 : 0;
    a.kv_rec = kv8 ? DSA_KV_FP8_RECORD_BYTES(d->d) : d->d * (d->mode == DSA_F32 ? 4 : 2);
    const bool ok = attn_uses_tc(*d) ? launch_attn_tc(a, stream, launches) : launch_attn_simt(a, stream, launches);
    return ok ? DSA_OK : DSA_ERR_LAUNCH;
}

// ------------------------------------------------------------------------------------------------
// scratch of dsa_indexer_topk_noalloc: one static device buffer per device, resolved once
// ------------------------------------------------------------------------------------------------

constexpr size_t kNoAllocScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_base[kMaxDevices];

// Device address of the static scratch on the current device; the first call per device looks it
// up (this may load the module on that device, so it belongs before any stream capture).
static void* noalloc_scratch() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        if (reinterpret_cast<uintptr_t>(p) & 255u) return nullptr;
        g_noalloc_base[dev] = p;
    }
    return g_noalloc_base[dev];
}

// ------------------------------------------------------------------------------------------------
// hierarchical selection: the coarse and fine problems and the workspace that holds both
// ------------------------------------------------------------------------------------------------

struct HierLayout {
    dsa_dims coarse, fine;
    int pages;            // summary pages per sequence: ceil(max_blocks / 64)
    size_t coarse_ws;     // at offset 0: its error word is the call's
    size_t coarse_table;  // int32 [B][pages]
    size_t coarse_lens;   // int32 [B]
    size_t coarse_pos;    // int32 [T]
    size_t bidx;          // int32 [T][n_sel] chosen blocks
    size_t vtable;        // int32 [T][n_sel] virtual block tables
    size_t vlen;          // int32 [T]
    size_t vidx;          // int32 [T][K] fine Top-K in virtual positions
    size_t fine_ws;
    size_t total;
};

static HierLayout hier_layout(const dsa_dims& d, int T, int n_sel) {
    HierLayout h{};
    h.pages = (d.max_blocks + kBlock - 1) / kBlock;
    h.coarse = d;
    h.coarse.mode = DSA_BF16;
    h.coarse.max_blocks = h.pages;
    h.coarse.num_blocks = d.B * h.pages;
    h.coarse.K = n_sel;
    h.fine = d;
    h.fine.B = T;
    h.fine.max_blocks = n_sel;
    size_t off = 0;
    h.coarse_ws = off;
    off = align256(off + ws_layout(h.coarse, T).total);
    h.coarse_table = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(d.B) * h.pages);
    h.coarse_lens = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(d.B));
    h.coarse_pos = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T));
    h.bidx = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T) * n_sel);
    h.vtable = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T) * n_sel);
    h.vlen = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T));
    h.vidx = off;
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(T) * d.K);
    h.fine_ws = off;
    off = align256(off + (T > 0 ? ws_layout(h.fine, T).total : 256));
    h.total = off;
    return h;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

size_t dsa_workspace_size(const dsa_dims* dims_in, int32_t T) {
    dsa_dims D;
    bool kv8;
    if (!dims_in || split_mode(dims_in, &D, &kv8) != DSA_OK) return 0;
    const dsa_dims* dims = &D;
    if (T < 0 || check_common(dims) != DSA_OK) return 0;
    return ws_layout(*dims, T).total;
}

dsa_status dsa_workspace_init(void* ws, size_t ws_bytes, dsa_stream_t stream) {
    if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)) return DSA_ERR_WORKSPACE;
    return cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DSA_OK
                                                                                              : DSA_ERR_LAUNCH;
}

dsa_status dsa_indexer_topk(const dsa_dims* dims_in, const void* q_I, const float* w, const void* k_I_cache,
                            const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_seq, const int32_t* q_pos, int32_t T, int32_t* idx, void* ws,
                            size_t ws_bytes, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_indexer_dims(dims);
    if (st != DSA_OK) return st;
    if (T < 0) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    if (T > 0 && (!q_I || !w || !k_I_cache || !block_table || !seq_lens || !idx)) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_I) || !aligned16(w) || !aligned16(k_I_cache)) return DSA_ERR_INVALID_ARG;
    st = check_ws(dims, T, ws, ws_bytes);
    if (st != DSA_OK) return st;
    int launches = 0;
    if (T > 0)
        st = run_indexer(dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, idx, ws,
                         reinterpret_cast<cudaStream_t>(stream), &launches, true, q_mx_ready(dims_in));
    g_last_launches = launches;
    return st;
}

dsa_status dsa_sparse_attn(const dsa_dims* dims_in, const void* q, const void* kv_cache, const int32_t* block_table,
                           const int32_t* seq_lens, const int32_t* q_seq, const int32_t* idx, int32_t T,
                           float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_attn_dims(dims);
    if (st != DSA_OK) return st;
    if (T < 0) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !kv_cache || !block_table || !seq_lens || !idx || !out)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    st = check_ws(dims, T, ws, ws_bytes);
    if (st != DSA_OK) return st;
    int launches = 0;
    if (T > 0)
        st = run_attn(dims, kv8, q, kv_cache, block_table, seq_lens, q_seq, idx, T, sm_scale, out, lse, ws,
                      reinterpret_cast<cudaStream_t>(stream), &launches, false);
    g_last_launches = launches;
    return st;
}

dsa_status dsa_decode(const dsa_dims* dims_in, const void* q_I, const float* w, const void* k_I_cache,
                      const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens, const void* q,
                      const void* kv_cache, float sm_scale, int32_t* idx, void* out, float* lse, void* ws,
                      size_t ws_bytes, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_indexer_dims(dims);
    if (st != DSA_OK) return st;
    st = check_attn_dims(dims);
    if (st != DSA_OK) return st;
    const int T = dims->B;
    if (!q_I || !w || !k_I_cache || !block_table || !seq_lens || !q || !kv_cache || !out) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_I) || !aligned16(w) || !aligned16(k_I_cache) || !aligned16(q) || !aligned16(kv_cache) ||
        !aligned16(out))
        return DSA_ERR_INVALID_ARG;
    st = check_ws(dims, T, ws, ws_bytes);
    if (st != DSA_OK) return st;
    const WsLayout L = ws_layout(*dims, T);
    int32_t* idx_buf = idx ? idx : reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.idx);
    int launches = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = run_indexer(dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, nullptr, nullptr, T, idx_buf, ws, s,
                     &launches, true, q_mx_ready(dims_in));
    if (st == DSA_OK)
        st = run_attn(dims, kv8, q, kv_cache, block_table, seq_lens, nullptr, idx_buf, T, sm_scale, out, lse, ws, s,
                      &launches, true);
    g_last_launches = launches;
    return st;
}

dsa_status dsa_indexer_topk_noalloc(const dsa_dims* dims_in, const void* q_I, const float* w, const void* k_I_cache,
                                    const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                                    const int32_t* q_seq, const int32_t* q_pos, int32_t T, int32_t* idx,
                                    int32_t* fault_word, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_indexer_dims(dims);
    if (st != DSA_OK) return st;
    if (T < 0) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    // the indexer uses the workspace regions up to the attention's (error word, plan, candidates);
    // checked before the pointers, so that a size query with null buffers never launches anything
    if (ws_layout(*dims, T, false).idx > kNoAllocScratchBytes) return DSA_ERR_TOO_LARGE;
    if (T > 0 && (!q_I || !w || !k_I_cache || !block_table || !seq_lens || !idx)) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_I) || !aligned16(w) || !aligned16(k_I_cache)) return DSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(fault_word) & 3u) return DSA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {  // no rows: no kernel and no scratch; only the caller's fault word is cleared
        g_last_launches = 0;
        if (fault_word && cudaMemsetAsync(fault_word, 0, sizeof(int32_t), s) != cudaSuccess) return DSA_ERR_LAUNCH;
        return DSA_OK;
    }
    void* ws = noalloc_scratch();
    if (!ws) return DSA_ERR_LAUNCH;
    int launches = 0;
    // the error word is the only scratch that must start at zero (every other region is written
    // before it is read within the call)
    if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return DSA_ERR_LAUNCH;
    st = run_indexer(dims, q_I, w, k_I_cache, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, idx, ws, s,
                     &launches, /*allow_prefill=*/false);
    if (st == DSA_OK && fault_word &&
        cudaMemcpyAsync(fault_word, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        st = DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return st;
}

dsa_status dsa_cache_append(const dsa_dims* dims_in, const void* k_I_new, const void* kv_new,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                            const int32_t* q_pos, int32_t T, void* k_I_cache, void* k_I_scale, void* kv_cache,
                            void* ws, size_t ws_bytes, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_common(dims);
    if (st != DSA_OK) return st;
    if (T < 0 || dims->d_I <= 0 || dims->d <= 0) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    if (T > 0 && (!k_I_new || !kv_new || !block_table || !seq_lens || !k_I_cache || !kv_cache)) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    const int act = dims->mode == DSA_F32 ? 4 : 2;
    if ((dims->d * act) % 16 || (dims->d_I * act) % 16) return DSA_ERR_UNSUPPORTED;
    if (dims->mode == DSA_MXFP8 && dims->d_I % 32) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(k_I_new) || !aligned16(kv_new) || !aligned16(k_I_cache) || !aligned16(kv_cache))
        return DSA_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return DSA_ERR_WORKSPACE;
    int launches = 0;
    if (!launch_cache_append(*dims, kv8, k_I_new, kv_new, block_table, seq_lens, q_seq, q_pos, T, k_I_cache,
                             k_I_scale, kv_cache, static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream),
                             &launches))
        st = DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return st;
}

dsa_status dsa_indexer_prolog(const dsa_dims* dims_in, const void* k_I_new, const void* kv_new,
                              const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                              const int32_t* q_pos, int32_t T_new, void* k_I_cache, void* k_I_scale, void* kv_cache,
                              const void* q_I, int32_t T_q, void* q_I_mx, void* ws, size_t ws_bytes,
                              dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_common(dims);
    if (st != DSA_OK) return st;
    if (T_new < 0 || T_q < 0 || dims->d_I <= 0 || dims->d <= 0) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T_new != dims->B) return DSA_ERR_INVALID_ARG;
    if (T_new > 0 && (!k_I_new || !kv_new || !block_table || !seq_lens || !k_I_cache || !kv_cache))
        return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    const int act = dims->mode == DSA_F32 ? 4 : 2;
    if ((dims->d * act) % 16 || (dims->d_I * act) % 16) return DSA_ERR_UNSUPPORTED;
    if (dims->mode == DSA_MXFP8 && dims->d_I % 32) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(k_I_new) || !aligned16(kv_new) || !aligned16(k_I_cache) || !aligned16(kv_cache))
        return DSA_ERR_INVALID_ARG;
    if (q_I_mx) {  // the query quantisation: MXFP8 only, both buffers [T_q][H_I][d_I] bf16
        if (dims->mode != DSA_MXFP8) return DSA_ERR_UNSUPPORTED;
        if (T_q > 0 && (!q_I || !aligned16(q_I) || !aligned16(q_I_mx))) return DSA_ERR_INVALID_ARG;
    }
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return DSA_ERR_WORKSPACE;
    int launches = 0;
    const int64_t q_elements = q_I_mx ? static_cast<int64_t>(T_q) * dims->H_I * dims->d_I : 0;
    if (!launch_indexer_prolog(*dims, kv8, k_I_new, kv_new, block_table, seq_lens, q_seq, q_pos, T_new, k_I_cache,
                               k_I_scale, kv_cache, q_I, q_I_mx, q_elements, static_cast<int*>(ws),
                               reinterpret_cast<cudaStream_t>(stream), &launches))
        st = DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return st;
}

size_t dsa_hier_workspace_size(const dsa_dims* dims_in, int32_t T, int32_t n_sel) {
    dsa_dims D;
    bool kv8;
    if (!dims_in || split_mode(dims_in, &D, &kv8) != DSA_OK) return 0;
    const dsa_dims* dims = &D;
    if (T <= 0 || n_sel <= 0 || n_sel > 2048 || check_common(dims) != DSA_OK) return 0;
    return hier_layout(*dims, T, n_sel).total;
}

dsa_status dsa_block_summaries(const dsa_dims* dims_in, const void* k_I_cache, const void* k_I_scale,
                               const int32_t* block_table, const int32_t* seq_lens, uint16_t* summaries, void* ws,
                               size_t ws_bytes, dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_common(dims);
    if (st != DSA_OK) return st;
    if (dims->d_I <= 0) return DSA_ERR_INVALID_ARG;
    if (dims->mode == DSA_MXFP8 && dims->d_I % 32) return DSA_ERR_UNSUPPORTED;
    if (!k_I_cache || !block_table || !seq_lens || !summaries) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return DSA_ERR_WORKSPACE;
    int launches = 0;
    if (!launch_block_summaries(*dims, k_I_cache, k_I_scale, block_table, seq_lens, summaries, static_cast<int*>(ws),
                                reinterpret_cast<cudaStream_t>(stream), &launches))
        st = DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return st;
}

dsa_status dsa_block_summaries_append(const dsa_dims* dims_in, const void* k_I_cache, const void* k_I_scale,
                                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                                      const int32_t* q_pos, int32_t T, uint16_t* summaries, void* ws, size_t ws_bytes,
                                      dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_common(dims);
    if (st != DSA_OK) return st;
    if (T < 0 || dims->d_I <= 0) return DSA_ERR_INVALID_ARG;
    if (dims->mode == DSA_MXFP8 && dims->d_I % 32) return DSA_ERR_UNSUPPORTED;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    if (T > 0 && (!k_I_cache || !block_table || !seq_lens || !summaries)) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return DSA_ERR_WORKSPACE;
    int launches = 0;
    if (!launch_summaries_append(*dims, k_I_cache, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, summaries,
                                 static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream), &launches))
        st = DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return st;
}

dsa_status dsa_indexer_topk_hier(const dsa_dims* dims_in, const void* q_I, const float* w, const void* k_I_cache,
                                 const void* k_I_scale, const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* q_seq, const int32_t* q_pos, int32_t T, const uint16_t* summaries,
                                 int32_t n_sel, int32_t* idx, int32_t* blocks_out, void* ws, size_t ws_bytes,
                                 dsa_stream_t stream) {
    dsa_dims D;
    bool kv8;
    {
        const dsa_status split = split_mode(dims_in, &D, &kv8);
        if (split != DSA_OK) return split;
    }
    const dsa_dims* dims = &D;
    dsa_status st = check_indexer_dims(dims);
    if (st != DSA_OK) return st;
    if (dims->mode == DSA_F32) return DSA_ERR_UNSUPPORTED;  // the coarse stage scores bf16 summaries with bf16 q_I
    if (T < 0 || n_sel <= 0 || n_sel > 2048) return DSA_ERR_INVALID_ARG;
    if (!q_seq && T != dims->B) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (!q_I || !w || !k_I_cache || !block_table || !seq_lens || !summaries || !idx) return DSA_ERR_INVALID_ARG;
    if (!scale_ok(dims, k_I_scale)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_I) || !aligned16(w) || !aligned16(k_I_cache) || !aligned16(summaries)) return DSA_ERR_INVALID_ARG;
    const HierLayout H = hier_layout(*dims, T, n_sel);
    if (check_indexer_dims(&H.coarse) != DSA_OK) return DSA_ERR_UNSUPPORTED;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < H.total) return DSA_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(ws);
    auto at = [&](size_t off) { return reinterpret_cast<int32_t*>(base + off); };
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int launches = 0;
    int* fine_err = reinterpret_cast<int*>(base + H.fine_ws);
    if (!launch_hier_setup(dims->B, H.pages, T, seq_lens, q_seq, q_pos, at(H.coarse_table), at(H.coarse_lens),
                           at(H.coarse_pos), fine_err, s, &launches))
        return DSA_ERR_LAUNCH;
    // coarse: the indexer over the summaries, Top-n_sel blocks per row
    st = run_indexer(&H.coarse, q_I, w, summaries, nullptr, at(H.coarse_table), at(H.coarse_lens), q_seq,
                     at(H.coarse_pos), T, at(H.bidx), base + H.coarse_ws, s, &launches);
    if (st != DSA_OK) return st;
    if (!launch_hier_virtualize(dims->B, dims->max_blocks, n_sel, T, block_table, seq_lens, q_seq, q_pos, at(H.bidx),
                                at(H.vtable), at(H.vlen), blocks_out, s, &launches))
        return DSA_ERR_LAUNCH;
    // fine: the indexer over the tokens of the chosen blocks (one virtual sequence per row)
    st = run_indexer(&H.fine, q_I, w, k_I_cache, k_I_scale, at(H.vtable), at(H.vlen), nullptr, nullptr, T, at(H.vidx),
                     base + H.fine_ws, s, &launches);
    if (st != DSA_OK) return st;
    if (!launch_hier_remap(T, n_sel, dims->K, at(H.bidx), at(H.vidx), idx, fine_err, reinterpret_cast<int*>(base), s,
                           &launches))
        return DSA_ERR_LAUNCH;
    g_last_launches = launches;
    return DSA_OK;
}

dsa_status dsa_read_error(void* ws, int32_t* fault_bits, dsa_stream_t stream) {
    if (!ws) return DSA_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_LAUNCH;
    if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_LAUNCH;
    if (cudaMemset(ws, 0, sizeof v) != cudaSuccess) return DSA_ERR_LAUNCH;
    if (fault_bits) *fault_bits = v;
    if (v & DSA_FAULT_TIMEOUT) return DSA_ERR_TIMEOUT;
    return v ? DSA_ERR_DEVICE : DSA_OK;
}

dsa_status dsa_selftest_wait_timeout(void* ws, size_t ws_bytes, dsa_stream_t stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return DSA_ERR_WORKSPACE;
    int launches = 0;
    const bool ok = launch_wait_timeout(static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream), &launches);
    g_last_launches = launches;
    return ok ? DSA_OK : DSA_ERR_LAUNCH;
}

int32_t dsa_last_launch_count(void) { return g_last_launches; }

const char* dsa_status_string(dsa_status status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case DSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DSA_ERR_LAUNCH: return "kernel launch failed";
        case DSA_ERR_DEVICE: return "device-side fault (bad block-table entry or index)";
        case DSA_ERR_TIMEOUT: return "a pipeline wait inside a kernel timed out";
        case DSA_ERR_TOO_LARGE: return "call needs more scratch than the static buffer of dsa_indexer_topk_noalloc";
    }
    return "unknown status";
}

int32_t dsa_version(void) { return 100; }

}  // extern "C"
