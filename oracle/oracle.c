/*
 * fp64 CPU oracle for index-selection sparse attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py load this library.  It shares no
 * code, header, table or helper with the CUDA path and is never called by it.
 *
 * What it computes (the plain definition; every step in fp64 on exactly
 * decoded inputs, no blocking, fusion or reordering beyond the definition):
 *
 *  1. Paged addressing ("Non-contiguous Layout of the KV Cache", Day-0 accelerator
 *     page §3.2): logical position s of sequence b lives in physical row
 *     block_table[b][s / bs] * bs + s % bs of the cache.
 *  2. Indexer score ("Core Pipeline Operator Fusion", Ascend CANN page §2.1 --
 *     relevance scoring, head-weight weighting, Top-K selection; formula fixed
 *     by the problem statement):
 *         S[t,s] = sum_j w[t,j] * max(0, sum_d q_I[t,j,d] * k_I[s,d])
 *     for every causal s in [0, pos(t)], with k_I = e4m3 code * block scale
 *     when the indexer keys are FP8 (Ascend CANN page §3).
 *  3. Top-K ("Integration of the Index Selection Operator", Day-0 accelerator
 *     page §3.1): the K largest S, ties to the lower s; fewer than K causal
 *     positions -> all of them, rest of the row -1.  The selection is a full
 *     library sort (qsort) under the total order (S descending, s ascending).
 *  4. Sparse attention (lightweight indexer page §1, "sparse flash attention"
 *     reads the KV pairs at the selected positions):
 *         z_i = sm_scale * q[t,h,:] . row_i,  p = softmax(z),
 *         out[t,h,:] = sum_i p_i * row_i[0:d_v],  lse = log sum_i exp(z_i)
 *     over the valid (!= -1) entries of idx[t]; V is the first d_v columns of
 *     the same shared latent row.  No valid entry -> out = 0, lse = -inf.
 *
 *  H. Hierarchical selection (coarse -> fine, Day-0 accelerator page §3.1 and the
 *     adaptation page §3.1: blocks shortlisted by summary scores, then fine
 *     filtering inside them): a block's summary key is the mean of its valid
 *     keys (fp32 sum in token order, fp32 division by the count, bf16 round to
 *     nearest even); the coarse stage is the indexer over the summaries, the
 *     fine stage the indexer over the tokens of the chosen blocks.  This file
 *     holds the summary; the two stages reuse steps 1-3 (oracle/__init__.py).
 *  0. Cache append (the step before the path: "Residual and normalization ...
 *     fused with the cache-update flow", Ascend adaptation page §2.2 table; the
 *     indexer prolog quantises keys, Ascend CANN page §2.2/§3): each new token t
 *     of sequence b sits at position pos(t) of the sequence's tail; its latent
 *     row and (fp32 / bf16 modes) its indexer key are copied to the paged slot.
 *     With FP8 indexer keys every touched 64-token block is requantised: with
 *     x = code * scale_old (fp32) for the block's earlier tokens and the new keys'
 *     values, scale = amax / 448 (fp32; 1 when amax is 0) and every code of the
 *     block becomes RNE_e4m3(x / scale), saturating at +-448.
 *
 * MXFP8 indexer (mode 3; "MXFP8 dynamic quantization in the indexing stage",
 * Ascend CANN page §3: groups of 32 adjacent elements share one scale): the
 * indexer keys are OCP MX E4M3 codes with one E8M0 scale byte (2^(byte-127))
 * per 32 elements of a key, and the bf16 query q_I is quantised the same way
 * before scoring (OCP Microscaling Formats: shared exponent
 * X = floor(log2(amax)) - 8 for E4M3, clamped to [-127, 127], -127 for an
 * all-zero group; element = RNE_e4m3(v * 2^-X), saturating at +-448; value =
 * element * 2^X).  Attention stays bf16.
 *
 * FP8 latent cache (flag 16 of mode, with any bf16 mode; "FP8 block quantization
 * in the attention stage", Ascend CANN page §3: per token and head, independent
 * blocks of 128 elements): every latent row is stored as one record of d e4m3
 * codes, then ceil(d/128) fp32 scales (tile j covers elements 128j..128j+127;
 * the last tile the remaining d mod 128 ones), then zero bytes up to a multiple
 * of 16 bytes.  Element e of the row is code[e] * scale[e / 128].  Appending a
 * row quantises each tile on its own, every step in fp32: scale = amax / 448
 * (1 when amax is 0), code = RNE_e4m3(x / scale), saturating at +-448.
 *
 * Input decoding:
 *  - bf16: the 16 bits are the top half of an IEEE binary32 (exact widening).
 *  - e4m3 (OCP 8-bit floating point spec, E4M3): sign, 4 exponent bits with
 *    bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111
 *    is NaN; there is no infinity; largest finite value 448.
 *
 * Multithreaded over independent work items with POSIX threads.  Build with
 * -ffp-contract=off so no fused multiply-add changes a result between hosts.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t mode; /* 0: fp32 everything; 1: bf16 (w fp32); 2: bf16 with e4m3 indexer keys; 3: MXFP8 indexer;
                   * + 16: FP8 latent cache (bf16 modes only) */
    int32_t B, max_blocks, num_blocks, block_size;
    int32_t H_I, d_I, H, d, d_v, K;
} odims;

enum { O_OK = 0, O_BAD_ARG = -1, O_BAD_IDX = -2, O_NOMEM = -3 };

#define OMODE(D) ((D)->mode & 15)          /* storage of activations and indexer keys */
#define KV_FP8(D) (((D)->mode & 16) != 0)  /* latent rows stored as FP8 records */

/* a valid mode: 0..3, plus the FP8-latent-cache flag on the bf16 modes */
static int mode_ok(const void* dims) {
    const int m = *(const int32_t*)dims;
    if (m & ~31) return 0;
    if ((m & 15) > 3) return 0;
    if ((m & 16) && (m & 15) == 0) return 0;
    return 1;
}

/* bytes of one FP8 latent record: d codes, one fp32 scale per 128-element tile, padded to 16 */
static size_t kv_record_bytes(int d) { return ((size_t)d + 4 * (size_t)((d + 127) / 128) + 15) / 16 * 16; }

/* ------------------------------------------------------------------------- */
/* exact decoders                                                            */
/* ------------------------------------------------------------------------- */

double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* (m/8) * 2^(1-7) */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* e4m3 encoder (same spec): round to nearest, ties to even, values beyond the
 * largest finite (448) saturate to it; NaN -> S.1111.111. */
uint8_t oracle_f32_to_e4m3(float f) {
    if (isnan(f)) return 0x7F;
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    const double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                    /* subnormal: multiples of 2^-9 */
        const double m = rint(ldexp(a, 9));      /* 0..8; 8 is the smallest normal, 0x08 */
        return sign | (uint8_t)m;
    }
    int e;
    frexp(a, &e);                                /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                               /* a = 1.m * 2^E, E >= -6 */
    double m = rint((ldexp(a, -E) - 1.0) * 8.0); /* 0..8 */
    if (m == 8.0) {
        m = 0.0;
        E += 1;
    }
    int code = ((E + 7) << 3) | (int)m;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* OCP MX (E4M3 elements, E8M0 scale) quantisation of 32 fp32 values: returns the shared
 * exponent X and writes the element codes. */
static int mx_quantize32(const float* v, uint8_t* codes) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i)
        if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
    int X = -127;
    if (amax > 0.0f) {
        int e;
        frexpf(amax, &e);  /* amax = f * 2^e, f in [0.5, 1): floor(log2(amax)) = e - 1 */
        X = (e - 1) - 8;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
    }
    for (int i = 0; i < 32; ++i) codes[i] = oracle_f32_to_e4m3(ldexpf(v[i], -X));
    return X;
}

/* the MXFP8 value of 32 bf16 values (quantise, then decode exactly) */
static void mx_roundtrip32(const uint16_t* bits, double* out) {
    float v[32];
    uint8_t c[32];
    for (int i = 0; i < 32; ++i) v[i] = (float)oracle_bf16_to_f64(bits[i]);
    const int X = mx_quantize32(v, c);
    for (int i = 0; i < 32; ++i) out[i] = ldexp(oracle_e4m3_to_f64(c[i]), X);
}

int oracle_mx_quantize32(const float* v, uint8_t* codes) { return mx_quantize32(v, codes); }

static double f32_at(const void* p, size_t i) { return (double)((const float*)p)[i]; }
static double bf16_at(const void* p, size_t i) { return oracle_bf16_to_f64(((const uint16_t*)p)[i]); }

/* value i of an activation / latent-cache tensor in the mode's storage type */
static double act_at(const odims* D, const void* p, size_t i) {
    return OMODE(D) == 0 ? f32_at(p, i) : bf16_at(p, i);
}

/* element e of latent row r: the activation type, or code * tile scale of an FP8 record */
static double kv_at(const odims* D, const void* kv, int64_t r, int e) {
    if (!KV_FP8(D)) return act_at(D, kv, (size_t)r * D->d + e);
    const uint8_t* rec = (const uint8_t*)kv + (size_t)r * kv_record_bytes(D->d);
    float scale;
    memcpy(&scale, rec + D->d + 4 * (e / 128), sizeof scale);
    return oracle_e4m3_to_f64(rec[e]) * (double)scale;
}

/* ------------------------------------------------------------------------- */
/* tiny work-queue thread pool                                               */
/* ------------------------------------------------------------------------- */

typedef void (*item_fn)(void* ctx, int64_t item, void* scratch);

typedef struct {
    item_fn fn;
    void* ctx;
    int64_t n_items;
    int64_t next;
    size_t scratch_bytes;
    pthread_mutex_t mu;
    int failed;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* P = (pool_t*)arg;
    void* scratch = P->scratch_bytes ? malloc(P->scratch_bytes) : NULL;
    if (P->scratch_bytes && !scratch) {
        pthread_mutex_lock(&P->mu);
        P->failed = 1;
        pthread_mutex_unlock(&P->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&P->mu);
        int64_t it = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (it >= P->n_items) break;
        P->fn(P->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

static int run_items(item_fn fn, void* ctx, int64_t n_items, size_t scratch_bytes, int threads) {
    pool_t P;
    P.fn = fn; P.ctx = ctx; P.n_items = n_items; P.next = 0; P.scratch_bytes = scratch_bytes; P.failed = 0;
    pthread_mutex_init(&P.mu, NULL);
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((int64_t)threads > n_items) threads = (int)(n_items > 0 ? n_items : 1);
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < threads; ++i) {
        if (pthread_create(&tid[i], NULL, pool_worker, &P) == 0) started = i;
        else break;
    }
    pool_worker(&P);
    for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
    pthread_mutex_destroy(&P.mu);
    return P.failed ? O_NOMEM : O_OK;
}

/* ------------------------------------------------------------------------- */
/* step 1+2: paged key fetch and indexer score                               */
/* ------------------------------------------------------------------------- */

typedef struct {
    const odims* D;
    const void* q_I; const float* w; const void* k_I; const float* k_I_scale;
    const int32_t* block_table; const int32_t* seq_lens; const int32_t* q_seq; const int32_t* q_pos;
    int T;
    double* S; const int64_t* row_off;  /* S[row_off[t] + s] */
    int64_t chunk;                       /* keys per work item */
    const int64_t* item_first;           /* first item index of row t (T+1 entries) */
    int bad;
} score_ctx;

/* physical cache row of logical position s in sequence b; -1 if the table entry is invalid */
static int64_t phys_row(const odims* D, const int32_t* block_table, int b, int64_t s, int32_t* blk_out) {
    int32_t blk = block_table[(int64_t)b * D->max_blocks + s / D->block_size];
    if (blk < 0 || blk >= D->num_blocks) return -1;
    if (blk_out) *blk_out = blk;
    return (int64_t)blk * D->block_size + s % D->block_size;
}

static void score_item(void* vctx, int64_t item, void* scratch) {
    score_ctx* C = (score_ctx*)vctx;
    const odims* D = C->D;
    /* find the row of this item */
    int lo = 0, hi = C->T - 1;               /* last row t with item_first[t] <= item */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (C->item_first[mid] <= item) lo = mid; else hi = mid - 1;
    }
    int t = lo;
    while (t + 1 <= C->T - 1 && C->item_first[t + 1] <= item) ++t;  /* skip empty rows */
    int64_t s0 = (item - C->item_first[t]) * C->chunk;
    int64_t pos = C->q_pos[t];
    int64_t s1 = s0 + C->chunk;
    if (s1 > pos + 1) s1 = pos + 1;
    int b = C->q_seq[t];
    double* q = (double*)scratch;            /* [H_I][d_I] decoded query */
    double* k = q + (size_t)D->H_I * D->d_I;  /* [d_I] decoded key */
    for (int j = 0; j < D->H_I; ++j)
        for (int e = 0; e < D->d_I; ++e) {
            size_t i = ((size_t)t * D->H_I + j) * D->d_I + e;
            q[(size_t)j * D->d_I + e] = act_at(D, C->q_I, i);
        }
    if (OMODE(D) == 3)  /* the MXFP8 query: every group of 32 quantised and decoded */
        for (int j = 0; j < D->H_I; ++j)
            for (int g = 0; g < D->d_I / 32; ++g)
                mx_roundtrip32((const uint16_t*)C->q_I + ((size_t)t * D->H_I + j) * D->d_I + 32 * g,
                               q + (size_t)j * D->d_I + 32 * g);
    for (int64_t s = s0; s < s1; ++s) {
        int32_t blk;
        int64_t row = phys_row(D, C->block_table, b, s, &blk);
        if (row < 0) { C->bad = 1; C->S[C->row_off[t] + s] = NAN; continue; }
        double scale = (OMODE(D) == 2) ? (double)C->k_I_scale[blk] : 1.0;
        for (int e = 0; e < D->d_I; ++e) {
            size_t i = (size_t)row * D->d_I + e;
            double v;
            if (OMODE(D) == 0) v = f32_at(C->k_I, i);
            else if (OMODE(D) == 1) v = bf16_at(C->k_I, i);
            else v = oracle_e4m3_to_f64(((const uint8_t*)C->k_I)[i]);
            if (OMODE(D) == 3)  /* E8M0 byte of the key's group of 32 */
                v = ldexp(v, (int)((const uint8_t*)C->k_I_scale)[(size_t)row * (D->d_I / 32) + e / 32] - 127);
            k[e] = v * scale;
        }
        double total = 0.0;
        for (int j = 0; j < D->H_I; ++j) {
            double dot = 0.0;
            for (int e = 0; e < D->d_I; ++e) dot += q[(size_t)j * D->d_I + e] * k[e];
            double relu = dot > 0.0 ? dot : 0.0;
            total += (double)C->w[(size_t)t * D->H_I + j] * relu;
        }
        C->S[C->row_off[t] + s] = total;
    }
}

static int check_dims(const odims* D) {
    if (!D || D->block_size <= 0 || D->H_I <= 0 || D->d_I <= 0 || D->K <= 0) return 0;
    if (!mode_ok(D)) return 0;
    if (OMODE(D) == 3 && D->d_I % 32) return 0;
    return 1;
}

static int check_rows(const odims* D, const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, int T) {
    for (int t = 0; t < T; ++t) {
        int b = q_seq[t];
        if (b < 0 || b >= D->B) return 0;
        if (q_pos[t] >= seq_lens[b]) return 0;
        if ((int64_t)seq_lens[b] > (int64_t)D->max_blocks * D->block_size) return 0;
    }
    return 1;
}

/* Scores of all causal positions of every query row.
 * S[row_off[t] + s] for s in [0, q_pos[t]]; q_pos[t] < 0 means an empty prefix. */
static int scores_all(const odims* D, const void* q_I, const float* w, const void* k_I, const float* k_I_scale,
                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos,
                      int T, double* S, const int64_t* row_off, int threads) {
    const int64_t chunk = 4096;
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + 1));
    if (!first) return O_NOMEM;
    first[0] = 0;
    for (int t = 0; t < T; ++t) {
        int64_t n = (int64_t)q_pos[t] + 1;
        if (n < 0) n = 0;
        first[t + 1] = first[t] + (n + chunk - 1) / chunk;
    }
    score_ctx C = {D, q_I, w, k_I, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, S, row_off, chunk, first, 0};
    size_t scratch = sizeof(double) * ((size_t)D->H_I * D->d_I + D->d_I);
    int rc = run_items(score_item, &C, first[T], scratch, threads);
    free(first);
    if (rc) return rc;
    return C.bad ? O_BAD_IDX : O_OK;
}

int oracle_index_scores(const odims* D, const void* q_I, const float* w, const void* k_I, const float* k_I_scale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                        const int32_t* q_pos, int T, int64_t row_stride, double* S, int threads) {
    if (!check_dims(D) || T < 0 || !check_rows(D, seq_lens, q_seq, q_pos, T)) return O_BAD_ARG;
    if ((OMODE(D) == 2 || OMODE(D) == 3) && !k_I_scale) return O_BAD_ARG;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    if (!off) return O_NOMEM;
    for (int t = 0; t < T; ++t) {
        if ((int64_t)q_pos[t] + 1 > row_stride) { free(off); return O_BAD_ARG; }
        off[t] = (int64_t)t * row_stride;
    }
    int rc = scores_all(D, q_I, w, k_I, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, S, off, threads);
    free(off);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* step 3: Top-K under (S descending, s ascending)                           */
/* ------------------------------------------------------------------------- */

typedef struct { double s; int32_t pos; } scored;

static int by_score_desc_pos_asc(const void* a, const void* b) {
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

typedef struct {
    const odims* D; const double* S; const int64_t* row_off; const int32_t* q_pos;
    int32_t* idx; double* kth;
} topk_ctx;

static void topk_row(void* vctx, int64_t t, void* scratch) {
    topk_ctx* C = (topk_ctx*)vctx;
    int64_t n = (int64_t)C->q_pos[t] + 1;
    if (n < 0) n = 0;
    scored* a = (scored*)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    int K = C->D->K;
    int32_t* out = C->idx + (int64_t)t * K;
    (void)scratch;
    if (!a) { for (int i = 0; i < K; ++i) out[i] = -2; return; }
    for (int64_t s = 0; s < n; ++s) { a[s].s = C->S[C->row_off[t] + s]; a[s].pos = (int32_t)s; }
    qsort(a, (size_t)n, sizeof(scored), by_score_desc_pos_asc);
    for (int i = 0; i < K; ++i) out[i] = (i < n) ? a[i].pos : -1;
    if (C->kth) {
        C->kth[2 * t + 0] = (K - 1 < n) ? a[K - 1].s : NAN;
        C->kth[2 * t + 1] = (K < n) ? a[K].s : NAN;
    }
    free(a);
}

/* idx[t][0:K): the selected logical positions in (S desc, s asc) order, -1 padded.
 * kth[t] (optional): {S_(K), S_(K+1)}, NaN where that rank does not exist. */
int oracle_indexer_topk(const odims* D, const void* q_I, const float* w, const void* k_I, const float* k_I_scale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_seq,
                        const int32_t* q_pos, int T, int32_t* idx, double* kth, int threads) {
    if (!check_dims(D) || T < 0 || !check_rows(D, seq_lens, q_seq, q_pos, T)) return O_BAD_ARG;
    if ((OMODE(D) == 2 || OMODE(D) == 3) && !k_I_scale) return O_BAD_ARG;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T + 1));
    if (!off) return O_NOMEM;
    off[0] = 0;
    for (int t = 0; t < T; ++t) off[t + 1] = off[t] + ((int64_t)q_pos[t] + 1 > 0 ? (int64_t)q_pos[t] + 1 : 0);
    double* S = (double*)malloc(sizeof(double) * (size_t)(off[T] > 0 ? off[T] : 1));
    if (!S) { free(off); return O_NOMEM; }
    int rc = scores_all(D, q_I, w, k_I, k_I_scale, block_table, seq_lens, q_seq, q_pos, T, S, off, threads);
    if (rc == O_OK) {
        topk_ctx C = {D, S, off, q_pos, idx, kth};
        rc = run_items(topk_row, &C, T, 0, threads);
    }
    free(S);
    free(off);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* step 4: gathered softmax attention                                        */
/* ------------------------------------------------------------------------- */

typedef struct {
    const odims* D; const void* q; const void* kv; const int32_t* block_table; const int32_t* seq_lens;
    const int32_t* q_seq; const int32_t* idx; int idx_stride; double sm_scale;
    double* out; double* lse; double* psum; int bad;
} attn_ctx;

static void attn_row(void* vctx, int64_t t, void* scratch) {
    attn_ctx* C = (attn_ctx*)vctx;
    const odims* D = C->D;
    int b = C->q_seq[t];
    int K = C->idx_stride;
    const int32_t* row_idx = C->idx + (int64_t)t * K;
    double* rows = (double*)scratch;                    /* [K][d] decoded selected rows */
    double* z = rows + (size_t)K * D->d;                /* [K] logits */
    double* qh = z + K;                                 /* [d] decoded query head */
    int n = 0;
    for (int i = 0; i < K; ++i) {
        int32_t s = row_idx[i];
        if (s == -1) continue;
        if (s < 0 || s >= C->seq_lens[b]) { C->bad = 1; return; }
        int64_t r = phys_row(D, C->block_table, b, s, NULL);
        if (r < 0) { C->bad = 1; return; }
        for (int e = 0; e < D->d; ++e) rows[(size_t)n * D->d + e] = kv_at(D, C->kv, r, e);
        ++n;
    }
    for (int h = 0; h < D->H; ++h) {
        double* o = C->out + ((size_t)t * D->H + h) * D->d_v;
        if (n == 0) {
            for (int c = 0; c < D->d_v; ++c) o[c] = 0.0;
            C->lse[(size_t)t * D->H + h] = -INFINITY;
            if (C->psum) C->psum[(size_t)t * D->H + h] = 0.0;
            continue;
        }
        for (int e = 0; e < D->d; ++e) qh[e] = act_at(D, C->q, ((size_t)t * D->H + h) * D->d + e);
        double m = -INFINITY;
        for (int i = 0; i < n; ++i) {
            double dot = 0.0;
            for (int e = 0; e < D->d; ++e) dot += qh[e] * rows[(size_t)i * D->d + e];
            z[i] = C->sm_scale * dot;
            if (z[i] > m) m = z[i];
        }
        double l = 0.0;
        for (int i = 0; i < n; ++i) { z[i] = exp(z[i] - m); l += z[i]; }
        for (int c = 0; c < D->d_v; ++c) o[c] = 0.0;
        double ps = 0.0;
        for (int i = 0; i < n; ++i) {
            double p = z[i] / l;
            ps += p;
            for (int c = 0; c < D->d_v; ++c) o[c] += p * rows[(size_t)i * D->d + c];
        }
        C->lse[(size_t)t * D->H + h] = m + log(l);
        if (C->psum) C->psum[(size_t)t * D->H + h] = ps;
    }
}

/* out[T][H][d_v], lse[T][H], psum[T][H] (optional) from idx[T][idx_stride]. */
int oracle_sparse_attn(const odims* D, const void* q, const void* kv, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* q_seq, const int32_t* idx, int idx_stride, int T,
                       double sm_scale, double* out, double* lse, double* psum, int threads) {
    if (!D || D->H <= 0 || D->d <= 0 || D->d_v <= 0 || D->d_v > D->d || idx_stride <= 0 || T < 0) return O_BAD_ARG;
    if (!mode_ok(D) || D->block_size <= 0) return O_BAD_ARG;
    for (int t = 0; t < T; ++t)
        if (q_seq[t] < 0 || q_seq[t] >= D->B) return O_BAD_ARG;
    attn_ctx C = {D, q, kv, block_table, seq_lens, q_seq, idx, idx_stride, sm_scale, out, lse, psum, 0};
    size_t scratch = sizeof(double) * ((size_t)idx_stride * D->d + idx_stride + D->d);
    int rc = run_items(attn_row, &C, T, scratch, threads);
    if (rc) return rc;
    return C.bad ? O_BAD_IDX : O_OK;
}

/* ------------------------------------------------------------------------- */
/* step 0: cache append                                                      */
/* ------------------------------------------------------------------------- */

/* position of new token t (the sequence's tail when q_pos is NULL: one row per sequence) */
static int append_pos(const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, int t, int* b_out) {
    const int b = q_seq ? q_seq[t] : t;
    *b_out = b;
    return q_pos ? q_pos[t] : seq_lens[b] - 1;
}

/* k_new[T][d_I] (fp32 in mode 0, bf16 otherwise), kv_new[T][d] (act type); the caches are updated
 * in place. Rows must name valid sequences, positions inside their block-table rows, and every
 * block's table entry must be valid (returns O_BAD_ARG otherwise, before writing anything). */
int oracle_cache_append(const odims* D, const void* k_new, const void* kv_new, const int32_t* block_table,
                        const int32_t* seq_lens, const int32_t* q_seq, const int32_t* q_pos, int T, void* k_cache,
                        float* k_scale, void* kv_cache) {
    if (!check_dims(D) || T < 0 || D->block_size > 1024) return O_BAD_ARG;
    const int bs = D->block_size;
    const size_t act = OMODE(D) == 0 ? 4 : 2;
    const size_t kb = OMODE(D) == 0 ? 4 : (OMODE(D) == 1 ? 2 : 1);
    if (OMODE(D) == 3 && D->d_I % 32) return O_BAD_ARG;
    for (int t = 0; t < T; ++t) {  /* validate first */
        int b;
        const int pos = append_pos(seq_lens, q_seq, q_pos, t, &b);
        if (b < 0 || b >= D->B || pos < 0 || pos >= seq_lens[b] || pos / bs >= D->max_blocks) return O_BAD_ARG;
        const int blk = block_table[(int64_t)b * D->max_blocks + pos / bs];
        if (blk < 0 || blk >= D->num_blocks) return O_BAD_ARG;
    }
    /* latent rows, and indexer keys in the fp32 / bf16 modes: copies */
    for (int t = 0; t < T; ++t) {
        int b;
        const int pos = append_pos(seq_lens, q_seq, q_pos, t, &b);
        const int64_t row = (int64_t)block_table[(int64_t)b * D->max_blocks + pos / bs] * bs + pos % bs;
        if (KV_FP8(D)) {  /* FP8 latent record: each 128-element tile quantised on its own */
            const size_t rb = kv_record_bytes(D->d);
            uint8_t* rec = (uint8_t*)kv_cache + (size_t)row * rb;
            const uint16_t* x = (const uint16_t*)kv_new + (int64_t)t * D->d;
            memset(rec, 0, rb);
            for (int j = 0; j < (D->d + 127) / 128; ++j) {
                const int e0 = 128 * j, e1 = e0 + 128 < D->d ? e0 + 128 : D->d;
                float amax = 0.0f;
                for (int e = e0; e < e1; ++e) {
                    const float v = fabsf((float)oracle_bf16_to_f64(x[e]));
                    if (v > amax) amax = v;
                }
                const float tile_scale = amax > 0.0f ? amax / 448.0f : 1.0f;
                for (int e = e0; e < e1; ++e) rec[e] = oracle_f32_to_e4m3((float)oracle_bf16_to_f64(x[e]) / tile_scale);
                memcpy(rec + D->d + 4 * j, &tile_scale, sizeof tile_scale);
            }
        } else {
            memcpy((char*)kv_cache + row * D->d * act, (const char*)kv_new + (int64_t)t * D->d * act, D->d * act);
        }
        if (OMODE(D) <= 1)
            memcpy((char*)k_cache + row * D->d_I * kb, (const char*)k_new + (int64_t)t * D->d_I * kb, D->d_I * kb);
        if (OMODE(D) == 3) {  /* MXFP8 keys: each group of 32 quantised on its own (no block state) */
            for (int g = 0; g < D->d_I / 32; ++g) {
                float v[32];
                for (int i = 0; i < 32; ++i)
                    v[i] = (float)oracle_bf16_to_f64(((const uint16_t*)k_new)[(int64_t)t * D->d_I + 32 * g + i]);
                const int X = mx_quantize32(v, (uint8_t*)k_cache + row * D->d_I + 32 * g);
                ((uint8_t*)k_scale)[row * (D->d_I / 32) + g] = (uint8_t)(X + 127);
            }
        }
    }
    if (OMODE(D) != 2) return O_OK;
    /* FP8 keys: every block that receives new tokens, once (at its first new token) */
    uint8_t* codes = (uint8_t*)k_cache;
    const uint16_t* knew = (const uint16_t*)k_new;
    for (int t = 0; t < T; ++t) {
        int b;
        const int pos = append_pos(seq_lens, q_seq, q_pos, t, &b);
        const int lb = pos / bs;
        int seen = 0;
        for (int u = 0; u < t && !seen; ++u) {
            int b2;
            const int p2 = append_pos(seq_lens, q_seq, q_pos, u, &b2);
            seen = (b2 == b && p2 / bs == lb);
        }
        if (seen) continue;
        /* the block's new tokens (slot -> row) and its first new position */
        int row_of_slot[1024];
        int first_new = pos;
        for (int i = 0; i < bs; ++i) row_of_slot[i] = -1;
        for (int u = 0; u < T; ++u) {
            int b2;
            const int p2 = append_pos(seq_lens, q_seq, q_pos, u, &b2);
            if (b2 == b && p2 / bs == lb) {
                row_of_slot[p2 % bs] = u;
                if (p2 < first_new) first_new = p2;
            }
        }
        const int blk = block_table[(int64_t)b * D->max_blocks + lb];
        const float old_scale = k_scale[blk];
        const int n_old = first_new - lb * bs; /* earlier tokens of the block: slots [0, n_old) */
        /* values of the block's tokens (fp32), then amax */
        float amax = 0.0f;
        for (int i = 0; i < bs; ++i) {
            const int u = row_of_slot[i];
            if (u < 0 && i >= n_old) continue;
            for (int d = 0; d < D->d_I; ++d) {
                float x;
                if (u >= 0) x = (float)oracle_bf16_to_f64(knew[(int64_t)u * D->d_I + d]);
                else x = (float)oracle_e4m3_to_f64(codes[((int64_t)blk * bs + i) * D->d_I + d]) * old_scale;
                const float ax = fabsf(x);
                if (ax > amax) amax = ax;
            }
        }
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int i = 0; i < bs; ++i) {
            const int u = row_of_slot[i];
            if (u < 0 && i >= n_old) continue;
            for (int d = 0; d < D->d_I; ++d) {
                uint8_t* c = &codes[((int64_t)blk * bs + i) * D->d_I + d];
                float x;
                if (u >= 0) x = (float)oracle_bf16_to_f64(knew[(int64_t)u * D->d_I + d]);
                else x = (float)oracle_e4m3_to_f64(*c) * old_scale;
                *c = oracle_f32_to_e4m3(x / scale);
            }
        }
        k_scale[blk] = scale;
    }
    return O_OK;
}

/* ------------------------------------------------------------------------- */
/* hierarchical selection: block summaries                                   */
/* ------------------------------------------------------------------------- */

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* summaries[b][lb][d] (bf16 bits) for every logical block lb < ceil(seq_lens[b] / bs): the mean
 * over the block's valid tokens (fp32 sum in token order, fp32 division, bf16 RNE). Blocks past a
 * sequence's end are left untouched. */
int oracle_block_summaries(const odims* D, const void* k_I, const float* k_I_scale, const int32_t* block_table,
                           const int32_t* seq_lens, uint16_t* summaries) {
    if (!check_dims(D)) return O_BAD_ARG;
    const int bs = D->block_size;
    for (int b = 0; b < D->B; ++b) {
        const int L = seq_lens[b];
        for (int lb = 0; lb * bs < L && lb < D->max_blocks; ++lb) {
            const int blk = block_table[(int64_t)b * D->max_blocks + lb];
            if (blk < 0 || blk >= D->num_blocks) return O_BAD_ARG;
            const int cnt = (L - lb * bs) < bs ? (L - lb * bs) : bs;
            for (int d = 0; d < D->d_I; ++d) {
                float acc = 0.0f;
                for (int i = 0; i < cnt; ++i) {
                    const size_t e = ((size_t)blk * bs + i) * D->d_I + d;
                    float x;
                    if (OMODE(D) == 0) x = ((const float*)k_I)[e];
                    else if (OMODE(D) == 1) x = (float)oracle_bf16_to_f64(((const uint16_t*)k_I)[e]);
                    else if (OMODE(D) == 2) x = (float)oracle_e4m3_to_f64(((const uint8_t*)k_I)[e]) * k_I_scale[blk];
                    else x = ldexpf((float)oracle_e4m3_to_f64(((const uint8_t*)k_I)[e]),
                                    (int)((const uint8_t*)k_I_scale)[((size_t)blk * bs + i) * (D->d_I / 32) + d / 32] - 127);
                    acc = acc + x;
                }
                summaries[((size_t)b * D->max_blocks + lb) * D->d_I + d] = f32_to_bf16_rne(acc / (float)cnt);
            }
        }
    }
    return O_OK;
}
