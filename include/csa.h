/*
 * csa.h -- C ABI of libcsa: the CSA / HCA attention layer of DeepSeek-V4 on
 * one NVIDIA B300 (sm_103a).
 *
 * The layer (sources are web pages about the DeepSeek-V4 report):
 *   1. compression: every m tokens' KV rows become one entry by a per-channel
 *      softmax over the block of (compression logit + per-slot bias)
 *      ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
 *      Key design 1 and Key design 2 equations; DeepSeek-V4 book ch.5 "How
 *      CSA Compresses Memory"];
 *   2. lightning indexer: score[t,j] = sum_h w[t,h] * ReLU(qI[t,h] . kI[j]),
 *      then top-k per query (CSA only) [same page, Key design 1 index-score
 *      equation; book ch.6 "How CSA Selects and Reads Memory"];
 *   3. shared-KV multi-query attention over the selected (CSA) or all
 *      visible (HCA) entries, plus the last n_win raw rows, plus a per-head
 *      sink logit in the denominator, with partial RoPE and output
 *      de-rotation [book ch.6 "Shared key-value MQA", ch.7 "HCA, Local
 *      Attention, and Position"].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer to a dense row-major array
 *    (innermost dimension contiguous, batch outermost), 16-byte aligned.
 *    The caller owns all memory, including workspaces; the library never
 *    allocates or frees device memory.
 *  - `stream` is a cudaStream_t passed as void*.  Every call only enqueues
 *    work on it and returns; no call synchronises the host, except
 *    csa_stream_status.  Calls from several host threads are safe.
 *  - Argument validation happens before anything is enqueued; on failure
 *    the call returns a non-zero csa_status, enqueues nothing, and
 *    csa_last_error() describes the problem.  A launch failure returns
 *    CSA_ERR_CUDA.
 *  - Conditions only the GPU can see (an index outside the cache, a window
 *    position missing from kv_raw, a bounded wait that ran out) never trap:
 *    the offending read is skipped and a bit is set in the status word at
 *    the start of the workspace; csa_stream_status() reports and clears it.
 *  - Storage dtype: CSA_F32 or CSA_BF16 for q, qI, C, Z, caches and outputs.
 *    bias, w, sink and scores are always float32; positions are int64;
 *    selected indices and counts are int32.
 *  - Positions: q_pos[b,t] is the absolute position of query t of sequence
 *    b.  Entry j of a cache compressed with rate m covers positions
 *    j*m .. j*m+m-1 and is visible to a query at t iff (j+1)*m <= t+1.  The
 *    window of a query at t is the raw rows at positions
 *    max(0, t-n_win+1) .. t; raw row l of sequence b holds position
 *    raw_pos0[b] + l.
 *  - RoPE rotates adjacent pairs (c-r+2i, c-r+2i+1) of the last r dims by
 *    p * theta^(-2i/r).  Stored caches carry their rotation: csa_compress
 *    rotates entry j at its block's last position (j+1)*m-1 and its raw-row
 *    output at each row's position; attention rotates q at t, and rotates
 *    the output's rotary dims back by -t when derotate = 1.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer   */
    CSA_ERR_UNSUPPORTED = 2, /* valid but outside the supported shapes       */
    CSA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required   */
    CSA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed         */
    CSA_ERR_TIMEOUT = 5,     /* (status word) a bounded device wait ran out  */
    CSA_ERR_DEVICE = 6       /* (status word) a device-side range check hit  */
} csa_status;

typedef enum { CSA_F32 = 0, CSA_BF16 = 1 } csa_dtype;

/* Layer hyper-parameters. */
typedef struct csa_params {
    int32_t m;          /* compression rate: 1, 2, 4, 8, ..., 128            */
    int32_t overlap;    /* 0: one branch (block i only); 1: two branches,   *
                         * entry i also pools branch b of block i-1         */
    int32_t top_k;      /* CSA selection budget k, 1 .. 2048                */
    int32_t n_win;      /* window length, 0 .. 1024                         */
    int32_t rope_dims;  /* r, even, 0 .. c                                  */
    int32_t derotate;   /* 1: rotate the output's rotary dims by -t         */
    double rope_theta;  /* RoPE base (> 1)                                  */
    float scale;        /* attention logit scale; 0 means 1/sqrt(c)         */
    int32_t batch_invariant; /* 1: a query's output and selection do not   *
                         * depend on the batch around it at any batch size  *
                         * (long lists are always split the same way); 0:   *
                         * large batches may skip the split, which changes  *
                         * the fp32 summation order                         */
    int64_t spin_limit; /* polls a kernel's wait on another of its warps    *
                         * may take before it gives up, records a timeout   *
                         * in the status word and unwinds; 0 = 2^24 (about  *
                         * a second)                                        */
    int32_t cache_format; /* CSA_CACHE_DTYPE or CSA_CACHE_LOWP (section 6)  */
    /* RMSNorm gains (device pointers to c floats, or NULL for no norm)
     * [book ch.7 "Query and KV normalization"]: y = x / sqrt(mean(x^2) +
     * norm_eps) * g over the c coordinates of a vector, applied to the vector
     * as produced, before RoPE.  q_norm: each query head (shared by the
     * heads), in every attention entry point.  kv_norm: each compressed KV
     * entry after pooling and each stored raw row, in csa_compress,
     * csa_prefill, hca_prefill and decode_append (caches passed to attention
     * are already stored normalised). */
    const float *q_norm;
    const float *kv_norm;
    float norm_eps;     /* 0 means 1e-6                                     */
} csa_params;

/* Storage of the compressed caches an entry point reads (section 6). */
typedef enum {
    CSA_CACHE_DTYPE = 0, /* entries and indexer keys in the call's dtype; fp32 scores */
    CSA_CACHE_LOWP = 1   /* FP8 KV records, MXFP4 indexer keys, BF16 scores      */
} csa_cache_format;

/* Supported sizes: c (main head dim) in {64, 128, 256, 512}; dI (indexer
 * dim) in {32, 64, 128}; H (query heads) 1 .. 128; hI (indexer heads)
 * 1 .. 64.  Anything else returns CSA_ERR_UNSUPPORTED. */

/* Workspace bytes for the entry points that take one. */
#define CSA_STATUS_BYTES 256

const char *csa_last_error(void);   /* thread-local message of the last failure */
const char *csa_version(void);
/* Number of kernels this library has launched in this process (all devices). */
int64_t csa_launch_count(void);

/*
 * Synchronise `stream`, read the status word at the start of `ws`, clear it
 * and return CSA_OK, CSA_ERR_DEVICE or CSA_ERR_TIMEOUT.
 */
csa_status csa_stream_status(void *ws, void *stream);

/* Zero the status word of a fresh workspace (enqueued on stream). */
csa_status csa_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Check of the bounded-wait path every tensor-core kernel uses between its
 * warps (the pages have no counterpart; this is a property of the library).
 * Enqueues one small kernel whose thread waits on a shared-memory barrier
 * that nothing completes, polling at most spin_limit times (0: the default
 * of csa_params), then records the timeout bit in the status word of `ws`
 * and returns.  csa_stream_status() then reports CSA_ERR_TIMEOUT and the
 * context stays usable.  Nothing is copied or multiplied while it waits.
 */
csa_status csa_wait_probe(int64_t spin_limit, void *ws, size_t ws_bytes, void *stream);

/*
 * Per-stage device timing, for profiling.  While enabled, every entry point
 * records a CUDA event before and after each kernel stage it enqueues (on
 * the call's stream).  csa_timing_read() waits for the recorded events, adds
 * their elapsed milliseconds and launch counts per stage into ms[s] and
 * launches[s] for s < nstages (either may be NULL), and forgets them.  Do
 * not enable it while a stream is being captured into a CUDA graph.
 */
typedef enum {
    CSA_STAGE_COMPRESS = 0,
    CSA_STAGE_INDEXER = 1,
    CSA_STAGE_TOPK = 2,
    CSA_STAGE_SPARSE_ATTN = 3,
    CSA_STAGE_HCA_ATTN = 4,
    CSA_NUM_STAGES = 5
} csa_stage;
csa_status csa_timing_enable(int32_t on);
csa_status csa_timing_read(double *ms, int64_t *launches, int32_t nstages);

/* --------------------------------------------------------------------- */
/* 1. Compression.                                                        */
/* --------------------------------------------------------------------- */
/*
 * ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
 * Key design 1 (two-branch CSA equation) and Key design 2 (HCA equation);
 * DeepSeek-V4 book ch.5 "One weight distribution per coordinate", "Which
 * positions enter a compressed block"; "DeepSeek-V4" explainer: "every m
 * consecutive tokens".]
 *
 * For each sequence b, block i < n/m and channel ch:
 *   a_s = Z[b, m*i+s, ch] + bias[s, ch]            (s < m)
 *   overlap = 1 also: b_s = Zb[b, m*(i-1)+s, ch] + biasb[s, ch]
 *                     (for i = 0: logit -inf, content 0)
 *   entry = sum softmax(a, b)_s * content_s   (content C, and Cb for b_s)
 * then RoPE at position (i+1)*m-1 on the last rope_dims dims, rounded to
 * dtype.  Trailing tokens that do not fill a block produce no entry.
 *
 *   C, Z       [B, n, c]  dtype      Cb, Zb [B, n, c] (overlap = 1 only)
 *   bias       [m, c]     float32    biasb  [m, c]    (overlap = 1 only)
 *   out        [B, n/m, c] dtype     compressed entries (stored, rotated)
 *   raw_out    [B, n, c]  dtype or NULL: the raw rows C rotated at their
 *              own positions, i.e. the stored rows a window reads
 * Uses params->m, overlap, rope_dims, rope_theta.
 */
csa_status csa_compress(csa_dtype dtype, int64_t B, int64_t n, int32_t c,
                        const void *C, const void *Z, const float *bias,
                        const void *Cb, const void *Zb, const float *biasb,
                        void *out, void *raw_out,
                        const csa_params *params, void *stream);

/* --------------------------------------------------------------------- */
/* 2. Indexer scores and top-k.                                           */
/* --------------------------------------------------------------------- */
/*
 * [Key design 1 index-score equation; book ch.6 "The index score".]
 *   scores[b,t,j] = sum_h w[b,t,h] * ReLU(qI[b,t,h,:] . kI[b,j,:])
 * for visible j ((j+1)*m <= q_pos[b,t]+1), -inf otherwise.  No RoPE, no scale.
 *   qI [B, T, hI, dI] dtype;  w [B, T, hI] float32;  kI [B, E, dI] dtype;
 *   q_pos [B, T] int64;  scores [B, T, E] float32.
 * ws: at least indexer_score_ws_size() bytes (status word).
 */
size_t indexer_score_ws_size(void);
csa_status indexer_score(csa_dtype dtype, int64_t B, int64_t T, int32_t hI, int32_t dI,
                         int64_t E, int32_t m,
                         const void *qI, const float *w, const void *kI,
                         const int64_t *q_pos, float *scores,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * [Key design 1, C_t = TopK_k(I[t,:]); book ch.6 "Top-k is a budget over
 * compressed entries".]  Per query: if at most k entries are visible, all
 * are kept; otherwise the k best by (score descending, index ascending),
 * -0.0 equal to +0.0.  idx [B, T, k] int32 holds the kept indices in
 * ascending order, padded with -1; cnt [B, T] int32 the number kept.
 * scores [B, T, E] float32 (entries beyond the visible prefix are ignored).
 */
size_t topk_select_ws_size(int64_t B, int64_t T, int64_t E, int32_t k);
csa_status topk_select(int64_t B, int64_t T, int64_t E, int32_t k, int32_t m,
                       const float *scores, const int64_t *q_pos,
                       int32_t *idx, int32_t *cnt,
                       void *ws, size_t ws_bytes, void *stream);

/*
 * topk_select without a workspace: the same selection and outputs as
 * topk_select, for callers that cannot allocate device memory (for example
 * code that runs where cudaMalloc is unavailable or forbidden and only gets
 * its input and output buffers from someone else).  The pages have no
 * counterpart; this is a property of the library, not of the method.
 *  - Scratch lives in a 17 MiB device array inside the library, held by every
 *    GPU that loads it until the process exits.  Rows of more than 16384
 *    entries (the multi-CTA path) need it; they are limited to at most 64
 *    rows and 2^21 row x entry products, and larger requests return
 *    CSA_ERR_UNSUPPORTED with nothing enqueued.
 *  - The first call on a device looks up that array's device address (with
 *    the device current); make that first call before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (two
 *    streams, or two threads) race and corrupt each other.  Serialise them.
 *  - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    call.
 *  - The looked-up address is kept for the life of the process: a device
 *    reset (cudaDeviceReset) after the first call on that device is not
 *    supported, because the array may then live at another address.
 */
csa_status topk_select_noalloc(int64_t B, int64_t T, int64_t E, int32_t k, int32_t m,
                               const float *scores, const int64_t *q_pos,
                               int32_t *idx, int32_t *cnt, void *stream);

/* --------------------------------------------------------------------- */
/* 3. Core attention.                                                     */
/* --------------------------------------------------------------------- */
/*
 * [book ch.6 "Shared key-value MQA"; ch.7 "The sliding window", "Partial
 * rotary position embeddings", "Why the output is de-rotated", "Attention
 * sinks".]  For query t of sequence b and head h, over the set S of
 * compressed entries (sparse_attn: idx[b,t,:] >= 0; hca_attn: every visible
 * entry) and the window rows W:
 *   q~ = RoPE(q[b,t,h], t);  l_u = scale * (q~ . u)  for u in S and W
 *   out[b,t,h] = sum e^l_u u / (e^sink[h] + sum e^l_u)
 *   derotate:  out[rotary dims] = RoPE(out, -t)[rotary dims]
 *   lse[b,t,h] = log(e^sink[h] + sum e^l_u)          (lse may be NULL)
 * Entries serve as both key and value (K = V).
 *   q [B, T, H, c];  kvc [B, E, c] stored entries;  idx [B, T, k] int32;
 *   kv_raw [B, L, c] stored raw rows;  raw_pos0 [B] int64;  sink [H] f32;
 *   out [B, T, H, c] dtype;  lse [B, T, H] float32 or NULL.
 * Uses params->m, n_win, rope_dims, rope_theta, scale, derotate.
 */
size_t attn_ws_size(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c,
                    int64_t E, int32_t k, const csa_params *params);
csa_status sparse_attn(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c,
                       int64_t E, int32_t k, int64_t L,
                       const void *q, const int64_t *q_pos, const void *kvc,
                       const int32_t *idx, const void *kv_raw, const int64_t *raw_pos0,
                       const float *sink, void *out, float *lse,
                       const csa_params *params, void *ws, size_t ws_bytes, void *stream);
csa_status hca_attn(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c,
                    int64_t E, int64_t L,
                    const void *q, const int64_t *q_pos, const void *kvc,
                    const void *kv_raw, const int64_t *raw_pos0,
                    const float *sink, void *out, float *lse,
                    const csa_params *params, void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------- */
/* 4. Fused layer entry points (one stream, graph-capturable).            */
/* --------------------------------------------------------------------- */
/*
 * CSA prefill of B sequences of n tokens, query t at position t:
 *   csa_compress(C, Z, bias[, Cb, Zb, biasb]) -> kvc (+ rotated raw rows)
 *   csa_compress(Ck, Zk, biask[, Ckb, Zkb, biaskb]) -> kIc   (no RoPE)
 *   indexer_score -> topk_select -> sparse_attn -> out
 *   C, Z [B,n,c]; Ck, Zk [B,n,dI]; bias [m,c]; biask [m,dI];
 *   q [B,n,H,c]; qI [B,n,hI,dI]; w [B,n,hI] f32; sink [H] f32;
 *   out [B,n,H,c]; idx_out [B,n,k] int32 or NULL (the selected indices).
 */
size_t csa_prefill_ws_size(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c,
                           int32_t hI, int32_t dI, const csa_params *params);
csa_status csa_prefill(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c,
                       int32_t hI, int32_t dI,
                       const void *C, const void *Z, const float *bias,
                       const void *Cb, const void *Zb, const float *biasb,
                       const void *Ck, const void *Zk, const float *biask,
                       const void *Ckb, const void *Zkb, const float *biaskb,
                       const void *q, const void *qI, const float *w, const float *sink,
                       void *out, int32_t *idx_out,
                       const csa_params *params, void *ws, size_t ws_bytes, void *stream);

/*
 * HCA prefill: csa_compress(C, Z, bias) with params->m (e.g. 128) ->
 * hca_attn over every visible entry + window + sink.
 */
size_t hca_prefill_ws_size(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c,
                           const csa_params *params);
csa_status hca_prefill(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c,
                       const void *C, const void *Z, const float *bias,
                       const void *q, const float *sink, void *out,
                       const csa_params *params, void *ws, size_t ws_bytes, void *stream);

/*
 * One decode step for B sequences, one query each at q_pos[b]:
 *   CSA layer: indexer_score(qI, w, kIc) -> topk_select -> sparse_attn(q,
 *   kvc, kv_raw, sink) -> out.
 *   HCA layer (skipped when q2 == NULL): hca_attn(q2, kvc2, kv_raw2, sink2)
 *   -> out2, with compression rate params2->m.
 *   q [B,1,H,c]; qI [B,1,hI,dI]; w [B,1,hI]; kvc [B,E,c]; kIc [B,E,dI];
 *   kv_raw [B,L,c]; raw_pos0 [B]; q2 [B,1,H,c]; kvc2 [B,E2,c];
 *   kv_raw2 [B,L,c]; out, out2 [B,1,H,c]; idx_out [B,1,k] or NULL.
 */
size_t hybrid_decode_ws_size(csa_dtype dtype, int64_t B, int32_t H, int32_t c, int32_t hI,
                             int32_t dI, int64_t E, int64_t E2,
                             const csa_params *params, const csa_params *params2);
csa_status hybrid_decode(csa_dtype dtype, int64_t B, int32_t H, int32_t c, int32_t hI,
                         int32_t dI, int64_t E, int64_t E2, int64_t L,
                         const void *q, const void *qI, const float *w,
                         const void *kvc, const void *kIc, const void *kv_raw,
                         const float *sink,
                         const void *q2, const void *kvc2, const void *kv_raw2,
                         const float *sink2,
                         const int64_t *q_pos, const int64_t *raw_pos0,
                         void *out, void *out2, int32_t *idx_out,
                         const csa_params *params, const csa_params *params2,
                         void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------- */
/* 5. Incremental decode state.                                           */
/* --------------------------------------------------------------------- */
/*
 * [DeepSeek-V4 book ch.5 "What is retained during decode"; ch.13 "Bounded
 * state per request": when a token arrives the window advances and the
 * compression state changes; when a block completes, its summary moves into
 * the growing cache.]
 *
 * decode_append takes one new token per sequence, at position t[b] (the
 * number of tokens the sequence held before it), for one compressed layer:
 *   - its raw row C, rotated at t, goes into the window ring `win` at row
 *     t mod n_win;
 *   - its compressor inputs (C, Z; the indexer keys' Ck, Zk when Ck is not
 *     NULL; the second-branch rows Cb, Zb, Ckb, Zkb when overlap = 1) go into
 *     the tail, which holds the current block's rows (and, for overlap = 1,
 *     the previous block's second-branch rows);
 *   - when t+1 is a multiple of m, block i = (t+1)/m - 1 is compressed
 *     exactly as csa_compress compresses it (same arithmetic, bitwise the
 *     same entry), rotated at (i+1)*m-1 and stored at kvc[b, i] (and the
 *     key, without rotation, at kIc[b, i]).
 * Sizes: C, Z, Cb, Zb [B, c]; Ck, Zk, Ckb, Zkb [B, dI]; bias, biasb [m, c];
 * biask, biaskb [m, dI]; win [B, n_win, c]; tail: decode_tail_bytes();
 * kvc [B, E_cap, c]; kIc [B, E_cap, dI]; all in dtype.  Uses params->m,
 * overlap, n_win, rope_dims, rope_theta.  The tail needs no initialisation:
 * every slot is written before it is read.  A block past E_cap sets the
 * range bit of the status word and is not stored.
 *
 * The ring is the window hybrid_decode reads: pass kv_raw = win, L = n_win
 * and raw_pos0[b] = max(0, t - n_win + 1) for the query at t.  While
 * t < n_win - 1, row l holds position l, as raw_pos0 = 0 says; once the
 * window is full every row of the ring is in it, in rotated rather than
 * positional order, which attention does not depend on (it sums over the
 * set, and stored rows carry their own rotation).  Pass E = E_cap: entries
 * past the visible prefix are never read.
 */
size_t decode_tail_bytes(csa_dtype dtype, int64_t B, int32_t c, int32_t dI,
                         const csa_params *params);
csa_status decode_append(csa_dtype dtype, int64_t B, int32_t c, int32_t dI, const int64_t *t,
                         const void *C, const void *Z, const float *bias,
                         const void *Cb, const void *Zb, const float *biasb,
                         const void *Ck, const void *Zk, const float *biask,
                         const void *Ckb, const void *Zkb, const float *biaskb,
                         void *win, void *tail, void *kvc, void *kIc, int64_t E_cap,
                         const csa_params *params, void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------- */
/* 6. Low-precision caches.                                               */
/* --------------------------------------------------------------------- */
/*
 * [DeepSeek-V4 book ch.8 "The main compressed-entry payload": an entry keeps
 * its non-rotary dims in FP8 and its 64 rotary dims in BF16, 576 bytes at
 * c = 512; ch.16 "The two main FP4 targets", "Why use fine-grained scales?":
 * indexer queries and keys in FP4 with one scale per 1 x 32 tile; "BF16
 * index scores".]
 *
 * FP8 KV record, one per entry of c = 512 with rope_dims = 64, KV_FP8_BYTES
 * bytes: bytes 0..447 the E4M3 codes of dims 0..447 (finite variant,
 * largest 448, nearest-even, saturating); bytes 448..575 dims 448..511 in
 * BF16; bytes 576..591 four fp32 scales for dims [0,128), [128,256),
 * [256,384), [384,448): scale = amax / 448 (1 for an all-zero group), code =
 * E4M3(x / scale) with the quotient formed in fp32.  A cache of E entries
 * per sequence is [B, E, KV_FP8_BYTES].
 *
 * MXFP4 rows of 128 values, planar over `rows` rows (rows = B * E for a key
 * cache), index_fp4_bytes(rows) bytes: first the codes, 64 bytes a row,
 * value 2i in the low nibble of byte i and 2i+1 in the high nibble (E2M1:
 * sign bit 3, magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; nearest-even,
 * saturating); then the scales, 4 bytes a row (one per block of 32 values,
 * the row count rounded up to a multiple of 4): the exponent e + 127 of the
 * block's scale 2^e, e = floor(log2 amax) - 2 clipped to [-127, 127] (0 for
 * an all-zero block).
 *
 * With params->cache_format = CSA_CACHE_LOWP:
 *   - sparse_attn, hca_attn and hybrid_decode read kvc (and kvc2) as FP8
 *     records (dtype bf16, c = 512, rope_dims = 64); the window rows stay in
 *     dtype.  A record's codes are dequantised to bf16 (code * scale rounded
 *     once) for the tensor-core products;
 *   - hybrid_decode reads kIc as MXFP4 keys (hI = 64, dI = 128), quantises
 *     the query qI to MXFP4 the same way, and ranks BF16 scores
 *     bf16(sum_h w * ReLU(q4 . k4)): equal BF16 scores tie and the lower
 *     index wins.
 * csa_prefill and hca_prefill take CSA_CACHE_DTYPE only.
 */
#define KV_FP8_BYTES 592
size_t index_fp4_bytes(int64_t rows);
/* src [rows, 512] in dtype -> dst [rows, KV_FP8_BYTES] */
csa_status quantize_kv_fp8(csa_dtype dtype, int64_t rows, int32_t c, int32_t rope_dims,
                           const void *src, void *dst, void *stream);
/* src [rows, 128] in dtype -> dst (index_fp4_bytes(rows) bytes) */
csa_status quantize_index_fp4(csa_dtype dtype, int64_t rows, int32_t d, const void *src, void *dst,
                              void *stream);
/*
 * Decode index scores over MXFP4 keys: one query per sequence, qI [B, 1, 64,
 * 128] bf16 (quantised to MXFP4 inside), w [B, 1, 64] f32, kI4 the MXFP4
 * cache of B * E keys, q_pos [B, 1]; scores [B, 1, E] f32 holding BF16
 * values for visible entries and -inf past them.  ws: the status word.
 */
csa_status indexer_score_fp4(int64_t B, int64_t E, int32_t m, const void *qI, const float *w,
                             const void *kI4, const int64_t *q_pos, float *scores, void *ws,
                             size_t ws_bytes, void *stream);

/* --------------------------------------------------------------------- */
/* 7. Grouped output projection.                                          */
/* --------------------------------------------------------------------- */
/*
 * [DeepSeek-V4 book ch.6 "Why output projection is a large cost": the heads
 * are split into groups, each group's concatenated outputs are projected to
 * a width d_g, and the concatenation of the group results is projected to
 * the hidden width d; "DeepSeek-V4 technical preview" blog: 16 groups for
 * Pro.]  For token t, G = H / heads_per_group groups:
 *   u[t, g*d_g + j] = sum_i o[t, g*hg*c + i] * w_g[g, j, i]     (hg = heads_per_group)
 *   y[t, n]         = sum_i u[t, i] * w_o[n, i]
 * o [T, H, c] bf16 (the attention output, de-rotated); w_g [G, d_g, hg*c]
 * and w_o [d, G*d_g] bf16 in the out-features-major layout of a linear
 * layer; y [T, d] bf16.  u is kept in bf16 in the workspace, after the
 * status word (out_proj_ws_size bytes in all).  Both products run on the
 * tensor cores with fp32 accumulation.  d_g and d must be multiples of 256,
 * hg*c a multiple of 64.
 */
size_t out_proj_ws_size(int64_t T, int32_t H, int32_t heads_per_group, int32_t d_g);
csa_status out_proj(int64_t T, int32_t H, int32_t c, int32_t heads_per_group, int32_t d_g,
                    int32_t d, const void *o, const void *w_g, const void *w_o, void *y,
                    void *ws, size_t ws_bytes, void *stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
