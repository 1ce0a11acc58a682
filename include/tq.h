/*
 * tq.h -- C ABI of the GB300 (sm_103a) TurboQuant-style online KV-cache
 * quantizer and decode-attention library (libtq.so).
 *
 * Method sources (web pages, cited by title and section):
 *   [P2] "생각정리 209 (TurboQuant)", uiyeonassociation.blogspot.com: the
 *        two-stage method (rotation + codebook, then QJL on the residual).
 *   [P4] "[LLM Serving] TurboQuant란 무엇이며, 어떻게 KV Cache 양자화로 메모리를
 *        5배 줄일 수 있을까?", riverfrot.github.io: §2.2 attention, §2.4 KV
 *        size, §3.1 paged blocks, §4.1 rotation, §4.2 Lloyd-Max, §4.3 QJL.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must be CUDA device pointers on the current
 *     device; "host" pointers are ordinary CPU memory.  The library never
 *     takes ownership of caller memory.
 *   - Quantize and decode are stream-ordered on `stream` (0 = legacy default
 *     stream), allocate nothing and never synchronise the host.
 *   - Argument errors are reported synchronously (TQ_ERR_INVALID_ARG) and
 *     launch nothing.  Launch failures return TQ_ERR_CUDA.
 *   - Corrupt device-side inputs (a page id outside [0, num_pages), a position
 *     beyond the block table, a sequence length beyond max_seq_len) are never
 *     dereferenced: the affected token is skipped and a bit is set in the
 *     context's device error word, read back by tq_check_device_status().
 *   - Every entry point returns a tq_status; tq_status_string() names it.
 *
 * Data layout (little-endian):
 *   K/V inputs    [batch][n_new][num_kv_heads][d], bf16 or fp32, dense.
 *   queries       [batch][num_q_heads][d], bf16 or fp32, dense.
 *   output        [batch][num_q_heads][d], fp32.
 *   block table   int32 [batch][max_pages_per_seq]: physical page of each
 *                 16-token block of a sequence ([P4] §3.1).
 *   caches        bytes; page p, KV head h starts at
 *                 p * page_bytes + h * (page_bytes / num_kv_heads).
 *   One (page, head) block of the K cache holds, for its 16 token slots:
 *     codes[16][code_bytes_k] | signs[16][m/8] | norm fp16[16] | rnorm fp16[16]
 *   and of the V cache:  codes[16][code_bytes_v] | norm fp16[16].
 *   Codes of one vector form one bit stream (byte k = stream bits 8k..8k+7,
 *   LSB first): channels [0, split) of the rotated vector first (bits_hi
 *   each), then [split, d) (bits_lo).  Within a group, channel c's stored value
 *   sits at group bits [b*c, b*c+b) for b = 1, 2, 4; for b = 3 channels come in
 *   octets of 8 (24 bits at group bit 24*o): octet channel i < 6 at bits
 *   4i..4i+2, channel 6 at bits 3/11/19, channel 7 at bits 7/15/23.  Codes are
 *   0-based, ascending with the centroid; the stored value is the code, except
 *   b = 4 which stores sign-magnitude (code >= 8 -> code-8, else 15-code).
 *   QJL sign i is bit i%8 of byte i/8 (1 = projection >= 0).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,   /* bad pointer, size or configuration */
  TQ_ERR_CUDA = 2,          /* a CUDA runtime call or launch failed */
  TQ_ERR_OOM = 3,           /* tq_create could not allocate its tables */
  TQ_ERR_UNSUPPORTED = 4,   /* valid but not implemented (e.g. d = 48) */
  TQ_ERR_DEVICE_CHECK = 5,  /* a kernel skipped out-of-range device input */
  TQ_ERR_WORKSPACE = 6      /* workspace too small for the requested call */
} tq_status;

typedef enum { TQ_BF16 = 0, TQ_F32 = 1 } tq_dtype;

/* Density the Lloyd-Max codebooks are fitted to, in unit-variance units
 * u = sqrt(d) y / ||x||: N(0,1) (the high-d limit), or the exact density of a
 * coordinate of a uniformly rotated vector, f(u) ~ (1 - u^2/d)^((d-3)/2) on
 * |u| < sqrt(d) ([P4] §4.2: a Beta distribution, close to Gaussian at high d). */
#define TQ_CODEBOOK_GAUSSIAN 0
#define TQ_CODEBOOK_SPHERE 1

/* Method configuration.  d is a multiple of 32 in [32, 256]; page_size = 16.
 * d = 128 runs on the tensor-core kernels (tcgen05 quantize, mma.sync LUT
 * decode); every other d on generic CUDA-core kernels that compute the same
 * records and the same attention (tq_causal_attention and tq_search: d = 128
 * only).  Bits per channel in [1, 4]; channels [0, split) of the rotated
 * vector use bits_hi, channels [split, d) bits_lo; split is a multiple of 32.
 * m (QJL projections) is a multiple of 32 in [32, 128].  k_qjl = 0 gives
 * MSE-only keys (no signs, no residual norm stored).  codebook: one of the
 * TQ_CODEBOOK_* densities (tq_config_init: TQ_CODEBOOK_GAUSSIAN). */
typedef struct {
  int d, m, page_size;
  int k_bits_hi, k_bits_lo, k_split;
  int v_bits_hi, v_bits_lo, v_split;
  int k_qjl;
  uint64_t seed;
  int codebook;
} tq_config;

typedef struct tq_ctx tq_ctx;   /* opaque; immutable after creation */

/* Fill `cfg` with head dimension d, page_size = 16, b bits on every channel
 * for keys and values (split = d/2 rounded down to a multiple of 32), QJL on
 * keys with m projections, the Gaussian codebook and `seed`. */
tq_status tq_config_init(tq_config* cfg, int d, int b, int m, uint64_t seed);

/* Build the context on the current device ([P4] §4.1-§4.3): the random
 * rotation Pi (Householder QR of a d x d Gaussian, positive R diagonal) and
 * the QJL matrix S (m x d Gaussian), drawn from the SplitMix64/Box-Muller
 * streams 1 and 2 of `seed`, and the Lloyd-Max codebooks for cfg->codebook's
 * density (tq_create: Gaussian).  The only call
 * that allocates device memory (about 0.5 MB) and the only one that copies
 * host to device; no later call creates anything (streams, events, memory).
 * `*out` receives the context; free it with tq_destroy. */
tq_status tq_create(int d, int b, int m, uint64_t seed, tq_ctx** out);
tq_status tq_create_ex(const tq_config* cfg, tq_ctx** out);
tq_status tq_destroy(tq_ctx* ctx);
tq_status tq_get_config(const tq_ctx* ctx, tq_config* cfg);

/* Bytes of one cache page (16 tokens x num_kv_heads) for K and for V.  A
 * cache of P pages is P * page_bytes; per-head blocks are page_bytes/H. */
tq_status tq_cache_layout(const tq_ctx* ctx, int num_kv_heads,
                          size_t* k_page_bytes, size_t* v_page_bytes);

/* Host-only copies of the tables tq_create builds (no GPU needed).
 * pi: d*d doubles, row-major (y = Pi x).  s: m*d doubles, row-major.
 * centroids: 2^bits doubles ascending; boundaries: 2^bits - 1 doubles. */
tq_status tq_host_rotation(int d, uint64_t seed, double* pi);
tq_status tq_host_qjl(int m, int d, uint64_t seed, double* s);
tq_status tq_host_codebook(int bits, double* centroids, double* boundaries);
/* The codebook for `density` (TQ_CODEBOOK_*) at dimension d (d >= 4; d is
 * ignored for the Gaussian density). */
tq_status tq_host_codebook_ex(int bits, int d, int density, double* centroids, double* boundaries);

/* Online quantize-and-append ([P2] stages 1-2; [P4] §4.1-§4.3, §3.1).
 * k, v (device): [batch][n_new][num_kv_heads][d] in `dtype`; either may be
 * NULL to skip that cache.  Token t of sequence b is written at position
 * start_pos[b] + t, i.e. page block_table[b*max_pages_per_seq + pos/16],
 * slot pos%16.  start_pos, block_table: device int32.  num_pages bounds the
 * page ids.  Per vector: y = Pi x; code_j = #{k : sqrt(d) y_j/||x|| >= t_k};
 * norm = fp16(||x||); keys also get r = y - norm/sqrt(d) * c[code],
 * sign bits of S r and fp16(||r||).  Codes and signs are decided exactly:
 * a value the fp32 fast path finds close to a boundary is recomputed in
 * fp64 before it is stored. */
tq_status tq_quantize(const tq_ctx* ctx, const void* k, const void* v, tq_dtype dtype,
                      int batch, int n_new, int num_kv_heads,
                      const int32_t* start_pos, const int32_t* block_table,
                      int max_pages_per_seq, int num_pages,
                      void* k_cache, void* v_cache, void* stream);

/* Workspace bytes tq_decode_attention needs for these sizes: the query
 * projections and the split-K partials (max, sum, acc[d]) per chunk. */
tq_status tq_workspace_size(const tq_ctx* ctx, int batch, int num_q_heads,
                            int max_seq_len, int chunk_tokens, size_t* bytes);

/* Split-K chunk for a decode over sequences totalling total_tokens (host
 * value, e.g. the scheduler's sum of the lengths; <= batch * max_seq_len)
 * with lengths <= max_seq_len: the chunk (multiple of 16, >= 256 unless the
 * sequences are shorter) that balances the work of the partials kernel over
 * the GPU.  Passing 0 as chunk_tokens to the decode calls assumes every
 * sequence has max_seq_len tokens; with very unequal lengths this call gives
 * a better split.  fused_append is accepted for compatibility and changes
 * nothing (tq_append_decode's partials kernel has the whole GPU).  No
 * counterpart in the pages (an implementation detail of the split-K decode).
 * Host only, no CUDA work. */
tq_status tq_decode_chunk(const tq_ctx* ctx, int batch, int num_q_heads, int num_kv_heads,
                          long long total_tokens, int max_seq_len, int fused_append, int* chunk_tokens);

/* Decode attention over the compressed cache ([P4] §2.2, §4.3; [P2] stage 2).
 * q (device): [batch][num_q_heads][d]; query head h reads KV head
 * h / (num_q_heads / num_kv_heads).  seq_lens (device int32 [batch]) <=
 * max_seq_len.  Score of cached key t: (norm_t/sqrt(d)) <Pi q, c[code_t]>
 * + sqrt(pi/2)/m * rnorm_t * <S Pi q, +-1 signs_t>; weights are
 * softmax(score * softmax_scale) (pass 1/sqrt(d) for the usual scale);
 * out = Pi^T sum_t w_t (vnorm_t/sqrt(d)) c_v[code_t], fp32.  The context is
 * split into chunks of chunk_tokens (a multiple of 16; 0 picks one) merged
 * with a log-sum-exp reduction.  A sequence of length 0 yields zeros.
 * Accuracy: max_j |out_j - exact_j| / max_j |exact_j| <= 2e-3 against the
 * same scores in fp64.  With d = 128 and |softmax_scale| <= 1/sqrt(d) the
 * tensor-core kernels run (fp16 q~, u and centroids, fp32 accumulation: their
 * logit error grows with the scale); a larger |softmax_scale| runs the fp32
 * CUDA-core kernels (slower), which keep the bound at any scale.
 * workspace (device) of at least tq_workspace_size() bytes. */
tq_status tq_decode_attention(const tq_ctx* ctx, const void* q, tq_dtype dtype,
                              int batch, int num_q_heads, int num_kv_heads,
                              const int32_t* seq_lens, int max_seq_len,
                              const int32_t* block_table, int max_pages_per_seq, int num_pages,
                              const void* k_cache, const void* v_cache,
                              int chunk_tokens, float softmax_scale,
                              float* out, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Same as tq_decode_attention, restricted to a subset of its three
 * stream-ordered stages (bit mask): TQ_STAGE_QPREP (q~ = Pi q, S q~ into the
 * workspace), TQ_STAGE_PARTIALS (per-chunk scores, online softmax and value
 * sums into the workspace), TQ_STAGE_MERGE (log-sum-exp merge, inverse
 * rotation, out).  Running the stages in order in separate calls with the
 * same arguments equals one tq_decode_attention call; a later stage reads
 * what the earlier one left in the workspace. */
#define TQ_STAGE_QPREP 1
#define TQ_STAGE_PARTIALS 2
#define TQ_STAGE_MERGE 4
#define TQ_STAGE_ALL 7
tq_status tq_decode_attention_ex(const tq_ctx* ctx, const void* q, tq_dtype dtype,
                                 int batch, int num_q_heads, int num_kv_heads,
                                 const int32_t* seq_lens, int max_seq_len,
                                 const int32_t* block_table, int max_pages_per_seq, int num_pages,
                                 const void* k_cache, const void* v_cache,
                                 int chunk_tokens, float softmax_scale,
                                 float* out, void* workspace, size_t workspace_bytes,
                                 int stages, void* stream);

/* Decode attention for callers that cannot allocate device memory.  The
 * paper has no counterpart: this entry point exists for callers that have no
 * way to call cudaMalloc when they run decode (code running inside a custom
 * allocator or memory pool, runtimes whose arena already owns the whole
 * device, embeddings that only pass pointers they already own).  Same
 * arguments and result as tq_decode_attention, without the workspace: the
 * query projections and split-K partials go to a fixed array of
 * TQ_NOALLOC_SCRATCH_BYTES that the library image holds on every device that
 * loads it, until the process exits.  Nothing is allocated, by this call or
 * by the library.  Returns TQ_ERR_WORKSPACE, launching nothing, when the
 * sizes need more than TQ_NOALLOC_SCRATCH_BYTES (tq_workspace_size gives the
 * need).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device); make that first call before any
 * stream capture.  Every call on a device shares the array and it keeps the
 * last call's contents (decode writes every byte it reads, so nothing needs
 * clearing); calls whose work overlaps on the GPU race on it. */
#define TQ_NOALLOC_SCRATCH_BYTES (16u << 20)
tq_status tq_decode_attention_noalloc(const tq_ctx* ctx, const void* q, tq_dtype dtype,
                                      int batch, int num_q_heads, int num_kv_heads,
                                      const int32_t* seq_lens, int max_seq_len,
                                      const int32_t* block_table, int max_pages_per_seq, int num_pages,
                                      const void* k_cache, const void* v_cache,
                                      int chunk_tokens, float softmax_scale,
                                      float* out, void* stream);

/* One decode step in one call ([P4] §2.3: the new token's K/V join the cache,
 * then its query attends over every cached token): quantize-and-append
 * k_new/v_new ([batch][1][H][d]) at position seq_lens[b] (lengths before the
 * append, device int32), then decode attention over seq_lens[b] + 1 tokens.
 * max_seq_len bounds the lengths after the append.  Same layouts, workspace
 * and errors as tq_quantize + tq_decode_attention; stream-ordered, no host
 * synchronisation. */
tq_status tq_append_decode(const tq_ctx* ctx, const void* k_new, const void* v_new, const void* q,
                           tq_dtype dtype, int batch, int num_q_heads, int num_kv_heads,
                           const int32_t* seq_lens, int max_seq_len,
                           const int32_t* block_table, int max_pages_per_seq, int num_pages,
                           void* k_cache, void* v_cache, int chunk_tokens, float softmax_scale,
                           float* out, void* workspace, size_t workspace_bytes, void* stream);

/* tq_append_decode with two optional CUDA events (cudaEvent_t, may be NULL)
 * recorded on `stream` just before and just after the split-K partials kernel,
 * for timing it inside the fused step (an event between two launches keeps the
 * second from starting early, so a step with events takes a little longer).
 * Execution, all on `stream`: the append (a warp per new K/V vector; d = 128
 * with the channel split a multiple of 8, else the tile quantize kernels),
 * the query prep launched dependent on it (it overlaps the append and ends
 * after it), the partials kernel over all seq_lens[b] + 1 positions and the
 * merge, each launched dependent on the one before.  Results equal
 * tq_quantize + tq_decode_attention over L+1 tokens bit for bit. */
tq_status tq_append_decode_ex(const tq_ctx* ctx, const void* k_new, const void* v_new, const void* q,
                              tq_dtype dtype, int batch, int num_q_heads, int num_kv_heads,
                              const int32_t* seq_lens, int max_seq_len,
                              const int32_t* block_table, int max_pages_per_seq, int num_pages,
                              void* k_cache, void* v_cache, int chunk_tokens, float softmax_scale,
                              float* out, void* workspace, size_t workspace_bytes, void* stream,
                              void* partials_begin_event, void* partials_end_event);

/* Multi-query causal attention over the compressed cache ([P4] §2.3: a new
 * token's query attends over every cached token; with T new tokens of one
 * sequence, the t-th attends over its prefix).  q (device): [batch][n_new][Hq][d]
 * in `dtype`, the queries of the tokens at positions start_pos[b] + t
 * (start_pos: device int32 [batch]); the caches must already hold positions
 * 0 .. start_pos[b] + n_new - 1 (append the new tokens' K/V with tq_quantize
 * first).  Query t of sequence b attends over positions 0 .. start_pos[b] + t
 * with the scores, softmax and value sums of tq_decode_attention; out (device,
 * fp32): [batch][n_new][Hq][d].  start_pos[b] + n_new <= max_seq_len.  The
 * context is split into chunks of chunk_tokens (0 picks one, 256 to 1024 tokens)
 * merged per query.  Runs the bit-width combinations of the persistent decode
 * kernel (d = 128, m = 128, split 64; K/V bits 3/3, 4-3/4-3, 3-2/3-2, 4/4, 2/2,
 * 4/2) with |softmax_scale| <= 1/sqrt(d) (the 2e-3 bar of tq_decode_attention;
 * its query is fp16 hi + lo), else TQ_ERR_UNSUPPORTED; query heads per KV head
 * <= 8.  Chunks of at most 1024 tokens run on the tensor cores (blocks of 128
 * query rows t * G + g of one sequence and KV head against 64-token tiles);
 * longer chunks on the lookup-table kernel (blocks of 8 rows).  q needs no
 * particular alignment (16-byte aligned rows load faster).  workspace (device)
 * of tq_causal_workspace_size bytes for the same chunk_tokens; stream-ordered,
 * no allocation.  Errors as tq_decode_attention. */
tq_status tq_causal_workspace_size(const tq_ctx* ctx, int batch, int n_new, int num_q_heads, int max_seq_len,
                                   int chunk_tokens, size_t* bytes);
tq_status tq_causal_attention(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch, int n_new,
                              int num_q_heads, int num_kv_heads, const int32_t* start_pos, int max_seq_len,
                              const int32_t* block_table, int max_pages_per_seq, int num_pages,
                              const void* k_cache, const void* v_cache, int chunk_tokens, float softmax_scale,
                              float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise the device and report (then clear) the context's device error
 * word: TQ_OK, or TQ_ERR_DEVICE_CHECK with the bits in *flags (may be NULL):
 * 1 = page id out of range, 2 = position beyond the block table,
 * 4 = sequence length beyond max_seq_len or the block table, 8 = a bounded
 * wait inside a kernel gave up (that launch's results are incomplete),
 * 16 = a kernel's shared-memory layout did not fit (it did no work). */
tq_status tq_check_device_status(const tq_ctx* ctx, uint32_t* flags);

/* Counters of the decisions the quantize kernels took again exactly (fp64 or
 * double-float) because their fast arithmetic found them inside its guard,
 * since creation (or the last reset): out[0] codes near a boundary, out[1]
 * sign bits near zero (the CUDA-core fp32-input kernel counts key vectors
 * with any such sign).  Synchronises the device. */
tq_status tq_refine_counters(const tq_ctx* ctx, unsigned long long out[2], int reset);

const char* tq_status_string(tq_status status);

/* Name and message of the last CUDA error behind a TQ_ERR_CUDA returned to the
 * calling host thread ("none" before any); the string stays valid until that
 * thread's next failing call.  No counterpart in the pages (a diagnostic). */
const char* tq_last_cuda_error(void);

/* Inner-product search over a quantized key database ([P2] "생각정리 209
 * (TurboQuant)": the vector-search use; [P4] §4.3: the two-stage estimate is
 * unbiased).  For every query i and database vector t the score is the
 * decode's estimate of <q_i, x_t> without any softmax or scale,
 *   (n16_t/sqrt(d)) <Pi q_i, c[code_t]> + sqrt(pi/2)/m rho16_t <S Pi q_i, +-1_t>,
 * then the k_top largest per query, best first (equal scores: lower t first).
 * The database is a K cache of ONE KV head written by tq_quantize (batch 1,
 * num_kv_heads 1, start_pos 0, n_new = n_db): vector t is in page
 * block_table[t / 16], slot t % 16 (device int32 [ceil(n_db/16)]); num_pages
 * bounds the page ids (an id outside [0, num_pages) is skipped, its score is
 * -inf and the device error word is set).  q: device [nq][d] in `dtype`.
 * top_scores (fp32) and top_index (int32): device [nq][k_top].
 *
 * Two paths, chosen from the configuration and k_top:
 *  - tensor cores (d = m = 128, channel split 64, key groups of 2-4 bits,
 *    k_top <= 16): 64 queries at a time, a tile of 128 vectors' codes turned
 *    into fp16 centroids and sign operands in shared memory and multiplied on
 *    tcgen05 (the decode's fp16 operands: scores within about 1e-3 of the
 *    query's largest |score|), the best 16 per query kept per CTA thread and
 *    merged; no score array is written;
 *  - CUDA cores (every other case, k_top <= 1024): fp32 scores into the
 *    workspace, then a radix-select top k.
 * Workspace (device, 16-byte aligned): tq_search_workspace_size(ctx, nq,
 * n_db, k_top) bytes (k_top = 0: the size tq_search_scores needs).  Stream-
 * ordered; no allocation.  Errors: null pointers, k_top out of range,
 * n_db > 16 num_pages, misaligned buffers -> TQ_ERR_INVALID_ARG; a small
 * workspace -> TQ_ERR_WORKSPACE; d != 128 or nq > 524280 ->
 * TQ_ERR_UNSUPPORTED.  All checked before any launch. */
tq_status tq_search_workspace_size(const tq_ctx* ctx, int nq, int n_db, int k_top, size_t* bytes);
tq_status tq_search(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, const void* k_cache,
                    const int32_t* block_table, int num_pages, int n_db, int k_top,
                    float* top_scores, int32_t* top_index, void* workspace, size_t workspace_bytes,
                    void* stream);
/* Every score of the same search, scores: device fp32 [nq][n_db], by the
 * arithmetic of the path tq_search takes with this k_top (so tq_search's
 * result is the stable ranking of these scores).  Workspace: the size
 * tq_search_workspace_size gives for k_top = 0.  Same errors as tq_search. */
tq_status tq_search_scores(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, const void* k_cache,
                           const int32_t* block_table, int num_pages, int n_db, int k_top, float* scores,
                           void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
