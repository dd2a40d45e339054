/*
 * kvdecode: one generation step of attention over a KV cache on one GB300.
 *
 * C ABI. Every pointer is plain memory owned by the caller (device memory
 * unless stated otherwise); the library allocates nothing and keeps no state
 * between calls, so it is reentrant. All GPU work is queued asynchronously on
 * the caller's stream; no call synchronises with the host.
 *
 * Problem statement (page titles and sections of the sources):
 *   - During generation each sequence produces one new token: its key and
 *     value projections are appended to the KV cache, and its query attends
 *     over every cached token (All About Transformer Inference, "Transformer
 *     inference basics", the Generation bullet; "Implementation: JetStream",
 *     the generate method).
 *   - Cache layout K[B, S, K, H], V likewise: batch, sequence position, KV
 *     head, head dimension (All About Transformer Inference, "Sharding the KV
 *     cache"). Here: bf16 [batch, s_max, n_heads_kv, head_dim], contiguous.
 *   - Query heads are grouped onto KV heads by the reshape [N] -> [K, M],
 *     M = N / K: query head n reads KV head n / M (same section, attention
 *     algorithm; multiquery attention is K = 1: Efficiently Scaling
 *     Transformer Inference, section 3.3).
 *   - Reads are ragged: only the first seq_lens[b] cached tokens of sequence b
 *     are read (All About Transformer Inference, "Tricks for improving
 *     generation throughput and latency", ragged HBM reads).
 *
 * Status handling: host-checkable faults are reported synchronously by the
 * return value, before anything is launched. Values that live on the device
 * (seq_lens, pos) cannot be checked on the host: out-of-range values are
 * clamped or skipped by the kernels, which then set a bit in the optional
 * device status word (never a trap).
 */
#ifndef KVDECODE_H
#define KVDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvd_status {
    KVD_OK = 0,
    KVD_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size or value */
    KVD_ERR_UNSUPPORTED = 2,          /* valid but not implemented (head_dim, group size) */
    KVD_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below kvd_decode_plan's figure */
    KVD_ERR_CUDA = 4                  /* a CUDA runtime call or launch failed */
} kvd_status;

typedef enum kvd_out_dtype {
    KVD_OUT_BF16 = 0,  /* bf16 output, round-to-nearest-even from fp32 */
    KVD_OUT_F32 = 1    /* fp32 output, with softmax weights carried to ~2^-17 */
} kvd_out_dtype;

/* cudaStream_t, passed as an opaque pointer (0 = the legacy default stream). */
typedef void* kvd_stream_t;

/* Bits of the optional device status word (int32, caller-owned, OR-ed in). */
#define KVD_STATUS_SEQ_LEN_CLAMPED 0x1  /* some seq_lens[b] outside [0, min(s_max, max_seq_len)] */
#define KVD_STATUS_POS_OUT_OF_RANGE 0x2 /* some pos[b] outside [0, s_max): that row not written */
#define KVD_STATUS_TIMEOUT 0x4          /* an internal pipeline wait gave up (~2 s): outputs invalid */
#define KVD_STATUS_BAD_PAGE 0x8         /* paged cache: a needed block-table entry named no page of the pool */
#define KVD_STATUS_UMAX_FALLBACK 0x10   /* unified-maximum calls: some row's scores left the window around phi */

/* Supported shapes: head_dim in {64, 128, 256}; n_heads_q a multiple of
 * n_heads_kv with group size n_heads_q / n_heads_kv <= 64. */
#define KVD_MAX_GROUP 64
/* Query tokens per sequence of the multi-token calls: 1 .. KVD_MAX_TOKENS. */
#define KVD_MAX_TOKENS 64

/*
 * kvd_decode_plan: split count and workspace size for kvd_decode_attention.
 *
 * The context of all (sequence, KV head) pairs is laid end to end and cut into
 * n_split contiguous, equal runs of tokens, one per CTA; each run's partial
 * softmax results are merged afterwards (All About Transformer Inference,
 * "Sharding the KV cache", sequence sharding accumulated like Flash Attention;
 * the split count adapts to shape and hardware as in the heuristic dataflow of
 * FlashDecoding++). n_split_request = 0 picks the heuristic (one CTA per
 * resident slot on num_sms SMs, capped by the work); > 0 forces that count.
 * num_sms = 0 queries the current CUDA device (needs a GPU); > 0 uses it as
 * given (host-only planning). max_seq_len is the largest seq_lens value the
 * call may see (<= s_max).
 * Outputs: *n_split_out (>= 1) and *workspace_bytes_out (0 when n_split is 1).
 * Errors: KVD_ERR_INVALID_ARG for null outputs, non-positive sizes, a group
 * that does not divide, max_seq_len < 0 or out_dtype unknown;
 * KVD_ERR_UNSUPPORTED for head_dim / group size outside the list above;
 * KVD_ERR_CUDA if num_sms = 0 and the device query fails.
 */
kvd_status kvd_decode_plan(int batch, int n_heads_q, int n_heads_kv, int head_dim,
                           int max_seq_len, int num_sms, int n_split_request,
                           kvd_out_dtype out_dtype,
                           int* n_split_out, size_t* workspace_bytes_out);

/*
 * kvd_kv_append: write the new token's key and value rows into the cache.
 *   k_cache[b, pos[b], h, :] = k_new[b, h, :]; v_cache likewise.
 * (All About Transformer Inference, "Transformer inference basics": the new
 * token's KV is appended to the KV cache.) A bit copy: no arithmetic.
 *   k_cache, v_cache : bf16 [batch, s_max, n_heads_kv, head_dim], 16-byte aligned
 *   k_new, v_new     : bf16 [batch, n_heads_kv, head_dim], 16-byte aligned
 *   pos              : device int32 [batch], the pre-append length of each
 *                      sequence; not modified. Rows with pos[b] outside
 *                      [0, s_max) are skipped and flag KVD_STATUS_POS_OUT_OF_RANGE.
 *   status_word      : optional device int32 (may be NULL).
 * batch = 0 is a no-op. Errors: KVD_ERR_INVALID_ARG for null or misaligned
 * pointers, negative sizes, head_dim not a multiple of 8; KVD_ERR_CUDA if the
 * launch fails.
 */
kvd_status kvd_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* pos, int batch, int s_max, int n_heads_kv,
                         int head_dim, int32_t* status_word, kvd_stream_t stream);

/*
 * kvd_decode_attention: attention of one new token per sequence over its cache.
 *   out[b, h, :] = sum_{t < L_b} softmax_t(scale * q[b, h, :] . K[b, t, g, :]) V[b, t, g, :]
 *   with g = h / (n_heads_q / n_heads_kv) and L_b = seq_lens[b] (clamped),
 * computed as the pages describe the fused attention: read q, read the K and
 * V cache once, q.K, softmax over the sequence, weights times V, write the
 * output, never writing the score matrix (All About Transformer Inference,
 * "What about attention?"; the softmax is evaluated in base 2 with log2(e)
 * folded into the scale, Efficiently Scaling Transformer Inference, section
 * 3.5). The context is split into n_split runs whose partial softmax results
 * (run maximum, sum of exponentials, unnormalised weighted sum of V) are
 * merged by log-sum-exp.
 *   q               : bf16 [batch, n_heads_q, head_dim], 16-byte aligned
 *   k_cache/v_cache : bf16 [batch, s_max, n_heads_kv, head_dim], 16-byte aligned;
 *                     only rows t < L_b are read
 *   seq_lens        : device int32 [batch]; clamped to [0, min(s_max, max_seq_len)]
 *                     (KVD_STATUS_SEQ_LEN_CLAMPED). L_b = 0 gives a zero row and
 *                     lse = -inf.
 *   scale           : finite softmax scale (typically 1/sqrt(head_dim))
 *   n_split         : 0 = heuristic, else the count to use (see kvd_decode_plan)
 *   workspace       : device scratch of at least kvd_decode_plan's bytes for the
 *                     same (batch, heads, head_dim, max_seq_len, n_split,
 *                     out_dtype), 256-byte aligned; may be NULL when that is 0.
 *                     Contents need no initialisation and are not preserved.
 *   out             : [batch, n_heads_q, head_dim], bf16 or fp32 per out_dtype,
 *                     16-byte aligned
 *   lse_out         : optional fp32 [batch, n_heads_q], natural-log
 *                     log(sum_t exp(scale * q.k_t))
 *   status_word     : optional device int32
 * batch = 0 is a no-op. Call order for a generation step: kvd_kv_append with
 * pos = old length, then this with seq_lens = old length + 1, same stream.
 * Errors (nothing launched): KVD_ERR_INVALID_ARG for null or misaligned
 * pointers, non-positive sizes, max_seq_len outside [0, s_max], a group that
 * does not divide, a non-finite scale, n_split < 0 or an unknown out_dtype;
 * KVD_ERR_UNSUPPORTED as for kvd_decode_plan; KVD_ERR_WORKSPACE_TOO_SMALL;
 * KVD_ERR_CUDA if a launch fails.
 */
kvd_status kvd_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                                int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                int n_split, void* workspace, size_t workspace_bytes,
                                void* out, kvd_out_dtype out_dtype, float* lse_out,
                                int32_t* status_word, kvd_stream_t stream);

/*
 * kvd_decode_step: one generation step's cache work in one call, exactly
 * kvd_kv_append(k_cache, v_cache, k_new, v_new, pos, ...) followed by
 * kvd_decode_attention(q, k_cache, v_cache, seq_lens, ...) on the same stream
 * (All About Transformer Inference, "Transformer inference basics",
 * Generation: the new token's key and value join the cache, then its query
 * attends over it). Arguments, layouts and errors are those of the two calls;
 * nothing is launched if either call's arguments are rejected.
 * Difference in timing only: the attention launch begins while the append
 * runs. It works out its schedule and loads q and seq_lens before the append
 * has finished, and waits for the append only before loading cache rows. So
 * q, seq_lens and pos must be complete when this call's work starts on the
 * stream (as for any stream-ordered input), and only the cache rows may be
 * produced by the append.
 */
kvd_status kvd_decode_step(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                           const int32_t* pos, const void* q, const int32_t* seq_lens, int batch,
                           int s_max, int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                           float scale, int n_split, void* workspace, size_t workspace_bytes,
                           void* out, kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                           kvd_stream_t stream);

/*
 * Unified-maximum softmax: kvd_decode_attention and kvd_decode_step with the
 * partial softmax of every split taken against one caller-given maximum phi
 * (in the units of the logits scale * q.k) instead of each split's own,
 * FlashDecoding++'s asynchronized softmax with a unified maximum (the
 * FlashDecoding++ summary page, solution 1: partial softmax results need no
 * synchronised update when they share the maximum). Where a row's scores
 * stay within [phi - 64 ln 2, phi + 8 ln 2] every partial of the row holds
 * exp(s - phi) sums, so the merge is a plain sum; the pages leave the
 * out-of-range case open, and here a row whose scores leave that window falls
 * back to the usual running maximum in the kernel (no recomputation; the
 * result is the same softmax either way) and KVD_STATUS_UMAX_FALLBACK is set.
 * phi must be finite (KVD_ERR_INVALID_ARG); bf16 caches only. Arguments,
 * results and errors otherwise as kvd_decode_attention and kvd_decode_step.
 */
kvd_status kvd_decode_attention_umax(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                                     int n_heads_q, int n_heads_kv, int head_dim, float scale, float phi,
                                     int n_split, void* workspace, size_t workspace_bytes, void* out,
                                     kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                     kvd_stream_t stream);
kvd_status kvd_decode_step_umax(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                const int32_t* pos, const void* q, const int32_t* seq_lens, int batch, int s_max,
                                int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                float phi, int n_split, void* workspace, size_t workspace_bytes, void* out,
                                kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                kvd_stream_t stream);

/*
 * Paged KV cache. The pages describe keeping the KV cache in an
 * operating-system-style page table, so that each sequence holds only the
 * memory it uses instead of a padded maximum (All About Transformer Inference,
 * "Tricks for improving generation throughput and latency", the ragged HBM
 * reads and Paged Attention bullet). They give no layout; this library's is:
 *   k_pages, v_pages : bf16 [num_pages, page_size, n_heads_kv, head_dim], a pool
 *                      of pages, each laid out like a cache of capacity
 *                      page_size; 16-byte aligned. num_pages * page_size must
 *                      be below 2^31.
 *   block_table      : device int32 [batch, max_blocks], 4-byte aligned. Entry
 *                      (b, j) names the page that holds tokens
 *                      [j * page_size, (j + 1) * page_size) of sequence b, so
 *                      token t of sequence b is row t % page_size of page
 *                      block_table[b * max_blocks + t / page_size]. Only the
 *                      entries of blocks holding tokens t < L_b (or pos[b])
 *                      are read; others may hold anything.
 *   page_size        : a power of two in [16, 4096]; the capacity of a
 *                      sequence (s_max of the contiguous calls) is
 *                      max_blocks * page_size.
 * A needed entry outside [0, num_pages) is never dereferenced: attention
 * reads zero key and value rows for that block's tokens, an append to it is
 * skipped, and either sets KVD_STATUS_BAD_PAGE.
 * Each paged call is the contiguous call with the cache replaced by the pool
 * and the table; the other arguments, the results (bit for bit: the same
 * kernels and schedule run, only the row addresses differ), the workspace
 * (kvd_decode_plan with the same max_seq_len) and the errors are the same,
 * plus KVD_ERR_INVALID_ARG for a bad page_size, max_blocks < 1 or
 * num_pages < 1.
 */
kvd_status kvd_kv_append_paged(void* k_pages, void* v_pages, const void* k_new, const void* v_new,
                               const int32_t* block_table, const int32_t* pos, int batch,
                               int max_blocks, int page_size, int num_pages, int n_heads_kv,
                               int head_dim, int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_decode_attention_paged(const void* q, const void* k_pages, const void* v_pages,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      int batch, int max_blocks, int page_size, int num_pages,
                                      int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                                      float scale, int n_split, void* workspace,
                                      size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                                      float* lse_out, int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_decode_step_paged(void* k_pages, void* v_pages, const void* k_new, const void* v_new,
                                 const int32_t* pos, const void* q, const int32_t* block_table,
                                 const int32_t* seq_lens, int batch, int max_blocks, int page_size,
                                 int num_pages, int max_seq_len, int n_heads_q, int n_heads_kv,
                                 int head_dim, float scale, int n_split, void* workspace,
                                 size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                                 float* lse_out, int32_t* status_word, kvd_stream_t stream);

/*
 * int8 KV cache. The pages name quantizing the KV cache (int8, fp8, ...) as
 * a way to cut the memory traffic of every generation step (All About
 * Transformer Inference, "Tricks for improving generation throughput and
 * latency", the quantization bullet) but give no scheme; this library's is
 * symmetric absmax per (token, KV head) row:
 *   a = max_d |x_d|, scale = a / 127, code_d = round-half-even(x_d / scale)
 *   clamped to [-127, 127], both divisions IEEE float32 (a = 0: scale 0 and
 *   codes 0); the row reads back as scale * code_d.
 *   k_codes, v_codes   : int8 [batch, s_max, n_heads_kv, head_dim], 16-byte aligned
 *   k_scales, v_scales : float32 [batch, s_max, n_heads_kv], 4-byte aligned
 * kvd_kv_quantize_q8 converts rows t < seq_lens[b] (clamped to max_seq_len)
 * of one bf16 cache (K or V) into codes and scales, leaving other rows
 * untouched (a prefill's cache, say). kvd_kv_append_q8 quantizes the new
 * token's rows and writes them at pos[b], as kvd_kv_append. The attention
 * and step calls are kvd_decode_attention and kvd_decode_step over the rows
 * read back: q stays bf16, the cache rows are exact small integers times
 * their scale, and the kernels compute in f16 MMAs with fp32 accumulation,
 * with each score multiplied by its key row's scale and each weight by its
 * value row's scale. Every supported group: groups of 17 to 64 query heads
 * at head_dim 128, or 17 to 48 at 256, on the tcgen05 kernel's converting
 * variant (the codes converted exactly to f16 in shared memory), others on
 * the mma.sync kernel (one CTA per 16 query heads of a group and token run);
 * head_dim 64, 128 or 256. The
 * split count and workspace are kvd_decode_plan's. A paged int8 cache (code
 * pools [num_pages, page_size, n_heads_kv, head_dim] and scale pools
 * [num_pages, page_size, n_heads_kv], one block table for both) is appended
 * to by kvd_kv_append_q8_paged and read by kvd_decode_ex; its rows are found
 * as kvd_kv_append_paged's, and an entry that names no page reads as zero
 * rows (KVD_STATUS_BAD_PAGE).
 * q must lie in f16's range (|q| < 65504). Results and errors otherwise as the
 * bf16 calls, plus
 * KVD_ERR_INVALID_ARG for null or misaligned scale arrays.
 */
kvd_status kvd_kv_quantize_q8(const void* cache, void* codes, float* scales, const int32_t* seq_lens, int batch,
                              int s_max, int max_seq_len, int n_heads_kv, int head_dim, kvd_stream_t stream);
kvd_status kvd_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                            const void* v_new, const int32_t* pos, int batch, int s_max, int n_heads_kv,
                            int head_dim, int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_kv_append_q8_paged(void* k_code_pages, void* v_code_pages, float* k_scale_pages,
                                  float* v_scale_pages, const void* k_new, const void* v_new,
                                  const int32_t* block_table, const int32_t* pos, int batch, int max_blocks,
                                  int page_size, int num_pages, int n_heads_kv, int head_dim,
                                  int32_t* status_word, kvd_stream_t stream);

/*
 * fp8 KV cache: the int8 scheme above with the OCP 8-bit floating-point
 * format E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * subnormals, largest finite 448, no infinities) in place of int8, the other
 * 8-bit format the same page names:
 *   a = max_d |x_d|, scale = a / 448, code_d = x_d / scale rounded to the
 *   nearest E4M3 value (ties to the even code, magnitudes past 448 saturate to
 *   448), a result of zero stored as +0 (0x00); both divisions IEEE float32
 *   (a = 0: scale 0 and codes 0); the row reads back as scale * value(code_d).
 * Codes are bytes (uint8, bit-compatible with a float8 e4m3 "fn" tensor);
 * layouts, alignment, row selection, status and errors exactly as the int8
 * calls. Attention over an fp8 cache goes through kvd_decode_ex with
 * kvd_cache.fp8 = 1 (contiguous or paged, any supported group, T query
 * tokens, with or without the append); the kernels convert the codes to f16
 * exactly and compute as for int8.
 */
kvd_status kvd_kv_quantize_fp8(const void* cache, void* codes, float* scales, const int32_t* seq_lens, int batch,
                               int s_max, int max_seq_len, int n_heads_kv, int head_dim, kvd_stream_t stream);
kvd_status kvd_kv_append_fp8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                             const void* v_new, const int32_t* pos, int batch, int s_max, int n_heads_kv,
                             int head_dim, int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_kv_append_fp8_paged(void* k_code_pages, void* v_code_pages, float* k_scale_pages,
                                   float* v_scale_pages, const void* k_new, const void* v_new,
                                   const int32_t* block_table, const int32_t* pos, int batch, int max_blocks,
                                   int page_size, int num_pages, int n_heads_kv, int head_dim,
                                   int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_decode_attention_q8(const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                                   const float* v_scales, const int32_t* seq_lens, int batch, int s_max,
                                   int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                   int n_split, void* workspace, size_t workspace_bytes, void* out,
                                   kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                   kvd_stream_t stream);
kvd_status kvd_decode_step_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                              const void* v_new, const int32_t* pos, const void* q, const int32_t* seq_lens,
                              int batch, int s_max, int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                              float scale, int n_split, void* workspace, size_t workspace_bytes, void* out,
                              kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                              kvd_stream_t stream);

/*
 * Multi-token decode: n_tokens = T new tokens per sequence at once, as when a
 * large model checks T drafted tokens in one pass over the shared KV cache
 * (All About Transformer Inference, appendix "Speculative Sampling"). The T
 * rows of each sequence are appended at pos[b] .. pos[b] + T - 1, and query
 * token i attends to the first L_b - T + 1 + i cached tokens (the cache plus
 * the new tokens up to itself; L_b = seq_lens[b] after the append, so
 * seq_lens = old length + T). Layouts:
 *   q, out    : [batch, T, n_heads_q, head_dim] (bf16 q; out as out_dtype)
 *   lse_out   : optional fp32 [batch, T, n_heads_q]
 *   k_new, v_new : bf16 [batch, T, n_heads_kv, head_dim]
 * A query token that sees no token (L_b < T - i) gets a zero row and lse -inf.
 * T from 1 to KVD_MAX_TOKENS (above: KVD_ERR_UNSUPPORTED), any supported
 * group. Groups of up to 16 run on the mma.sync kernel, one CTA per 16 of a
 * pair's T * G rows and token run; wider groups on the tcgen05 kernel, with
 * the T tokens' rows stacked in one 128-row tile when T times the group
 * (rounded up to 8) is at most 128 (bf16 caches), else each query token as a
 * sequence of its own over the shared cache rows. T = 1 is
 * exactly the single-token call. The split count is the single-token plan's,
 * and the workspace holds T times the rows: size it with
 * kvd_decode_plan_multi. Rows of the append outside [0, s_max) are skipped
 * with KVD_STATUS_POS_OUT_OF_RANGE.
 * Other arguments, results and errors as the single-token calls, plus
 * KVD_ERR_INVALID_ARG for n_tokens < 1.
 */
kvd_status kvd_decode_plan_multi(int batch, int n_tokens, int n_heads_q, int n_heads_kv, int head_dim,
                                 int max_seq_len, int num_sms, int n_split_request, kvd_out_dtype out_dtype,
                                 int* n_split_out, size_t* workspace_bytes_out);
kvd_status kvd_kv_append_multi(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                               const int32_t* pos, int batch, int n_tokens, int s_max, int n_heads_kv,
                               int head_dim, int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* seq_lens, int batch, int n_tokens, int s_max,
                                      int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                      int n_split, void* workspace, size_t workspace_bytes, void* out,
                                      kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                      kvd_stream_t stream);
kvd_status kvd_decode_step_multi(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                 const int32_t* pos, const void* q, const int32_t* seq_lens, int batch,
                                 int n_tokens, int s_max, int max_seq_len, int n_heads_q, int n_heads_kv,
                                 int head_dim, float scale, int n_split, void* workspace, size_t workspace_bytes,
                                 void* out, kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                 kvd_stream_t stream);

/*
 * kvd_decode_ex: one entry point for every combination of the cache forms and
 * options above that the kernels support, with the cache described by a
 * struct:
 *   - bf16, int8 (k_scales and v_scales non-NULL: k and v hold int8 codes) or
 *     fp8 (the scales and fp8 = 1: k and v hold E4M3 codes);
 *   - contiguous (block_table NULL: k, v [batch, s_max, Hkv, D]) or paged
 *     (k, v are page pools, and for int8 k_scales, v_scales too);
 *   - n_tokens query tokens per sequence (layouts as kvd_decode_attention_multi;
 *     1 .. KVD_MAX_TOKENS; workspace from kvd_decode_plan_multi);
 *   - with the step's append (k_new, v_new and pos all non-NULL; the new rows,
 *     [batch, n_tokens, Hkv, D] bf16, are appended, quantized for an int8
 *     cache, before the attention, as kvd_decode_step) or without it (all three
 *     NULL).
 * Each combination is bit-identical to the dedicated call where one exists.
 * Errors: KVD_ERR_INVALID_ARG for a NULL cache, a cache description that fails
 * the dedicated calls' checks (fp8 set without scales included), or only some
 * of k_new, v_new, pos given; the rest as the dedicated calls.
 */
typedef struct kvd_cache {
    void* k;                       /* bf16 cache or page pool, or int8 codes */
    void* v;
    float* k_scales;               /* int8: float32 [batch, s_max, Hkv] (paged: [num_pages, page_size, Hkv]); NULL for bf16 */
    float* v_scales;
    const int32_t* block_table;    /* paged: int32 [batch, max_blocks]; NULL for contiguous */
    int s_max;                     /* contiguous: capacity of each sequence */
    int max_blocks, page_size, num_pages;  /* paged */
    int fp8;                       /* with the scales: 1 = k, v hold fp8 E4M3 codes, 0 = int8 codes */
} kvd_cache;

kvd_status kvd_decode_ex(const kvd_cache* cache, const void* q, const int32_t* seq_lens, int batch, int n_tokens,
                         int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale, int n_split,
                         void* workspace, size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                         float* lse_out, const void* k_new, const void* v_new, const int32_t* pos,
                         int32_t* status_word, kvd_stream_t stream);

/*
 * The two launches of kvd_decode_attention, exposed separately so that each
 * can be timed on its own. Arguments and errors are those of
 * kvd_decode_attention; calling kvd_split_kv_chunk then kvd_split_kv_merge on
 * one stream with the same arguments is exactly kvd_decode_attention.
 *  - kvd_split_kv_chunk: every CTA streams its run of K/V rows and either
 *    writes final rows (pairs it covers entirely) or partial (m, l, o) states
 *    into the workspace.
 *  - kvd_split_kv_merge: merges the partial states of every split pair by
 *    log-sum-exp: M = max_j m_j, w_j = 2^(m_j - M), out = sum_j w_j o_j /
 *    sum_j w_j l_j, skipping empty partials. A no-op when n_split is 1. It
 *    recomputes from seq_lens which CTAs wrote partials for each pair (and
 *    reads seq_lens before waiting for the chunk launch), so seq_lens must hold
 *    the values the chunk call used and must not be written in between.
 */
kvd_status kvd_split_kv_chunk(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                              int n_heads_q, int n_heads_kv, int head_dim, float scale,
                              int n_split, void* workspace, size_t workspace_bytes,
                              void* out, kvd_out_dtype out_dtype, float* lse_out,
                              int32_t* status_word, kvd_stream_t stream);
kvd_status kvd_split_kv_merge(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                              int n_heads_q, int n_heads_kv, int head_dim, float scale,
                              int n_split, void* workspace, size_t workspace_bytes,
                              void* out, kvd_out_dtype out_dtype, float* lse_out,
                              int32_t* status_word, kvd_stream_t stream);

/*
 * kvd_schedule_describe: host-only replica of the device work schedule, for
 * inspection and tests (no GPU needed). seq_lens_host is HOST int32 [batch].
 * Writes up to max_rows rows of 8 int32 each to rows_out:
 *   {cta, b, h, tok_lo, tok_hi, kind, slot, c_last}
 * one row per segment (a CTA's tokens [tok_lo, tok_hi) of pair (b, h)) and one
 * per empty pair, where kind is 0 = final (the CTA owns and covers the pair),
 * 1 = partial written by the pair's owner, 2 = partial written by another CTA,
 * 3 = empty pair (zero output). slot is the partial's workspace slot (-1 if
 * none); c_last is the last CTA contributing to the pair (owner rows of kind 1).
 * *n_rows_out receives the total number of rows (even if > max_rows) and
 * *n_split_eff_out the number of CTAs that do work. Errors as kvd_decode_plan.
 */
kvd_status kvd_schedule_describe(const int32_t* seq_lens_host, int batch, int s_max,
                                 int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                                 int n_split, kvd_out_dtype out_dtype,
                                 int32_t* rows_out, int max_rows, int* n_rows_out,
                                 int* n_split_eff_out);

/*
 * kvd_kernel_info: launch shape of the attention kernel chosen for a shape:
 * threads per CTA, dynamic shared memory bytes, tokens per pipeline tile, the
 * CTAs per SM the heuristic assumes, and the unit and start-up charge of its
 * work schedule. The schedule lays the (sequence, KV head) pairs on a line of
 * positions of seg_unit tokens each (1, or tile_tokens when the kernel's time
 * is set by its tile count): a non-empty pair occupies
 * seg_cost + ceil(len / seg_unit) positions, and the CTAs get balanced runs of
 * positions. Any out pointer may be NULL. Host only. Errors as kvd_decode_plan.
 */
kvd_status kvd_kernel_info(int n_heads_q, int n_heads_kv, int head_dim, kvd_out_dtype out_dtype,
                           int* threads_out, int* smem_bytes_out, int* tile_tokens_out,
                           int* ctas_per_sm_out, int* seg_unit_out, int* seg_cost_out);

/*
 * kvd_merge_attention: attention results over disjoint shards of each
 * sequence's tokens combined into the result over all of them, the exchange
 * step of sequence-sharded KV (All About Transformer Inference, "Sharding the
 * KV cache": the shards' results accumulate as in Flash Attention): given, per
 * shard j, the normalised output out_j and its natural-log normaliser lse_j
 * (as kvd_decode_attention returns them in out and lse_out), with
 * L = ln sum_j exp(lse_j):  out = sum_j exp(lse_j - L) out_j,  lse = L.
 * A shard with lse = -inf holds no token and adds nothing; a row with no token
 * in any shard gets a zero row and lse -inf. A row where any shard's lse is
 * NaN or +inf (no valid attention result) gets NaN in every column and in
 * lse_out, so that a corrupted shard cannot pass for a plausible result.
 *   outs    : [n_shards, rows, head_dim] bf16 or fp32 (in_dtype), 16-byte aligned
 *   lses    : fp32 [n_shards, rows]
 *   out     : [rows, head_dim] (out_dtype), 16-byte aligned; lse_out: optional fp32 [rows]
 * rows is B * Hq (or B * T * Hq) of the shards' calls. The shards may come
 * from other devices (copied here first) or from separate caches on this one
 * (a shared prefix and a per-sequence suffix). The call cannot work in place:
 * out and lse_out must overlap neither outs, lses nor each other. Errors:
 * KVD_ERR_INVALID_ARG for NULL or misaligned pointers, overlapping written and
 * read ranges, n_shards < 1, rows < 0 or a bad dtype;
 * KVD_ERR_UNSUPPORTED for head_dim outside {64, 128, 256}; KVD_ERR_CUDA if the
 * launch fails.
 */
kvd_status kvd_merge_attention(const void* outs, const float* lses, int n_shards, long long rows, int head_dim,
                               kvd_out_dtype in_dtype, void* out, kvd_out_dtype out_dtype, float* lse_out,
                               kvd_stream_t stream);

/*
 * kvd_decode_step_host: one step whose per-step inputs come from the host and
 * whose result goes back to it, in one call (a deployment convenience, not
 * part of the method): q_host [batch, n_tokens, Hq, D] bf16, k_new_host,
 * v_new_host [batch, n_tokens, Hkv, D] bf16, pos_host and seq_lens_host
 * int32 [batch] are copied (cudaMemcpyAsync on `stream`; pinned host memory
 * makes the copies asynchronous) into `staging`, a device buffer of at least
 * kvd_step_staging_bytes(...) bytes, 256-byte aligned; then the step runs as
 * kvd_decode_step_multi on the staged inputs (n_tokens = 1: kvd_decode_step),
 * writing `out` on the device, and `out` is copied to out_host (same size).
 * Host inputs laid out like the staging buffer (q | k_new | v_new | pos |
 * seq_lens, each 256-byte aligned, one host packet starting at q_host) are
 * copied with one cudaMemcpyAsync instead of five; if that packet is
 * page-locked memory the device addresses (256-byte aligned), nothing is
 * copied ahead: the append kernel reads k_new, v_new and pos from it and pulls
 * q into `staging` over the host link while the attention's cache loads run,
 * and the attention reads pos and seq_lens from it (q's loads wait for the
 * append). The packet must then stay unchanged until the call's work on
 * `stream` is done. With out = NULL the kernels
 * write the result straight into out_host, which must then be page-locked
 * host memory the device can address (cudaHostAlloc / cudaHostRegister, 16-byte
 * aligned; else KVD_ERR_INVALID_ARG), and no copy back is queued.
 * Nothing is synchronised: out_host is valid once `stream` has reached the end
 * of this call's work. Every argument is checked before any copy is queued;
 * errors as kvd_decode_step_multi, plus KVD_ERR_INVALID_ARG for a NULL host
 * pointer or a missing, small or misaligned staging buffer. The caller owns
 * all buffers; the cache, workspace, out and lse_out are device memory.
 */
size_t kvd_step_staging_bytes(int batch, int n_tokens, int n_heads_q, int n_heads_kv, int head_dim);
kvd_status kvd_decode_step_host(void* k_cache, void* v_cache, const void* q_host, const void* k_new_host,
                                const void* v_new_host, const int32_t* pos_host, const int32_t* seq_lens_host,
                                void* staging, size_t staging_bytes, int batch, int n_tokens, int s_max,
                                int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                int n_split, void* workspace, size_t workspace_bytes, void* out, void* out_host,
                                kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                kvd_stream_t stream);

/*
 * kvd_decode_attention_static: kvd_decode_attention for callers that cannot
 * allocate device memory. (The sources have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * Some callers may not allocate at decode time: a serving loop whose device
 * memory is budgeted and frozen at start-up, a plugin handed only the tensors
 * it works on, or a path that must not risk the device-wide synchronisation
 * that cudaMalloc/cudaFree can cause. This entry point takes the same
 * arguments as kvd_decode_attention without workspace/workspace_bytes and
 * uses instead a scratch array inside the library: a __device__ array of
 * KVD_STATIC_WORKSPACE_BYTES that every GPU loading the library holds until
 * the process exits. It allocates nothing (no cudaMalloc, cudaFree or
 * allocating library call); inputs and outputs stay the caller's.
 *   - Limit: if kvd_decode_plan's workspace for the call exceeds
 *     KVD_STATIC_WORKSPACE_BYTES, the call returns KVD_ERR_WORKSPACE_TOO_SMALL
 *     and launches nothing (a smaller n_split lowers the need).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is cached per device and
 *     context: after the device's context is destroyed and re-created
 *     (cudaDeviceReset), the next call looks it up again (make that call
 *     outside stream capture as well).
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero, but calls that overlap on the GPU
 *     (e.g. on two streams) race on it: serialise them.
 * Other arguments, errors and results as kvd_decode_attention.
 */
#define KVD_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)
kvd_status kvd_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                                       int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                       int n_split, void* out, kvd_out_dtype out_dtype, float* lse_out,
                                       int32_t* status_word, kvd_stream_t stream);

/*
 * kvd_probe_read: a measurement aid, not part of the method. One pass that only
 * reads [src, src + bytes) into shared memory, the way the attention kernels
 * read the KV cache (bulk asynchronous copies into a ring of 32 KB stages, one
 * CTA per SM with a contiguous slice each; L2 evict-first), so that the time
 * of one launch bounds from below what any kernel reading those bytes once
 * can take, its launch, first-data latency and drain included. Decode
 * attention is bound by that read (Efficiently Scaling Transformer Inference,
 * section 2; All About Transformer Inference, "What about attention?").
 *   src         : device memory, 16-byte aligned; bytes rounded down to 16
 *   ctas        : CTAs launched (0 = the device's SM count)
 *   sink        : optional device u64[ctas]: a word per CTA derived from the
 *                 data read (so the reads have a consumer); 8-byte aligned
 *   status_word : optional; KVD_STATUS_TIMEOUT if a copy wait gave up (~2 s)
 * Errors: KVD_ERR_INVALID_ARG for a NULL src, misaligned pointers or
 * ctas < 0; KVD_ERR_CUDA if the launch fails. Fewer than 16 bytes: no launch.
 */
kvd_status kvd_probe_read(const void* src, size_t bytes, int ctas, unsigned long long* sink,
                          int32_t* status_word, kvd_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* kvd_status_string(kvd_status s);

/* Library version string (static). */
const char* kvd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVDECODE_H */
