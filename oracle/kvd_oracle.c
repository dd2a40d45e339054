/*
 * CPU oracle for single-token decode attention over a KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this library. The CUDA path never
 * calls it and shares no code, header or constant with it.
 *
 * Plain, slow and direct: every value is widened from bf16 to double and every
 * sum is a left-to-right loop in double precision. No blocking, fusion or
 * reordering beyond what the definitions below state. OpenMP (when compiled
 * with it) only splits the independent (sequence, query head) problems over
 * threads; each problem is still computed by one thread in the order written.
 *
 * Definitions followed:
 *
 *  - Attention of one decode token, per query head, over the cached keys and
 *    values: scores = q . k_t (contraction over the head dimension H), softmax
 *    over the sequence axis S, then the softmax-weighted sum of the value rows.
 *    All About Transformer Inference, "Sharding the KV cache", the attention
 *    algorithm (steps "O = Q *_H K", "Softmax_S", "O *_S V").
 *  - Head grouping: query heads are reshaped from [N] to [K, M] with M = N/K,
 *    so query head n uses KV head n / M (same algorithm, the Reshape step;
 *    multiquery is K = 1: Efficiently Scaling Transformer Inference, section
 *    3.3; grouped-query: All About Transformer Inference, "Tricks for
 *    improving generation throughput and latency").
 *  - Cache layout K[B, S, K, H] and V likewise (All About Transformer
 *    Inference, "Sharding the KV cache"); a token only attends to tokens
 *    already in the cache, so the decode token attends to all L_b cached rows
 *    including its own appended one (All About Transformer Inference,
 *    "Transformer inference basics").
 *  - Appending the new token's key/value projections to the cache is a plain
 *    copy (All About Transformer Inference, "Transformer inference basics",
 *    the Generation bullet; "Implementation: JetStream", the generate method).
 *  - The chunked path splits the sequence axis into pieces whose partial
 *    softmax results are combined afterwards, the way sequence-sharded KV is
 *    accumulated "like Flash Attention" (All About Transformer Inference,
 *    "Sharding the KV cache", the sequence-sharding bullet). The pages give no
 *    formula for the combination; the one used is the textbook log-sum-exp
 *    identity: with chunk maxima m_j, sums l_j = sum exp(s - m_j) and
 *    unnormalised outputs o_j = sum exp(s - m_j) v, the result is
 *    sum_j exp(m_j - M) o_j / sum_j exp(m_j - M) l_j with M = max_j m_j, and
 *    empty chunks skipped.
 *  - Paged cache: the cache is kept in an operating-system-style page table,
 *    so a sequence only holds the pages it uses (All About Transformer
 *    Inference, "Tricks for improving generation throughput and latency", the
 *    ragged HBM reads and Paged Attention bullet). The pages give no layout;
 *    the one used is: pages of P tokens, each laid out like a cache of
 *    capacity P ([P, K, H]), and a block table whose entry (b, j) names the
 *    page that holds tokens [j P, (j + 1) P) of sequence b, so token t sits in
 *    row t mod P of page table[b][t / P]. A token whose entry is not a page
 *    of the pool reads zero key and value rows (and an append to it is
 *    skipped); both are counted.
 *  - int8 cache: the pages name int8 (and fp8, int4) quantization of the
 *    KV cache as a way to cut its memory traffic (All About Transformer
 *    Inference, "Tricks for improving generation throughput and latency",
 *    the quantization bullet) but give no scheme. The one used is symmetric
 *    absmax per (token, KV head) row: with a = max_d |x_d| (float32),
 *    scale = a / 127 and code_d = round-half-even(x_d / scale) clamped to
 *    [-127, 127], both divisions in IEEE float32 (a = 0: scale 0, codes 0).
 *    A row is read back as scale * code_d. Attention over an int8 cache is
 *    the attention above over the rows read back, in double precision.
 *
 * All functions return 0 on success and a negative value on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int check_dims(int B, int S_max, int Hq, int Hkv, int D)
{
    if (B < 0 || S_max < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -2;
    return 0;
}

/* Address of element (b, t, g, 0) of a [B, S_max, Hkv, D] cache. */
static const uint16_t* cache_row(const uint16_t* c, int b, int t, int g,
                                 int S_max, int Hkv, int D)
{
    return c + (((size_t)b * (size_t)S_max + (size_t)t) * (size_t)Hkv + (size_t)g) * (size_t)D;
}

/* Softmax weights of one query head over the first L cached tokens.
 * w[t] = exp(s_t - max s) / sum_u exp(s_u - max s), s_t = scale * q . k_t.
 * Returns the natural-log normaliser log sum_t exp(s_t) (or -inf if L == 0). */
static double head_weights(const uint16_t* qrow, const uint16_t* k, int b, int g,
                           int L, int S_max, int Hkv, int D, double scale, double* w)
{
    if (L == 0) return -INFINITY;
    double mx = -INFINITY;
    for (int t = 0; t < L; ++t) {
        const uint16_t* kr = cache_row(k, b, t, g, S_max, Hkv, D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(qrow[d]) * bf16_to_double(kr[d]);
        w[t] = scale * dot;
        if (w[t] > mx) mx = w[t];
    }
    double sum = 0.0;
    for (int t = 0; t < L; ++t) {
        w[t] = exp(w[t] - mx);
        sum += w[t];
    }
    for (int t = 0; t < L; ++t) w[t] /= sum;
    return mx + log(sum);
}

/* Attention weights of one (sequence b, query head h): w[0..L_b). */
int kvo_attention_weights(const uint16_t* q, const uint16_t* k, const int32_t* seq_lens,
                          int B, int S_max, int Hq, int Hkv, int D, double scale,
                          int b, int h, double* w)
{
    if (check_dims(B, S_max, Hq, Hkv, D)) return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq) return -3;
    int L = seq_lens[b];
    if (L < 0 || L > S_max) return -4;
    int g = h / (Hq / Hkv);
    head_weights(q + ((size_t)b * Hq + h) * D, k, b, g, L, S_max, Hkv, D, scale, w);
    return 0;
}

/* out[b, h, :] = sum_t w_t V[b, t, h / (Hq/Hkv), :] for t < seq_lens[b];
 * lse[b, h] = log sum_t exp(s_t) (natural log), -inf for an empty sequence,
 * where the output row is all zeros. n_threads <= 0 means "all available". */
int kvo_decode_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* seq_lens, int B, int S_max, int Hq, int Hkv, int D,
                         double scale, double* out, double* lse, int n_threads)
{
    if (check_dims(B, S_max, Hq, Hkv, D)) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > S_max) return -4;
    const int G = Hq / Hkv;
    const long n_problems = (long)B * Hq;
    int fail = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(|:fail)
#endif
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)(S_max > 0 ? S_max : 1));
        if (!w) {
            fail = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (long p = 0; p < n_problems; ++p) {
                const int b = (int)(p / Hq), h = (int)(p % Hq), g = h / G;
                const int L = seq_lens[b];
                double* o = out + (size_t)p * D;
                const double norm = head_weights(q + (size_t)p * D, k, b, g, L,
                                                 S_max, Hkv, D, scale, w);
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int t = 0; t < L; ++t) {
                    const uint16_t* vr = cache_row(v, b, t, g, S_max, Hkv, D);
                    for (int d = 0; d < D; ++d) o[d] += w[t] * bf16_to_double(vr[d]);
                }
                if (lse) lse[p] = norm;
            }
            free(w);
        }
    }
    return fail ? -5 : 0;
}

/* The same attention computed chunk by chunk: the first L_b tokens are cut into
 * n_chunks pieces of ceil(L_b / n_chunks) tokens (trailing pieces may be
 * empty). Each piece yields (m_j, l_j, o_j); the pieces are then combined with
 * the log-sum-exp identity in the header comment. */
int kvo_decode_attention_chunked(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const int32_t* seq_lens, int B, int S_max, int Hq, int Hkv,
                                 int D, double scale, int n_chunks, double* out, double* lse)
{
    if (check_dims(B, S_max, Hq, Hkv, D)) return -1;
    if (n_chunks <= 0) return -3;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > S_max) return -4;
    const int G = Hq / Hkv;
    double* m = (double*)malloc(sizeof(double) * (size_t)n_chunks);
    double* l = (double*)malloc(sizeof(double) * (size_t)n_chunks);
    double* o = (double*)malloc(sizeof(double) * (size_t)n_chunks * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(S_max > 0 ? S_max : 1));
    if (!m || !l || !o || !s) { free(m); free(l); free(o); free(s); return -5; }

    for (long p = 0; p < (long)B * Hq; ++p) {
        const int b = (int)(p / Hq), h = (int)(p % Hq), g = h / G;
        const int L = seq_lens[b];
        const uint16_t* qrow = q + (size_t)p * D;
        const int chunk = (L + n_chunks - 1) / n_chunks;

        /* Partial softmax state of each chunk. */
        for (int j = 0; j < n_chunks; ++j) {
            const int t0 = j * chunk;
            const int t1 = (t0 + chunk < L) ? t0 + chunk : L;
            double* oj = o + (size_t)j * D;
            for (int d = 0; d < D; ++d) oj[d] = 0.0;
            m[j] = -INFINITY;
            l[j] = 0.0;
            if (t0 >= t1) continue;
            for (int t = t0; t < t1; ++t) {
                const uint16_t* kr = cache_row(k, b, t, g, S_max, Hkv, D);
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += bf16_to_double(qrow[d]) * bf16_to_double(kr[d]);
                s[t] = scale * dot;
                if (s[t] > m[j]) m[j] = s[t];
            }
            for (int t = t0; t < t1; ++t) {
                const double e = exp(s[t] - m[j]);
                const uint16_t* vr = cache_row(v, b, t, g, S_max, Hkv, D);
                l[j] += e;
                for (int d = 0; d < D; ++d) oj[d] += e * bf16_to_double(vr[d]);
            }
        }

        /* Combine: M = max over non-empty chunks; weights exp(m_j - M). */
        double M = -INFINITY;
        for (int j = 0; j < n_chunks; ++j)
            if (l[j] > 0.0 && m[j] > M) M = m[j];
        double* orow = out + (size_t)p * D;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        if (M == -INFINITY) {              /* empty sequence */
            if (lse) lse[p] = -INFINITY;
            continue;
        }
        double denom = 0.0;
        for (int j = 0; j < n_chunks; ++j) {
            if (!(l[j] > 0.0)) continue;
            const double a = exp(m[j] - M);
            denom += a * l[j];
            for (int d = 0; d < D; ++d) orow[d] += a * o[(size_t)j * D + d];
        }
        for (int d = 0; d < D; ++d) orow[d] /= denom;
        if (lse) lse[p] = M + log(denom);
    }
    free(m); free(l); free(o); free(s);
    return 0;
}

/* Append one token per sequence: K[b, pos[b], h, :] = k_new[b, h, :] and the
 * same for V, a byte-for-byte copy of the bf16 rows. Sequences whose pos lies
 * outside [0, S_max) are left untouched and counted in the return value. */
int kvo_kv_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                  const uint16_t* v_new, const int32_t* pos, int B, int S_max,
                  int Hkv, int D)
{
    if (B < 0 || S_max < 0 || Hkv <= 0 || D <= 0) return -1;
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        const int t = pos[b];
        if (t < 0 || t >= S_max) { ++skipped; continue; }
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)b * S_max + (size_t)t) * Hkv + h) * (size_t)D;
            const size_t src = ((size_t)b * Hkv + h) * (size_t)D;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    return skipped;
}

/* Paged cache -> contiguous cache: out[b, t, h, :] = pages[table[b][t / P],
 * t mod P, h, :] for t < seq_lens[b]; zero rows where table[b][t / P] is not
 * in [0, num_pages); rows t >= seq_lens[b] are left as the caller filled them.
 * out is [B, max_blocks * P, Hkv, D]. Returns the number of tokens that read
 * zero rows (or a negative value on bad arguments). */
int kvo_paged_gather(const uint16_t* pages, const int32_t* table, const int32_t* seq_lens,
                     int B, int max_blocks, int P, int num_pages, int Hkv, int D, uint16_t* out)
{
    if (B < 0 || max_blocks < 0 || P <= 0 || num_pages < 0 || Hkv <= 0 || D <= 0) return -1;
    const size_t row = (size_t)Hkv * (size_t)D;  /* elements per token */
    const size_t S = (size_t)max_blocks * (size_t)P;
    int zeroed = 0;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        if (L < 0 || (size_t)L > S) return -2;
        for (int t = 0; t < L; ++t) {
            const int page = table[(size_t)b * max_blocks + t / P];
            uint16_t* dst = out + ((size_t)b * S + (size_t)t) * row;
            if (page < 0 || page >= num_pages) {
                memset(dst, 0, sizeof(uint16_t) * row);
                ++zeroed;
                continue;
            }
            const uint16_t* src = pages + ((size_t)page * (size_t)P + (size_t)(t % P)) * row;
            memcpy(dst, src, sizeof(uint16_t) * row);
        }
    }
    return zeroed;
}

/* Paged append: pages[table[b][pos[b] / P], pos[b] mod P, h, :] = new[b, h, :]
 * for K and V. Sequences whose pos lies outside [0, max_blocks * P), or whose
 * entry is not a page of the pool, are skipped; *bad_page counts the latter.
 * Returns the number of skipped sequences. */
int kvo_kv_append_paged(uint16_t* k_pages, uint16_t* v_pages, const uint16_t* k_new,
                        const uint16_t* v_new, const int32_t* table, const int32_t* pos,
                        int B, int max_blocks, int P, int num_pages, int Hkv, int D, int* bad_page)
{
    if (B < 0 || max_blocks < 0 || P <= 0 || num_pages < 0 || Hkv <= 0 || D <= 0) return -1;
    int skipped = 0, bad = 0;
    for (int b = 0; b < B; ++b) {
        const int t = pos[b];
        if (t < 0 || (long long)t >= (long long)max_blocks * P) { ++skipped; continue; }
        const int page = table[(size_t)b * max_blocks + t / P];
        if (page < 0 || page >= num_pages) { ++skipped; ++bad; continue; }
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)page * P + (size_t)(t % P)) * Hkv + h) * (size_t)D;
            const size_t src = ((size_t)b * Hkv + h) * (size_t)D;
            memcpy(k_pages + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
            memcpy(v_pages + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    if (bad_page) *bad_page = bad;
    return skipped;
}

/* Quantize rows of D bf16 values to int8 codes and one float32 scale each
 * (the scheme in the header comment). */
int kvo_quantize_q8(const uint16_t* x, long rows, int D, int8_t* codes, float* scales)
{
    if (rows < 0 || D <= 0) return -1;
    for (long r = 0; r < rows; ++r) {
        const uint16_t* xr = x + (size_t)r * D;
        float a = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float v = fabsf((float)bf16_to_double(xr[d]));
            if (v > a) a = v;
        }
        volatile float sc = a / 127.0f;  /* one IEEE float32 division, rounded to nearest */
        scales[r] = sc;
        for (int d = 0; d < D; ++d) {
            int c = 0;
            if (a > 0.0f) {
                volatile float y = (float)bf16_to_double(xr[d]) / sc;
                c = (int)rintf(y);  /* round half to even (default rounding mode) */
                if (c > 127) c = 127;
                if (c < -127) c = -127;
            }
            codes[(size_t)r * D + d] = (int8_t)c;
        }
    }
    return 0;
}

/* Rows read back from int8 codes: out[r, d] = scales[r] * codes[r, d]. */
int kvo_dequantize_q8(const int8_t* codes, const float* scales, long rows, int D, double* out)
{
    if (rows < 0 || D <= 0) return -1;
    for (long r = 0; r < rows; ++r)
        for (int d = 0; d < D; ++d)
            out[(size_t)r * D + d] = (double)scales[r] * (double)codes[(size_t)r * D + d];
    return 0;
}

/* ---- fp8 (E4M3) KV cache ----
 * The OCP 8-bit floating-point format E4M3: a sign bit, 4 exponent bits with
 * bias 7 and 3 mantissa bits; exponent field 0 holds the subnormals
 * m/8 * 2^-6, the all-ones pattern S.1111.111 is NaN, there are no
 * infinities, and the largest finite magnitude is 1.75 * 2^8 = 448. */
static double e4m3_value(int code)
{
    const int e = (code >> 3) & 15, m = code & 7;
    const double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return (code & 0x80) ? -v : v;
}

/* The E4M3 code nearest to y: round to nearest, ties to the code with the even
 * low bit (adjacent codes alternate), magnitudes past 448 saturate to 448, and
 * a value that rounds to zero is stored as +0 (code 0). A search over the 127
 * finite magnitudes, in order, so the comparison is plain. */
int kvo_e4m3_encode(float y)
{
    const double a = fabs((double)y);
    int best = 0;
    double bd = a;  /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs(e4m3_value(c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    if (best == 0) return 0;
    return (y < 0.0f) ? (best | 0x80) : best;
}

double kvo_e4m3_value(int code) { return e4m3_value(code & 0xFF); }

/* fp8 rows: a = max_d |x_d|, scale = a / 448, code_d = E4M3(x_d / scale), both
 * divisions IEEE float32 (a = 0: scale 0 and codes 0). */
int kvo_quantize_fp8(const uint16_t* x, long rows, int D, uint8_t* codes, float* scales)
{
    if (rows < 0 || D <= 0) return -1;
    for (long r = 0; r < rows; ++r) {
        const uint16_t* xr = x + (size_t)r * D;
        float a = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float v = fabsf((float)bf16_to_double(xr[d]));
            if (v > a) a = v;
        }
        volatile float sc = a / 448.0f;
        scales[r] = sc;
        for (int d = 0; d < D; ++d) {
            int c = 0;
            if (a > 0.0f) {
                volatile float y = (float)bf16_to_double(xr[d]) / sc;
                c = kvo_e4m3_encode(y);
            }
            codes[(size_t)r * D + d] = (uint8_t)c;
        }
    }
    return 0;
}

/* Rows read back from fp8 codes: out[r, d] = scales[r] * E4M3 value of codes[r, d]. */
int kvo_dequantize_fp8(const uint8_t* codes, const float* scales, long rows, int D, double* out)
{
    if (rows < 0 || D <= 0) return -1;
    for (long r = 0; r < rows; ++r)
        for (int d = 0; d < D; ++d)
            out[(size_t)r * D + d] = (double)scales[r] * e4m3_value(codes[(size_t)r * D + d]);
    return 0;
}

/* kvo_decode_attention with the caches given as doubles (e.g. rows read back
 * from int8): the same definition, the same loops. */
int kvo_decode_attention_f64kv(const uint16_t* q, const double* k, const double* v,
                               const int32_t* seq_lens, int B, int S_max, int Hq, int Hkv, int D,
                               double scale, double* out, double* lse, int n_threads)
{
    if (check_dims(B, S_max, Hq, Hkv, D)) return -1;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > S_max) return -4;
    const int G = Hq / Hkv;
    const long n_problems = (long)B * Hq;
    int fail = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(|:fail)
#endif
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)(S_max > 0 ? S_max : 1));
        if (!w) {
            fail = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (long p = 0; p < n_problems; ++p) {
                const int b = (int)(p / Hq), h = (int)(p % Hq);
                const int kvh = h / G;  /* KV head of query head h */
                const int len = seq_lens[b];
                const uint16_t* qrow = q + (size_t)p * D;
                double* o = out + (size_t)p * D;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (len == 0) {
                    if (lse) lse[p] = -INFINITY;
                    continue;
                }
                double top = -INFINITY;
                for (int t = 0; t < len; ++t) {
                    const double* kr = k + (((size_t)b * S_max + t) * Hkv + kvh) * (size_t)D;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += bf16_to_double(qrow[d]) * kr[d];
                    w[t] = acc * scale;
                    if (w[t] > top) top = w[t];
                }
                double total = 0.0;
                for (int t = 0; t < len; ++t) {
                    const double e = exp(w[t] - top);
                    w[t] = e;
                    total += e;
                }
                for (int t = 0; t < len; ++t) {
                    const double* vr = v + (((size_t)b * S_max + t) * Hkv + kvh) * (size_t)D;
                    const double wt = w[t] / total;
                    for (int d = 0; d < D; ++d) o[d] += wt * vr[d];
                }
                if (lse) lse[p] = top + log(total);
            }
            free(w);
        }
    }
    return fail ? -5 : 0;
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int kvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
