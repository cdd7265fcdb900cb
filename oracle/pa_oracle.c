/*
 * pa_oracle.c -- plain fp64 CPU oracle for one decode step of paged attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file. The CUDA library never includes, links
 * or calls it, and it includes nothing from the CUDA library.
 *
 * What it computes, and where the definition comes from:
 *
 *  append   Each new token's K and V row is copied, bit for bit, into its slot
 *           of the paged pool. A slot is block * block_size + offset, the flat
 *           form of the paged indexing in "MLSys Engineer -- Inference Systems
 *           Q&A", Q1 "How does PagedAttention work?" (the kernel rewrite). The
 *           decode step appends before it attends: "LLM inference and
 *           serving", "Code from memory", the naive incremental decoder (the
 *           cache append, then softmax over every row seen so far).
 *
 *  copy     Copy-on-write of whole blocks: for each (src, dst) pair, every
 *           KV head's block_size rows of K and of V in block src are copied,
 *           bit for bit, over block dst. A block shared by several sequences
 *           is copied before one of them writes into it ("MLSys Engineer --
 *           Inference Systems Q&A", Q1, "Why this helps": copy-on-write
 *           sharing; "Forward Deployed Engineering Interview", Chapter 2
 *           "Batching and the KV Cache": the block manager's append copies a
 *           shared last block first). Pairs are applied in order.
 *
 *  fp8      An FP8 cache stores each element as an e4m3 code with one scale
 *           per tensor (K and V each): value = scale * e4m3(code); an
 *           uncalibrated scale is 1.0 ("Forward Deployed Engineering
 *           Interview", Chapter 2: an FP8 cache halves the bytes per token,
 *           scales per tensor). The pages name the format only; e4m3 is read
 *           as the OCP 8-bit format: 1 sign bit, 4 exponent bits with bias 7,
 *           3 mantissa bits, subnormals at exponent 0, no infinities, the
 *           all-ones exponent-and-mantissa pattern (0x7F, 0xFF) is NaN, so
 *           the largest finite magnitude is 448. Appending into an FP8 cache
 *           divides each new value by the scale in fp32 (IEEE division) and
 *           rounds the quotient to the nearest e4m3 value, ties to the even
 *           code, magnitudes beyond 448 saturating to 448 (pao_e4m3_encode).
 *
 *  gather   Row i of a sequence's K (and V) lives in physical block
 *           block_table[i / block_size] at offset i % block_size (same Q1).
 *           The oracle rebuilds the sequence's contiguous K and V this way.
 *
 *  attend   Textbook single-query attention per query head, in fp64, from the
 *           values stored in the cache dtype: S_i = scale * <q, K_i>,
 *           w_i = exp(S_i - max S), out = sum_i (w_i / sum w) V_i (the naive
 *           decoder above, with the running-max subtraction of Q4 "How would
 *           you write a fused attention kernel?" used only for stability).
 *           Grouped-query attention: query head qh reads KV head
 *           qh / (num_heads / num_kv_heads) ("LLM inference and serving", Q7
 *           "What are MQA and GQA"; consecutive grouping is this library's
 *           reading of "each shared by H/H_kv query heads").
 *
 *  multi    Several query tokens per sequence (pao_decode_multi): the last Q
 *           of a sequence's n rows are new tokens verified together, as in
 *           speculative decoding ("MLSys Engineer -- Inference Systems Q&A",
 *           Q6: verifying K draft tokens in one pass reads the cache once; Q2,
 *           phase 3: each draft token attends only to its ancestors). Query j
 *           (0-based) sits at row n - Q + j and attends to rows 0 .. n - Q + j,
 *           each by the single-query definition above.
 *
 *  int8     An INT8 cache stores each (token, KV head) row of K (and of V) as
 *           int8 codes with one fp32 scale per row: scale = max|x| / 127 and
 *           code = x / scale rounded to the nearest integer, ties to even
 *           (the division in fp32), so value = scale * code ("MLSys Engineer
 *           -- Inference Systems Q&A", Q3: INT8 KV with per-token scaling,
 *           scale = max(|K_row|) / 127, dequantised before the softmax). An
 *           all-zero row gets scale 0 and codes 0.
 *
 *  window   Sliding-window attention (pao_decode_window): a sequence of n rows
 *           attends only to its last W rows, n - W .. n - 1 ("MLSys Engineer
 *           -- Inference Systems Q&A", Q3: local-attention layers need only
 *           the last W tokens; Q4: tiles wholly before the window are skipped).
 *
 *  split    pao_decode_partitions / pao_combine_partitions restate the same
 *           attention as per-partition (max, sum, unnormalised output)
 *           triples merged by rescaling with exp(m_p - M), the rescale rule of
 *           Q4's online softmax. They exist to pin the split-K identity.
 *
 * Layouts (row-major, element type = cache dtype):
 *   q, out         [num_seqs][num_heads][head_dim]     (out is fp64 here)
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim]
 *   k/v cache      [num_blocks][num_kv_heads][block_size][head_dim]
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs], counting the token appended this step
 * dtype: 0 = fp32, 1 = bf16 (raw 16-bit patterns), 2 = fp8 e4m3 (raw 8-bit
 * codes, caches only; see "fp8" above). Context length 0 gives a
 * zero output row (a reading: the pages say nothing about empty sequences).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PAO_OK 0
#define PAO_BAD_ARG (-1)
#define PAO_BAD_BLOCK (-2)
#define PAO_BAD_LEN (-3)
#define PAO_NO_MEMORY (-4)

/* The value of an e4m3 code (NaN for 0x7F and 0xFF). */
double pao_e4m3_decode(int code) {
    const int c = code & 0xFF;
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? -mag : mag;
}

/* Nearest e4m3 code of a binary32 value: round to nearest, ties to the even
 * code; |x| >= 448 gives +-448; NaN gives 0x7F. Within a binade of exponent
 * E (2^E <= |x| < 2^(E+1), E >= -6) the codes are spaced 2^(E-3); below 2^-6
 * they are spaced 2^-9 (subnormals). Rounding |x| / spacing to an integer q
 * then gives code (E + 7) * 8 + (q - 8), or q below 2^-6; q = 16 carries into
 * the next binade by the same formula. */
int pao_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    const int sign = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int ex;
    (void)frexp(a, &ex);                    /* a = f * 2^ex, f in [0.5, 1) */
    const int E = ex - 1;
    int code;
    if (a == 0.0 || E < -6) {
        code = (int)nearbyint(ldexp(a, 9));  /* exact quotient; ties to even */
    } else {
        const int q = (int)nearbyint(ldexp(a, 3 - E));
        code = (E + 7) * 8 + (q - 8);
    }
    return sign | code;
}

static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    if (dtype == 2) return pao_e4m3_decode(((const uint8_t*)base)[idx]);
    /* bf16: the 16 stored bits are the high half of an IEEE binary32. */
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int elem_bytes_of(int dtype) { return dtype == 0 ? 4 : dtype == 1 ? 2 : 1; }

/* Copy every new K/V row into its slot. Negative slots are skipped (padding);
 * a slot past the pool is skipped and counted. Returns that count. */
int pao_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
               void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
               int head_dim, int block_size, int num_blocks, int dtype) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || dtype < 0 || dtype > 2)
        return PAO_BAD_ARG;
    const size_t row = (size_t)head_dim * (size_t)elem_bytes_of(dtype);
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    int bad = 0;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { ++bad; continue; }
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * num_kv_heads + h) * row;
            const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row;
            memcpy((char*)k_cache + dst, (const char*)k_new + src, row);
            memcpy((char*)v_cache + dst, (const char*)v_new + src, row);
        }
    }
    return bad;
}

/* Copy-on-write: block dst of K and V becomes a copy of block src, for each
 * (src, dst) pair of block_mapping ([num_pairs][2]). A pair with a negative
 * entry is skipped; a pair with an entry >= num_blocks is skipped and
 * counted. Returns that count, or PAO_BAD_ARG. */
int pao_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int num_pairs,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || dtype < 0 || dtype > 2)
        return PAO_BAD_ARG;
    const size_t block_bytes =
        (size_t)num_kv_heads * block_size * head_dim * (size_t)elem_bytes_of(dtype);
    int bad = 0;
    for (int i = 0; i < num_pairs; ++i) {
        const int64_t src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || dst < 0) continue;
        if (src >= num_blocks || dst >= num_blocks) { ++bad; continue; }
        memmove((char*)k_cache + (size_t)dst * block_bytes,
                (const char*)k_cache + (size_t)src * block_bytes, block_bytes);
        memmove((char*)v_cache + (size_t)dst * block_bytes,
                (const char*)v_cache + (size_t)src * block_bytes, block_bytes);
    }
    return bad;
}

/* Per-row INT8 quantisation of one row of n binary32 values. */
static float quantize_row_int8(const float* x, int n, int8_t* codes) {
    float amax = 0.0f;
    for (int d = 0; d < n; ++d) {
        const float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    const float scale = amax / 127.0f;
    for (int d = 0; d < n; ++d) {
        if (scale == 0.0f) { codes[d] = 0; continue; }
        float c = nearbyintf(x[d] / scale);
        if (c > 127.0f) c = 127.0f;
        if (c < -127.0f) c = -127.0f;
        codes[d] = (int8_t)c;
    }
    return scale;
}

/* Append into an INT8 cache: codes [NB][Hkv][bs][D] int8, scales [NB][Hkv][bs]
 * fp32, one per (row, KV head), for K and for V. k_new/v_new in new_dtype (0
 * or 1). Returns the out-of-range slot count, or PAO_BAD_ARG. */
int pao_append_int8(const void* k_new, const void* v_new, int new_dtype,
                    const int64_t* slot_mapping, int8_t* k_cache, int8_t* v_cache,
                    float* k_scales, float* v_scales, int num_tokens, int num_kv_heads,
                    int head_dim, int block_size, int num_blocks) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || (new_dtype != 0 && new_dtype != 1))
        return PAO_BAD_ARG;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    float* row = (float*)malloc(sizeof(float) * (size_t)head_dim);
    if (!row) return PAO_NO_MEMORY;
    int bad = 0;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { ++bad; continue; }
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * num_kv_heads + h) * (size_t)head_dim;
            const size_t r = ((size_t)blk * num_kv_heads + h) * block_size + off;
            for (int d = 0; d < head_dim; ++d) row[d] = (float)load_elem(k_new, src + d, new_dtype);
            k_scales[r] = quantize_row_int8(row, head_dim, k_cache + r * head_dim);
            for (int d = 0; d < head_dim; ++d) row[d] = (float)load_elem(v_new, src + d, new_dtype);
            v_scales[r] = quantize_row_int8(row, head_dim, v_cache + r * head_dim);
        }
    }
    free(row);
    return bad;
}

/* Rebuild the contiguous K and V rows 0..n-1 of (seq, kv_head) as fp64. */
static int gather(const void* k_cache, const void* v_cache, const int32_t* table, int n,
                  int kv_head, int num_kv_heads, int head_dim, int block_size,
                  int num_blocks, int dtype, double k_scale, double v_scale, double* Kc,
                  double* Vc) {
    for (int i = 0; i < n; ++i) {
        const int32_t blk = table[i / block_size];
        if (blk < 0 || blk >= num_blocks) return PAO_BAD_BLOCK;
        const int off = i % block_size;
        const size_t base =
            (((size_t)blk * num_kv_heads + kv_head) * block_size + off) * (size_t)head_dim;
        for (int d = 0; d < head_dim; ++d) {
            Kc[(size_t)i * head_dim + d] = k_scale * load_elem(k_cache, base + d, dtype);
            Vc[(size_t)i * head_dim + d] = v_scale * load_elem(v_cache, base + d, dtype);
        }
    }
    return PAO_OK;
}

/* Softmax weights of one query against n contiguous keys: w_i = exp(S_i - M) / Z. */
static void softmax_weights(const double* qv, const double* Kc, int n, int head_dim,
                            double scale, double* w) {
    double M = -INFINITY;
    for (int i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qv[d] * Kc[(size_t)i * head_dim + d];
        w[i] = scale * dot;
        if (w[i] > M) M = w[i];
    }
    double Z = 0.0;
    for (int i = 0; i < n; ++i) {
        w[i] = exp(w[i] - M);
        Z += w[i];
    }
    for (int i = 0; i < n; ++i) w[i] /= Z;
}

static int check_shapes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, int max_blocks_per_seq, int dtype) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
        (dtype != 0 && dtype != 1) || num_heads % num_kv_heads != 0)
        return PAO_BAD_ARG;
    return PAO_OK;
}

/* Full decode attention. out: fp64 [num_seqs][num_heads][head_dim].
 * q in q_dtype (0 or 1); K and V in kv_dtype (0, 1 or 2), their values
 * multiplied by k_scale and v_scale. num_threads <= 0 lets OpenMP (when
 * compiled in) choose. */
int pao_decode_kv(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                  int kv_dtype, double k_scale, double v_scale, const int32_t* block_tables,
                  const int32_t* context_lens, double scale, double* out, int num_seqs,
                  int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                  int max_blocks_per_seq, int num_threads) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, q_dtype);
    if (rc != PAO_OK) return rc;
    if (kv_dtype < 0 || kv_dtype > 2) return PAO_BAD_ARG;
    const int G = num_heads / num_kv_heads;
    const int units = num_seqs * num_kv_heads;
    int err = PAO_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    const int nt = 1;
    (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int u = 0; u < units; ++u) {
        const int s = u / num_kv_heads, h = u % num_kv_heads;
        const int n = context_lens[s];
        if (n < 0 || (long)n > (long)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            err = PAO_BAD_LEN;
            continue;
        }
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* w = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!Kc || !Vc || !w || !qv) {
#pragma omp atomic write
            err = PAO_NO_MEMORY;
            free(Kc); free(Vc); free(w); free(qv);
            continue;
        }
        int grc = gather(k_cache, v_cache, block_tables + (size_t)s * max_blocks_per_seq, n, h,
                         num_kv_heads, head_dim, block_size, num_blocks, kv_dtype, k_scale,
                         v_scale, Kc, Vc);
        if (grc != PAO_OK) {
#pragma omp atomic write
            err = grc;
        }
        for (int g = 0; g < G; ++g) {
            const int qh = h * G + g;
            double* o = out + ((size_t)s * num_heads + qh) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n == 0 || grc != PAO_OK) continue;
            for (int d = 0; d < head_dim; ++d)
                qv[d] = load_elem(q, ((size_t)s * num_heads + qh) * head_dim + d, q_dtype);
            softmax_weights(qv, Kc, n, head_dim, scale, w);
            for (int i = 0; i < n; ++i)
                for (int d = 0; d < head_dim; ++d) o[d] += w[i] * Vc[(size_t)i * head_dim + d];
        }
        free(Kc); free(Vc); free(w); free(qv);
    }
    return err;
}

/* Multi-query decode. q: [num_seqs][num_queries][num_heads][head_dim] in
 * q_dtype; out: fp64, same shape. Query j of sequence s attends to rows
 * 0 .. n - num_queries + j (n = context_lens[s]). n == 0 gives zero rows;
 * 0 < n < num_queries is PAO_BAD_LEN (that sequence's rows are left zero). */
int pao_decode_multi(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                     int kv_dtype, double k_scale, double v_scale,
                     const int32_t* block_tables, const int32_t* context_lens, double scale,
                     double* out, int num_seqs, int num_queries, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                     int max_blocks_per_seq, int num_threads) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, q_dtype);
    if (rc != PAO_OK) return rc;
    if (kv_dtype < 0 || kv_dtype > 2 || num_queries < 1) return PAO_BAD_ARG;
    const int G = num_heads / num_kv_heads;
    const int Q = num_queries;
    const int units = num_seqs * num_kv_heads;
    int err = PAO_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    const int nt = 1;
    (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int u = 0; u < units; ++u) {
        const int s = u / num_kv_heads, h = u % num_kv_heads;
        const int n = context_lens[s];
        for (int j = 0; j < Q; ++j)
            for (int g = 0; g < G; ++g) {
                double* o = out + (((size_t)s * Q + j) * num_heads + h * G + g) * head_dim;
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            }
        if (n < 0 || (long)n > (long)max_blocks_per_seq * block_size || (n > 0 && n < Q)) {
#pragma omp atomic write
            err = PAO_BAD_LEN;
            continue;
        }
        if (n == 0) continue;
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* w = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!Kc || !Vc || !w || !qv) {
#pragma omp atomic write
            err = PAO_NO_MEMORY;
            free(Kc); free(Vc); free(w); free(qv);
            continue;
        }
        const int grc = gather(k_cache, v_cache, block_tables + (size_t)s * max_blocks_per_seq,
                               n, h, num_kv_heads, head_dim, block_size, num_blocks, kv_dtype,
                               k_scale, v_scale, Kc, Vc);
        if (grc != PAO_OK) {
#pragma omp atomic write
            err = grc;
        } else {
            for (int j = 0; j < Q; ++j) {
                const int rows = n - Q + j + 1;       /* rows 0 .. n - Q + j */
                for (int g = 0; g < G; ++g) {
                    const int qh = h * G + g;
                    const size_t qrow = ((size_t)s * Q + j) * num_heads + qh;
                    double* o = out + qrow * head_dim;
                    for (int d = 0; d < head_dim; ++d)
                        qv[d] = load_elem(q, qrow * head_dim + d, q_dtype);
                    softmax_weights(qv, Kc, rows, head_dim, scale, w);
                    for (int i = 0; i < rows; ++i)
                        for (int d = 0; d < head_dim; ++d) o[d] += w[i] * Vc[(size_t)i * head_dim + d];
                }
            }
        }
        free(Kc); free(Vc); free(w); free(qv);
    }
    return err;
}

/* Sliding-window decode: sequence s attends to rows max(0, n - window) ..
 * n - 1 (window >= 1). Same layouts and errors as pao_decode. */
int pao_decode_window(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, double scale,
                      int window, double* out, int num_seqs, int num_heads, int num_kv_heads,
                      int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                      int dtype, int num_threads) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, dtype);
    if (rc != PAO_OK) return rc;
    if (window < 1) return PAO_BAD_ARG;
    const int G = num_heads / num_kv_heads;
    const int units = num_seqs * num_kv_heads;
    int err = PAO_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    const int nt = 1;
    (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int u = 0; u < units; ++u) {
        const int s = u / num_kv_heads, h = u % num_kv_heads;
        const int n = context_lens[s];
        for (int g = 0; g < G; ++g) {
            double* o = out + ((size_t)s * num_heads + h * G + g) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        }
        if (n < 0 || (long)n > (long)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            err = PAO_BAD_LEN;
            continue;
        }
        if (n == 0) continue;
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* w = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!Kc || !Vc || !w || !qv) {
#pragma omp atomic write
            err = PAO_NO_MEMORY;
            free(Kc); free(Vc); free(w); free(qv);
            continue;
        }
        const int grc = gather(k_cache, v_cache, block_tables + (size_t)s * max_blocks_per_seq,
                               n, h, num_kv_heads, head_dim, block_size, num_blocks, dtype, 1.0,
                               1.0, Kc, Vc);
        if (grc != PAO_OK) {
#pragma omp atomic write
            err = grc;
        } else {
            const int first = n > window ? n - window : 0;   /* rows first .. n - 1 */
            const int rows = n - first;
            for (int g = 0; g < G; ++g) {
                const int qh = h * G + g;
                double* o = out + ((size_t)s * num_heads + qh) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    qv[d] = load_elem(q, ((size_t)s * num_heads + qh) * head_dim + d, dtype);
                softmax_weights(qv, Kc + (size_t)first * head_dim, rows, head_dim, scale, w);
                for (int i = 0; i < rows; ++i)
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += w[i] * Vc[(size_t)(first + i) * head_dim + d];
            }
        }
        free(Kc); free(Vc); free(w); free(qv);
    }
    return err;
}

/* Decode attention over an INT8 cache with per-row scales: K_i = k_scale_i *
 * code_i (fp64), same for V. q in q_dtype (0 or 1); out fp64. */
int pao_decode_int8(const void* q, int q_dtype, const int8_t* k_cache, const int8_t* v_cache,
                    const float* k_scales, const float* v_scales,
                    const int32_t* block_tables, const int32_t* context_lens, double scale,
                    double* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq, int num_threads) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, q_dtype);
    if (rc != PAO_OK) return rc;
    const int G = num_heads / num_kv_heads;
    const int units = num_seqs * num_kv_heads;
    int err = PAO_OK;
#ifdef _OPENMP
    const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    const int nt = 1;
    (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int u = 0; u < units; ++u) {
        const int s = u / num_kv_heads, h = u % num_kv_heads;
        const int n = context_lens[s];
        for (int g = 0; g < G; ++g) {
            double* o = out + ((size_t)s * num_heads + h * G + g) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        }
        if (n < 0 || (long)n > (long)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            err = PAO_BAD_LEN;
            continue;
        }
        if (n == 0) continue;
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* w = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!Kc || !Vc || !w || !qv) {
#pragma omp atomic write
            err = PAO_NO_MEMORY;
            free(Kc); free(Vc); free(w); free(qv);
            continue;
        }
        int grc = PAO_OK;
        const int32_t* table = block_tables + (size_t)s * max_blocks_per_seq;
        for (int i = 0; i < n && grc == PAO_OK; ++i) {
            const int32_t blk = table[i / block_size];
            if (blk < 0 || blk >= num_blocks) { grc = PAO_BAD_BLOCK; break; }
            const size_t r = ((size_t)blk * num_kv_heads + h) * block_size + i % block_size;
            for (int d = 0; d < head_dim; ++d) {
                Kc[(size_t)i * head_dim + d] = (double)k_scales[r] * (double)k_cache[r * head_dim + d];
                Vc[(size_t)i * head_dim + d] = (double)v_scales[r] * (double)v_cache[r * head_dim + d];
            }
        }
        if (grc != PAO_OK) {
#pragma omp atomic write
            err = grc;
        } else {
            for (int g = 0; g < G; ++g) {
                const int qh = h * G + g;
                double* o = out + ((size_t)s * num_heads + qh) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    qv[d] = load_elem(q, ((size_t)s * num_heads + qh) * head_dim + d, q_dtype);
                softmax_weights(qv, Kc, n, head_dim, scale, w);
                for (int i = 0; i < n; ++i)
                    for (int d = 0; d < head_dim; ++d) o[d] += w[i] * Vc[(size_t)i * head_dim + d];
            }
        }
        free(Kc); free(Vc); free(w); free(qv);
    }
    return err;
}

int pao_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, const int32_t* context_lens, double scale,
               double* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
               int block_size, int num_blocks, int max_blocks_per_seq, int dtype,
               int num_threads) {
    if (dtype != 0 && dtype != 1) return PAO_BAD_ARG;
    return pao_decode_kv(q, dtype, k_cache, v_cache, dtype, 1.0, 1.0, block_tables,
                         context_lens, scale, out, num_seqs, num_heads, num_kv_heads, head_dim,
                         block_size, num_blocks, max_blocks_per_seq, num_threads);
}

/* Append into an FP8 cache: code = e4m3(x / scale) for each new element x
 * (k_new, v_new in new_dtype 0 or 1; the division in fp32), into the slots as
 * pao_append. Returns the out-of-range slot count, or PAO_BAD_ARG. */
int pao_append_fp8(const void* k_new, const void* v_new, int new_dtype,
                   const int64_t* slot_mapping, uint8_t* k_cache, uint8_t* v_cache,
                   int num_tokens, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, float k_scale, float v_scale) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || (new_dtype != 0 && new_dtype != 1) || !(k_scale > 0.0f) ||
        !(v_scale > 0.0f))
        return PAO_BAD_ARG;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    int bad = 0;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { ++bad; continue; }
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)t * num_kv_heads + h) * (size_t)head_dim;
            const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                const float kx = (float)load_elem(k_new, src + d, new_dtype);
                const float vx = (float)load_elem(v_new, src + d, new_dtype);
                k_cache[dst + d] = (uint8_t)pao_e4m3_encode(kx / k_scale);
                v_cache[dst + d] = (uint8_t)pao_e4m3_encode(vx / v_scale);
            }
        }
    }
    return bad;
}

/* The normalised softmax weights of one (seq, query head): w[0..n-1]. */
int pao_attention_weights(const void* q, const void* k_cache, const int32_t* block_tables,
                          const int32_t* context_lens, double scale, int seq, int head,
                          double* w, int num_seqs, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, int dtype) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, dtype);
    if (rc != PAO_OK) return rc;
    if (seq < 0 || seq >= num_seqs || head < 0 || head >= num_heads) return PAO_BAD_ARG;
    const int G = num_heads / num_kv_heads, h = head / G;
    const int n = context_lens[seq];
    if (n <= 0 || (long)n > (long)max_blocks_per_seq * block_size) return PAO_BAD_LEN;
    double* Kc = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)n * head_dim);
    double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!Kc || !Vc || !qv) { free(Kc); free(Vc); free(qv); return PAO_NO_MEMORY; }
    /* V is gathered along with K and ignored: one gather routine for both. */
    rc = gather(k_cache, k_cache, block_tables + (size_t)seq * max_blocks_per_seq, n, h,
                num_kv_heads, head_dim, block_size, num_blocks, dtype, 1.0, 1.0, Kc, Vc);
    if (rc == PAO_OK) {
        for (int d = 0; d < head_dim; ++d)
            qv[d] = load_elem(q, ((size_t)seq * num_heads + head) * head_dim + d, dtype);
        softmax_weights(qv, Kc, n, head_dim, scale, w);
    }
    free(Kc); free(Vc); free(qv);
    return rc;
}

/* Per-partition state of the split form. Partition p of a sequence covers tokens
 * [p*P, min(n, (p+1)*P)). For each (seq, head, p) it stores
 *   m = max_i S_i,  l = sum_i exp(S_i - m),  o[d] = sum_i exp(S_i - m) V_i[d]
 * into m/l [num_seqs][num_heads][max_parts] and o [..][max_parts][head_dim].
 * Partitions past the sequence get m = -inf, l = 0, o = 0. */
int pao_decode_partitions(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          double scale, int partition_size, int max_parts, double* m,
                          double* l, double* o, int num_seqs, int num_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, int dtype) {
    int rc = check_shapes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, dtype);
    if (rc != PAO_OK) return rc;
    if (partition_size <= 0 || max_parts < 0) return PAO_BAD_ARG;
    const int G = num_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        const int n = context_lens[s];
        if (n < 0 || (long)n > (long)max_blocks_per_seq * block_size) return PAO_BAD_LEN;
        if ((long)n > (long)partition_size * max_parts) return PAO_BAD_ARG;
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)n * head_dim + 1));
        double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
        double* S = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        if (!Kc || !Vc || !qv || !S) { free(Kc); free(Vc); free(qv); free(S); return PAO_NO_MEMORY; }
        for (int h = 0; h < num_kv_heads && rc == PAO_OK; ++h) {
            rc = gather(k_cache, v_cache, block_tables + (size_t)s * max_blocks_per_seq, n, h,
                        num_kv_heads, head_dim, block_size, num_blocks, dtype, 1.0, 1.0, Kc, Vc);
            if (rc != PAO_OK) break;
            for (int g = 0; g < G; ++g) {
                const int qh = h * G + g;
                for (int d = 0; d < head_dim; ++d)
                    qv[d] = load_elem(q, ((size_t)s * num_heads + qh) * head_dim + d, dtype);
                for (int i = 0; i < n; ++i) {
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d) dot += qv[d] * Kc[(size_t)i * head_dim + d];
                    S[i] = scale * dot;
                }
                for (int p = 0; p < max_parts; ++p) {
                    const size_t mi = ((size_t)s * num_heads + qh) * max_parts + p;
                    double* op = o + mi * head_dim;
                    double mp = -INFINITY, lp = 0.0;
                    for (int d = 0; d < head_dim; ++d) op[d] = 0.0;
                    const int lo = p * partition_size;
                    const int hi = lo + partition_size < n ? lo + partition_size : n;
                    for (int i = lo; i < hi; ++i)
                        if (S[i] > mp) mp = S[i];
                    for (int i = lo; i < hi; ++i) {
                        const double e = exp(S[i] - mp);
                        lp += e;
                        for (int d = 0; d < head_dim; ++d) op[d] += e * Vc[(size_t)i * head_dim + d];
                    }
                    m[mi] = mp;
                    l[mi] = lp;
                }
            }
        }
        free(Kc); free(Vc); free(qv); free(S);
        if (rc != PAO_OK) return rc;
    }
    return PAO_OK;
}

/* Merge per-partition triples: M = max_p m_p, c_p = exp(m_p - M),
 * out = (sum_p c_p o_p) / (sum_p c_p l_p). parts[s] partitions are used for
 * sequence s; a sequence with none gets zeros. */
int pao_combine_partitions(const double* m, const double* l, const double* o,
                           const int32_t* parts, int max_parts, double* out, int num_seqs,
                           int num_heads, int head_dim) {
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_parts < 0) return PAO_BAD_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        if (parts[s] < 0 || parts[s] > max_parts) return PAO_BAD_ARG;
        for (int qh = 0; qh < num_heads; ++qh) {
            const size_t base = ((size_t)s * num_heads + qh) * max_parts;
            double* y = out + ((size_t)s * num_heads + qh) * head_dim;
            for (int d = 0; d < head_dim; ++d) y[d] = 0.0;
            if (parts[s] == 0) continue;
            double M = -INFINITY;
            for (int p = 0; p < parts[s]; ++p)
                if (m[base + p] > M) M = m[base + p];
            double L = 0.0;
            for (int p = 0; p < parts[s]; ++p) {
                const double c = exp(m[base + p] - M);
                L += c * l[base + p];
                for (int d = 0; d < head_dim; ++d) y[d] += c * o[(base + p) * head_dim + d];
            }
            for (int d = 0; d < head_dim; ++d) y[d] /= L;
        }
    }
    return PAO_OK;
}
