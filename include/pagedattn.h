/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode library.
 *
 * One decode step of paged attention is two calls on one CUDA stream
 * (three when a shared block must first be copied, pa_copy_blocks):
 *
 *   pa_reshape_and_cache  writes each sequence's new K and V row into its slot
 *                         of the paged pool (the cache append of the naive
 *                         incremental decoder in "LLM inference and serving",
 *                         "Code from memory");
 *   pa_decode             single-query attention for every sequence, reading K
 *                         and V through the sequence's block table
 *                         ("MLSys Engineer -- Inference Systems Q&A", Q1 "How
 *                         does PagedAttention work?": row i of a sequence is
 *                         row i % block_size of physical block
 *                         block_table[i / block_size]).
 *
 * Data layouts (row-major; "T" is the cache dtype, fp32 or bf16):
 *   k_cache, v_cache  T [num_blocks][num_kv_heads][block_size][head_dim]
 *   k_new, v_new      T [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping      int64 [num_tokens]; slot = block * block_size + offset,
 *                     a negative slot means "no append for this token"
 *   q, out            T [num_seqs][num_heads][head_dim]
 *   block_tables      int32 [num_seqs][max_blocks_per_seq]; entries past
 *                     ceil(context_len / block_size) are never read
 *   context_lens      int32 [num_seqs]; the number of rows attended, counting
 *                     the row appended this step (0 gives a zero output row)
 * Query head qh uses KV head qh / (num_heads / num_kv_heads): consecutive
 * groups of query heads share one KV head ("LLM inference and serving", Q7
 * "What are MQA and GQA").
 *
 * Ownership and synchronisation: every pointer is a device pointer owned by
 * the caller. The library allocates no memory and keeps no state between
 * calls beyond cached driver entry points and kernel attributes. Calls only
 * enqueue work on `stream` (NULL = legacy default stream) and return without
 * waiting for it.
 *
 * Errors: invalid arguments are rejected on the host before anything is
 * enqueued, with a pa_status and no side effects. Problems only visible on
 * the device (a block-table entry outside the pool, a slot past the pool, a
 * context length past the block table, a wait that hit its time limit) are
 * OR-ed into *error_word (an int32 in device memory, may be NULL) as
 * PA_DEVERR_* bits; the affected sequence or token is skipped and nothing
 * outside the caller's buffers is touched. The kernels never trap.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer, ... */
    PA_ERR_UNSUPPORTED = 2,  /* a valid shape this build has no kernel for */
    PA_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned */
    PA_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed */
    PA_ERR_DEVICE_BOUNDS = 5 /* returned by pa_check_error_word: PA_DEVERR_* set */
} pa_status;

/* Element types. PA_DTYPE_FP8_E4M3 is a cache type only: each element is an
 * 8-bit e4m3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * subnormals, largest finite 448, 0x7F/0xFF NaN) and the cached value is
 * scale * e4m3(code) with one scale per tensor (pa_reshape_and_cache_fp8,
 * pa_decode_fp8). An FP8 cache halves the bytes per token ("Forward Deployed
 * Engineering Interview", Chapter 2 "Batching and the KV Cache": FP8 KV, scales
 * per tensor, 1.0 when uncalibrated). */
typedef enum pa_dtype {
    PA_DTYPE_F32 = 0,
    PA_DTYPE_BF16 = 1,
    PA_DTYPE_FP8_E4M3 = 2,
    PA_DTYPE_INT8 = 3 /* cache type only: int8 codes with one fp32 scale per (row, KV head);
                         pa_reshape_and_cache_int8, pa_decode_int8 */
} pa_dtype;

/* Bits the kernels OR into *error_word. */
#define PA_DEVERR_BLOCK_ID 0x1  /* a block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 0x2      /* a slot >= num_blocks * block_size */
#define PA_DEVERR_CONTEXT 0x4   /* context_len < 0, or > max_context_len, or past the table */
#define PA_DEVERR_TIMEOUT 0x8   /* a shared-memory barrier wait gave up after its limit */

/*
 * Append one K and one V row per token into the paged pool:
 *   k_cache[s / bs][h][s % bs][:] = k_new[t][h][:]   (same for V), s = slot_mapping[t]
 * for every t with s >= 0 and every KV head h. A bit copy: no rounding.
 * Tokens with s >= num_blocks * block_size are skipped and flagged
 * PA_DEVERR_SLOT. Two tokens with the same slot race (last writer wins).
 * head_dim * sizeof(T) must be a multiple of 16 and every buffer 16-byte
 * aligned. dtype may be PA_DTYPE_FP8_E4M3 (k_new/v_new then hold codes,
 * copied as they are). Returns PA_OK or an error; never blocks.
 */
pa_status pa_reshape_and_cache(const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               int num_tokens, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, pa_dtype dtype,
                               int32_t* error_word, struct CUstream_st* stream);

/*
 * Quantising append into an FP8 (e4m3) cache:
 *   k_cache[s / bs][h][s % bs][d] = e4m3(k_new[t][h][d] / k_scale)   (same for V)
 * with the division in fp32 (IEEE, round to nearest) and the conversion
 * rounding to the nearest e4m3 value, ties to even, saturating at +-448.
 * k_new, v_new: new_dtype (PA_DTYPE_F32 or PA_DTYPE_BF16) [num_tokens]
 * [num_kv_heads][head_dim]; k_cache, v_cache: uint8 codes
 * [num_blocks][num_kv_heads][block_size][head_dim]. Scales > 0 and finite.
 * Slots as in pa_reshape_and_cache; head_dim a multiple of 16; buffers
 * 16-byte aligned. Returns PA_OK or an error; never blocks.
 */
pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                                   const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                   int num_tokens, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, float k_scale, float v_scale,
                                   int32_t* error_word, struct CUstream_st* stream);

/*
 * Quantising append into an INT8 cache with one scale per (row, KV head)
 * ("MLSys Engineer -- Inference Systems Q&A", Q3: INT8 KV with per-token
 * scaling, scale = max(|K_row|) / 127):
 *   scale = max_d |x[d]| / 127,  code[d] = round_half_even(x[d] / scale)
 * for the new K row x = k_new[t][h] (and V), both divisions in fp32 (IEEE),
 * codes clamped to [-127, 127]; an all-zero row gets scale 0 and codes 0.
 * k_cache, v_cache: int8 [num_blocks][num_kv_heads][block_size][head_dim];
 * k_scales, v_scales: fp32 [num_blocks][num_kv_heads][block_size], 16-byte
 * aligned. k_new, v_new: new_dtype (PA_DTYPE_F32 or PA_DTYPE_BF16). head_dim
 * 16..256, a multiple of 16. Slots as in pa_reshape_and_cache.
 */
pa_status pa_reshape_and_cache_int8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                                    const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                    float* k_scales, float* v_scales, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int32_t* error_word,
                                    struct CUstream_st* stream);

/*
 * pa_decode over an INT8 cache with per-row scales, bf16 q and out:
 *   K_i = k_scales[row i] * code(K_i), V_i likewise, then the pa_decode sum.
 * Codes are widened to f16 in registers (exact) and multiplied on tensor
 * cores with fp32 accumulation; each score row is multiplied by its K scale
 * and each probability by its V scale before the P.V product. Same
 * partitioning, merge, workspace and error behaviour as pa_decode. Supported:
 * head_dim 128, block_size a multiple of 16, 1, 2, 4 or 8 query heads per KV
 * head (else PA_ERR_UNSUPPORTED).
 */
pa_status pa_decode_int8(const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scales, const float* v_scales,
                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                         void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, int max_blocks_per_seq,
                         int max_context_len, void* workspace, size_t workspace_bytes,
                         int32_t* error_word, struct CUstream_st* stream);

/*
 * Copy-on-write of whole blocks: for each pair i,
 *   k_cache[dst][:][:][:] = k_cache[src][:][:][:]   (same for V),
 *   src = block_mapping[2 i], dst = block_mapping[2 i + 1],
 * every KV head's block_size rows, bit for bit. A block shared by several
 * sequences (after a fork, or a shared prompt prefix) is copied before one of
 * them appends into it ("MLSys Engineer -- Inference Systems Q&A", Q1, "Why
 * this helps": copy-on-write sharing). block_mapping is int64 [num_pairs][2]
 * in device memory, 8-byte aligned. A pair with a negative entry is skipped;
 * a pair with an entry >= num_blocks is skipped and flagged PA_DEVERR_BLOCK_ID.
 * Destinations must be distinct and no destination may be a source of
 * another pair in the same call (such pairs race). head_dim * sizeof(T) must
 * be a multiple of 16 and the pools 16-byte aligned. Returns PA_OK or an
 * error; never blocks. For an INT8 cache (dtype PA_DTYPE_INT8) this copies
 * the codes; copy the row scales with a second call on the two scale arrays
 * viewed as fp32 pools of one KV head, one row and num_kv_heads * block_size
 * values per block (num_kv_heads * block_size a multiple of 4).
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                         int num_pairs, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, pa_dtype dtype, int32_t* error_word,
                         struct CUstream_st* stream);

/*
 * Decode attention for num_seqs sequences:
 *   out[s][qh][:] = sum_i softmax_i(scale * <q[s][qh], K_i>) * V_i[:]
 * over the context_lens[s] rows of sequence s (K_i, V_i gathered through
 * block_tables[s]), accumulated in fp32, stored in the cache dtype with
 * round-to-nearest-even.
 *
 * Long sequences are split into fixed partitions of 512 rows (1024 over the
 * FP8 caches of pa_decode_fp8: the same bytes per partition;
 * pa_default_partition_size) whose partial
 * results (running max, sum and unnormalised output, the online-softmax state
 * of Q4 "How would you write a fused attention kernel?") are merged by a
 * second kernel. Partition boundaries and the merge order depend only on the
 * sequence's own length, so a sequence's result does not depend on the rest
 * of the batch.
 *
 * max_context_len: an upper bound on every context_lens[s] (sizes the work
 *   list and the workspace); must not exceed max_blocks_per_seq * block_size.
 * workspace: device scratch of at least
 *   pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len)
 *   bytes, 16-byte aligned (non-zero for any non-empty batch: it holds the
 *   call's work list, and the partition partials when a sequence can span
 *   more than one partition). Its contents on entry do not matter; calls that
 *   share one workspace must not overlap on the GPU.
 * Supported: fp32 and bf16; any block_size >= 1; head_dim 1..256; any
 * num_heads that is a multiple of num_kv_heads. The fastest kernels need
 * block_size a multiple of 16, head_dim 64 or 128 and at most 8 query heads
 * per KV head; other shapes run a plain kernel that loads through the block
 * table directly.
 */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq,
                    int max_context_len, pa_dtype dtype, void* workspace,
                    size_t workspace_bytes, int32_t* error_word, struct CUstream_st* stream);

/*
 * pa_append_decode -- one decode step in one call: pa_reshape_and_cache of one
 * new token per sequence followed by pa_decode (the token is the last of the
 * context_lens[s] rows attended), as in the naive decoder of "MLSys Engineer
 * -- Inference Systems Q&A", Q1: append the step's K and V, then attend over
 * every cached row including them.
 *
 * k_new, v_new: [num_seqs][num_kv_heads][head_dim] in `dtype` (device,
 *   16-byte aligned); slot_mapping: int64 [num_seqs], slot_mapping[s] the slot
 *   of row context_lens[s] - 1 of sequence s, i.e.
 *   block_tables[s][(n - 1) / block_size] * block_size + (n - 1) % block_size,
 *   or negative (nothing appended for s). Every other argument as pa_decode.
 * The tile-ring kernels write each new row from the CTA that attends to the
 * sequence's last partition, just before it loads that tile: no separate
 * append kernel, no extra pass over HBM. Other shapes run pa_reshape_and_cache's
 * kernel, then pa_decode's plain kernel. Results (cache bytes and output) are
 * those of the two calls in sequence.
 * Errors: host checks as pa_reshape_and_cache and pa_decode. A slot that is
 * non-negative but not the slot of row n - 1 (or of an empty sequence) sets
 * PA_DEVERR_SLOT in error_word and is not written (fused path; the unfused
 * path writes any slot inside the pool, as pa_reshape_and_cache does).
 * Supported dtypes: fp32 and bf16 (one query token per sequence).
 */
pa_status pa_append_decode(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           void* k_cache, void* v_cache, const void* q,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, int32_t* error_word,
                           struct CUstream_st* stream);

/*
 * pa_append_decode over an FP8 (e4m3) cache (pa_reshape_and_cache_fp8 of one
 * bf16 row per sequence, then pa_decode_fp8) and over an INT8 cache with row
 * scales (pa_reshape_and_cache_int8, then pa_decode_int8). The rows are
 * quantised by the decode kernel with the append kernels' arithmetic (codes
 * and scales bit-identical to theirs) before the tiles that hold them load.
 * k_new, v_new: bf16 [num_seqs][num_kv_heads][head_dim]; slot_mapping as in
 * pa_append_decode; every other argument as the decode call.
 */
pa_status pa_append_decode_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               void* k_cache, void* v_cache, float k_scale, float v_scale,
                               const void* q, const int32_t* block_tables,
                               const int32_t* context_lens, float scale, void* out, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, int max_blocks_per_seq, int max_context_len,
                               void* workspace, size_t workspace_bytes, int32_t* error_word,
                               struct CUstream_st* stream);
pa_status pa_append_decode_int8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                const void* q, const int32_t* block_tables,
                                const int32_t* context_lens, float scale, void* out, int num_seqs,
                                int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, int max_blocks_per_seq, int max_context_len,
                                void* workspace, size_t workspace_bytes, int32_t* error_word,
                                struct CUstream_st* stream);

/*
 * pa_decode over an FP8 (e4m3) cache with bf16 q and out:
 *   out[s][qh][:] = sum_i softmax_i(scale * <q, k_scale * e4m3(K_i)>) * v_scale * e4m3(V_i)[:]
 * The codes are widened to f16 in registers (exact) and multiplied on tensor
 * cores with fp32 accumulation; q * scale * k_scale is rounded to f16 once per
 * sequence and KV head. Same partitioning, merge, workspace
 * (pa_decode_workspace_size) and error behaviour as pa_decode. Supported:
 * head_dim 128, block_size a multiple of 16, 1, 2, 4 or 8 query heads per KV
 * head (else PA_ERR_UNSUPPORTED). Scales > 0 and finite.
 */
pa_status pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        float k_scale, float v_scale, void* out, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        int max_blocks_per_seq, int max_context_len, void* workspace,
                        size_t workspace_bytes, int32_t* error_word,
                        struct CUstream_st* stream);

/* pa_decode_fp8 with explicit options (NULL = defaults; declared below):
 * kernel PA_KERNEL_AUTO, PA_KERNEL_MMA (the tile ring with per-tile mma.sync
 * on codes widened to f16) or PA_KERNEL_TC (tcgen05: 128-row chunks, e4m3
 * products straight from the TMA-staged codes, q and the probabilities as
 * three e4m3 terms each, accumulators in tensor memory); partition options as
 * pa_decode_ex. */
struct pa_decode_options;
pa_status pa_decode_fp8_ex(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens, float scale,
                           float k_scale, float v_scale, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, void* workspace,
                           size_t workspace_bytes, int32_t* error_word,
                           const struct pa_decode_options* options, struct CUstream_st* stream);

/*
 * Multi-query decode: num_queries (Q) new tokens per sequence verified
 * together, as speculative decoding does ("MLSys Engineer -- Inference Systems
 * Q&A", Q6: verifying K draft tokens in one pass costs about one decode's
 * bandwidth; Q2, phase 3: each draft token attends only to its ancestors).
 * The last Q of a sequence's n = context_lens[s] rows are the new tokens
 * (appended beforehand, e.g. by pa_reshape_and_cache with Q tokens per
 * sequence); query token j (0-based) sits at row n - Q + j and attends to
 * rows 0 .. n - Q + j:
 *   out[s][j][qh][:] = sum_{i <= n-Q+j} softmax_i(scale * <q[s][j][qh], K_i>) * V_i[:]
 * q, out: [num_seqs][num_queries][num_heads][head_dim], bf16 (dtype must be
 * PA_DTYPE_BF16). Each sequence's K/V rows are read once for all its query
 * tokens. 0 < n < Q is flagged PA_DEVERR_CONTEXT (those rows are left
 * unspecified); n == 0 gives zero rows. Workspace:
 * pa_decode_workspace_size_multi. Supported: head_dim 64 or 128, block_size a
 * multiple of 16, (num_heads / num_kv_heads) * num_queries <= 8 (else
 * PA_ERR_UNSUPPORTED); 1 <= num_queries <= 8. Same merge order and batch
 * invariance as pa_decode.
 */
pa_status pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          void* out, int num_seqs, int num_queries, int num_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                          void* workspace, size_t workspace_bytes, int32_t* error_word,
                          struct CUstream_st* stream);

size_t pa_decode_workspace_size_multi(int num_seqs, int num_queries, int num_heads,
                                      int head_dim, int max_context_len);

/*
 * Sliding-window decode: pa_decode where sequence s attends only to its last
 * `window` rows, max(0, n - window) .. n - 1 (n = context_lens[s]), as
 * local-attention layers do ("MLSys Engineer -- Inference Systems Q&A", Q3:
 * local layers need only the last W tokens; Q4: tiles wholly before the
 * window are never loaded). Partitions start at the 16-row tile holding the
 * window's first row, so only about window rows per sequence are read.
 * window >= 1 (window >= n attends to every row, as pa_decode). Same
 * arguments, layouts, workspace (pa_decode_workspace_size is enough) and
 * error behaviour as pa_decode; fp32 or bf16; block_size a multiple of 16,
 * head_dim 64 or 128 and 1, 2, 4 or 8 query heads per KV head (else
 * PA_ERR_UNSUPPORTED).
 */
pa_status pa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, int window, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, int32_t* error_word,
                           struct CUstream_st* stream);

/* Bytes of workspace pa_decode needs for these sizes (0 only for an empty
 * batch). */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len);

/*
 * pa_decode_noalloc -- pa_decode without a workspace argument. The pages have
 * no counterpart to this call: it exists for callers that cannot hand the
 * library a scratch buffer. A host program that links only this library and
 * the CUDA runtime may have no device allocator of its own to size one per
 * batch shape; a server that reserves almost all device memory for the paged
 * pool when it starts may have no room left to allocate per call, and a
 * cudaMalloc/cudaFree pair per step would stall its decode loop, because
 * cudaFree waits for the device to go idle.
 *
 * Same arguments, layouts and results as pa_decode (same kernels, same
 * partitioning). The scratch is a device array of PA_NOALLOC_SCRATCH_BYTES
 * inside the library, created by the CUDA runtime on each device where the
 * library's modules are loaded; no call allocates device or host memory.
 *   - Requests whose pa_decode_workspace_size(num_seqs, num_heads, head_dim,
 *     max_context_len) exceeds PA_NOALLOC_SCRATCH_BYTES return
 *     PA_ERR_WORKSPACE before anything is enqueued; use pa_decode with a
 *     caller-provided workspace for those.
 *   - The first call on a device looks up the scratch's address there (with
 *     that device current) and caches it: make that first call before any
 *     stream capture on that device. The cached address is that of the
 *     device's context at the time: no call may follow a cudaDeviceReset of
 *     that device in the same process.
 *   - There is ONE scratch per device. Calls whose work may overlap on the
 *     GPU (other streams, other host threads, or another pa_decode_noalloc
 *     call on a stream not ordered after this one) race on it and give wrong
 *     results. Calls on one stream are ordered and safe.
 * Returns PA_ERR_CUDA if the scratch's address cannot be obtained.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            float scale, void* out, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                            int32_t* error_word, struct CUstream_st* stream);

/* Kernel choice for pa_decode_ex (for measurement and tests; pa_decode uses
 * PA_KERNEL_AUTO). PA_KERNEL_MMA needs bf16. */
typedef enum pa_kernel {
    PA_KERNEL_AUTO = 0,
    PA_KERNEL_SIMT = 1,    /* TMA tile ring, CUDA-core dot products */
    PA_KERNEL_MMA = 2,     /* TMA tile ring, per-tile tensor-core MMA (mma.sync) */
    PA_KERNEL_GENERIC = 3, /* direct loads through the block table */
    PA_KERNEL_TC = 4       /* FP8 caches only: 128-row chunks on the tcgen05 tensor cores
                              (e4m3 x e4m3, accumulators in tensor memory) */
} pa_kernel;

typedef struct pa_decode_options {
    int kernel;          /* a pa_kernel value */
    int partition_size;  /* rows per split-K partition: a multiple of 16, 16..4096;
                            0 = pa_default_partition_size(dtype) */
    /* Optional larger partitions for long sequences: a sequence whose
     * partitions cover more than long_partition_from rows (its context length,
     * or for a sliding window the rows from the tile holding the window's
     * first row) is split into partitions of long_partition_size rows (a
     * multiple of 16, partition_size..4096). The choice depends on the
     * sequence's own length only, so its result stays independent of the rest
     * of the batch. 0 (the default) = one partition size for all. Measured on
     * the bench workloads it is no faster: fewer, larger items balance worse
     * across the persistent CTAs than they save in per-item work. */
    int long_partition_size;
    int long_partition_from;
} pa_decode_options;

/* pa_decode with explicit options (NULL = defaults). The workspace must be
 * sized with pa_decode_workspace_size_ex for the same partition size. */
pa_status pa_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, float scale,
                       void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_seq,
                       int max_context_len, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* error_word,
                       const pa_decode_options* options, struct CUstream_st* stream);

size_t pa_decode_workspace_size_ex(int num_seqs, int num_heads, int head_dim,
                                   int max_context_len, int partition_size);

/*
 * Failure test of the bounded waits (not for production use): pa_decode (or,
 * with dtype PA_DTYPE_FP8_E4M3, pa_decode_fp8 with unit scales) where CTA 0 of
 * the tile-ring decode kernel announces tile `withhold_tile` (>= 0) of its own
 * stream to its consumer but neither copies it nor completes its barrier.
 * Nothing faults and nothing waits without limit: the consumer's wait gives
 * up after about 2 s, the kernel sets PA_DEVERR_TIMEOUT in error_word
 * (required, device memory), its warps wind down and the call completes; the
 * output is unspecified. The CUDA context stays usable, and a following call
 * is exact. If CTA 0 streams fewer tiles, nothing is withheld. Returns
 * PA_ERR_INVALID_ARG for a negative withhold_tile or a null error_word, else
 * as pa_decode.
 */
pa_status pa_test_withhold_tile(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, void* out, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                                void* workspace, size_t workspace_bytes, int32_t* error_word,
                                int withhold_tile, struct CUstream_st* stream);

/* Human-readable name of a status. Never NULL. */
const char* pa_status_string(pa_status status);

/* PA_OK if error_word (host copy) is 0, else PA_ERR_DEVICE_BOUNDS. */
pa_status pa_check_error_word(int32_t error_word_value);

/* Library version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Rows per split-K partition the decode calls use for a cache of this type
 * when none is requested: 512 for fp32, bf16 and INT8, 1024 for FP8 (the same
 * bytes per partition as 512 bf16 rows). 0 for a type no cache holds. The
 * workspace size functions assume 512, which covers every case. */
int pa_default_partition_size(pa_dtype cache_dtype);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
