// pa_internal.h -- parameters and launchers shared between the host API and
// the kernel translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

namespace pa {

// Everything a decode kernel needs besides the tensor maps.
struct DecodeParams {
    const void* q;                 // [B][Hq][D], cache dtype
    void* out;                     // [B][Hq][D], cache dtype
    const void* k_cache;           // raw pool pointers (the generic kernel reads them directly)
    const void* v_cache;
    const int32_t* block_tables;   // [B][max_blocks_per_seq]
    const int32_t* context_lens;   // [B]
    float* part_o;                 // [B][Hq][max_parts][D] unnormalised partial outputs
    float* part_ml;                // [B][Hq][max_parts][2] (running max in log2 units, sum)
    int4* items;                   // work items (sequence, KV head, partition, context length)
    // Fused append (pa_append_decode; in-order stream kernels): each
    // sequence's new K and V rows [B][Hkv][D] (cache dtype) and their slots,
    // written by the CTA that loads them; null otherwise.
    const void* k_new;
    const void* v_new;
    const int64_t* slot_mapping;
    int32_t* error_word;           // nullable
    float scale_log2;              // scale * log2(e): scores are kept in base 2
    float k_scale;                 // FP8 caches: K value = k_scale * e4m3(code) (else 1)
    float v_scale;                 // FP8 caches: V value = v_scale * e4m3(code) (else 1)
    const float* k_row_scales;     // INT8 caches: [num_blocks][num_kv_heads][block_size] (else null)
    const float* v_row_scales;
    int num_seqs;
    int num_queries;               // query tokens per sequence, the last rows of each (>= 1)
    int window;                    // sliding window: attend to the last `window` rows (0 = all)
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int num_blocks;
    int max_blocks_per_seq;
    int context_cap;               // min(max_context_len, max_blocks_per_seq * block_size)
    int partition_size;            // rows per partition (seq_partition: of shorter sequences)
    int partition_long;            // rows per partition of sequences past partition_long_from
    int partition_long_from;       // span (rows from seq_row_base) above which partition_long applies
    int max_parts;                 // ceil(max_context_len / partition_size), >= 1: the partials' row stride
    // Failure test only (-1 otherwise): the tile-ring kernels' CTA 0 announces
    // its stream tile withhold_tile without copying it or completing its
    // barrier, so the consumer's bounded wait expires.
    int withhold_tile = -1;
};

// Launch result: cudaSuccess or the launch error.
cudaError_t launch_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                          int row_bytes, int block_size, int num_blocks, int32_t* error_word,
                          cudaStream_t stream);

// Copy-on-write block copies (block_bytes: one block of one pool, a multiple of 16).
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                               int num_pairs, long long block_bytes, int num_blocks,
                               int32_t* error_word, cudaStream_t stream);

// Persistent tile-ring kernels (one launch per call, sm_count SMs).
// Return cudaErrorNotSupported for shapes without an instance.
cudaError_t launch_decode_mma(const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, int sm_count, cudaStream_t stream);
cudaError_t launch_decode_simt(const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, pa_dtype dtype, int sm_count,
                               cudaStream_t stream);
bool has_tma_instance(pa_kernel kernel, pa_dtype dtype, int head_dim, int group,
                      int num_queries);

// FP8 (e4m3) cache, bf16 q/out: tensor-core tile math (head dim 128; 1, 2, 4
// or 8 query heads per KV head).
cudaError_t launch_decode_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, int sm_count, cudaStream_t stream);
bool has_fp8_instance(int head_dim, int group);

// FP8 (e4m3) cache on the tcgen05 tensor cores: 128-row chunks, e4m3 MMAs
// from the TMA-staged codes, accumulators in tensor memory (head dim 128; 1,
// 2, 4 or 8 query heads per KV head; one query token, no window).
cudaError_t launch_decode_fp8_tc(const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeParams& p, int sm_count, cudaStream_t stream);

// INT8 cache with per-row scales, bf16 q/out (head dim 128; 1, 2, 4 or 8
// query heads per KV head).
cudaError_t launch_decode_int8(const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int sm_count, cudaStream_t stream);

// Quantising append into an INT8 cache: one scale per (row, KV head).
cudaError_t launch_append_int8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               float* k_scales, float* v_scales, int num_tokens,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int32_t* error_word, cudaStream_t stream);

// Quantising append into an FP8 cache (new rows fp32 or bf16).
cudaError_t launch_append_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                              const int64_t* slot_mapping, void* k_cache, void* v_cache,
                              int num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float k_scale, float v_scale, int32_t* error_word,
                              cudaStream_t stream);

constexpr int kPlanMaxSeqs = 4096;   // sequences per persistent decode launch

// Direct-load kernel for any block size and head dim <= 256.
cudaError_t launch_decode_generic(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream);
size_t generic_smem_bytes(int group, int head_dim, int partition_size, int block_size);

// Merge of partition partials for sequences longer than one partition.
cudaError_t launch_combine(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream);

// Rows per partition of a sequence whose partitions cover `span` rows (its
// rows from seq_row_base on): partition_size, or partition_long for spans
// above partition_long_from. A function of the sequence's own length, so a
// sequence's partition boundaries and merge order never depend on the rest of
// the batch.
__host__ __device__ inline int seq_partition(const DecodeParams& p, int span) {
    return span > p.partition_long_from ? p.partition_long : p.partition_size;
}

// First row of a sequence's partitions: 0, or with a sliding window of W rows
// the window's first row rounded down to a 16-row tile (partition p covers
// rows base + p * partition_size ..). Depends only on n and W.
__host__ __device__ inline int seq_row_base(int n, int window) {
    return (window > 0 && n > window) ? ((n - window) / 16) * 16 : 0;
}

constexpr int kMaxHeadDim = 256;
constexpr int kMaxDevices = 64;      // devices whose per-kernel launch set-up is cached
constexpr int kDefaultPartition = 512;
// FP8 caches: twice the rows, the same bytes per partition as 512 bf16 rows
// (fewer items, merges and partials for the same traffic; faster on large and
// small batches alike). INT8 and multi-token calls keep 512: with fewer items
// than CTAs a small batch waits for its largest item, and there 1024 rows
// measured slower.
constexpr int kDefaultPartition8 = 1024;
constexpr int kNoLongPartitions = 0x7fffffff;   // partition_long_from: one size for all
// Kernel of pa_decode_fp8 and pa_append_decode_fp8 when none is requested.
constexpr pa_kernel kFp8DefaultKernel = PA_KERNEL_MMA;

}  // namespace pa
