// pa_append.cu -- the cache append (reshape_and_cache): each token's new K and
// V row is copied into slot_mapping[t] of the paged pool,
//   cache[slot / block_size][kv_head][slot % block_size][:] = new[t][kv_head][:],
// the flat-slot form of the paged indexing of "MLSys Engineer -- Inference
// Systems Q&A", Q1, and the cache append that precedes attention in the naive
// incremental decoder of "LLM inference and serving". A bit copy in 16-byte
// vectors: one thread per 16-byte chunk of one (token, KV head) row, K and V
// both. The read of k_new/v_new and the write into the pool are each one
// coalesced pass over the row.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
              const int64_t* __restrict__ slot_mapping, uint4* __restrict__ k_cache,
              uint4* __restrict__ v_cache, long long total_chunks, int chunks_per_row,
              int num_kv_heads, int block_size, long long num_slots, int32_t* error_word) {
    // A decode call launched next on the stream may start its set-up now; it
    // waits for this grid to finish before reading the cache.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < total_chunks; i += stride) {
        const long long rowi = i / chunks_per_row;           // (token, kv head)
        const int c = static_cast<int>(i - rowi * chunks_per_row);
        const long long t = rowi / num_kv_heads;
        const int h = static_cast<int>(rowi - t * num_kv_heads);
        const long long slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (c == 0 && h == 0) raise_error(error_word, PA_DEVERR_SLOT);
            continue;
        }
        const long long blk = slot / block_size;
        const long long off = slot - blk * block_size;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        k_cache[dst] = __ldg(k_new + i);
        v_cache[dst] = __ldg(v_new + i);
    }
}

}  // namespace

cudaError_t launch_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                          int row_bytes, int block_size, int num_blocks, int32_t* error_word,
                          cudaStream_t stream) {
    const int chunks_per_row = row_bytes / 16;
    const long long total = static_cast<long long>(num_tokens) * num_kv_heads * chunks_per_row;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 8192) blocks = 8192;
    append_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), total, chunks_per_row,
        num_kv_heads, block_size, static_cast<long long>(num_blocks) * block_size, error_word);
    return cudaGetLastError();
}

}  // namespace pa
