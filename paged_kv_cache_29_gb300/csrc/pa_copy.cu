// pa_copy.cu -- copy-on-write of whole cache blocks: for each (src, dst) pair,
// block dst of the K pool and of the V pool becomes a bit copy of block src
// (every KV head's block_size rows). A block shared by several sequences is
// copied before one of them appends into it ("MLSys Engineer -- Inference
// Systems Q&A", Q1, "Why this helps": copy-on-write sharing of blocks).
//
// One block of one pool is num_kv_heads * block_size * head_dim elements,
// contiguous in the [block][kv_head][block_size][head_dim] layout, so a pair
// is two contiguous copies. Threads take 16-byte chunks in a grid-stride loop
// over (pair, pool, chunk); consecutive threads touch consecutive chunks of
// one block, so both the read and the write are coalesced.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int64_t* __restrict__ block_mapping, long long total_chunks,
                   long long chunks_per_block, long long num_blocks, int32_t* error_word) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < total_chunks; i += stride) {
        const long long per_pair = 2 * chunks_per_block;
        const long long pair = i / per_pair;
        const long long rem = i - pair * per_pair;
        const bool is_v = rem >= chunks_per_block;
        const long long c = is_v ? rem - chunks_per_block : rem;
        const long long src = __ldg(block_mapping + 2 * pair);
        const long long dst = __ldg(block_mapping + 2 * pair + 1);
        if (src < 0 || dst < 0) continue;
        if (src >= num_blocks || dst >= num_blocks) {
            if (rem == 0) raise_error(error_word, PA_DEVERR_BLOCK_ID);
            continue;
        }
        uint4* pool = is_v ? v_cache : k_cache;
        pool[dst * chunks_per_block + c] = pool[src * chunks_per_block + c];
    }
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                               int num_pairs, long long block_bytes, int num_blocks,
                               int32_t* error_word, cudaStream_t stream) {
    const long long chunks_per_block = block_bytes / 16;
    const long long total = 2LL * num_pairs * chunks_per_block;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + kCopyThreads - 1) / kCopyThreads;
    if (blocks > 8192) blocks = 8192;   // grid-stride beyond
    copy_blocks_kernel<<<static_cast<unsigned>(blocks), kCopyThreads, 0, stream>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_mapping, total,
        chunks_per_block, num_blocks, error_word);
    return cudaGetLastError();
}

}  // namespace pa
