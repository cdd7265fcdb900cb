// pa_noalloc.cu -- pa_decode_noalloc: pa_decode with the library's own
// fixed-size device scratch in place of a caller-provided workspace.
//
// The scratch is one file-scope device array of PA_NOALLOC_SCRATCH_BYTES. The
// CUDA runtime creates it, once per device, when this translation unit's
// module is loaded there; nothing here calls cudaMalloc, cudaFree or any
// routine that allocates. Its address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached; after that a
// call only checks sizes and forwards to pa_decode.
//
// Nothing in the scratch has to start at zero: each CTA of the persistent
// decode kernel computes the launch's work list itself and writes every work
// item it later reads back (no CTA reads another's items), and every partition
// partial is written by the decode kernel before the merge kernel reads it.
// So the scratch is never cleared.
//
// The cached address belongs to the device's primary context of the moment.
// cudaDeviceReset (or anything else that destroys that context) unloads the
// module and may place the array elsewhere when it is loaded again, so no
// call may follow a device reset in the same process.
#include <atomic>
#include <cstdint>

#include "pa_internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

std::atomic<void*> g_scratch_ptr[pa::kMaxDevices];

// Device address of g_decode_scratch on the current device, or nullptr if the
// runtime could not provide it.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < pa::kMaxDevices) {
        void* cached = g_scratch_ptr[dev].load(std::memory_order_acquire);
        if (cached != nullptr) return cached;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();   // do not leave the lookup's error for the caller's next check
        return nullptr;
    }
    if (dev >= 0 && dev < pa::kMaxDevices) g_scratch_ptr[dev].store(ptr, std::memory_order_release);
    return ptr;
}

}  // namespace

extern "C" {

pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            float scale, void* out, int num_seqs, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                            int32_t* error_word, struct CUstream_st* stream) {
    if (num_seqs == 0) {
        return pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                         num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         max_blocks_per_seq, max_context_len, dtype, nullptr, 0, error_word,
                         stream);
    }
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len);
    if (need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) return PA_ERR_WORKSPACE;
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return PA_ERR_CUDA;
    return pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     max_blocks_per_seq, max_context_len, dtype, scratch,
                     static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES), error_word, stream);
}

}  // extern "C"
