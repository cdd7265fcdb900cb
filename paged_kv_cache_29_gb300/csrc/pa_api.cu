// pa_api.cu -- the C ABI declared in include/pagedattn.h: argument checks,
// TMA descriptor set-up, kernel choice and launches. Everything here runs on
// the host and only enqueues work on the caller's stream.
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "pa_internal.h"

namespace {

using pa::DecodeParams;

constexpr int kVersion = 10000;   // 1.0.0
constexpr float kLog2e = 1.4426950408889634f;
constexpr size_t kMaxDynamicSmem = 227 * 1024;

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pa_dtype d) { return d == PA_DTYPE_F32 ? 4 : 2; }

bool valid_dtype(pa_dtype d) { return d == PA_DTYPE_F32 || d == PA_DTYPE_BF16; }

// The pool viewed as a 2D tensor [rows][head_dim], rows = blocks * kv_heads *
// block_size; boxes of 16 rows x 128 bytes with the 128-byte swizzle.
pa_status make_pool_map(CUtensorMap* map, const void* base, pa_dtype dtype, int head_dim,
                        long long rows) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return PA_ERR_CUDA;
    const int es = elem_bytes(dtype);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), 16u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map,
                          dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

size_t workspace_bytes_for(int num_seqs, int num_heads, int head_dim, int max_context_len,
                           int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || partition_size <= 0 ||
        max_context_len <= partition_size)
        return 0;
    const long long parts = ceil_div(max_context_len, partition_size);
    return static_cast<size_t>(num_seqs) * num_heads * parts * (head_dim + 2) * sizeof(float);
}

}  // namespace

extern "C" {

const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_DEVICE_BOUNDS: return "device-side bounds or timeout error";
    }
    return "unknown status";
}

pa_status pa_check_error_word(int32_t error_word_value) {
    return error_word_value == 0 ? PA_OK : PA_ERR_DEVICE_BOUNDS;
}

int pa_version(void) { return kVersion; }

size_t pa_decode_workspace_size_ex(int num_seqs, int num_heads, int head_dim,
                                   int max_context_len, int partition_size) {
    if (partition_size == 0) partition_size = pa::kDefaultPartition;
    return workspace_bytes_for(num_seqs, num_heads, head_dim, max_context_len, partition_size);
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len) {
    return workspace_bytes_for(num_seqs, num_heads, head_dim, max_context_len,
                               pa::kDefaultPartition);
}

pa_status pa_reshape_and_cache(const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               int num_tokens, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, pa_dtype dtype, int32_t* error_word,
                               struct CUstream_st* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !valid_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    const cudaError_t err =
        pa::launch_append(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads,
                          row_bytes, block_size, num_blocks, error_word,
                          reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, float scale,
                       void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_seq,
                       int max_context_len, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* error_word,
                       const pa_decode_options* options, struct CUstream_st* stream) {
    const int kernel_req = options ? options->kernel : PA_KERNEL_AUTO;
    const int partition = (options && options->partition_size) ? options->partition_size
                                                               : pa::kDefaultPartition;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 || max_context_len < 0 ||
        !valid_dtype(dtype) || num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (kernel_req < PA_KERNEL_AUTO || kernel_req > PA_KERNEL_GENERIC) return PA_ERR_INVALID_ARG;
    if (partition < 16 || partition > 4096 || partition % 16 != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;   // NaN scale
    if (head_dim > pa::kMaxHeadDim) return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(max_context_len) >
        static_cast<long long>(max_blocks_per_seq) * block_size)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u) != 0)
        return PA_ERR_INVALID_ARG;

    const int group = num_heads / num_kv_heads;
    const long long max_parts = max_context_len > 0 ? ceil_div(max_context_len, partition) : 1;
    const long long grid = max_parts * num_seqs * num_kv_heads;
    if (grid > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (max_parts > 1 && num_seqs > 65535) return PA_ERR_UNSUPPORTED;

    const size_t need = workspace_bytes_for(num_seqs, num_heads, head_dim, max_context_len, partition);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_WORKSPACE;

    const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    const bool tma_shape = block_size % 16 == 0 && rows < 0x7fffffffLL &&
                           (head_dim * elem_bytes(dtype)) % 128 == 0;
    pa_kernel kernel = static_cast<pa_kernel>(kernel_req);
    if (kernel == PA_KERNEL_AUTO) {
        if (tma_shape && pa::has_tma_instance(PA_KERNEL_MMA, dtype, head_dim, group))
            kernel = PA_KERNEL_MMA;
        else if (tma_shape && pa::has_tma_instance(PA_KERNEL_SIMT, dtype, head_dim, group))
            kernel = PA_KERNEL_SIMT;
        else
            kernel = PA_KERNEL_GENERIC;
    } else if (kernel != PA_KERNEL_GENERIC &&
               (!tma_shape || !pa::has_tma_instance(kernel, dtype, head_dim, group))) {
        return PA_ERR_UNSUPPORTED;
    }
    if (kernel == PA_KERNEL_GENERIC &&
        pa::generic_smem_bytes(group, head_dim, partition, block_size) > kMaxDynamicSmem)
        return PA_ERR_UNSUPPORTED;

    DecodeParams p{};
    p.q = q;
    p.out = out;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    const size_t ml_floats = static_cast<size_t>(num_seqs) * num_heads * max_parts * 2;
    p.part_ml = need ? static_cast<float*>(workspace) : nullptr;
    p.part_o = need ? static_cast<float*>(workspace) + ml_floats : nullptr;
    p.error_word = error_word;
    p.scale_log2 = scale * kLog2e;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_cap = max_context_len;
    p.partition_size = partition;
    p.max_parts = static_cast<int>(max_parts);

    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (kernel == PA_KERNEL_GENERIC) {
        err = pa::launch_decode_generic(p, dtype, st);
    } else {
        CUtensorMap tk, tv;
        pa_status ps = make_pool_map(&tk, k_cache, dtype, head_dim, rows);
        if (ps == PA_OK) ps = make_pool_map(&tv, v_cache, dtype, head_dim, rows);
        if (ps != PA_OK) return ps;
        err = kernel == PA_KERNEL_MMA ? pa::launch_decode_mma(tk, tv, p, st)
                                      : pa::launch_decode_simt(tk, tv, p, dtype, st);
    }
    if (err == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    if (err != cudaSuccess) return PA_ERR_CUDA;
    if (max_parts > 1) {
        err = pa::launch_combine(p, dtype, st);
        if (err != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int max_blocks_per_seq,
                    int max_context_len, pa_dtype dtype, void* workspace,
                    size_t workspace_bytes, int32_t* error_word, struct CUstream_st* stream) {
    return pa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out, num_seqs,
                        num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                        max_blocks_per_seq, max_context_len, dtype, workspace, workspace_bytes,
                        error_word, nullptr, stream);
}

}  // extern "C"
