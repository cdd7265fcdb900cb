// pa_api.cu -- the C ABI declared in include/pagedattn.h: argument checks,
// TMA descriptor set-up, kernel choice and launches. Everything here runs on
// the host and only enqueues work on the caller's stream.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "pa_internal.h"

namespace {

using pa::DecodeParams;

constexpr int kVersion = 10100;   // 1.1.0
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

int elem_bytes(pa_dtype d) { return d == PA_DTYPE_F32 ? 4 : d == PA_DTYPE_BF16 ? 2 : 1; }

// Types of q, out and new rows.
bool valid_dtype(pa_dtype d) { return d == PA_DTYPE_F32 || d == PA_DTYPE_BF16; }

// Types a cache may hold (an INT8 cache also carries per-row scales, so the
// plain row copies leave it out).
bool valid_cache_dtype(pa_dtype d) { return valid_dtype(d) || d == PA_DTYPE_FP8_E4M3; }
bool valid_decode_cache_dtype(pa_dtype d) { return valid_cache_dtype(d) || d == PA_DTYPE_INT8; }

// The pool viewed as a 3D tensor for TMA: x = element within a 128-byte
// column half of a row, y = row (rows = blocks * kv_heads * block_size, stride
// one row), z = which 128-byte half (stride 128 bytes). One box {128 B, 16
// rows, all halves} is one 16-row tile of one (block, KV head), landing in
// shared memory as [half][row][128 B] with the 128-byte swizzle.
pa_status make_pool_map(CUtensorMap* map, const void* base, pa_dtype dtype, int head_dim,
                        long long rows) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return PA_ERR_CUDA;
    const int es = elem_bytes(dtype);
    const int row_bytes = head_dim * es;
    const int halves = row_bytes / 128;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(128 / es), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(halves)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), 128};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 16u, static_cast<cuuint32_t>(halves)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(map,
                          dtype == PA_DTYPE_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                          : dtype == PA_DTYPE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                  : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Workspace layout (per launch of at most kPlanMaxSeqs sequences, reused by
// consecutive launches of one call):
//   [0, 256)              reserved
//   items                 int4 per (sequence, KV head, partition), written and
//                         read by the decode kernel: num_heads bounds
//                         num_kv_heads
//   part_ml, part_o       partition partials, only when a sequence can span
//                         more than one partition
struct WorkspaceLayout {
    size_t items_off, ml_off, o_off, total;
};

WorkspaceLayout layout_for(int num_seqs, int num_heads, int head_dim, int max_context_len,
                           int partition_size, int num_queries = 1) {
    WorkspaceLayout w{0, 0, 0, 0};
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || partition_size <= 0 ||
        max_context_len < 0 || num_queries < 1)
        return w;
    const long long seqs = num_seqs < pa::kPlanMaxSeqs ? num_seqs : pa::kPlanMaxSeqs;
    const long long parts = max_context_len > 0 ? ceil_div(max_context_len, partition_size) : 1;
    const size_t units = static_cast<size_t>(seqs) * num_heads * parts;   // items (bounded)
    const size_t prows = units * static_cast<size_t>(num_queries);          // partial rows
    w.items_off = 256;
    w.ml_off = w.items_off + 16 * units;
    w.o_off = w.ml_off + (parts > 1 ? 8 * prows : 0);
    w.total = w.o_off + (parts > 1 ? 4 * prows * static_cast<size_t>(head_dim) : 0);
    return w;
}

size_t workspace_bytes_for(int num_seqs, int num_heads, int head_dim, int max_context_len,
                           int partition_size, int num_queries = 1) {
    return layout_for(num_seqs, num_heads, head_dim, max_context_len, partition_size, num_queries)
        .total;
}

// One decode call: q/out in act_dtype, the caches in dtype (act_dtype, or FP8
// with bf16 q/out), K/V values scaled by k_scale/v_scale (1 unless FP8).
pa_status decode_call(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, float scale,
                      float k_scale, float v_scale, void* out, int num_seqs, int num_heads,
                      int num_kv_heads, int head_dim, int block_size, int num_blocks,
                      int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                      pa_dtype act_dtype, void* workspace, size_t workspace_bytes,
                      int32_t* error_word, const pa_decode_options* options,
                      struct CUstream_st* stream, int num_queries = 1, int window = 0,
                      const float* k_row_scales = nullptr, const float* v_row_scales = nullptr,
                      const void* k_new = nullptr, const void* v_new = nullptr,
                      const int64_t* slot_mapping = nullptr, int withhold_tile = -1) {
    const int kernel_req = options ? options->kernel : PA_KERNEL_AUTO;
    const int partition = (options && options->partition_size) ? options->partition_size
                          : dtype == PA_DTYPE_FP8_E4M3          ? pa::kDefaultPartition8
                                                               : pa::kDefaultPartition;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 || max_context_len < 0 ||
        !valid_decode_cache_dtype(dtype) || !valid_dtype(act_dtype) ||
        num_heads % num_kv_heads != 0 || num_queries < 1 || window < 0 ||
        (window > 0 && num_queries > 1))
        return PA_ERR_INVALID_ARG;
    if (kernel_req < PA_KERNEL_AUTO || kernel_req > PA_KERNEL_TC) return PA_ERR_INVALID_ARG;
    if (partition < 16 || partition > 4096 || partition % 16 != 0) return PA_ERR_INVALID_ARG;
    if (options && options->long_partition_from != 0 &&
        (options->long_partition_from < 0 || options->long_partition_size < partition ||
         options->long_partition_size > 4096 || options->long_partition_size % 16 != 0))
        return PA_ERR_INVALID_ARG;
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
    const long long chunk = num_seqs < pa::kPlanMaxSeqs ? num_seqs : pa::kPlanMaxSeqs;
    if (max_parts * chunk * num_kv_heads > 0x3fffffffLL) return PA_ERR_UNSUPPORTED;

    const WorkspaceLayout lay =
        layout_for(num_seqs, num_heads, head_dim, max_context_len, partition, num_queries);
    if (workspace == nullptr || workspace_bytes < lay.total || !aligned16(workspace))
        return PA_ERR_WORKSPACE;

    const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    const bool tma_shape = block_size % 16 == 0 && rows < 0x7fffffffLL &&
                           (head_dim * elem_bytes(dtype)) % 128 == 0;
    pa_kernel kernel = static_cast<pa_kernel>(kernel_req);
    const bool fp8 = dtype == PA_DTYPE_FP8_E4M3;
    const bool int8 = dtype == PA_DTYPE_INT8;
    if (int8) {
        // One kernel family: the INT8 tensor-core tile ring.
        if (!tma_shape || !pa::has_fp8_instance(head_dim, group) || num_queries > 1 ||
            window > 0 || !k_row_scales || !v_row_scales || !aligned16(k_row_scales) ||
            !aligned16(v_row_scales) || (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_MMA))
            return (!k_row_scales || !v_row_scales) ? PA_ERR_INVALID_ARG : PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_MMA;
    } else if (num_queries > 1) {
        // Several query tokens per sequence: the bf16 tensor-core tile ring.
        if (fp8 || !tma_shape ||
            !pa::has_tma_instance(PA_KERNEL_MMA, dtype, head_dim, group, num_queries) ||
            (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_MMA))
            return PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_MMA;
    } else if (fp8) {
        // The FP8 tile ring (mma.sync on widened codes) or the tcgen05 kernel.
        if (!tma_shape || !pa::has_fp8_instance(head_dim, group) ||
            (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_MMA && kernel != PA_KERNEL_TC))
            return PA_ERR_UNSUPPORTED;
        if (kernel == PA_KERNEL_AUTO) kernel = pa::kFp8DefaultKernel;
    } else if (kernel == PA_KERNEL_AUTO) {
        if (tma_shape && pa::has_tma_instance(PA_KERNEL_MMA, dtype, head_dim, group, 1))
            kernel = PA_KERNEL_MMA;
        else if (tma_shape && pa::has_tma_instance(PA_KERNEL_SIMT, dtype, head_dim, group, 1))
            kernel = PA_KERNEL_SIMT;
        else
            kernel = PA_KERNEL_GENERIC;
    } else if (kernel == PA_KERNEL_TC ||
               (kernel != PA_KERNEL_GENERIC &&
                (!tma_shape || !pa::has_tma_instance(kernel, dtype, head_dim, group, 1)))) {
        return PA_ERR_UNSUPPORTED;
    }
    const int largest_partition =
        (options && options->long_partition_from > 0) ? options->long_partition_size : partition;
    if (kernel == PA_KERNEL_GENERIC &&
        (window > 0 ||   // the direct-load kernel has no sliding window
         pa::generic_smem_bytes(group, head_dim, largest_partition, block_size) > kMaxDynamicSmem))
        return PA_ERR_UNSUPPORTED;

    // Fused append: the in-order tile-ring kernels write each sequence's new
    // row themselves; the direct-load kernel gets a separate append first.
    const bool append = k_new != nullptr;
    const bool fused_append = append && kernel != PA_KERNEL_GENERIC;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (append && !fused_append) {
        if (pa::launch_append(k_new, v_new, slot_mapping, const_cast<void*>(k_cache),
                              const_cast<void*>(v_cache), num_seqs, num_kv_heads, row_bytes,
                              block_size, num_blocks, error_word,
                              reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return PA_ERR_CUDA;
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams base{};
    base.k_cache = k_cache;
    base.v_cache = v_cache;
    base.part_ml = max_parts > 1 ? reinterpret_cast<float*>(ws + lay.ml_off) : nullptr;
    base.part_o = max_parts > 1 ? reinterpret_cast<float*>(ws + lay.o_off) : nullptr;
    base.items = reinterpret_cast<int4*>(ws + lay.items_off);
    base.error_word = error_word;
    base.scale_log2 = scale * kLog2e;
    base.k_scale = k_scale;
    base.v_scale = v_scale;
    base.num_queries = num_queries;
    base.window = window;
    base.withhold_tile = withhold_tile;
    base.k_row_scales = k_row_scales;
    base.v_row_scales = v_row_scales;
    base.num_heads = num_heads;
    base.num_kv_heads = num_kv_heads;
    base.head_dim = head_dim;
    base.block_size = block_size;
    base.num_blocks = num_blocks;
    base.max_blocks_per_seq = max_blocks_per_seq;
    base.context_cap = max_context_len;
    base.partition_size = partition;
    // Larger partitions for long sequences by default (tile-ring kernels); an
    // explicit partition size, and the direct-load kernel, keep one size.
    // Optional larger partitions for long sequences (checked above).
    const bool tiered = options && options->long_partition_from > 0;
    base.partition_long = tiered ? options->long_partition_size : partition;
    base.partition_long_from = tiered ? options->long_partition_from : pa::kNoLongPartitions;
    base.max_parts = static_cast<int>(max_parts);

    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tk, tv;
    int sm_count = 0;
    if (kernel != PA_KERNEL_GENERIC) {
        pa_status ps = make_pool_map(&tk, k_cache, dtype, head_dim, rows);
        if (ps == PA_OK) ps = make_pool_map(&tv, v_cache, dtype, head_dim, rows);
        if (ps != PA_OK) return ps;
        static std::atomic<int> cached_sms[pa::kMaxDevices];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
        sm_count = dev < pa::kMaxDevices ? cached_sms[dev].load(std::memory_order_relaxed) : 0;
        if (sm_count <= 0) {
            if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                sm_count <= 0)
                return PA_ERR_CUDA;
            if (dev < pa::kMaxDevices) cached_sms[dev].store(sm_count, std::memory_order_relaxed);
        }
    }
    const size_t es = static_cast<size_t>(elem_bytes(act_dtype));   // q, out and new rows
    // Batches above kPlanMaxSeqs sequences run as consecutive launches over
    // slices of the batch; they reuse the workspace in stream order.
    for (int s0 = 0; s0 < num_seqs; s0 += pa::kPlanMaxSeqs) {
        const int bs_n = num_seqs - s0 < pa::kPlanMaxSeqs ? num_seqs - s0 : pa::kPlanMaxSeqs;
        DecodeParams p = base;
        const size_t qoff = static_cast<size_t>(s0) * num_queries * num_heads * head_dim * es;
        p.q = static_cast<const uint8_t*>(q) + qoff;
        p.out = static_cast<uint8_t*>(out) + qoff;
        p.block_tables = block_tables + static_cast<size_t>(s0) * max_blocks_per_seq;
        p.context_lens = context_lens + s0;
        p.num_seqs = bs_n;
        if (fused_append) {
            // New rows are in the activation dtype (bf16 over 8-bit pools).
            const size_t roff = static_cast<size_t>(s0) * num_kv_heads * head_dim * es;
            p.k_new = static_cast<const uint8_t*>(k_new) + roff;
            p.v_new = static_cast<const uint8_t*>(v_new) + roff;
            p.slot_mapping = slot_mapping + s0;
        }
        cudaError_t err;
        if (kernel == PA_KERNEL_GENERIC) {
            err = pa::launch_decode_generic(p, dtype, st);
        } else {
            err = (fp8 && kernel == PA_KERNEL_TC) ? pa::launch_decode_fp8_tc(tk, tv, p, sm_count, st)
                  : fp8                      ? pa::launch_decode_fp8(tk, tv, p, sm_count, st)
                  : int8                    ? pa::launch_decode_int8(tk, tv, p, sm_count, st)
                  : kernel == PA_KERNEL_MMA ? pa::launch_decode_mma(tk, tv, p, sm_count, st)
                                            : pa::launch_decode_simt(tk, tv, p, dtype, sm_count, st);
        }
        if (err == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
        if (err != cudaSuccess) return PA_ERR_CUDA;
        if (max_parts > 1) {
            err = pa::launch_combine(p, act_dtype, st);
            if (err != cudaSuccess) return PA_ERR_CUDA;
        }
    }
    return PA_OK;
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

int pa_default_partition_size(pa_dtype cache_dtype) {
    if (!valid_decode_cache_dtype(cache_dtype)) return 0;
    return cache_dtype == PA_DTYPE_FP8_E4M3 ? pa::kDefaultPartition8 : pa::kDefaultPartition;
}



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
        num_blocks <= 0 || !valid_cache_dtype(dtype))
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

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                         int num_pairs, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, pa_dtype dtype, int32_t* error_word,
                         struct CUstream_st* stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !valid_decode_cache_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    const int row_bytes = head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    const long long block_bytes = static_cast<long long>(num_kv_heads) * block_size * row_bytes;
    const cudaError_t err =
        pa::launch_copy_blocks(k_cache, v_cache, block_mapping, num_pairs, block_bytes,
                               num_blocks, error_word, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens, float scale,
                       void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_seq,
                       int max_context_len, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* error_word,
                       const pa_decode_options* options, struct CUstream_st* stream) {
    if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, dtype, workspace,
                       workspace_bytes, error_word, options, stream);
}

pa_status pa_test_withhold_tile(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, void* out, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                                void* workspace, size_t workspace_bytes, int32_t* error_word,
                                int withhold_tile, struct CUstream_st* stream) {
    const bool fp8 = dtype == PA_DTYPE_FP8_E4M3;
    if (withhold_tile < 0 || error_word == nullptr || (!fp8 && !valid_dtype(dtype)))
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, fp8 ? PA_DTYPE_BF16 : dtype,
                       workspace, workspace_bytes, error_word, nullptr, stream, 1, 0, nullptr,
                       nullptr, nullptr, nullptr, nullptr, withhold_tile);
}

pa_status pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        float k_scale, float v_scale, void* out, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        int max_blocks_per_seq, int max_context_len, void* workspace,
                        size_t workspace_bytes, int32_t* error_word,
                        struct CUstream_st* stream) {
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || k_scale == INFINITY || v_scale == INFINITY)
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                       out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_DTYPE_FP8_E4M3, PA_DTYPE_BF16,
                       workspace, workspace_bytes, error_word, nullptr, stream);
}

pa_status pa_decode_fp8_ex(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens, float scale,
                           float k_scale, float v_scale, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, void* workspace,
                           size_t workspace_bytes, int32_t* error_word,
                           const pa_decode_options* options, struct CUstream_st* stream) {
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || k_scale == INFINITY || v_scale == INFINITY)
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                       out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_DTYPE_FP8_E4M3, PA_DTYPE_BF16,
                       workspace, workspace_bytes, error_word, options, stream);
}

pa_status pa_append_decode_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               void* k_cache, void* v_cache, float k_scale, float v_scale,
                               const void* q, const int32_t* block_tables,
                               const int32_t* context_lens, float scale, void* out, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, int max_blocks_per_seq, int max_context_len,
                               void* workspace, size_t workspace_bytes, int32_t* error_word,
                               struct CUstream_st* stream) {
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || k_scale == INFINITY || v_scale == INFINITY)
        return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping || !aligned16(k_new) ||
                         !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0))
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                       out, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_DTYPE_FP8_E4M3, PA_DTYPE_BF16,
                       workspace, workspace_bytes, error_word, nullptr, stream, 1, 0, nullptr,
                       nullptr, k_new, v_new, slot_mapping);
}

pa_status pa_append_decode_int8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                const void* q, const int32_t* block_tables,
                                const int32_t* context_lens, float scale, void* out, int num_seqs,
                                int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, int max_blocks_per_seq, int max_context_len,
                                void* workspace, size_t workspace_bytes, int32_t* error_word,
                                struct CUstream_st* stream) {
    if (num_seqs > 0 && (!k_scales || !v_scales || !k_new || !v_new || !slot_mapping ||
                         !aligned16(k_new) || !aligned16(v_new) ||
                         (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0))
        return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_DTYPE_INT8, PA_DTYPE_BF16,
                       workspace, workspace_bytes, error_word, nullptr, stream, 1, 0, k_scales,
                       v_scales, k_new, v_new, slot_mapping);
}

pa_status pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens, float scale,
                          void* out, int num_seqs, int num_queries, int num_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                          void* workspace, size_t workspace_bytes, int32_t* error_word,
                          struct CUstream_st* stream) {
    if (!valid_dtype(dtype) || num_queries < 1 || num_queries > 8) return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, dtype, workspace,
                       workspace_bytes, error_word, nullptr, stream, num_queries);
}

pa_status pa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, int window, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, int32_t* error_word,
                           struct CUstream_st* stream) {
    if (!valid_dtype(dtype) || window < 1) return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, dtype, workspace,
                       workspace_bytes, error_word, nullptr, stream, 1, window);
}

pa_status pa_decode_int8(const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scales, const float* v_scales,
                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                         void* out, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, int max_blocks_per_seq,
                         int max_context_len, void* workspace, size_t workspace_bytes,
                         int32_t* error_word, struct CUstream_st* stream) {
    if (num_seqs > 0 && (!k_scales || !v_scales)) return PA_ERR_INVALID_ARG;
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.0f, 1.0f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, PA_DTYPE_INT8, PA_DTYPE_BF16,
                       workspace, workspace_bytes, error_word, nullptr, stream, 1, 0, k_scales,
                       v_scales);
}

pa_status pa_reshape_and_cache_int8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                                    const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                    float* k_scales, float* v_scales, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int32_t* error_word,
                                    struct CUstream_st* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !valid_dtype(new_dtype))
        return PA_ERR_INVALID_ARG;
    if (head_dim % 16 != 0 || head_dim > pa::kMaxHeadDim) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scales || !v_scales)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(k_scales) || !aligned16(v_scales) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    const cudaError_t err = pa::launch_append_int8(
        k_new, v_new, new_dtype, slot_mapping, k_cache, v_cache, k_scales, v_scales, num_tokens,
        num_kv_heads, head_dim, block_size, num_blocks, error_word,
        reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size_multi(int num_seqs, int num_queries, int num_heads,
                                      int head_dim, int max_context_len) {
    return workspace_bytes_for(num_seqs, num_heads, head_dim, max_context_len,
                               pa::kDefaultPartition, num_queries);
}

pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                                   const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                   int num_tokens, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, float k_scale, float v_scale,
                                   int32_t* error_word, struct CUstream_st* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || !valid_dtype(new_dtype) || !(k_scale > 0.0f) ||
        !(v_scale > 0.0f) || k_scale == INFINITY || v_scale == INFINITY)
        return PA_ERR_INVALID_ARG;
    if (head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    const cudaError_t err = pa::launch_append_fp8(
        k_new, v_new, new_dtype, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads,
        head_dim, block_size, num_blocks, k_scale, v_scale, error_word,
        reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_append_decode(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           void* k_cache, void* v_cache, const void* q,
                           const int32_t* block_tables, const int32_t* context_lens,
                           float scale, void* out, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int max_context_len, pa_dtype dtype,
                           void* workspace, size_t workspace_bytes, int32_t* error_word,
                           struct CUstream_st* stream) {
    if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0) {
        if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
        if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
            !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
            return PA_ERR_INVALID_ARG;
        if ((head_dim * elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    }
    return decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, 1.f, 1.f, out,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_context_len, dtype, dtype, workspace,
                       workspace_bytes, error_word, nullptr, stream, 1, 0, nullptr, nullptr,
                       k_new, v_new, slot_mapping);
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
