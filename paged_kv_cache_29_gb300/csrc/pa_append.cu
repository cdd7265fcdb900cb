// pa_append.cu -- the cache append (reshape_and_cache): each token's new K and
// V row is copied into slot_mapping[t] of the paged pool,
//   cache[slot / block_size][kv_head][slot % block_size][:] = new[t][kv_head][:],
// the flat-slot form of the paged indexing of "MLSys Engineer -- Inference
// Systems Q&A", Q1, and the cache append that precedes attention in the naive
// incremental decoder of "LLM inference and serving". A bit copy in 16-byte
// vectors: one thread per 16-byte chunk of one (token, KV head) row, K and V
// both. The read of k_new/v_new and the write into the pool are each one
// coalesced pass over the row.
#include <cuda_fp8.h>

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

// Quantising append into an FP8 (e4m3) cache: code = e4m3(x / scale), the
// division in fp32 (IEEE, round to nearest), the conversion rounding to
// nearest even and saturating at +-448. One thread per 16 codes (one 16-byte
// store) of one (token, KV head) row; TIn is the new rows' type.
template <typename TIn>
__global__ void __launch_bounds__(kAppendThreads)
append_fp8_kernel(const TIn* __restrict__ k_new, const TIn* __restrict__ v_new,
                  const int64_t* __restrict__ slot_mapping, uint4* __restrict__ k_cache,
                  uint4* __restrict__ v_cache, long long total_chunks, int chunks_per_row,
                  int num_kv_heads, int block_size, long long num_slots, float k_scale,
                  float v_scale, int32_t* error_word) {
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
        const TIn* ks = k_new + i * 16;
        const TIn* vs = v_new + i * 16;
        uint32_t kw[4], vw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t kb = 0, vb = 0;
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const float2 kx = make_float2(__fdiv_rn(ElemTraits<TIn>::load(ks + 4 * w + e), k_scale),
                                              __fdiv_rn(ElemTraits<TIn>::load(ks + 4 * w + e + 1), k_scale));
                const float2 vx = make_float2(__fdiv_rn(ElemTraits<TIn>::load(vs + 4 * w + e), v_scale),
                                              __fdiv_rn(ElemTraits<TIn>::load(vs + 4 * w + e + 1), v_scale));
                kb |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(kx, __NV_SATFINITE, __NV_E4M3)) << (8 * e);
                vb |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(vx, __NV_SATFINITE, __NV_E4M3)) << (8 * e);
            }
            kw[w] = kb;
            vw[w] = vb;
        }
        k_cache[dst] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
        v_cache[dst] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
    }
}

// Quantising append into an INT8 cache with one scale per (row, KV head):
// scale = max|x| / 127 and code = x / scale rounded to the nearest integer,
// ties to even (both divisions in fp32, IEEE), clamped to [-127, 127]; an
// all-zero row gets scale 0 and codes 0. One warp per (token, KV head, K or
// V) row: the lanes hold the row, a butterfly max gives the scale.
constexpr int kInt8MaxPerLane = kMaxHeadDim / 32;

template <typename TIn>
__global__ void __launch_bounds__(kAppendThreads)
append_int8_kernel(const TIn* __restrict__ k_new, const TIn* __restrict__ v_new,
                   const int64_t* __restrict__ slot_mapping, int8_t* __restrict__ k_cache,
                   int8_t* __restrict__ v_cache, float* __restrict__ k_scales,
                   float* __restrict__ v_scales, long long rows, int head_dim,
                   int num_kv_heads, int block_size, long long num_slots, int32_t* error_word) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < 2 * rows; w += warps) {
        const bool is_v = w >= rows;
        const long long rowi = is_v ? w - rows : w;          // (token, kv head)
        const long long t = rowi / num_kv_heads;
        const int h = static_cast<int>(rowi - t * num_kv_heads);
        const long long slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (lane == 0 && h == 0 && !is_v) raise_error(error_word, PA_DEVERR_SLOT);
            continue;
        }
        const TIn* src = (is_v ? v_new : k_new) + rowi * head_dim;
        float x[kInt8MaxPerLane];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kInt8MaxPerLane; ++i) {
            const int d = lane + 32 * i;
            x[i] = d < head_dim ? ElemTraits<TIn>::load(src + d) : 0.f;
            amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = __fdiv_rn(amax, 127.0f);
        const long long blk = slot / block_size;
        const long long r = (blk * num_kv_heads + h) * block_size + (slot - blk * block_size);
        int8_t* dst = (is_v ? v_cache : k_cache) + r * head_dim;
#pragma unroll
        for (int i = 0; i < kInt8MaxPerLane; ++i) {
            const int d = lane + 32 * i;
            if (d < head_dim) {
                int c = 0;
                if (scale != 0.f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], scale))));
                dst[d] = static_cast<int8_t>(c);
            }
        }
        if (lane == 0) (is_v ? v_scales : k_scales)[r] = scale;
    }
}

}  // namespace

cudaError_t launch_append_int8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               float* k_scales, float* v_scales, int num_tokens,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int32_t* error_word, cudaStream_t stream) {
    const long long rows = static_cast<long long>(num_tokens) * num_kv_heads;
    if (rows == 0) return cudaSuccess;
    long long blocks = (2 * rows * 32 + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 8192) blocks = 8192;
    const long long num_slots = static_cast<long long>(num_blocks) * block_size;
    if (new_dtype == PA_DTYPE_BF16) {
        append_int8_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
            slot_mapping, static_cast<int8_t*>(k_cache), static_cast<int8_t*>(v_cache), k_scales,
            v_scales, rows, head_dim, num_kv_heads, block_size, num_slots, error_word);
    } else {
        append_int8_kernel<float><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
            static_cast<const float*>(k_new), static_cast<const float*>(v_new), slot_mapping,
            static_cast<int8_t*>(k_cache), static_cast<int8_t*>(v_cache), k_scales, v_scales,
            rows, head_dim, num_kv_heads, block_size, num_slots, error_word);
    }
    return cudaGetLastError();
}

cudaError_t launch_append_fp8(const void* k_new, const void* v_new, pa_dtype new_dtype,
                              const int64_t* slot_mapping, void* k_cache, void* v_cache,
                              int num_tokens, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, float k_scale, float v_scale, int32_t* error_word,
                              cudaStream_t stream) {
    const int chunks_per_row = head_dim / 16;
    const long long total = static_cast<long long>(num_tokens) * num_kv_heads * chunks_per_row;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 8192) blocks = 8192;
    const long long num_slots = static_cast<long long>(num_blocks) * block_size;
    if (new_dtype == PA_DTYPE_BF16) {
        append_fp8_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
            slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), total,
            chunks_per_row, num_kv_heads, block_size, num_slots, k_scale, v_scale, error_word);
    } else {
        append_fp8_kernel<float><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
            static_cast<const float*>(k_new), static_cast<const float*>(v_new), slot_mapping,
            static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), total, chunks_per_row,
            num_kv_heads, block_size, num_slots, k_scale, v_scale, error_word);
    }
    return cudaGetLastError();
}

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
