// pa_decode_simt.cu -- instances of the tile-ring decode kernel with the
// CUDA-core tile math (fp32 or bf16 caches; head dim 64 or 128; 1, 2, 4 or 8
// query heads per KV head).
#include "pa_decode_stream.cuh"

namespace pa {

namespace {
constexpr int kWarps = 4;

// Ring depth: one stage per consumer warp (short rings, several CTAs per SM).
template <typename T, int D>
constexpr int stages_for() {
    return kWarps;
}

template <typename T, int D, int G>
cudaError_t run(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                int sm_count, cudaStream_t stream) {
    return launch_stream_instance<SimtMath<T, D, G>, D, G, kWarps, stages_for<T, D>(), 1, false>(
        tk, tv, p, sm_count, stream);
}

template <typename T, int D>
cudaError_t by_group(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                     int sm_count, cudaStream_t stream) {
    switch (p.num_heads / p.num_kv_heads) {
        case 1: return run<T, D, 1>(tk, tv, p, sm_count, stream);
        case 2: return run<T, D, 2>(tk, tv, p, sm_count, stream);
        case 4: return run<T, D, 4>(tk, tv, p, sm_count, stream);
        case 8: return run<T, D, 8>(tk, tv, p, sm_count, stream);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t by_dim(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                   int sm_count, cudaStream_t stream) {
    switch (p.head_dim) {
        case 64: return by_group<T, 64>(tk, tv, p, sm_count, stream);
        case 128: return by_group<T, 128>(tk, tv, p, sm_count, stream);
        default: return cudaErrorNotSupported;
    }
}
}  // namespace

cudaError_t launch_decode_simt(const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, pa_dtype dtype, int sm_count,
                               cudaStream_t stream) {
    return dtype == PA_DTYPE_BF16 ? by_dim<__nv_bfloat16>(tk, tv, p, sm_count, stream)
                                  : by_dim<float>(tk, tv, p, sm_count, stream);
}

bool has_tma_instance(pa_kernel kernel, pa_dtype dtype, int head_dim, int group,
                      int num_queries) {
    const bool dims = head_dim == 64 || head_dim == 128;
    const bool pow2_group = group == 1 || group == 2 || group == 4 || group == 8;
    if (kernel == PA_KERNEL_MMA) {
        // Query columns (heads x query tokens) fill the 8 MMA columns.
        const bool cols = num_queries == 1 ? pow2_group : group * num_queries <= 8;
        return dims && cols && dtype == PA_DTYPE_BF16;
    }
    if (kernel == PA_KERNEL_SIMT) return dims && pow2_group && num_queries == 1;
    return false;
}

}  // namespace pa
