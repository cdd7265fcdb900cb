// pa_decode_mma.cu -- instances of the tile-ring decode kernel with the
// tensor-core tile math (bf16 caches; head dim 64 or 128; up to 8 query
// columns per item: 1, 2, 4 or 8 query heads per KV head, times the query
// tokens per sequence).
#include "pa_decode_stream.cuh"

namespace pa {

namespace {
constexpr int kWarps = 4;     // consumer warps per CTA
constexpr int kStages = 4;    // ring depth, a multiple of kWarps: 4 x (K + V) tiles = 32 KiB at d=128
constexpr int kMinCtasPerSm = 4;   // four rings per SM (register budget 96 per thread)

template <int D, int G>
cudaError_t run(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                int sm_count, cudaStream_t stream) {
    if constexpr (G > 1) {   // several query tokens fill at least two columns
        if (p.num_queries > 1)
            return launch_stream_instance<MmaMath<D, G, true>, D, G, kWarps, kStages,
                                          kMinCtasPerSm, false>(tk, tv, p, sm_count, stream);
    }
    return launch_stream_instance<MmaMath<D, G>, D, G, kWarps, kStages, kMinCtasPerSm, false>(
        tk, tv, p, sm_count, stream);
}

// The instance's column capacity: the query columns of an item (group heads x
// query tokens per sequence) rounded up to 1, 2, 4 or 8.
template <int D>
cudaError_t by_group(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                     int sm_count, cudaStream_t stream) {
    const int cols = (p.num_heads / p.num_kv_heads) * p.num_queries;
    if (cols <= 1) return run<D, 1>(tk, tv, p, sm_count, stream);
    if (cols <= 2) return run<D, 2>(tk, tv, p, sm_count, stream);
    if (cols <= 4) return run<D, 4>(tk, tv, p, sm_count, stream);
    if (cols <= 8) return run<D, 8>(tk, tv, p, sm_count, stream);
    return cudaErrorNotSupported;
}
}  // namespace

cudaError_t launch_decode_mma(const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, int sm_count, cudaStream_t stream) {
    switch (p.head_dim) {
        case 64: return by_group<64>(tk, tv, p, sm_count, stream);
        case 128: return by_group<128>(tk, tv, p, sm_count, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
