// pa_decode_int8.cu -- instances of the tile-ring decode kernel for an INT8
// cache with per-row scales and bf16 q and output (head dim 128; 1, 2, 4 or 8
// query heads per KV head).
#include "pa_decode_stream.cuh"
#include "pa_tile_math_quant.cuh"

namespace pa {

namespace {
constexpr int kWarps = 4;          // consumer warps per CTA
constexpr int kStages = 8;         // a multiple of kWarps: 8 x (K + V) tiles of codes = 32 KiB
constexpr int kMinCtasPerSm = 4;   // four rings per SM (register budget 96 per thread)

template <int G>
cudaError_t run(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                int sm_count, cudaStream_t stream) {
    return launch_stream_instance<Int8MmaMath<128, G>, 128, G, kWarps, kStages, kMinCtasPerSm, true>(
        tk, tv, p, sm_count, stream);
}
}  // namespace

cudaError_t launch_decode_int8(const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int sm_count, cudaStream_t stream) {
    if (p.head_dim != 128) return cudaErrorNotSupported;
    switch (p.num_heads / p.num_kv_heads) {
        case 1: return run<1>(tk, tv, p, sm_count, stream);
        case 2: return run<2>(tk, tv, p, sm_count, stream);
        case 4: return run<4>(tk, tv, p, sm_count, stream);
        case 8: return run<8>(tk, tv, p, sm_count, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
