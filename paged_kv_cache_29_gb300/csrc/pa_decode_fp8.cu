// pa_decode_fp8.cu -- instances of the tile-ring decode kernel for an FP8
// (e4m3) cache with bf16 q and output (head dim 128; 1, 2, 4 or 8 query heads
// per KV head).
#include "pa_decode_stream.cuh"
#include "pa_tile_math_quant.cuh"

namespace pa {

namespace {
constexpr int kWarps = 4;          // consumer warps per CTA
// Three tiles in flight per consumer warp (12 x (K + V) tiles = 48 KiB of
// codes), three CTAs per SM: with per-warp refills this beats 8 stages at four
// CTAs per SM (93 vs 101 us on the 8B GQA batch); more registers alone (8
// stages, three CTAs) do not help.
constexpr int kStages = 12;
constexpr int kMinCtasPerSm = 3;

template <int G>
cudaError_t run(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                int sm_count, cudaStream_t stream) {
    return launch_stream_instance<Fp8MmaMath<128, G>, 128, G, kWarps, kStages, kMinCtasPerSm, true>(
        tk, tv, p, sm_count, stream);
}
}  // namespace

bool has_fp8_instance(int head_dim, int group) {
    return head_dim == 128 && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
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
