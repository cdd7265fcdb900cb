// pa_decode_generic.cu -- the plain decode kernel (any block size, head dim up
// to 256, any group size) and the split-K combine kernel.
//
// Generic kernel: one CTA per (sequence, KV head, partition). It reads the
// partition's rows straight from the pool through the block table (row i is
// row i % block_size of block block_tables[s][i / block_size], "MLSys
// Engineer -- Inference Systems Q&A", Q1), computes all scores of the
// partition into shared memory, takes the softmax over them in base 2 and
// accumulates P.V in fp32. It exists for shapes the tile-ring kernels do not
// cover (block sizes that are not a multiple of 16, other head dims); it is
// not tuned.
//
// Combine kernel: for a sequence split into partitions p = 0..P-1 with states
// (m_p, l_p, o_p) -- running max (base 2), sum of exp2(s - m_p), unnormalised
// output -- the result is sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p with
// M = max_p m_p: the rescale rule of the online softmax in Q4 "How would you
// write a fused attention kernel?", applied per partition. The summation
// order is fixed by the sequence's own partition count.
#include <cfloat>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kGenericThreads = 128;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

template <typename T>
__global__ void __launch_bounds__(kGenericThreads)
decode_generic_kernel(const DecodeParams p, int group) {
    using E = ElemTraits<T>;
    extern __shared__ float sm[];
    const int D = p.head_dim;
    const int PS = max(p.partition_size, p.partition_long);   // score row stride
    float* qf = sm;                           // [group][D]
    float* sc = qf + group * D;               // [group][PS]
    float* red = sc + group * PS;             // [group][2]: max, sum
    int32_t* ids = reinterpret_cast<int32_t*>(red + 2 * group);   // partition's block ids
    __shared__ int bad;

    const int bh = p.num_seqs * p.num_kv_heads;
    const int part = blockIdx.x / bh;
    const int rem = blockIdx.x - part * bh;
    const int s = rem / p.num_kv_heads;
    const int h = rem - s * p.num_kv_heads;
    const int n = __ldg(p.context_lens + s);
    if (n < 0 || n > p.context_cap) {
        if (threadIdx.x == 0 && part == 0 && h == 0) raise_error(p.error_word, PA_DEVERR_CONTEXT);
        return;
    }
    const int P = seq_partition(p, n);        // rows per partition of this sequence
    const int lo = part * P;
    const size_t row0 = static_cast<size_t>(s) * p.num_heads + static_cast<size_t>(h) * group;
    if (n == 0) {
        if (part == 0)
            for (int i = threadIdx.x; i < group * D; i += blockDim.x)
                E::store(static_cast<T*>(p.out) + row0 * D + i, 0.f);
        return;
    }
    if (lo >= n) return;
    const int hi = min(n, lo + P);
    const int len = hi - lo;
    const int nparts = (n + P - 1) / P;
    const int bs = p.block_size;
    const int b0 = lo / bs;
    const int nblk = (hi - 1) / bs - b0 + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;

    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
        const int id = __ldg(p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq + b0 + j);
        if (id < 0 || id >= p.num_blocks) bad = 1;
        ids[j] = id;
    }
    const T* q = static_cast<const T*>(p.q) + row0 * D;
    for (int i = threadIdx.x; i < group * D; i += blockDim.x) qf[i] = E::load(q + i) * p.scale_log2;
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) raise_error(p.error_word, PA_DEVERR_BLOCK_ID);
        return;
    }
    const T* kc = static_cast<const T*>(p.k_cache);
    const T* vc = static_cast<const T*>(p.v_cache);
    auto row_of = [&](int i) -> size_t {
        const int tok = lo + i;
        const size_t blk = static_cast<size_t>(ids[tok / bs - b0]);
        return ((blk * p.num_kv_heads + h) * bs + (tok % bs)) * static_cast<size_t>(D);
    };

    // scores, base 2: one warp per row, lanes over head dims
    for (int i = warp; i < len; i += nwarps) {
        const T* krow = kc + row_of(i);
        for (int g = 0; g < group; ++g) {
            float acc = 0.f;
            for (int d = lane; d < D; d += 32) acc = fmaf(qf[g * D + d], E::load(krow + d), acc);
            acc = warp_sum(acc);
            if (lane == 0) sc[g * PS + i] = acc;
        }
    }
    __syncthreads();
    // softmax per query head: one warp per head
    for (int g = warp; g < group; g += nwarps) {
        float mx = -INFINITY;
        for (int i = lane; i < len; i += 32) mx = fmaxf(mx, sc[g * PS + i]);
        mx = warp_max(mx);
        float sum = 0.f;
        for (int i = lane; i < len; i += 32) {
            const float e = fast_exp2(sc[g * PS + i] - mx);
            sc[g * PS + i] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            red[2 * g] = mx;
            red[2 * g + 1] = sum;
        }
    }
    __syncthreads();
    // P.V: threads over (head, dim)
    for (int idx = threadIdx.x; idx < group * D; idx += blockDim.x) {
        const int g = idx / D, d = idx - g * D;
        float acc = 0.f;
        for (int i = 0; i < len; ++i) acc = fmaf(sc[g * PS + i], E::load(vc + row_of(i) + d), acc);
        const size_t row = row0 + g;
        if (nparts == 1) {
            E::store(static_cast<T*>(p.out) + row * D + d, acc / red[2 * g + 1]);
        } else {
            const size_t slot = row * p.max_parts + part;
            p.part_o[slot * D + d] = acc;
            if (d == 0) {
                p.part_ml[2 * slot] = red[2 * g];
                p.part_ml[2 * slot + 1] = red[2 * g + 1];
            }
        }
    }
}

constexpr int kCombineChunk = 32;          // partitions per warp per pass (one per lane)
constexpr int kCombineMaxWarps = 16;
constexpr int kCombineMaxElems = kMaxHeadDim / 32;   // output elements per lane
constexpr int kCombineBatch = 8;           // partitions whose o rows are loaded before use
// Query heads per CTA (one warp each) when every sequence fits one warp's
// chunk of partitions: fewer, larger CTAs for the same per-head work.
constexpr int kCombineHeadsPerCta = 4;

// Warps used for a sequence of np partitions: warp w takes chunks w, w + nw,
// ... of 32 consecutive partitions. Depends on np only, so a sequence's
// summation order does not depend on the rest of the batch.
__host__ __device__ __forceinline__ int combine_warps(int np) {
    const int w = (np + kCombineChunk - 1) / kCombineChunk;
    return w < kCombineMaxWarps ? w : kCombineMaxWarps;
}

// One CTA per (sequence, query token, query head) of a sequence longer than
// one partition (one query token per sequence for plain decode), or with
// HPB > 1 (every sequence within one warp's chunk of partitions) one CTA per
// HPB query heads, a warp each.
// Each warp merges its chunks (lane q holds partition q's max and sum; the o
// rows are loaded kCombineBatch partitions at a time), then the warp results
// are merged in warp order.
template <typename T, int E, int HPB>
__global__ void __launch_bounds__(kCombineMaxWarps * 32) combine_kernel(const DecodeParams p) {
    extern __shared__ float sm[];                // [nw][2 + head_dim]
    const int qh = HPB > 1 ? blockIdx.x * HPB + (threadIdx.x >> 5) : blockIdx.x;
    const int sq = blockIdx.y;                 // s * num_queries + query token
    const int s = sq / p.num_queries;
    // Launched as a programmatic dependent of a decode kernel. The context
    // lengths are read before griddepcontrol.wait, which is safe because no
    // decode kernel writes them and every decode kernel either triggers this
    // grid only after its own griddepcontrol.wait (the tile-ring kernels:
    // every kernel before them has completed by then) or never triggers it
    // (the direct-load kernel, which therefore completes first). A decode
    // kernel that triggered earlier would break this. A sequence of one
    // partition (written directly by the decode kernel) leaves at once. CTA
    // (0, 0) always waits, so that this grid never completes before the
    // decode kernel does.
    const int n = __ldg(p.context_lens + s);
    const int span = n - seq_row_base(n, p.window);       // rows of the partitions
    const int P = seq_partition(p, span);
    const bool merge = n <= p.context_cap && n >= p.num_queries && span > P;   // else flagged or one partition
    if (!merge && (blockIdx.x | blockIdx.y) != 0) return;
    asm volatile("griddepcontrol.wait;" ::: "memory");    // the partials are the decode kernel's output
    if (!merge) return;
    const int np = (span + P - 1) / P;
    const int nw = HPB > 1 ? 1 : combine_warps(np);
    const int D = p.head_dim;
    const size_t row = static_cast<size_t>(sq) * p.num_heads + qh;
    const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + row * p.max_parts;
    const float* o = p.part_o + row * p.max_parts * static_cast<size_t>(D);
    const int warp = HPB > 1 ? 0 : threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < nw) {
        float M = -INFINITY, L = 0.f;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        for (int c0 = warp * kCombineChunk; c0 < np; c0 += nw * kCombineChunk) {
            const int cnt = min(kCombineChunk, np - c0);
            const float2 v = lane < cnt ? ml[c0 + lane] : make_float2(-INFINITY, 0.f);
            // The first o rows are loaded together with the maxima.
            float ov[kCombineBatch][E];
#pragma unroll
            for (int k = 0; k < kCombineBatch; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int d = lane + 32 * e;
                    ov[k][e] = (k < cnt && d < D) ? o[static_cast<size_t>(c0 + k) * D + d] : 0.f;
                }
            const float Mc = fmaxf(M, warp_max(v.x));
            // Partitions a query token does not reach (several tokens per
            // sequence) hold m = -inf, l = 0: weight 0, never NaN.
            const float ref = Mc == -INFINITY ? 0.f : Mc;
            const float w = lane < cnt ? fast_exp2(v.x - ref) : 0.f;
            const float rescale = fast_exp2(M - ref);         // 0 on the first chunk
            L = L * rescale + warp_sum(w * v.y);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] *= rescale;
            M = Mc;
            for (int i = 0; i < cnt; i += kCombineBatch) {
                if (i > 0) {
#pragma unroll
                    for (int k = 0; k < kCombineBatch; ++k)
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const int d = lane + 32 * e;
                            ov[k][e] = (i + k < cnt && d < D)
                                           ? o[static_cast<size_t>(c0 + i + k) * D + d] : 0.f;
                        }
                }
#pragma unroll
                for (int k = 0; k < kCombineBatch; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, w, (i + k) & 31);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, ov[k][e], acc[e]);
                }
            }
        }
        if (nw == 1) {
            // One warp merged every partition: store from its registers (the
            // same values the cross-warp merge below would give: 2^0 = 1).
            T* out = static_cast<T*>(p.out) + row * D;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int d = lane + 32 * e;
                if (d < D) ElemTraits<T>::store(out + d, acc[e] / L);
            }
        } else {
            float* st = sm + warp * (D + 2);
            if (lane == 0) {
                st[0] = M;
                st[1] = L;
            }
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int d = lane + 32 * e;
                if (d < D) st[2 + d] = acc[e];
            }
        }
    }
    if (nw == 1) return;                       // the same for every thread of the CTA
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, sm[w * (D + 2)]);
    float L = 0.f;
    for (int w = 0; w < nw; ++w) L = fmaf(fast_exp2(sm[w * (D + 2)] - M), sm[w * (D + 2) + 1], L);
    T* out = static_cast<T*>(p.out) + row * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.f;
        for (int w = 0; w < nw; ++w) a = fmaf(fast_exp2(sm[w * (D + 2)] - M), sm[w * (D + 2) + 2 + d], a);
        ElemTraits<T>::store(out + d, a / L);
    }
}

}  // namespace

size_t generic_smem_bytes(int group, int head_dim, int partition_size, int block_size) {
    const size_t floats = static_cast<size_t>(group) * head_dim +
                          static_cast<size_t>(group) * partition_size + 2 * static_cast<size_t>(group);
    const size_t ids = static_cast<size_t>(partition_size) / block_size + 2;
    return 4 * (floats + ids);
}

cudaError_t launch_decode_generic(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream) {
    const int group = p.num_heads / p.num_kv_heads;
    const size_t smem = generic_smem_bytes(group, p.head_dim,
                                           max(p.partition_size, p.partition_long), p.block_size);
    const long long grid = static_cast<long long>(p.max_parts) * p.num_seqs * p.num_kv_heads;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t err;
    if (dtype == PA_DTYPE_BF16) {
        err = cudaFuncSetAttribute(decode_generic_kernel<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        decode_generic_kernel<__nv_bfloat16>
            <<<static_cast<unsigned>(grid), kGenericThreads, smem, stream>>>(p, group);
    } else {
        err = cudaFuncSetAttribute(decode_generic_kernel<float>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        decode_generic_kernel<float>
            <<<static_cast<unsigned>(grid), kGenericThreads, smem, stream>>>(p, group);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream) {
    if (p.max_parts <= 1 || p.num_seqs == 0) return cudaSuccess;
    const int warps = combine_warps(p.max_parts);   // enough for the longest sequence
    // One warp per head merges every partition: several heads per CTA.
    const bool packed = warps == 1 && kCombineHeadsPerCta > 1 &&
                        p.num_heads % kCombineHeadsPerCta == 0;
    const size_t smem = packed ? 0 : static_cast<size_t>(warps) * (p.head_dim + 2) * sizeof(float);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(packed ? p.num_heads / kCombineHeadsPerCta : p.num_heads,
                       p.num_seqs * p.num_queries);
    cfg.blockDim = dim3(packed ? 32 * kCombineHeadsPerCta : 32 * warps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Output elements per lane: exact for head dims 64 and 128, else the maximum.
    auto pick = [&](auto tag) -> cudaError_t {
        using T = decltype(tag);
        // At most 16 warps x (256 + 2) floats: within the default shared-memory limit.
        auto run = [&](auto kernel) -> cudaError_t { return cudaLaunchKernelEx(&cfg, kernel, p); };
        constexpr int H = kCombineHeadsPerCta;
        if (p.head_dim == 128) return packed ? run(combine_kernel<T, 4, H>) : run(combine_kernel<T, 4, 1>);
        if (p.head_dim == 64) return packed ? run(combine_kernel<T, 2, H>) : run(combine_kernel<T, 2, 1>);
        return packed ? run(combine_kernel<T, kCombineMaxElems, H>)
                      : run(combine_kernel<T, kCombineMaxElems, 1>);
    };
    cudaError_t err = dtype == PA_DTYPE_BF16 ? pick(__nv_bfloat16{}) : pick(float{});
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pa
