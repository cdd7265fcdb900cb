// pa_plan.cu -- the work list of one decode call.
//
// A work item is one (sequence, KV head, partition) of at most partition_size
// rows. One CTA reads the context lengths and writes, into the workspace, the
// item count and the items in processing order:
//   1. every full partition (partition_size rows), by sequence, partition,
//      KV head;
//   2. then the partial last partitions, in 16 buckets of decreasing size, so
//      that the last items a persistent CTA picks up are the smallest.
// The order only decides which CTA does what and when; every item's result
// and the merge order of a sequence's partitions are fixed by the sequence's
// own length, so the output does not depend on the rest of the batch.
//
// It also writes the zero output rows of empty sequences and flags context
// lengths outside [0, max_context_len] (those sequences get no items).
#include <atomic>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kPlanThreads = 256;
constexpr int kBuckets = 16;

__device__ __forceinline__ void grid_dependency_wait_() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents_() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const DecodeParams p) {
    // The decode kernel may launch and set up its rings now; it reads nothing
    // this kernel writes before its own griddepcontrol.wait.
    grid_launch_dependents_();
    extern __shared__ int sm[];
    const int B = p.num_seqs;
    int* lens = sm;              // [B], -1 = invalid
    int* pf = lens + B;          // [B + 1] exclusive prefix of full partitions
    int* rank = pf + B + 1;      // [B] position among partial items
    __shared__ int count[kBuckets], cursor[kBuckets];
    __shared__ int warp_sum[32];
    __shared__ int partials;
    const int P = p.partition_size;
    const int Hkv = p.num_kv_heads;
    const int tid = threadIdx.x;

    for (int s = tid; s < B; s += blockDim.x) {
        int n = __ldg(p.context_lens + s);
        if (n < 0 || n > p.context_cap) {
            raise_error(p.error_word, PA_DEVERR_CONTEXT);
            n = -1;
        }
        lens[s] = n;
    }
    if (tid < kBuckets) count[tid] = 0;
    __syncthreads();

    // Zero output rows of empty sequences (one warp per sequence).
    const int row_elems = p.num_heads * p.head_dim;
    for (int s = tid >> 5; s < B; s += blockDim.x >> 5) {
        if (lens[s] != 0) continue;
        T* out = static_cast<T*>(p.out) + static_cast<size_t>(s) * row_elems;
        for (int i = tid & 31; i < row_elems; i += 32) ElemTraits<T>::store(out + i, 0.f);
    }

    // Exclusive prefix of full partitions: each thread owns a contiguous run.
    const int per = (B + kPlanThreads - 1) / kPlanThreads;
    const int s0 = tid * per;
    int local = 0;
    for (int s = s0; s < min(B, s0 + per); ++s) local += lens[s] > 0 ? lens[s] / P : 0;
    int incl = local;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (kPlanThreads >> 5) ? warp_sum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += v;
        }
        if (lane < (kPlanThreads >> 5)) warp_sum[lane] = wi - w;   // exclusive prefix of warp totals
    }
    __syncthreads();
    int run = warp_sum[warp] + incl - local;
    for (int s = s0; s < min(B, s0 + per); ++s) {
        pf[s] = run;
        run += lens[s] > 0 ? lens[s] / P : 0;
    }
    if (s0 < B && s0 + per >= B) pf[B] = run;
    if (B == 0 && tid == 0) pf[0] = 0;

    // Partial partitions by decreasing size bucket.
    for (int s = tid; s < B; s += blockDim.x) {
        const int r = lens[s] > 0 ? lens[s] % P : 0;
        if (r > 0) atomicAdd(&count[min(kBuckets - 1, ((P - r) * kBuckets) / P)], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int b = 0; b < kBuckets; ++b) {
            cursor[b] = acc;
            acc += count[b];
        }
        partials = acc;
    }
    __syncthreads();
    for (int s = tid; s < B; s += blockDim.x) {
        const int r = lens[s] > 0 ? lens[s] % P : 0;
        rank[s] = r > 0 ? atomicAdd(&cursor[min(kBuckets - 1, ((P - r) * kBuckets) / P)], 1) : -1;
    }
    __syncthreads();

    const int full_items = pf[B] * Hkv;
    if (tid == 0) p.sched[0] = full_items + partials * Hkv;
    // One warp per sequence writes its items: the full partitions at
    // pf[s] * Hkv (partition-major, KV head fastest), the partial one at its
    // bucket rank.
    for (int s = warp; s < B; s += blockDim.x >> 5) {
        const int n = lens[s];
        if (n <= 0) continue;
        const int nfull = n / P;
        int4* dst = p.items + static_cast<size_t>(pf[s]) * Hkv;
        for (int i = lane; i < nfull * Hkv; i += 32) dst[i] = make_int4(s, i % Hkv, i / Hkv, n);
        if (rank[s] >= 0) {
            int4* pdst = p.items + full_items + static_cast<size_t>(rank[s]) * Hkv;
            for (int h = lane; h < Hkv; h += 32) pdst[h] = make_int4(s, h, nfull, n);
        }
    }
    // The next kernel's griddepcontrol.wait covers this grid only: wait for the
    // kernel before this one (the cache append) so that the chain stays whole.
    grid_dependency_wait_();
}

}  // namespace

size_t plan_smem_bytes(int num_seqs) { return 4 * (3 * static_cast<size_t>(num_seqs) + 1); }

cudaError_t launch_plan(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream) {
    const int smem = static_cast<int>(plan_smem_bytes(p.num_seqs));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // The shared-memory attribute is set once per device, for the largest
    // batch a launch takes.
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= kMaxDevices || !ready[dev].load(std::memory_order_relaxed)) {
        const int max_smem = static_cast<int>(plan_smem_bytes(kPlanMaxSeqs));
        err = cudaFuncSetAttribute(plan_kernel<__nv_bfloat16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(plan_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       max_smem);
        if (err != cudaSuccess) return err;
        if (dev < kMaxDevices) ready[dev].store(1, std::memory_order_relaxed);
    }
    err = dtype == PA_DTYPE_BF16 ? cudaLaunchKernelEx(&cfg, plan_kernel<__nv_bfloat16>, p)
                                 : cudaLaunchKernelEx(&cfg, plan_kernel<float>, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pa
