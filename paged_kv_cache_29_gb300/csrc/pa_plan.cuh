// pa_plan.cuh -- the work list of one persistent decode launch, computed by
// every CTA of that launch for itself.
//
// A work item is one (sequence, KV head, partition) of at most
// seq_partition(span) rows (partitions start at seq_row_base: row 0, or the
// tile holding the first row of a sliding window). The items of the batch
// are numbered in one global order, largest first:
//   1. every full partition of the sequences that take partition_long rows,
//      by sequence, partition, KV head;
//   2. every full partition of the others (partition_size rows), likewise;
//   3. then the partial last partitions, in kPlanBuckets buckets of
//      decreasing size (by sequence within a bucket), so that the last items
//      a persistent CTA picks up are the smallest.
// CTA c of C processes items c, 2C-1-c, 2C+c, ... (a snake, so that the
// per-CTA totals even out). Each CTA walks the context lengths twice (the
// prefix of full partitions, then the bucket ranks) and writes only its own
// items into the workspace, which it then reads back in order; no other CTA
// touches them. The order only decides which CTA does what and when: every
// item's result and the merge order of a sequence's partitions are fixed by
// the sequence's own length, so the output does not depend on the rest of the
// batch.
//
// The walk also writes the zero output rows of empty sequences (sequence s by
// CTA s % C) and flags context lengths outside [0, max_context_len] (those
// sequences get no items).
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kPlanBuckets = 16;

// CTA c's j-th item in a snake over C CTAs.
__device__ __forceinline__ int snake_item(int c, int j, int C) {
    return j * C + ((j & 1) ? (C - 1 - c) : c);
}

// Number of items CTA c owns when the launch has `total` items.
__device__ __forceinline__ int own_item_count(int c, int C, int total) {
    const int rounds = total / C;
    const int rem = total - rounds * C;
    const int pos = (rounds & 1) ? (C - 1 - c) : c;   // its slot in the last, partial round
    return rounds + (pos < rem ? 1 : 0);
}

// Shared ints plan_cta needs for NT threads.
__host__ __device__ constexpr int plan_scratch_ints(int nt) {
    return (nt / 32) * (1 + kPlanBuckets) + 3 * kPlanBuckets + 4;   // carry: 4
}

// Calls f(k) for every k in [a, e) that is one of CTA c's items.
template <typename F>
__device__ __forceinline__ void for_own_items(int a, int e, int c, int C, F&& f) {
    if (a >= e) return;
    for (int j = a / C; j * C < e; ++j) {
        const int k = snake_item(c, j, C);
        if (k >= a && k < e) f(k);
    }
}

// Context length of sequence s, or -1 (flagged) when it is out of range
// (negative, past max_context_len, or shorter than the query tokens it holds).
__device__ __forceinline__ int plan_len(const DecodeParams& p, int s, bool flag) {
    int n = __ldg(p.context_lens + s);
    if (n < 0 || n > p.context_cap || (n > 0 && n < p.num_queries)) {
        if (flag) raise_error(p.error_word, PA_DEVERR_CONTEXT);
        n = -1;
    }
    return n;
}

// Size bucket of a partial partition of r rows: 0 for the largest (r close to
// P, the partition size of short sequences, or above it: the partial last
// partitions of long sequences all fall in bucket 0), kPlanBuckets - 1 for the
// smallest.
__device__ __forceinline__ int plan_bucket(int r, int P) {
    return r > 0 ? min(kPlanBuckets - 1, max(0, ((P - r) * kPlanBuckets) / P)) : -1;
}

// Barrier among the plan's threads: the whole CTA (BAR = 0) or the first NT
// threads on named barrier BAR.
template <int NT, int BAR>
__device__ __forceinline__ void plan_sync() {
    if constexpr (BAR == 0) {
        __syncthreads();
    } else {
        named_barrier(BAR, NT);
    }
}

// Exclusive prefix of v over the plan's NT = 32 NW threads, starting at
// *carry, which then grows by their sum. All NT threads call it; wsum holds
// NW ints.
template <int NW, int BAR>
__device__ __forceinline__ int block_scan(int v, int* wsum, int* carry) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    plan_sync<NW * 32, BAR>();
    int base = *carry, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) base += wsum[w];
        total += wsum[w];
    }
    plan_sync<NW * 32, BAR>();
    if (tid == 0) *carry += total;
    return base + incl - v;
}

// Writes CTA c's items and returns the number of items of the launch; the
// CTA's first two items also go to `first` (shared memory), so that its work
// starts without a global-memory round trip. Threads 0 .. NT - 1 of the CTA
// call it (all of them with BAR = 0, else they meet on named barrier BAR);
// `sm` holds plan_scratch_ints(NT) ints. Row bytes of the output (num_heads *
// head_dim * sizeof(T)) are a multiple of 16.
template <typename T, int NT, int BAR = 0>
__device__ int plan_cta(const DecodeParams& p, int c, int C, int* sm, int4* first) {
    constexpr int NW = NT / 32;
    int* wsum = sm;                          // [NW]
    int* wcnt = wsum + NW;                   // [NW][kPlanBuckets]
    int* bcount = wcnt + NW * kPlanBuckets;  // [kPlanBuckets]
    int* bcursor = bcount + kPlanBuckets;    // [kPlanBuckets]
    int* brun = bcursor + kPlanBuckets;      // [kPlanBuckets]
    // [0] long full partitions so far, [1] short full partitions, [2] short
    // full partitions so far (pass 2, after the long ones), [3] total items
    int* carry = brun + kPlanBuckets;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.num_seqs, Hkv = p.num_kv_heads;
    const int Pb = p.partition_size;
    if (tid < kPlanBuckets) {
        bcount[tid] = 0;
        brun[tid] = 0;
    }
    if (tid < 4) carry[tid] = 0;
    plan_sync<NT, BAR>();

    // The order: full partitions of long sequences (partition_long rows),
    // then full partitions of the others (partition_size rows), each by
    // sequence, partition, KV head; then the partial last partitions by size
    // bucket, largest first, by sequence within a bucket.
    // Pass 1: exclusive prefix of the long full partitions, chunk by chunk;
    // emit those items; total the short full partitions; count partial
    // partitions per bucket.
    for (int s0 = 0; s0 < B; s0 += NT) {
        const int s = s0 + tid;
        const int n = s < B ? plan_len(p, s, s % C == c) : -1;
        const int span = n > 0 ? n - seq_row_base(n, p.window) : 0;   // rows of its partitions
        const int P = seq_partition(p, span);
        const bool lng = P != Pb;
        const int nf = span / P;
        const int pf = block_scan<NW, BAR>(lng ? nf : 0, wsum, &carry[0]);   // long full partitions before s
        if (!lng && nf > 0) atomicAdd(&carry[1], nf);
        if (lng)
            for_own_items(pf * Hkv, (pf + nf) * Hkv, c, C, [&](int k) {
                const int unit = k / Hkv;
                const int4 v = make_int4(s, k - unit * Hkv, unit - pf, n);
                p.items[k] = v;
                if (k < 2 * C) first[k / C] = v;
            });
        const int b = n > 0 ? plan_bucket(span % P, Pb) : -1;
        if (b >= 0) atomicAdd(&bcount[b], 1);
        if (n == 0 && s % C == c) {
            // A fused append for an empty sequence has no row to go to.
            if (p.slot_mapping != nullptr && __ldg(p.slot_mapping + s) >= 0)
                raise_error(p.error_word, PA_DEVERR_SLOT);
            // the sequence's num_queries output rows
            const int chunks =
                p.num_queries * p.num_heads * p.head_dim * static_cast<int>(sizeof(T)) / 16;
            uint4* row = reinterpret_cast<uint4*>(
                static_cast<T*>(p.out) +
                static_cast<size_t>(s) * p.num_queries * p.num_heads * p.head_dim);
            for (int i = 0; i < chunks; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    plan_sync<NT, BAR>();
    if (tid == 0) {
        int acc = 0;
        for (int b = 0; b < kPlanBuckets; ++b) {
            bcursor[b] = acc;
            acc += bcount[b];
        }
        carry[3] = (carry[0] + carry[1] + acc) * Hkv;
        carry[2] = carry[0];            // the short full partitions start here
    }
    plan_sync<NT, BAR>();
    const int full_items = (carry[0] + carry[1]) * Hkv;
    const int total = carry[3];

    // Pass 2: the short full partitions (prefix again, after the long ones),
    // and each partial partition's rank: bucket start, then earlier sequences
    // of the same bucket (earlier chunks, earlier warps, earlier lanes).
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int s0 = 0; s0 < B; s0 += NT) {
        const int s = s0 + tid;
        const int n = s < B ? plan_len(p, s, false) : -1;
        const int span = n > 0 ? n - seq_row_base(n, p.window) : 0;
        const int P = seq_partition(p, span);
        const bool lng = P != Pb;
        const int nf = span / P;
        const int pf = block_scan<NW, BAR>(lng ? 0 : nf, wsum, &carry[2]);
        if (!lng)
            for_own_items(pf * Hkv, (pf + nf) * Hkv, c, C, [&](int k) {
                const int unit = k / Hkv;
                const int4 v = make_int4(s, k - unit * Hkv, unit - pf, n);
                p.items[k] = v;
                if (k < 2 * C) first[k / C] = v;
            });
        const int b = n > 0 ? plan_bucket(span % P, Pb) : -1;
        const unsigned same = __match_any_sync(0xffffffffu, b);
        if (lane < kPlanBuckets) wcnt[warp * kPlanBuckets + lane] = 0;
        __syncwarp();
        if (b >= 0 && (same & lt_mask) == 0) wcnt[warp * kPlanBuckets + b] = __popc(same);
        plan_sync<NT, BAR>();
        if (b >= 0) {
            int j = bcursor[b] + brun[b] + __popc(same & lt_mask);
            for (int w = 0; w < warp; ++w) j += wcnt[w * kPlanBuckets + b];
            const int a = full_items + j * Hkv;
            for_own_items(a, a + Hkv, c, C, [&](int k) {
                const int4 v = make_int4(s, k - a, nf, n);
                p.items[k] = v;
                if (k < 2 * C) first[k / C] = v;
            });
        }
        plan_sync<NT, BAR>();
        if (tid < kPlanBuckets) {
            int add = 0;
            for (int w = 0; w < NW; ++w) add += wcnt[w * kPlanBuckets + tid];
            brun[tid] += add;
        }
        plan_sync<NT, BAR>();
    }
    return total;
}

}  // namespace pa
