// pa_decode_stream.cuh -- persistent paged decode attention with a TMA tile ring.
//
// Work item: one (sequence s, KV head h, partition p) of at most
// partition_size rows. A fixed set of CTAs (a few per SM) shares the items of
// the launch; each CTA computes and stores its own items (pa_plan.cuh: full
// partitions first, then the partial last partitions, largest first, dealt
// out in a snake) and streams all of their tiles through one ring without
// stopping between items.
//
// Start-up: the consumer warps compute the CTA's work list while the producer
// warp finds the CTA's first item alone where it can (first_item_by_warp: a
// warp scan of the context lengths), fetches its block ids, issues its first
// tiles and copies its q into the consumers' first q buffer (an mbarrier
// completed by the copies and by a note of which item it is). The producer
// reads the item count and the items after the first once the plan's
// mbarrier completes.
//
// Producer warp: for each item, loads its block ids (one coalesced load,
// validated against the pool, prefetched one item ahead), then for every
// 16-row tile issues 3D TMA loads of the K and V tile (16 rows x head_dim of
// one physical block and KV head, contiguous in the
// [block][kv_head][block_size][head_dim] pool) into the next ring stage. Row i
// of a sequence is row (i % block_size) of block block_tables[s][i /
// block_size]: the paged gather of "MLSys Engineer -- Inference Systems Q&A",
// Q1. Stages are refilled in stream order, or per consumer warp
// (PER_WARP_ISSUE, below). With a fused append (pa_append_decode) the item
// holding a sequence's last row also writes (or quantises) that KV head's new
// K/V row into its slot before the tile holding it is loaded.
//
// Consumer warps: the CTA's tiles are numbered in stream order; tile t lives
// in stage t % STAGES and is consumed by warp t % W (STAGES is a multiple of
// W, so every stage has one owner and parity waits stay within one phase).
// At the end of an item every warp writes its online-softmax state to the
// merge area, the consumer warps meet at a named barrier, the merged result is
// written as the final output (one partition) or as the item's partial (max,
// sum, unnormalised output) for the combine kernel, and a second barrier frees
// the area for the next item (one buffer: with 8 query columns a second one
// would cost a CTA per SM).
//
// Sizing: a random 4 KB tile gather streams at 6.6-6.8 TB/s on GB300 only
// with three or more producers per SM: one producer's per-tile issue chain
// (wait for the oldest stage, arrive with the byte count, issue the copies)
// moves ~15 GB/s however deep its ring. So the kernel runs several small CTAs
// per SM, each with a short ring.
//
// Programmatic dependent launch: only ring and barrier set-up come before
// griddepcontrol.wait; every global access (context lengths, the work list,
// block tables, q, the KV pool, the output) comes after it, so a launch never
// touches memory that the kernel before it on the stream still uses. The
// merge kernel after it may launch at once (griddepcontrol.launch_dependents
// right after the wait) and waits for this grid itself.
#pragma once

#include <atomic>
#include <climits>

#include "pa_plan.cuh"
#include "pa_tile_math.cuh"

namespace pa {

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block ids of one item: partitions of up to 4096 rows span at most
// 4096 / 16 + 1 = 257 blocks when block_size is a multiple of 16.
constexpr int kMaxItemBlocks = 260;

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_group_1() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// CTA c's first item as one warp can find it without the plan, or x = -1.
// With one partition size for every sequence, item c of the launch (the
// snake's first round) is, while c is below the full partitions' count times
// Hkv, full partition c / Hkv in sequence order with KV head c % Hkv: the
// order the plan gives its full partitions. A warp-wide scan of the
// full-partition counts over the context lengths finds its sequence; a
// flagged length counts no partition, as in the plan.
__device__ __forceinline__ int4 first_item_by_warp(const DecodeParams& p, int c, int lane) {
    if (p.partition_long != p.partition_size) return make_int4(-1, 0, 0, 0);
    const int Hkv = p.num_kv_heads;
    const int unit = c / Hkv;
    int carry = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
        const int s = s0 + lane;
        const int n = s < p.num_seqs ? plan_len(p, s, false) : -1;
        const int nf = n > 0 ? (n - seq_row_base(n, p.window)) / p.partition_size : 0;
        int incl = nf;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += u;
        }
        const int first = carry + incl - nf;   // full partitions before sequence s
        const unsigned hit = __ballot_sync(0xffffffffu, unit >= first && unit < first + nf);
        if (hit != 0u) {
            const int src = __ffs(hit) - 1;
            return make_int4(s0 + src, c - unit * Hkv, unit - __shfl_sync(0xffffffffu, first, src),
                             __shfl_sync(0xffffffffu, n, src));
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    return make_int4(-1, 0, 0, 0);
}

template <int W, int STAGES, typename Geom, int G, int D, int Math_kQBufBytes, int XBYTES,
          bool PER_WARP_ISSUE>
struct StreamSmem {
    static constexpr int kRing = STAGES * Geom::kStageBytes;
    static constexpr int kState = 2 * G + G * D;        // m[G], l[G], o[G][D]
    static constexpr int kMerge = W * kState * 4;       // the warps' states at an item's end
    // full[STAGES], empty[STAGES], the plan's completion (+ 8 bytes of padding)
    static constexpr int kBarriers = (2 * STAGES + 2) * 8;
    // stage_bad[STAGES], warp_bad[2 W], abort flag (+7), with per-warp issue
    // last_t[STAGES] and imeta[16]; then (16-byte aligned) the CTA's first two
    // items
    static constexpr int kFlagInts = STAGES + 2 * W + 8 + (PER_WARP_ISSUE ? STAGES + 16 : 0);
    static constexpr int kFirstItemsOffset = (kFlagInts * 4 + 15) / 16 * 16;
    static constexpr int kFlags = kFirstItemsOffset + 2 * 16;
    static constexpr int kIds = 2 * kMaxItemBlocks * 4;
    static constexpr size_t kQBuf = 2 * Math_kQBufBytes;
    static constexpr size_t kExtra = static_cast<size_t>(STAGES) * XBYTES;   // per-stage side data
    static constexpr size_t kBytes =
        1024 + kRing + kMerge + kBarriers + kFlags + kIds + kQBuf + kExtra;
};

// MIN_CTAS: resident CTAs per SM the register budget is sized for (see
// "Sizing" above). PER_WARP_ISSUE: the producer refills each consumer warp's
// stages independently (instead of in stream order), which pays where the
// consumers' per-tile math is long (8-bit caches) and costs ~1 % where the
// kernel streams at the bandwidth limit (bf16).
template <class Math, int D, int G, int W, int STAGES, int MIN_CTAS, bool PER_WARP_ISSUE>
__global__ void __launch_bounds__((W + 1) * 32, MIN_CTAS)
decode_stream_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    static_assert(STAGES % W == 0, "each ring stage must belong to exactly one consumer warp");
    static_assert(STAGES <= 32 && W <= 32, "the producer warp keeps one lane per stage and per consumer warp");
    using T = typename Math::T;
    using Geom = typename Math::Geom;
    using Smem = StreamSmem<W, STAGES, Geom, G, D, Math::kQBufBytes, Math::kExtraStageBytes,
                            PER_WARP_ISSUE>;
    static_assert(Math::kExtraStageBytes % 16 == 0, "side data moves in 16-byte units");
    static_assert(Smem::kMerge >= 4 * plan_scratch_ints(W * 32),
                  "the plan's scratch lives in the merge area");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* merge = reinterpret_cast<float*>(ring + Smem::kRing);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + Smem::kRing + Smem::kMerge);
    uint64_t* empty = full + STAGES;
    uint64_t* plan_bar = empty + STAGES;                      // the consumers' plan is complete
    uint64_t* q0_bar = empty + STAGES + 1;                    // the producer's copy of item 0's q
    uint64_t* flags_base = empty + STAGES + 2;
    volatile int32_t* stage_bad = reinterpret_cast<volatile int32_t*>(flags_base);
    volatile int32_t* warp_bad = stage_bad + STAGES;          // [2][W]: per item parity
    volatile int32_t* abort_flag = warp_bad + 2 * W;
    volatile int32_t* total_sm = abort_flag + 1;              // the launch's item count (the plan's)
    volatile int32_t* q0_sm = abort_flag + 2;                 // (sequence, KV head) of that copy, or -1
    // per-warp issue only: the producer's last tile per stage, item meta [2][8]
    volatile int32_t* last_t = abort_flag + 8;
    volatile int32_t* imeta = last_t + STAGES;
    int4* first_items = reinterpret_cast<int4*>(
        reinterpret_cast<uint8_t*>(flags_base) + Smem::kFirstItemsOffset);   // [2]
    int32_t* ids_buf = reinterpret_cast<int32_t*>(
        reinterpret_cast<uint8_t*>(flags_base) + Smem::kFlags);   // [2][kMaxItemBlocks]
    uint8_t* qbuf = reinterpret_cast<uint8_t*>(ids_buf + 2 * kMaxItemBlocks);   // [2][kQBufBytes]
    // [STAGES][kExtraStageBytes]: per-row scales of a stage's K and V tiles
    const uint32_t xring = smem_addr(qbuf + Smem::kQBuf);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        mbar_init(smem_addr(plan_bar), 1);
        // the producer lanes' copies (one completion each) and lane 0's note
        mbar_init(smem_addr(q0_bar), 33);
        abort_flag[0] = 0;
        mbar_init_fence();
    }
    if (warp == W && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    __syncthreads();
    grid_dependency_wait();
    grid_launch_dependents();

    const int C = gridDim.x;
    const int c = blockIdx.x;
    // The CTA's work list, computed by the consumer warps (named barrier 1)
    // while the producer warp starts on the first item where it can find that
    // item alone (below); its scratch is the merge area, free until the first
    // item ends. The items are read back with plain (coherent) loads. The
    // producer reads the item count and any item after its first one only
    // after the plan barrier completes.
    int total = 0;
    if (warp < W) {
        total = plan_cta<T, W * 32, 1>(p, c, C, reinterpret_cast<int*>(merge), first_items);
        named_barrier(1, W * 32);       // every consumer's item writes precede the arrival
        if (threadIdx.x == 0) {
            total_sm[0] = total;
            mbar_arrive(smem_addr(plan_bar));
        }
    }
    // The CTA's j-th item (x = -1: none): the first two from shared memory.
    auto own_item = [&](int j) -> int4 {
        const int k = snake_item(c, j, C);
        if (k >= total) return make_int4(-1, 0, 0, 0);
        return j < 2 ? first_items[j] : p.items[k];
    };
    const int bs = p.block_size;
    // Rows per partition of the sequence an item belongs to (n rows).
    auto part_rows = [&](int n) { return seq_partition(p, n - seq_row_base(n, p.window)); };
    const uint32_t ring_addr = smem_addr(ring);

    if (warp == W) {
        // ------------------------------ producer ------------------------------
        // The CTA's first item where this warp can find it alone
        // (first_item_by_warp); its q goes to the consumers' first q buffer at
        // once (they take it from there if the plan gives them the same item,
        // after the completion of every lane's copies and lane 0's note of
        // which item it is).
        const int4 first = first_item_by_warp(p, c, lane);
        if constexpr (Math::kQInSmem) {
            if (first.x >= 0) {
                const int grp0 = Math::kCausal ? p.num_heads / p.num_kv_heads : G;
                Math().stage_q(p, first.x, first.y, Math::kCausal ? grp0 * p.num_queries : G, grp0,
                               smem_addr(qbuf), lane);
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(q0_bar))
                         : "memory");
            if (lane == 0) {
                q0_sm[0] = first.x;
                q0_sm[1] = first.y;
                mbar_arrive(smem_addr(q0_bar));
            }
        }
        if constexpr (PER_WARP_ISSUE) {
            // Consumer warp w takes tiles w, w + W, ... of every item, in ring
            // stages w, w + W, ... . Lane w < W of this warp issues warp w's tiles
            // in order; the W streams are independent, so a stage is refilled as
            // soon as its own consumer frees it, whatever the other consumer warps
            // are doing. The lanes stay converged: in every round each lane whose
            // next stage is free issues its tile (arrive.expect_tx, then the K and
            // V boxes); a round in which nothing moved sleeps on the empty barrier
            // of the oldest outstanding tile.
            //
            // Items: the consumer warps meet at the end of every item, so no lane
            // runs more than one item ahead of the slowest one. The block ids of
            // item j (one coalesced cp.async, checked against the pool) live in
            // buffer j & 1; those of item j + 1 are fetched once every lane has
            // entered item j. Item descriptors are read two items ahead, once
            // the consumers' plan is complete; the first item, where this warp
            // found it alone, starts before that (its item count unknown
            // until then: no lane leaves the first item before the plan).
            bool planned = false;
            int n_items = INT_MAX;
            auto load_item = own_item;
            if (first.x < 0) {
                bool plan_ok = true;
                if (lane == 0) plan_ok = mbar_wait(smem_addr(plan_bar), 0);
                plan_ok = __shfl_sync(0xffffffffu, plan_ok, 0);
                if (!plan_ok && lane == 0) {
                    raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                    abort_flag[0] = 1;
                }
                total = plan_ok ? total_sm[0] : 0;
                n_items = own_item_count(c, C, total);
                planned = true;
            }
            if (lane < STAGES) last_t[lane] = -1;
            // descriptor of item jl, the next whose ids to fetch, and the one after
            int4 d_req = planned ? load_item(0) : first;
            int4 d_req2 = planned ? load_item(1) : make_int4(-1, 0, 0, 0);
            int4 d_val = make_int4(-1, 0, 0, 0);   // descriptor of the requested, unchecked item
            // Fused append: this lane's share of that item's new K and V rows,
            // loaded at the request (used once its block ids are checked).
            uint2 new_k = make_uint2(0u, 0u), new_v = make_uint2(0u, 0u);
            int jl = 0;                     // items whose ids were requested
            int ready = 0;                  // items whose ids landed and were checked
            int t_req = 0;                  // stream index of item jl's first tile
            // Item meta in shared memory, slot j & 1: blocks, KV head, first row,
            // first block, tiles, tiles per consumer warp, first stream index, bad.
            auto request = [&]() {
                const int4 it = d_req;
                const int P = part_rows(it.w);
                const int lo = seq_row_base(it.w, p.window) + it.z * P;
                const int hi = min(it.w, lo + P);
                const int b0 = lo / bs;
                const int nblk = (hi - 1) / bs - b0 + 1;
                const int ntiles = (hi - lo + kTileRows - 1) / kTileRows;
                const int share = (ntiles + W - 1) / W;
                int32_t* buf = ids_buf + (jl & 1) * kMaxItemBlocks;
                const int32_t* bt = p.block_tables + static_cast<size_t>(it.x) * p.max_blocks_per_seq + b0;
                for (int i = lane; i < nblk; i += 32) cp_async_4(smem_addr(buf + i), bt + i);
                cp_async_commit();
                if (lane == 0) {
                    volatile int32_t* m = imeta + (jl & 1) * 8;
                    m[0] = nblk; m[1] = it.y; m[2] = lo; m[3] = b0;
                    m[4] = ntiles; m[5] = share; m[6] = t_req; m[7] = 0;
                }
                __syncwarp();
                t_req += share * W;
                ++jl;
                d_val = it;
                if constexpr (Math::kQuantAppend) {
                    if (p.k_new != nullptr && hi == it.w) {
                        const size_t src = (static_cast<size_t>(it.x) * p.num_kv_heads + it.y) * (D / 4);
                        new_k = __ldg(static_cast<const uint2*>(p.k_new) + src + lane);
                        new_v = __ldg(static_cast<const uint2*>(p.v_new) + src + lane);
                    }
                }
                if (planned) {
                    d_req = d_req2;
                    d_req2 = load_item(jl + 1);
                } else {
                    d_req = make_int4(-1, 0, 0, 0);   // read once the plan is complete
                }
            };
            auto validate = [&](int j) {
                cp_async_wait_all();
                __syncwarp();
                volatile int32_t* m = imeta + (j & 1) * 8;
                const int nblk = m[0];
                const int32_t* ids = ids_buf + (j & 1) * kMaxItemBlocks;
                bool bad_lane = false;
                for (int i = lane; i < nblk; i += 32) bad_lane |= (ids[i] < 0) | (ids[i] >= p.num_blocks);
                const bool bad = __any_sync(0xffffffffu, bad_lane);
                if (lane == 0) {
                    m[7] = bad ? 1 : 0;
                    if (bad) raise_error(p.error_word, PA_DEVERR_BLOCK_ID);
                }
                // Fused append: the item holding the sequence's last row
                // quantises this KV head's new rows into their slot (the slot
                // must be that row's) before any lane may load its tiles.
                if constexpr (Math::kQuantAppend) {
                    const int4 it = d_val;
                    const int lo = m[2];
                    if (p.k_new != nullptr && !bad && min(it.w, lo + part_rows(it.w)) == it.w) {
                        const long long slot = __ldg(p.slot_mapping + it.x);
                        if (slot >= 0) {
                            const int r = it.w - 1;
                            const int blk = ids[r / bs - m[3]];
                            if (slot == static_cast<long long>(blk) * bs + r % bs) {
                                Math::Codes::append_row(p, new_k, new_v,
                                                        (static_cast<size_t>(blk) * p.num_kv_heads + it.y) * bs + r % bs,
                                                        lane);
                                // visible to this warp's next copies (the async proxy)
                                asm volatile("fence.proxy.async.global;" ::: "memory");
                            } else if (lane == 0) {
                                raise_error(p.error_word, PA_DEVERR_SLOT);
                            }
                        }
                    }
                    __syncwarp();
                }
                ready = j + 1;
            };
            bool ok = true;
            if (n_items > 0) {
                request();
                validate(0);
                if (planned && jl < n_items) request();
                // lane w < W: warp w's item and next tile within it, and that item's meta
                int cj = 0, ci = 0;
                int h = 0, lo = 0, b0 = 0, ntiles = 0, share = 0, t0 = 0, bad = 0;
                auto enter = [&]() {
                    const volatile int32_t* m = imeta + (cj & 1) * 8;
                    h = m[1]; lo = m[2]; b0 = m[3]; ntiles = m[4]; share = m[5]; t0 = m[6]; bad = m[7];
                };
                if (lane < W) enter();
                uint32_t idle_rounds = 0;
                uint64_t idle_since = 0;
                while (true) {
                    if (!planned) {
                        // The plan (not waited for): the item count and the
                        // descriptors of the items after the first.
                        bool done = false;
                        if (lane == 0) done = mbar_test_wait(smem_addr(plan_bar), 0);
                        if (__shfl_sync(0xffffffffu, done, 0)) {
                            planned = true;
                            total = total_sm[0];
                            n_items = own_item_count(c, C, total);
                            d_req = load_item(jl);
                            d_req2 = load_item(jl + 1);
                        }
                    }
                    // Issue first (a lane woken by its stage's release refills it
                    // at once), then the item bookkeeping.
                    bool moved = false;
                    int t_wait = INT_MAX;                       // this lane's blocked tile, if any
                    if (lane < W && cj < n_items && ci < share) {
                        const int tt = lane + W * ci;           // tile within the item
                        const int t = t0 + tt;
                        const int stage = t % STAGES;
                        if (t < STAGES || mbar_test_wait(smem_addr(&empty[stage]), ((t / STAGES) - 1) & 1)) {
                            // A withheld tile (failure test) gets neither copies nor
                            // an arrival, and no wait for its copies at the end.
                            const bool withheld = c == 0 && t == p.withhold_tile;
                            const bool data = tt < ntiles && !bad && !withheld;
                            const uint32_t fb = smem_addr(&full[stage]);
                            stage_bad[stage] = bad;
                            last_t[stage] = withheld ? -1 : t;
                            if (data) {
                                mbar_arrive_expect_tx(fb, Geom::kStageBytes + Math::kExtraStageBytes);
                                const int tok = lo + kTileRows * tt;
                                const int id = ids_buf[(cj & 1) * kMaxItemBlocks + tok / bs - b0];
                                const int row = (id * p.num_kv_heads + h) * bs + (tok % bs);
                                const uint32_t dst = ring_addr + stage * Geom::kStageBytes;
                                // One 3D box each (all 128-byte column halves of 16 rows).
                                tma_load_3d(dst, &tmap_k, fb, 0, row, 0);
                                tma_load_3d(dst + Geom::kTileBytes, &tmap_v, fb, 0, row, 0);
                                if constexpr (Math::kExtraStageBytes > 0) {
                                    // The tile's 16 K and 16 V row scales (64 bytes each,
                                    // 64-byte aligned: the tile's first row is a multiple
                                    // of 16 within its block).
                                    const size_t r = static_cast<size_t>(row);
                                    const uint32_t xd = xring + stage * Math::kExtraStageBytes;
                                    constexpr int kHalf = Math::kExtraStageBytes / 2;
                                    asm volatile(
                                        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
                                        " [%0], [%1], %2, [%3];" ::"r"(xd), "l"(p.k_row_scales + r),
                                        "r"(kHalf), "r"(fb)
                                        : "memory");
                                    asm volatile(
                                        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
                                        " [%0], [%1], %2, [%3];" ::"r"(xd + kHalf),
                                        "l"(p.v_row_scales + r), "r"(kHalf), "r"(fb)
                                        : "memory");
                                }
                            } else if (!withheld) {
                                mbar_arrive(fb);                // no data: consumers skip the slot
                            }
                            ++ci;
                            moved = true;
                        } else {
                            t_wait = t;
                        }
                    }
                    if (__any_sync(0xffffffffu, abort_flag[0] != 0)) {
                        ok = false;
                        break;
                    }
                    const bool live = lane < W && cj < n_items;
                    const int jmin = __reduce_min_sync(0xffffffffu, live ? cj : INT_MAX);
                    if (jmin == INT_MAX) break;                 // every tile issued
                    // The ids of the next item: buffer jl & 1 last held item jl - 2,
                    // which every lane has left.
                    if (planned && jl < n_items && jl == ready && jl <= jmin + 1) {
                        request();
                        moved = true;
                    }
                    const bool wants_next = live && ci == share && cj == jmin && cj + 1 < n_items;
                    if (__any_sync(0xffffffffu, wants_next) && ready == jmin + 1 && jl > jmin + 1) {
                        validate(jmin + 1);
                        moved = true;
                    }
                    if (live && ci == share) {
                        if (cj + 1 == n_items) {
                            cj = n_items;                       // this warp's tiles are all issued
                            moved = true;
                        } else if (cj == jmin && cj + 1 < ready) {
                            ++cj;
                            ci = 0;
                            enter();
                            moved = true;
                        }
                    }
                    if (__any_sync(0xffffffffu, moved)) {
                        idle_rounds = 0;
                        continue;
                    }
                    // Nothing moved: sleep on the oldest blocked tile's empty barrier
                    // (a hardware-suspended wait that returns when it completes or
                    // after the system's time limit), then look at every lane again.
                    const int t_old = __reduce_min_sync(0xffffffffu, t_wait);
                    if (t_old != INT_MAX) {
                        if (lane == 0)
                            (void)mbar_try_wait(smem_addr(&empty[t_old % STAGES]),
                                                ((t_old / STAGES) - 1) & 1);
                        __syncwarp();
                    } else {
                        __nanosleep(64);
                    }
                    if ((idle_rounds++ & 15u) == 0) {
                        const uint64_t now = global_timer_ns();
                        if (idle_rounds == 1) {
                            idle_since = now;
                        } else if (now - idle_since > kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                    }
                }
            }
            cp_async_wait_all();
            __syncwarp();
            if (!ok) {
                if (lane == 0 && !abort_flag[0]) {
                    raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                    abort_flag[0] = 1;
                }
                // Copies still in flight must land before the CTA's shared memory
                // is released: wait (bounded) for each stage's last issued tile.
                if (lane < STAGES && last_t[lane] >= 0)
                    (void)mbar_wait(smem_addr(&full[lane]), (last_t[lane] / STAGES) & 1);
            }
        } else {
            // In stream order: one lane waits for each stage in turn.
            // Item info and block ids are loaded one item ahead of their use.
            auto load_item = own_item;
            // Block ids of an item are copied into a double-buffered shared array
            // with cp.async one item ahead of their use.
            auto prefetch_ids = [&](const int4& it, int32_t* buf) {
                if (it.x >= 0) {
                    const int P = part_rows(it.w);
                    const int lo = seq_row_base(it.w, p.window) + it.z * P;
                    const int hi = min(it.w, lo + P);
                    const int b0 = lo / bs;
                    const int nblk = (hi - 1) / bs - b0 + 1;
                    const int32_t* bt = p.block_tables + static_cast<size_t>(it.x) * p.max_blocks_per_seq + b0;
                    for (int i = lane; i < nblk; i += 32) cp_async_4(smem_addr(buf + i), bt + i);
                }
                cp_async_commit();
            };
            // The plan's completion: the item count, then items 0, 1, ... .
            bool planned = false;
            auto wait_plan = [&]() -> bool {
                bool done = true;
                if (lane == 0) done = mbar_wait(smem_addr(plan_bar), 0);
                done = __shfl_sync(0xffffffffu, done, 0);
                if (done) {
                    total = total_sm[0];
                    planned = true;
                }
                return done;
            };
            // The first item without the plan where the warp can find it
            // alone (first_item_by_warp); otherwise the warp waits for the plan.
            int4 cur = first;
            int4 nxt = make_int4(-1, 0, 0, 0);
            bool ok = true;
            if (cur.x < 0) {
                ok = wait_plan();
                if (ok) {
                    cur = load_item(0);
                    nxt = load_item(1);
                }
            }
            if (ok) prefetch_ids(cur, ids_buf);
            int t = 0;              // stream tile counter
            int issued = 0;
            for (int j = 0; cur.x >= 0 && ok; ++j) {
                int4 nxt2 = make_int4(-1, 0, 0, 0);   // used two items from now
                int32_t* ids = ids_buf + (j & 1) * kMaxItemBlocks;
                if (planned) {
                    nxt2 = load_item(j + 2);
                    prefetch_ids(nxt, ids_buf + ((j + 1) & 1) * kMaxItemBlocks);
                    cp_async_wait_group_1();            // this item's ids have landed
                } else {
                    cp_async_wait_all();                // the first item's ids, the only group
                }
                __syncwarp();
                const int P = part_rows(cur.w);
                const int lo = seq_row_base(cur.w, p.window) + cur.z * P;
                const int hi = min(cur.w, lo + P);
                const int b0 = lo / bs;
                const int nblk = (hi - 1) / bs - b0 + 1;
                bool bad_lane = false;
                for (int i = lane; i < nblk; i += 32) bad_lane |= (ids[i] < 0) | (ids[i] >= p.num_blocks);
                const int cur_bad = __any_sync(0xffffffffu, bad_lane) ? 1 : 0;
                const int ntiles = (hi - lo + kTileRows - 1) / kTileRows;
                if (cur_bad && lane == 0) raise_error(p.error_word, PA_DEVERR_BLOCK_ID);
                // Fused append: the item holding the sequence's last row writes
                // this KV head's new K and V rows into their slot before the
                // tile that holds them is loaded (the slot must be that row's).
                const long long new_slot =
                    (p.k_new != nullptr && hi == cur.w) ? __ldg(p.slot_mapping + cur.x) : -1;
                const int new_tile = (cur.w - 1 - lo) / kTileRows;
                // The new rows, 16-byte chunks dealt over the lanes (K, then V),
                // loaded now and stored when their tile comes up.
                constexpr int kChunks = D * static_cast<int>(sizeof(T)) / 16;   // per row
                constexpr int kNewPerLane = (2 * kChunks + 31) / 32;
                uint4 new_rows[kNewPerLane];
                if (new_slot >= 0) {
                    const size_t src = (static_cast<size_t>(cur.x) * p.num_kv_heads + cur.y) * kChunks;
#pragma unroll
                    for (int u = 0; u < kNewPerLane; ++u) {
                        const int i = lane + 32 * u;
                        if (i < 2 * kChunks) {
                            const bool v = i >= kChunks;
                            new_rows[u] = __ldg(static_cast<const uint4*>(v ? p.v_new : p.k_new) + src +
                                                (v ? i - kChunks : i));
                        }
                    }
                }
                // The item's tiles are padded with data-less slots up to a multiple
                // of W, so that every item starts at a stream index divisible by W
                // and warp w always takes tiles w, w + W, ... of the item: the
                // rounding of an item's result never depends on what the CTA
                // streamed before it.
                const int span = ((ntiles + W - 1) / W) * W;
                for (int tt = 0; tt < span; ++tt, ++t) {
                    const int tok = lo + kTileRows * tt;
                    // A withheld tile (failure test) gets neither copies nor an
                    // arrival, and no wait for its copies at the end.
                    const bool withheld = c == 0 && t == p.withhold_tile;
                    const bool data = tt < ntiles && !cur_bad && !withheld;
                    const int stage = t % STAGES;
                    const uint32_t fb = smem_addr(&full[stage]);
                    if (new_slot >= 0 && tt == new_tile && !cur_bad) {
                        const int r = cur.w - 1;                  // the new row
                        const int blk = ids[r / bs - b0];
                        if (new_slot == static_cast<long long>(blk) * bs + r % bs) {
                            const size_t dst = ((static_cast<size_t>(blk) * p.num_kv_heads + cur.y) * bs + r % bs) * kChunks;
#pragma unroll
                            for (int u = 0; u < kNewPerLane; ++u) {
                                const int i = lane + 32 * u;
                                if (i < 2 * kChunks) {
                                    const bool v = i >= kChunks;
                                    static_cast<uint4*>(const_cast<void*>(v ? p.v_cache : p.k_cache))
                                        [dst + (v ? i - kChunks : i)] = new_rows[u];
                                }
                            }
                            // The generic-proxy writes are visible to this
                            // warp's next TMA loads (the async proxy).
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                        } else if (lane == 0) {
                            raise_error(p.error_word, PA_DEVERR_SLOT);
                        }
                        __syncwarp();
                    }
                    if (lane == 0) {
                        if (t >= STAGES && !mbar_wait(smem_addr(&empty[stage]), ((t / STAGES) - 1) & 1)) {
                            ok = false;
                        } else if (abort_flag[0]) {
                            ok = false;
                        } else {
                            stage_bad[stage] = cur_bad;
                            if (data)
                                mbar_arrive_expect_tx(fb, Geom::kStageBytes + Math::kExtraStageBytes);
                            else if (!withheld)
                                mbar_arrive(fb);          // no data: consumers skip the slot
                            issued = t + 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    // Lane 0 copies the K tile, lane 1 the V tile: one 3D box each
                    // (all 128-byte column halves of 16 rows), issued after lane
                    // 0's expect_tx (ordered by the shuffle above).
                    if (data && lane < 2) {
                        const int id = ids[tok / bs - b0];
                        const int row = (id * p.num_kv_heads + cur.y) * bs + (tok % bs);
                        const uint32_t dst = ring_addr + stage * Geom::kStageBytes +
                                             (lane ? Geom::kTileBytes : 0);
                        tma_load_3d(dst, lane ? static_cast<const void*>(&tmap_v)
                                              : static_cast<const void*>(&tmap_k),
                                    fb, 0, row, 0);
                    }
                    if (!planned && tt == min(span, STAGES) - 1) {
                        // The ring is full with the first item's tiles: now the
                        // plan, then the next items as in every other round.
                        ok = wait_plan();
                        if (!ok) break;
                        nxt = load_item(1);
                        nxt2 = load_item(2);
                        prefetch_ids(nxt, ids_buf + kMaxItemBlocks);
                    }
                    if constexpr (Math::kExtraStageBytes > 0) {
                        // Lanes 2 and 3: the tile's 16 K and 16 V row scales (64 bytes
                        // each, 64-byte aligned: the tile's first row is a multiple of
                        // 16 within its block).
                        if (data && (lane == 2 || lane == 3)) {
                            const int id = ids[tok / bs - b0];
                            const size_t r = (static_cast<size_t>(id) * p.num_kv_heads + cur.y) * bs + (tok % bs);
                            const float* src = (lane == 2 ? p.k_row_scales : p.v_row_scales) + r;
                            const uint32_t dst = xring + stage * Math::kExtraStageBytes +
                                                 (lane - 2) * (Math::kExtraStageBytes / 2);
                            asm volatile(
                                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
                                " [%0], [%1], %2, [%3];" ::"r"(dst), "l"(src),
                                "r"(Math::kExtraStageBytes / 2), "r"(fb)
                                : "memory");
                        }
                    }
                }
                cur = nxt;
                nxt = nxt2;
            }
            cp_async_wait_all();
            if (lane == 0) {
                if (!ok) {
                    raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                    abort_flag[0] = 1;
                }
                // Copies still in flight must land before the CTA's shared memory
                // is released: wait (bounded) for the last issued stages.
                for (int u = issued > STAGES ? issued - STAGES : 0; u < issued; ++u)
                    if (!(c == 0 && u == p.withhold_tile))
                        (void)mbar_wait(smem_addr(&full[u % STAGES]), (u / STAGES) & 1);
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    // The next item's description and q are loaded one item ahead, so that an
    // item boundary costs no global-memory round trip.
    Math math;
    math.setup(lane, p);
    // Query columns of an item: the group's heads x the query tokens per
    // sequence, at most G (the state's capacity). Maths without causal
    // masking serve one query per sequence with exactly G heads.
    const int grp = Math::kCausal ? p.num_heads / p.num_kv_heads : G;
    const int Qn = Math::kCausal ? p.num_queries : 1;
    const int ncols = Math::kCausal ? grp * Qn : G;
    auto item_at = own_item;
    int4 it = item_at(0);
    int4 it_next = item_at(1);
    typename Math::QRegs q_next;
    bool aborted = false;
    if constexpr (Math::kQInSmem) {
        // q of item 0 now (unless the producer already copied it), then always
        // one item ahead, copied by warp 0.
        if (warp == 0 && it.x >= 0) {
            bool landed = true;
            if (lane == 0) landed = mbar_wait(smem_addr(q0_bar), 0);
            landed = __shfl_sync(0xffffffffu, landed, 0);
            if (!landed) {
                aborted = true;
                if (lane == 0) {
                    raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                    abort_flag[0] = 1;
                }
            }
            const bool have = landed && q0_sm[0] == it.x && q0_sm[1] == it.y;
            if (!have) {
                math.stage_q(p, it.x, it.y, ncols, grp, smem_addr(qbuf), lane);
                cp_async_wait_all();
            }
        }
        named_barrier(1, W * 32);
    } else {
        if (it.x >= 0) math.load_q(p, it.x, it.y, q_next);
    }
    int t0 = 0;                 // stream index of the current item's first tile (a multiple of W)
    for (int j = 0; it.x >= 0; ++j) {
        const int s = it.x, h = it.y, part = it.z, n = it.w;
        const int base = seq_row_base(n, p.window);
        const int P = seq_partition(p, n - base);
        const int lo = base + part * P;
        const int hi = min(n, lo + P);
        const int ntiles = (hi - lo + kTileRows - 1) / kTileRows;
        const int4 it_after = item_at(j + 2);
        if constexpr (Math::kQInSmem) {
            math.begin_staged(qbuf + (j & 1) * Math::kQBufBytes, ncols);
            // The other buffer was last read when item j - 1 began, before the
            // previous item's closing barrier.
            if (warp == 0 && it_next.x >= 0)
                math.stage_q(p, it_next.x, it_next.y, ncols, grp,
                             smem_addr(qbuf + ((j + 1) & 1) * Math::kQBufBytes), lane);
        } else {
            math.begin(p, q_next);
            if (it_next.x >= 0) math.load_q(p, it_next.x, it_next.y, q_next);
        }
        const int span = ((ntiles + W - 1) / W) * W;   // padded as the producer pads
        const int limit0 = n - Qn;                      // the last row query token 0 sees
        bool bad = false;
        if (!aborted) {
            for (int t = t0 + warp; t < t0 + span; t += W) {
                const int stage = t % STAGES;
                const bool got = mbar_wait(smem_addr(&full[stage]), (t / STAGES) & 1);
                if (!__all_sync(0xffffffffu, got)) {
                    aborted = true;
                    break;
                }
                if (stage_bad[stage]) {
                    bad = true;
                } else if (t - t0 < ntiles) {
                    const int row0 = lo + kTileRows * (t - t0);
                    const int valid = min(kTileRows, hi - row0);
                    const uint32_t kb = ring_addr + stage * Geom::kStageBytes;
                    // Rows of the tile before a sliding window (<= 0: none).
                    const int skip = p.window > 0 ? n - p.window - row0 : 0;
                    math.tile(kb, kb + Geom::kTileBytes, valid, p.scale_log2, lane, row0, limit0,
                              grp, skip, xring + stage * Math::kExtraStageBytes);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&empty[stage]));
            }
        }
        it = it_next;
        it_next = it_after;
        t0 += span;
        float* buf = merge;
        math.write_state(buf + warp * Smem::kState, lane, ncols);
        if constexpr (Math::kQInSmem) {
            if (warp == 0) cp_async_wait_all();   // next item's q is visible after the barrier
        }
        if (lane == 0) {
            warp_bad[(j & 1) * W + warp] = bad;
            if (aborted) {
                abort_flag[0] = 1;
                raise_error(p.error_word, PA_DEVERR_TIMEOUT);
            }
        }
        named_barrier(1, W * 32);
        if (abort_flag[0]) break;           // read after the barrier: one decision for all warps
        bool any_bad = false;
#pragma unroll
        for (int w = 0; w < W; ++w) any_bad |= warp_bad[(j & 1) * W + w] != 0;
        // any_bad: flagged by the producer; output left unspecified
        const int nparts = (n - base + P - 1) / P;
        for (int idx = any_bad ? ncols * D : threadIdx.x; idx < ncols * D; idx += W * 32) {
            const int g = idx / D;            // query column
            const int d = idx - g * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, buf[w * Smem::kState + g]);
            // A column that sees no row of this partition (several queries per
            // sequence) merges to m = -inf, l = 0, o = 0.
            const float ref = M == -INFINITY ? 0.f : M;
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float* sw = buf + w * Smem::kState;
                const float cw = fast_exp2(sw[g] - ref);
                L = fmaf(cw, sw[G + g], L);
                O = fmaf(cw, sw[2 * G + g * D + d], O);
            }
            const size_t row = Math::kCausal
                                   ? query_row(p, s, h, g, grp)
                                   : static_cast<size_t>(s) * p.num_heads + h * G + g;
            if (nparts == 1) {
                ElemTraits<T>::store(static_cast<T*>(p.out) + row * D + d, O / L);
            } else {
                const size_t slot = row * p.max_parts + part;
                p.part_o[slot * D + d] = O;
                if (d == 0) {
                    p.part_ml[2 * slot] = M;
                    p.part_ml[2 * slot + 1] = L;
                }
            }
        }
        // The next item's warp states overwrite the merge area.
        named_barrier(1, W * 32);
    }
}

// Host-side launch of one persistent instance: as many CTAs as fit on
// sm_count SMs, programmatic dependent launch on the stream.
template <class Math, int D, int G, int W, int STAGES, int MIN_CTAS, bool PER_WARP_ISSUE>
cudaError_t launch_stream_instance(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const DecodeParams& p, int sm_count, cudaStream_t stream) {
    using Smem = StreamSmem<W, STAGES, typename Math::Geom, G, D, Math::kQBufBytes,
                            Math::kExtraStageBytes, PER_WARP_ISSUE>;
    auto kernel = decode_stream_kernel<Math, D, G, W, STAGES, MIN_CTAS, PER_WARP_ISSUE>;
    const int smem = static_cast<int>(Smem::kBytes);
    // The shared-memory attribute and the resulting CTAs per SM are set up
    // once per device and instance.
    static std::atomic<int> cached_per_sm[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    int per_sm = dev < kMaxDevices ? cached_per_sm[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm == 0) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, (W + 1) * 32, smem);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        if (dev < kMaxDevices) cached_per_sm[dev].store(per_sm, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count * per_sm));
    cfg.blockDim = dim3((W + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, tk, tv, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pa
