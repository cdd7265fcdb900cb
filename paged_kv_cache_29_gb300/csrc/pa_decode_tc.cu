// pa_decode_tc.cu -- paged decode attention over an FP8 (e4m3) cache on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The same work items as the tile-ring kernels (pa_plan.cuh: one (sequence,
// KV head, partition) each) are cut into chunks of 128 rows: eight 16-row
// tiles of K and V, each a contiguous 2 KB TMA box of one (block, KV head) of
// the [block][kv_head][block_size][128] pool, row i of a sequence being row
// i % block_size of block block_tables[s][i / block_size] ("MLSys Engineer --
// Inference Systems Q&A", Q1). Per chunk:
//
//   QK   S[128 rows][N] = K_codes[128][128] . Qt^T on the tensor core
//        (kind::f8f6f4, e4m3 x e4m3 -> fp32): A is the chunk's K tiles
//        (K-major, 128-byte swizzle, as TMA stores them), B holds q in three
//        e4m3 terms per query head, q' * 2^a = t0 + t1/16 + t2/256, with
//        q' = q * scale * log2(e) * k_scale and a per-head power of two a, so
//        the scores keep about 12 significant bits.
//   softmax  four warps, one row per thread: the row's base-2 scores from its
//        tensor-memory lane, the chunk's maximum per head across the four
//        warps, p = 2^(s - m) against the running maximum (the online softmax
//        of Q4 "How would you write a fused attention kernel?"), the running
//        sum per thread, and p * 256 written back to shared memory as three
//        e4m3 terms per head (the B operand of the next product).
//   PV   O^T[128 dims][N] = V_codes^T . P^T on the tensor core: A is the
//        chunk's V tiles read MN-major (the tiles are [row][dim], dims
//        contiguous), B the three P terms. The same four warps then read
//        their dim's lane, rebuild p.V from the terms, rescale the running
//        output by 2^(m_old - m_new) and add.
//
// Warps: 0 loads (block ids, TMA boxes into a ring of NC chunk slots, the
// fused append's quantisation, and each item's q operand, prefetched one item
// ahead), 1 issues the QK products from one thread and owns the tensor-memory
// allocation, 2-5 do the softmax and the output and issue their own P.V
// product (one thread, right after the four warps meet) so that no hand-off
// sits on that path. Scores and outputs are double-buffered in tensor memory
// and the B operands in shared memory, so the tensor core computes the next
// chunk's scores while the softmax warps work on the current one. Item ends write the output (one
// partition) or the (max, sum, unnormalised output) partial the merge kernel
// reads, exactly as the tile-ring kernels do; v_scale is applied there.
//
// Rows past an item's end (in its last chunk) get p = 0, and their V rows are
// zeroed in shared memory before the P.V product, so stale or NaN codes in
// those rows never reach the output. Every wait is bounded; a wait that runs
// out sets PA_DEVERR_TIMEOUT and an abort flag, after which every role winds
// down through the same barriers without waiting again.
#include "pa_decode_stream.cuh"
#include "pa_tile_math_quant.cuh"

namespace pa {

namespace {

// ---- tcgen05 / UMMA helpers (inline PTX) ------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1 (bits 46-47),
// swizzle mode 2 (bits 61-63).
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
           (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B and an fp32
// accumulator: D format at bits 4-5 (1 = f32), A and B formats at 7-9 and
// 10-12 (0 = e4m3), A major at bit 15 (1 = MN-major), N / 8 at bits 17-22,
// M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, int a_mn) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier completes once every MMA this thread issued before has.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Generic-proxy shared-memory writes made visible to the async proxy (the
// tensor core's operand reads).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
        " [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two e4m3 codes (low byte first) for two floats: round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// The values of two e4m3 codes (low byte first), exactly.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t codes) {
    uint32_t h;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
        : "=r"(h)
        : "r"(codes));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// x0, x1 (|x| <= 448) as three e4m3 terms each: x ~ t0 + t1 / 16 + t2 / 256.
// Returns the three code pairs (low byte = x0's code).
__device__ __forceinline__ void split3(float x0, float x1, uint32_t (&c)[3]) {
#pragma unroll
    for (int t = 0; t < 3; ++t) {
        c[t] = e4m3x2(x0, x1);
        if (t < 2) {
            const float2 v = e4m3x2_value(c[t]);
            x0 = (x0 - v.x) * 16.f;
            x1 = (x1 - v.y) * 16.f;
        }
    }
}

// Order-preserving int key of a float (for integer max reductions).
__device__ __forceinline__ int fkey(float f) {
    const int b = __float_as_int(f);
    return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float fkey_value(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// Byte offset of element k (0..127) of row n of a 128-byte-swizzled K-major
// operand (n's 8-row group at 1024 * (n / 8)).
__device__ __forceinline__ uint32_t sw128_byte(int n, int k) {
    return static_cast<uint32_t>(n * 128 + (((k >> 4) ^ (n & 7)) << 4) + (k & 15));
}

constexpr int kRows = 128;                       // rows per chunk: the MMA's M
constexpr int kChunkTiles = kRows / kTileRows;   // 8
constexpr int kTileBytes8 = kTileRows * 128;     // one 16-row box of 1-byte codes
constexpr int kHalfSlot = kChunkTiles * kTileBytes8;   // 16 KB: a chunk's K (or V) tiles
constexpr int kSlotBytes = 2 * kHalfSlot;
constexpr int kSoftWarps = 4;
constexpr int kTcThreads = (2 + kSoftWarps) * 32;
constexpr int kTcMinCtas = 2;                    // resident CTAs per SM the registers are sized for
constexpr int kTerms = 3;

// Poll an mbarrier phase; gives up (false) after the kernel-wide wait limit
// or as soon as the abort flag is set.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < kWaitMaxIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

template <int G>
struct TcShape {
    static constexpr int kN = ((kTerms * G + 15) / 16) * 16;   // MMA N: 16 or 32
    static constexpr int kOpBytes = kN * 128;                  // a B operand: kN rows x 128 B
    // Tensor memory: two score and two output buffers of kN fp32 columns.
    static constexpr int kCols = 4 * kN;                       // 64 or 128: a power of 2 >= 32
};

template <int G, int NC>
struct TcSmem {
    using S = TcShape<G>;
    static constexpr int kSlots = 0;
    static constexpr int kQ = kSlots + NC * kSlotBytes;       // [2] q operands
    static constexpr int kP = kQ + 2 * S::kOpBytes;           // [2] P operands
    static constexpr int kBars = kP + 2 * S::kOpBytes;
    // kv_full[NC] (the K half), kv_empty[NC], s_full[2], s_free[2], o_full[2],
    // q_full[2], q_empty[2], done (QK issuer), done (P.V issuer), v_full[NC]
    static constexpr int kNumBars = 3 * NC + 10 + 2;
    static constexpr int kInts = kBars + 8 * kNumBars;        // abort, tmem slot, slot_bad[NC]
    static constexpr int kNumInts = 2 + NC;
    static constexpr int kFloats = (kInts + 4 * kNumInts + 15) / 16 * 16;
    // red_max[2][4][G] (ints), red_l[2][4][G], q_inv[2][G] (16-byte rows)
    static constexpr int kNumFloats = 2 * 2 * 4 * G + 2 * ((G + 3) / 4) * 4;
    static constexpr int kIds = (kFloats + 4 * kNumFloats + 15) / 16 * 16;   // [2][kMaxItemBlocks]
    static constexpr int kFirst = (kIds + 4 * 2 * kMaxItemBlocks + 15) / 16 * 16;   // int4[2]
    static constexpr int kPlan = kFirst + 32;
    static constexpr int kEnd = kPlan + 4 * plan_scratch_ints(kTcThreads);
    static constexpr size_t kBytes = 1024 + static_cast<size_t>(kEnd);
};

template <int G, int NC>
__global__ void __launch_bounds__(kTcThreads, kTcMinCtas)
decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    using S = TcShape<G>;
    using L = TcSmem<G, NC>;
    constexpr int D = 128;
    constexpr int N = S::kN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sm_addr = smem_addr(sm);
    const uint32_t slots = sm_addr + L::kSlots;
    const uint32_t qops = sm_addr + L::kQ;
    const uint32_t pops = sm_addr + L::kP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBars);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int KV_FULL = 0, KV_EMPTY = NC, S_FULL = 2 * NC, S_FREE = S_FULL + 2, O_FULL = S_FREE + 2,
              Q_FULL = O_FULL + 2, Q_EMPTY = Q_FULL + 2, DONE = Q_EMPTY + 2, DONE_PV = DONE + 1,
              V_FULL = DONE_PV + 1;
    volatile int32_t* ints = reinterpret_cast<volatile int32_t*>(sm + L::kInts);
    volatile int32_t* abort_flag = ints;
    volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(ints + 1);
    volatile int32_t* slot_bad = ints + 2;
    float* fl = reinterpret_cast<float*>(sm + L::kFloats);
    int* red_max = reinterpret_cast<int*>(fl);            // [2][4][G]
    float* red_l = fl + 2 * 4 * G;                        // [2][4][G]
    float* q_inv = red_l + 2 * 4 * G;                     // [2][G]: 2^-a per head of q buffer b
    int32_t* ids_buf = reinterpret_cast<int32_t*>(sm + L::kIds);
    int4* first_items = reinterpret_cast<int4*>(sm + L::kFirst);
    int* plan_sm = reinterpret_cast<int*>(sm + L::kPlan);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NC; ++i) {
            mbar_init(bar(KV_FULL + i), 1);
            mbar_init(bar(V_FULL + i), 1);
            mbar_init(bar(KV_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(S_FULL + i), 1);
            mbar_init(bar(S_FREE + i), kSoftWarps);
            mbar_init(bar(O_FULL + i), 1);
            mbar_init(bar(Q_FULL + i), 1);
            // the last QK of the buffer's item (a commit) and every softmax
            // warp's read of its scales
            mbar_init(bar(Q_EMPTY + i), 1 + kSoftWarps);
        }
        mbar_init(bar(DONE), 1);
        mbar_init(bar(DONE_PV), 1);
        abort_flag[0] = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        // Tensor memory for the score and output buffers (this CTA alone
        // allocates, once).
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(const_cast<uint32_t*>(tslot))),
                     "r"(S::kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    // The q and P operand rows past the 3 G term rows stay zero.
    for (int i = threadIdx.x; i < 4 * S::kOpBytes / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(sm + L::kQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot[0];
    grid_dependency_wait();
    grid_launch_dependents();

    const int C = gridDim.x;
    const int c = blockIdx.x;
    const int total = plan_cta<__nv_bfloat16, kTcThreads>(p, c, C, plan_sm, first_items);
    __syncthreads();
    auto own_item = [&](int j) -> int4 {
        const int k = snake_item(c, j, C);
        if (k >= total) return make_int4(-1, 0, 0, 0);
        return j < 2 ? first_items[j] : p.items[k];
    };
    const int n_items = own_item_count(c, C, total);
    const int bs = p.block_size;
    // Rows [lo, hi) of an item.
    auto item_rows = [&](const int4& it, int& lo, int& hi) {
        const int P = seq_partition(p, it.w);
        lo = it.z * P;
        hi = min(it.w, lo + P);
    };

    if (warp == 0) {
        // ------------------------------ loads ---------------------------------
        auto request_ids = [&](int j) {
            const int4 it = own_item(j);
            if (it.x >= 0) {
                int lo, hi;
                item_rows(it, lo, hi);
                const int b0 = lo / bs;
                const int nblk = (hi - 1) / bs - b0 + 1;
                int32_t* buf = ids_buf + (j & 1) * kMaxItemBlocks;
                const int32_t* bt = p.block_tables + static_cast<size_t>(it.x) * p.max_blocks_per_seq + b0;
                for (int i = lane; i < nblk; i += 32) cp_async_4(smem_addr(buf + i), bt + i);
            }
            cp_async_commit();
        };
        // q of an item, prefetched one item ahead: lane l holds dims 4 l ..
        // 4 l + 3 of each of the group's G heads.
        uint2 qraw[G];
        auto load_q = [&](int j) {
            const int4 it = own_item(j);
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                qraw[gg] = it.x < 0 ? make_uint2(0u, 0u)
                                    : __ldg(reinterpret_cast<const uint2*>(
                                                static_cast<const __nv_bfloat16*>(p.q) +
                                                (static_cast<size_t>(it.x) * p.num_heads + it.y * G + gg) * D) +
                                            lane);
        };
        // The q operand of item j (buffer j & 1, free once the item two back
        // is done with it): three e4m3 terms of q' * 2^a per head (row
        // t * G + head, element = dim), a per head chosen so that
        // max |q' * 2^a| is in [64, 128); q_inv holds 2^-a.
        const float qscale = p.scale_log2 * p.k_scale;
        auto write_q = [&](int j) -> bool {
            if (j >= 2) {
                bool free = true;
                if (lane == 0) free = tc_wait(bar(Q_EMPTY + (j & 1)), ((j - 2) >> 1) & 1, abort_flag);
                if (!__shfl_sync(0xffffffffu, free, 0)) return false;   // warp-uniform from here
            }
            const uint32_t qb = L::kQ + (j & 1) * S::kOpBytes;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float x[4] = {bf16_lo(qraw[gg].x) * qscale, bf16_hi(qraw[gg].x) * qscale,
                              bf16_lo(qraw[gg].y) * qscale, bf16_hi(qraw[gg].y) * qscale};
                float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
                amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
                int a = 0;
                if (amax > 0.f && amax < INFINITY) a = min(100, max(-100, 6 - ilogbf(amax)));
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = ldexpf(x[i], a);
                uint32_t c01[3], c23[3];
                split3(x[0], x[1], c01);
                split3(x[2], x[3], c23);
#pragma unroll
                for (int t = 0; t < kTerms; ++t)
                    *reinterpret_cast<uint32_t*>(sm + qb + sw128_byte(t * G + gg, 4 * lane)) =
                        (c01[t] & 0xffffu) | (c23[t] << 16);
                if (lane == 0) q_inv[(j & 1) * ((G + 3) / 4) * 4 + gg] = ldexpf(1.f, -a);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Q_FULL + (j & 1)));
            return true;
        };
        int g = 0;              // chunks issued
        bool ok = true;
        if (n_items > 0) {
            request_ids(0);
            load_q(0);
            ok = write_q(0);
            if (n_items > 1) load_q(1);
        }
        for (int j = 0; j < n_items && ok; ++j) {
            const int4 it = own_item(j);
            int lo, hi;
            item_rows(it, lo, hi);
            request_ids(j + 1);                 // the next item's ids, one item ahead
            cp_async_wait_group_1();
            __syncwarp();
            const int32_t* ids = ids_buf + (j & 1) * kMaxItemBlocks;
            const int b0 = lo / bs;
            const int nblk = (hi - 1) / bs - b0 + 1;
            bool bad_lane = false;
            for (int i = lane; i < nblk; i += 32) bad_lane |= (ids[i] < 0) | (ids[i] >= p.num_blocks);
            const bool bad = __any_sync(0xffffffffu, bad_lane);
            if (bad && lane == 0) raise_error(p.error_word, PA_DEVERR_BLOCK_ID);
            // Fused append: the item holding the sequence's last row quantises
            // this KV head's new K and V rows into their slot before any of
            // its boxes is loaded (the slot must be that row's).
            if (p.k_new != nullptr && !bad && hi == it.w) {
                const long long slot = __ldg(p.slot_mapping + it.x);
                if (slot >= 0) {
                    const int r = it.w - 1;
                    const int blk = ids[r / bs - b0];
                    if (slot == static_cast<long long>(blk) * bs + r % bs) {
                        const size_t src = (static_cast<size_t>(it.x) * p.num_kv_heads + it.y) * (D / 4);
                        const uint2 nk = __ldg(static_cast<const uint2*>(p.k_new) + src + lane);
                        const uint2 nv = __ldg(static_cast<const uint2*>(p.v_new) + src + lane);
                        E4m3Codes::append_row(p, nk, nv,
                                              (static_cast<size_t>(blk) * p.num_kv_heads + it.y) * bs + r % bs,
                                              lane);
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    } else if (lane == 0) {
                        raise_error(p.error_word, PA_DEVERR_SLOT);
                    }
                }
                __syncwarp();
            }
            const int nch = (hi - lo + kRows - 1) / kRows;
            // Each lane's tile of a chunk: lanes 0-7 the K boxes, 8-15 the V
            // boxes (one warp instruction issues all of them), the block-table
            // lookup done once per lane.
            const int tl = lane & (kChunkTiles - 1);
            for (int ch = 0; ch < nch && ok; ++ch, ++g) {
                const int s_ = g % NC;
                const int row0 = lo + ch * kRows;
                const int ntile = min(kChunkTiles, (hi - row0 + kTileRows - 1) / kTileRows);
                int row = 0;
                if (lane < 2 * kChunkTiles && tl < ntile) {
                    const int tok = row0 + tl * kTileRows;
                    const int id = ids[tok / bs - b0];
                    row = (id * p.num_kv_heads + it.y) * bs + (tok % bs);
                }
                // Separate completions for the K half (the QK product waits
                // only for its own boxes) and the V half (needed a softmax
                // later).
                const uint32_t fb = bar(KV_FULL + s_);
                const uint32_t vb = bar(V_FULL + s_);
                const bool withheld = c == 0 && g == p.withhold_tile;   // failure test
                if (lane == 0) {
                    if (g >= NC && !tc_wait(bar(KV_EMPTY + s_), ((g / NC) - 1) & 1, abort_flag))
                        ok = false;
                    if (ok) {
                        slot_bad[s_] = bad ? 1 : 0;
                        if (withheld) {
                            // neither copies nor an arrival: the MMA warp's wait runs out
                        } else if (bad) {
                            mbar_arrive(fb);
                            mbar_arrive(vb);
                        } else {
                            mbar_arrive_expect_tx(fb, ntile * kTileBytes8);
                            mbar_arrive_expect_tx(vb, ntile * kTileBytes8);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (!bad && !withheld && lane < 2 * kChunkTiles && tl < ntile) {
                    const bool v = lane >= kChunkTiles;
                    tma_load_3d(slots + s_ * kSlotBytes + (v ? kHalfSlot : 0) + tl * kTileBytes8,
                                v ? static_cast<const void*>(&tmap_v) : static_cast<const void*>(&tmap_k),
                                v ? vb : fb, 0, row, 0);
                }
            }
            // The next item's q, its rows prefetched one item ago; then the
            // rows of the item after it.
            if (ok && j + 1 < n_items) {
                ok = __shfl_sync(0xffffffffu, write_q(j + 1), 0);
                if (j + 2 < n_items) load_q(j + 2);
            }
        }
        cp_async_wait_all();
        if (lane == 0) {
            if (!ok && !abort_flag[0]) {
                raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                abort_flag[0] = 1;
            }
            // Copies in flight land before the CTA's shared memory is released:
            // wait (bounded, no abort shortcut) for the last NC chunks issued.
            for (int u = g > NC ? g - NC : 0; u < g; ++u)
                if (!(c == 0 && u == p.withhold_tile)) {
                    (void)mbar_wait(bar(KV_FULL + u % NC), (u / NC) & 1);
                    (void)mbar_wait(bar(V_FULL + u % NC), (u / NC) & 1);
                }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issue -----------------------------
        if (lane == 0) {
            // QK(0), QK(1), ... in order, each once its chunk has landed, its
            // item's q is written and its score buffer has been read back
            // (chunk g - 2). The softmax warps issue the P.V products
            // themselves (no hand-off on that path).
            constexpr uint32_t kIdQK = idesc_e4m3(kRows, N, 0);
            bool ok = true;
            int g = 0;
            for (int j = 0; j < n_items && ok; ++j) {
                int lo, hi;
                item_rows(own_item(j), lo, hi);
                const int nch = (hi - lo + kRows - 1) / kRows;
                if (!tc_wait(bar(Q_FULL + (j & 1)), (j >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t qb = qops + (j & 1) * S::kOpBytes;
                for (int ch = 0; ch < nch; ++ch, ++g) {
                    if (!tc_wait(bar(KV_FULL + g % NC), (g / NC) & 1, abort_flag) ||
                        (g >= 2 && !tc_wait(bar(S_FREE + (g & 1)), ((g - 2) >> 1) & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k0 = slots + (g % NC) * kSlotBytes;
                    const uint32_t d = tmem + (g & 1) * N;
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)       // 32 dims per MMA
                        umma_e4m3(d, umma_desc(k0 + 32 * k, 16, 1024), umma_desc(qb + 32 * k, 16, 1024),
                                  kIdQK, k > 0);
                    umma_commit(bar(S_FULL + (g & 1)));
                }
                if (ok) umma_commit(bar(Q_EMPTY + (j & 1)));   // the item's q operand is free
            }
            if (!ok && !abort_flag[0]) {
                raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                abort_flag[0] = 1;
            }
            // Every MMA issued completes before the tensor memory is freed.
            if (g > 0) {
                umma_commit(bar(DONE));
                (void)mbar_wait(bar(DONE), 0);
            }
        }
        __syncwarp();
    } else {
        // --------------------------- softmax and output ------------------------
        const int sw = warp - 2;                   // softmax warp 0..3
        const int quad = warp & 3;                 // its tensor-memory lane quadrant
        const int r = quad * 32 + lane;            // row of a chunk (QK), dim (PV)
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        bool aborted = false;
        bool issued_pv = false;
        // A wait that runs out (or finds the abort flag) leaves the whole
        // warp aborted: the tensor-memory loads are warp-collective. Aborted
        // warps still pass every named barrier, so the four warps never part.
        auto wait = [&](uint32_t b, uint32_t parity) {
            bool failed = !aborted && !tc_wait(b, parity, abort_flag);
            if (failed && !abort_flag[0]) {
                raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                abort_flag[0] = 1;
            }
            aborted = __any_sync(0xffffffffu, aborted || failed);
        };
        float qinv_cur[G];
        float m_sm[G], l_thr[G];                 // softmax side: running max and sums of this item
        // An item's sums and each chunk's maximum, by chunk parity (two named
        // copies: register arrays indexed at run time would live in memory).
        float l_done0[G], l_done1[G], m_hist0[G], m_hist1[G];
        float o_run[G], m_ep[G];                 // output side: running p.V of this item
        int g = 0;
        // Output side of chunk x (its P.V), merged into the running output;
        // at the item's last chunk the item's result is written.
        auto output_chunk = [&](int x, const int4& it, int part_lo, bool first, bool last,
                                bool bad) {
            wait(bar(O_FULL + (x & 1)), (x >> 1) & 1);
            float o[2][16];
            if (!aborted) {
                tc_fence_after();
                const uint32_t t = tmem + lane_base + 2 * N + (x & 1) * N;
                tmem_ld16(t, o[0]);
                if (N > 16) tmem_ld16(t + 16, o[1]);
                tmem_wait_ld();
            }
            tc_fence_before();
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                auto col = [&](int n) { return n < 16 ? o[0][n] : o[1][n - 16]; };
                const float oc = (col(gg) + col(G + gg) * 0.0625f + col(2 * G + gg) * 0.00390625f) *
                                 0.00390625f;
                const float mx = (x & 1) ? m_hist1[gg] : m_hist0[gg];
                o_run[gg] = first ? oc : fmaf(o_run[gg], fast_exp2(m_ep[gg] - mx), oc);
                m_ep[gg] = mx;
            }
            if (!last) return;
            // Item end: the sums of the four warps, then the output or the
            // partition's partial.
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float v = (x & 1) ? l_done1[gg] : l_done0[gg];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) red_l[(x & 1) * 4 * G + sw * G + gg] = v;
            }
            named_barrier(3, kSoftWarps * 32);
            if (bad || aborted) return;
            const int s = it.x, h = it.y, n = it.w;
            const int nparts = (n + seq_partition(p, n) - 1) / seq_partition(p, n);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float lsum = 0.f;
#pragma unroll
                for (int w = 0; w < kSoftWarps; ++w) lsum += red_l[(x & 1) * 4 * G + w * G + gg];
                const size_t row = static_cast<size_t>(s) * p.num_heads + h * G + gg;
                const float ov = o_run[gg] * p.v_scale;
                if (nparts == 1) {
                    ElemTraits<__nv_bfloat16>::store(static_cast<__nv_bfloat16*>(p.out) + row * D + r,
                                                     ov / lsum);
                } else {
                    const int part = part_lo;
                    const size_t slot = row * p.max_parts + part;
                    p.part_o[slot * D + r] = ov;
                    if (r == 0) {
                        p.part_ml[2 * slot] = m_ep[gg];
                        p.part_ml[2 * slot + 1] = lsum;
                    }
                }
            }
        };

        int4 prev_it = make_int4(-1, 0, 0, 0);
        bool prev_first = false, prev_last = false, prev_bad = false;
        for (int j = 0; j < n_items; ++j) {
            const int4 it = own_item(j);
            int lo, hi;
            item_rows(it, lo, hi);
            const int nch = (hi - lo + kRows - 1) / kRows;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                m_sm[gg] = -INFINITY;
                l_thr[gg] = 0.f;
            }
            bool bad = false;
            for (int ch = 0; ch < nch; ++ch, ++g) {
                // ---- scores of chunk g
                wait(bar(S_FULL + (g & 1)), (g >> 1) & 1);
                float acc[2][16];
                if (!aborted) {
                    tc_fence_after();
                    const uint32_t t = tmem + lane_base + (g & 1) * N;
                    tmem_ld16(t, acc[0]);
                    if (N > 16) tmem_ld16(t + 16, acc[1]);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(S_FREE + (g & 1)));
                // The item's q scales (written with its q operand), then the
                // buffer may be reused once the item's QKs are done too.
                if (ch == 0) {
                    wait(bar(Q_FULL + (j & 1)), (j >> 1) & 1);
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) qinv_cur[gg] = q_inv[(j & 1) * ((G + 3) / 4) * 4 + gg];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(Q_EMPTY + (j & 1)));
                }
                wait(bar(V_FULL + g % NC), (g / NC) & 1);   // the V half; orders slot_bad
                if (ch == 0) bad = slot_bad[g % NC] != 0;
                const int row = lo + ch * kRows + r;
                const bool valid = row < hi && !bad;
                float s[G];
                int wmax[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    auto col = [&](int n) { return n < 16 ? acc[0][n] : acc[1][n - 16]; };
                    s[gg] = valid ? (col(gg) + col(G + gg) * 0.0625f + col(2 * G + gg) * 0.00390625f) *
                                        qinv_cur[gg]
                                  : -INFINITY;
                    wmax[gg] = __reduce_max_sync(0xffffffffu, fkey(s[gg]));
                }
                if (lane == 0) {
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) red_max[(g & 1) * 4 * G + sw * G + gg] = wmax[gg];
                }
                named_barrier(1, kSoftWarps * 32);
#pragma unroll
                for (int w = 0; w < kSoftWarps; ++w) {
                    if (w == sw) continue;
                    const int* src = red_max + (g & 1) * 4 * G + w * G;
                    if constexpr (G % 4 == 0) {
#pragma unroll
                        for (int v = 0; v < G / 4; ++v) {
                            const int4 m4 = reinterpret_cast<const int4*>(src)[v];
                            wmax[4 * v] = max(wmax[4 * v], m4.x);
                            wmax[4 * v + 1] = max(wmax[4 * v + 1], m4.y);
                            wmax[4 * v + 2] = max(wmax[4 * v + 2], m4.z);
                            wmax[4 * v + 3] = max(wmax[4 * v + 3], m4.w);
                        }
                    } else {
#pragma unroll
                        for (int gg = 0; gg < G; ++gg) wmax[gg] = max(wmax[gg], src[gg]);
                    }
                }
                float pv[G];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    const float m_new = fmaxf(m_sm[gg], fkey_value(wmax[gg]));
                    const float ref = m_new == -INFINITY ? 0.f : m_new;
                    pv[gg] = valid ? fast_exp2(s[gg] - ref) : 0.f;
                    l_thr[gg] = fmaf(l_thr[gg], fast_exp2(m_sm[gg] - ref), pv[gg]);
                    m_sm[gg] = m_new;
                    if (g & 1) m_hist1[gg] = ref;
                    else m_hist0[gg] = ref;
                }
                // P as three e4m3 terms of p * 256 (row t * G + head, element r).
                const uint32_t pb = L::kP + (g & 1) * S::kOpBytes;
#pragma unroll
                for (int gg = 0; gg < G; gg += 2) {
                    uint32_t cc[3];
                    split3(pv[gg] * 256.f, gg + 1 < G ? pv[gg + 1] * 256.f : 0.f, cc);
#pragma unroll
                    for (int t = 0; t < kTerms; ++t) {
                        sm[pb + sw128_byte(t * G + gg, r)] = static_cast<uint8_t>(cc[t] & 0xffu);
                        if (gg + 1 < G) sm[pb + sw128_byte(t * G + gg + 1, r)] = static_cast<uint8_t>(cc[t] >> 8);
                    }
                }
                if (row >= hi && !bad) {
                    // Zero the V row past the item's end (stale or unloaded codes,
                    // possibly NaN) so that p = 0 meets a zero code.
                    uint4* v = reinterpret_cast<uint4*>(sm + L::kSlots + (g % NC) * kSlotBytes + kHalfSlot +
                                                        r * 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_async_smem();
                // P(g) is complete once all four warps are here; output
                // buffer g & 1 was read back (chunk g - 2) one iteration ago.
                named_barrier(4, kSoftWarps * 32);
                if (threadIdx.x == 2 * 32 && !aborted) {
                    tc_fence_after();
                    constexpr uint32_t kIdPV = idesc_e4m3(kRows, N, 1);
                    const uint32_t v0 = slots + (g % NC) * kSlotBytes + kHalfSlot;
                    const uint32_t b0 = pops + (g & 1) * S::kOpBytes;
                    const uint32_t d = tmem + 2 * N + (g & 1) * N;
#pragma unroll
                    for (int k = 0; k < kRows / 32; ++k)   // 32 rows of the chunk per MMA
                        umma_e4m3(d, umma_desc(v0 + k * 4 * 1024, 1024, 1024),
                                  umma_desc(b0 + 32 * k, 16, 1024), kIdPV, k > 0);
                    umma_commit(bar(O_FULL + (g & 1)));
                    umma_commit(bar(KV_EMPTY + g % NC));
                    issued_pv = true;
                }
                if (ch == nch - 1) {
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        if (g & 1) l_done1[gg] = l_thr[gg];
                        else l_done0[gg] = l_thr[gg];
                    }
                }
                // ---- output side of the previous chunk
                if (g >= 1) output_chunk(g - 1, prev_it, prev_it.z, prev_first, prev_last, prev_bad);
                prev_it = it;
                prev_first = ch == 0;
                prev_last = ch == nch - 1;
                prev_bad = bad;
            }
        }
        if (g >= 1) output_chunk(g - 1, prev_it, prev_it.z, prev_first, prev_last, prev_bad);
        // Every P.V issued completes before the tensor memory is freed (also
        // after an abort).
        if (threadIdx.x == 2 * 32 && issued_pv) {
            umma_commit(bar(DONE_PV));
            (void)mbar_wait(bar(DONE_PV), 0);
        }
    }

    // Every role is done with the tensor memory and the ring.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kCols)
                     : "memory");
}

template <int G, int NC>
cudaError_t run_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                   int sm_count, cudaStream_t stream) {
    using L = TcSmem<G, NC>;
    auto kernel = decode_tc_fp8_kernel<G, NC>;
    const int smem = static_cast<int>(L::kBytes);
    static std::atomic<int> cached_per_sm[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    int per_sm = dev < kMaxDevices ? cached_per_sm[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm == 0) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        // All of the SM's on-chip memory as shared memory: two CTAs' rings
        // fit only then.
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTcThreads, smem);
        if (err != cudaSuccess) return err;
        // The occupancy query has answered one CTA per SM where two fit (the
        // launch then runs two per SM): count from the SM's shared memory,
        // registers and the launch bounds as well, and take the larger.
        int smem_sm = 0, reserved = 0;
        cudaFuncAttributes fa{};
        if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
            return cudaErrorInvalidConfiguration;
        const int by_smem = smem_sm / (smem + reserved);
        const int by_regs = fa.numRegs > 0 ? 65536 / (fa.numRegs * kTcThreads) : 1;
        per_sm = max(per_sm, min(min(by_smem, by_regs), kTcMinCtas));
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        // Tensor memory: every resident CTA holds TcShape<G>::kCols of the
        // SM's 512 columns.
        per_sm = min(per_sm, 512 / TcShape<G>::kCols);
        if (dev < kMaxDevices) cached_per_sm[dev].store(per_sm, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count * per_sm));
    cfg.blockDim = dim3(kTcThreads);
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

// Chunk slots (32 KB each) per CTA: three keep more bytes in flight while a
// chunk is computed on; with 8 query heads per KV head the larger operands
// leave room for two (two CTAs per SM either way).
template <int G>
constexpr int kTcSlots = G <= 4 ? 3 : 2;

}  // namespace

cudaError_t launch_decode_fp8_tc(const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeParams& p, int sm_count, cudaStream_t stream) {
    if (p.head_dim != 128 || p.num_queries != 1 || p.window != 0) return cudaErrorNotSupported;
    switch (p.num_heads / p.num_kv_heads) {
        case 1: return run_tc<1, kTcSlots<1>>(tk, tv, p, sm_count, stream);
        case 2: return run_tc<2, kTcSlots<2>>(tk, tv, p, sm_count, stream);
        case 4: return run_tc<4, kTcSlots<4>>(tk, tv, p, sm_count, stream);
        case 8: return run_tc<8, kTcSlots<8>>(tk, tv, p, sm_count, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
