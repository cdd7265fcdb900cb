// pa_decode_tma.cuh -- paged decode attention with a TMA tile ring.
//
// Work item: one (sequence s, KV head h, partition) of at most partition_size
// rows. One CTA per work item, W consumer warps plus one producer warp.
//
// Producer: stages the partition's block ids in shared memory, then streams
// 16-row tiles of K and V (16 rows x head_dim of one physical block and KV
// head, contiguous in the [block][kv_head][block_size][head_dim] pool) into a
// ring of STAGES shared-memory stages with 2D TMA loads (128-byte swizzle, so
// any 8 rows of one 16-byte column land in 8 different bank groups). Row i of
// the sequence is row (i % block_size) of block block_tables[s][i / block_size]:
// the paged gather of "MLSys Engineer -- Inference Systems Q&A", Q1.
//
// Consumers: warp w takes tiles w, w + W, ... and keeps its own online-softmax
// state per query head of the group (running max m, running sum l, and an
// unnormalised output o rescaled by exp(m_old - m_new) when the max grows, as
// in Q4 "How would you write a fused attention kernel?"), with fp32
// accumulation throughout. Scores are kept in base 2 (scale * log2 e folded
// into the score scale). The math of one tile is a policy:
//   MmaMath   bf16: S^T = K_tile . Q^T and O^T += V_tile^T . P^T as
//             m16n8k16 tensor-core MMAs (tokens, then head-dim rows, as M;
//             the G <= 8 query heads of the group as N);
//   SimtMath  fp32 or bf16: CUDA-core dot products and warp-shuffle sums.
// At the end the W warp states are merged through shared memory and written
// either as the final normalised output (one partition) or as a partition
// partial (max, sum, unnormalised output) for the combine kernel.
#pragma once

#include <cfloat>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kTileRows = 16;
constexpr int kBoxBytes = kTileRows * 128;   // one 16 x 128-byte TMA box

// Byte address of 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled box that starts at a 1024-byte-aligned address.
__device__ __forceinline__ uint32_t swizzled(uint32_t box, int row, int chunk) {
    return box + static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <typename T, int D>
struct TileGeom {
    static constexpr int kElem = sizeof(T);
    static constexpr int kRowBytes = D * kElem;
    static constexpr int kBoxes = kRowBytes / 128;     // 128-byte column boxes per row
    static constexpr int kBoxElems = 128 / kElem;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;  // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte boxes");
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1,
                                        uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& a0, uint32_t& a1,
                                              uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}

// D (16x8, fp32) += A (16x16, bf16, row) . B (16x8, bf16, col)
__device__ __forceinline__ void mma_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// ---------------------------------------------------------------------------
// Tensor-core tile math (bf16). Fragment layouts are those of mma.m16n8k16:
// lane = 4 * gid + t4; accumulator c0,c1 = (row gid, cols 2t4, 2t4+1),
// c2,c3 = (row gid + 8, same cols).
//   QK:  C = S^T [16 tokens][8 heads], A = K tile [16 tokens][16 dims] per
//        k-step (ldmatrix), B = Q^T [16 dims][8 heads] (registers; heads >= G
//        are zero).
//   PV:  C = O^T [16 dims][8 heads] per m-tile of 16 dims, A = V^T [16 dims]
//        [16 tokens] (ldmatrix.trans of the V tile), B = P^T [16 tokens]
//        [8 heads], built from the QK accumulators with four shuffles.
// ---------------------------------------------------------------------------
template <int D, int G>
struct MmaMath {
    using T = __nv_bfloat16;
    using Geom = TileGeom<T, D>;
    static constexpr int kSteps = D / 16;
    static_assert(G >= 1 && G <= 8, "the MMA N dimension holds at most 8 query heads");

    uint32_t qb[kSteps][2];
    float o[kSteps][4];
    float m[2], l[2];
    int gid, t4;

    __device__ __forceinline__ void init(const DecodeParams& p, int s, int h, int lane) {
        gid = lane >> 2;
        t4 = lane & 3;
        // Lanes of padded heads (gid >= G) keep a valid row pointer and load nothing.
        const int head = h * G + (gid < G ? gid : G - 1);
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            static_cast<const T*>(p.q) + (static_cast<size_t>(s) * p.num_heads + head) * D);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            qb[kk][0] = gid < G ? __ldg(qrow + 8 * kk + t4) : 0u;
            qb[kk][1] = gid < G ? __ldg(qrow + 8 * kk + 4 + t4) : 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) o[kk][i] = 0.f;
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float scale_log2, int lane) {
        const int mi = lane >> 3;
        const int lr = lane & 7;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int r = lr + ((mi & 1) << 3);
#pragma unroll
            for (int kk = 0; kk < kSteps; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(swizzled(kbase + (kk >> 2) * kBoxBytes, r, 2 * (kk & 3) + (mi >> 1)),
                        a0, a1, a2, a3);
                mma_16816(c, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] *= scale_log2;
        if (valid < kTileRows) {
            if (gid >= valid) c[0] = c[1] = -INFINITY;
            if (gid + 8 >= valid) c[2] = c[3] = -INFINITY;
        }
        float mx0 = fmaxf(c[0], c[2]);
        float mx1 = fmaxf(c[1], c[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0);
        const float mn1 = fmaxf(m[1], mx1);
        const float al0 = fast_exp2(m[0] - mn0);
        const float al1 = fast_exp2(m[1] - mn1);
        const float p0 = fast_exp2(c[0] - mn0);
        const float p1 = fast_exp2(c[1] - mn1);
        const float p2 = fast_exp2(c[2] - mn0);
        const float p3 = fast_exp2(c[3] - mn1);
        l[0] = l[0] * al0 + (p0 + p2);
        l[1] = l[1] * al1 + (p1 + p3);
        m[0] = mn0;
        m[1] = mn1;
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
        }
        // P^T as the B operand: lane (gid, t4) needs P[token 2t4, 2t4+1][head gid]
        // (b0) and P[token 2t4+8, 2t4+9][head gid] (b1). Lane (g', t') holds
        // P[token g'][heads 2t', 2t'+1] and P[token g'+8][same heads].
        const uint32_t p01 = pack_bf16x2(p0, p1);
        const uint32_t p23 = pack_bf16x2(p2, p3);
        const int src_a = 8 * t4 + (gid >> 1);
        const uint32_t v0 = __shfl_sync(0xffffffffu, p01, src_a);
        const uint32_t v1 = __shfl_sync(0xffffffffu, p01, src_a + 4);
        const uint32_t w0 = __shfl_sync(0xffffffffu, p23, src_a);
        const uint32_t w1 = __shfl_sync(0xffffffffu, p23, src_a + 4);
        const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = prmt(v0, v1, sel);
        const uint32_t b1 = prmt(w0, w1, sel);
        const int r = lr + ((mi >> 1) << 3);
        if (valid == kTileRows) {
#pragma unroll
            for (int mt = 0; mt < kSteps; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(
                    swizzled(vbase + (mt >> 2) * kBoxBytes, r, 2 * (mt & 3) + (mi & 1)), a0, a1,
                    a2, a3);
                mma_16816(o[mt], a0, a1, a2, a3, b0, b1);
            }
        } else {
            // Rows past the sequence hold whatever the pool holds (possibly NaN
            // bit patterns): zero their V values so that 0 * V stays 0.
            const int tk = 2 * t4;
            const uint32_t mlo = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
            const uint32_t mhi = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < kSteps; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(
                    swizzled(vbase + (mt >> 2) * kBoxBytes, r, 2 * (mt & 3) + (mi & 1)), a0, a1,
                    a2, a3);
                mma_16816(o[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
            }
        }
    }

    // State layout: m[G], l[G], o[G][D] (fp32, base-2 max).
    __device__ __forceinline__ void write_state(float* st, int lane) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
        (void)lane;
        const int h0 = 2 * t4, h1 = 2 * t4 + 1;
        if (gid == 0) {
            if (h0 < G) { st[h0] = m[0]; st[G + h0] = l[0]; }
            if (h1 < G) { st[h1] = m[1]; st[G + h1] = l[1]; }
        }
        float* so = st + 2 * G;
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            const int d0 = 16 * mt + gid;
            if (h0 < G) { so[h0 * D + d0] = o[mt][0]; so[h0 * D + d0 + 8] = o[mt][2]; }
            if (h1 < G) { so[h1 * D + d0] = o[mt][1]; so[h1 * D + d0 + 8] = o[mt][3]; }
        }
    }
};

// ---------------------------------------------------------------------------
// CUDA-core tile math (fp32 or bf16). A row of the tile is split over LPR
// lanes, one 16-byte chunk each; RPP = 32 / LPR rows are processed per pass.
// Dot products are summed over the LPR lanes with butterfly shuffles, so every
// lane of a row group holds the row's scores; softmax runs on sub-tiles of at
// most 8 passes to bound registers.
// ---------------------------------------------------------------------------
template <typename TT, int D, int G>
struct SimtMath {
    using T = TT;
    using Geom = TileGeom<T, D>;
    using E = ElemTraits<T>;
    static constexpr int kEpc = E::kPerChunk;               // elements per 16-byte chunk
    static constexpr int kCpr = Geom::kRowBytes / 16;       // chunks per row
    static constexpr int kLpr = kCpr < 32 ? kCpr : 32;      // lanes per row
    static_assert(kCpr == kLpr, "one chunk per lane per row");
    static constexpr int kRpp = 32 / kLpr;                  // rows per pass
    static constexpr int kPasses = kTileRows / kRpp;
    static constexpr int kSub = kPasses < 8 ? kPasses : 8;  // passes per softmax sub-step

    float qf[G][kEpc];
    float o[G][kEpc];
    float m[G], l[G];
    int rr, ch;

    __device__ __forceinline__ void init(const DecodeParams& p, int s, int h, int lane) {
        rr = lane / kLpr;
        ch = lane % kLpr;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const T* qrow = static_cast<const T*>(p.q) +
                            (static_cast<size_t>(s) * p.num_heads + h * G + g) * D;
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow) + ch);
            E::unpack(raw, qf[g]);
#pragma unroll
            for (int e = 0; e < kEpc; ++e) {
                qf[g][e] *= p.scale_log2;
                o[g][e] = 0.f;
            }
            m[g] = -INFINITY;
            l[g] = 0.f;
        }
    }

    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float /*scale_log2*/, int /*lane*/) {
        const uint32_t kbox = kbase + (ch >> 3) * kBoxBytes;
        const uint32_t vbox = vbase + (ch >> 3) * kBoxBytes;
        const int cc = ch & 7;
#pragma unroll
        for (int sub = 0; sub < kPasses / kSub; ++sub) {
            float sc[kSub][G];
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                const int row = (sub * kSub + j) * kRpp + rr;
                float kv[kEpc];
                E::unpack(lds128(swizzled(kbox, row, cc)), kv);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < kEpc; ++e) acc = fmaf(qf[g][e], kv[e], acc);
                    sc[j][g] = acc;
                }
            }
#pragma unroll
            for (int j = 0; j < kSub; ++j)
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int off = 1; off < kLpr; off <<= 1)
                        sc[j][g] += __shfl_xor_sync(0xffffffffu, sc[j][g], off);
            if (valid < kTileRows) {
#pragma unroll
                for (int j = 0; j < kSub; ++j) {
                    const int row = (sub * kSub + j) * kRpp + rr;
                    if (row >= valid)
#pragma unroll
                        for (int g = 0; g < G; ++g) sc[j][g] = -INFINITY;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = sc[0][g];
#pragma unroll
                for (int j = 1; j < kSub; ++j) mx = fmaxf(mx, sc[j][g]);
#pragma unroll
                for (int off = kLpr; off < 32; off <<= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float mn = fmaxf(m[g], mx);
                const float al = fast_exp2(m[g] - mn);
                m[g] = mn;
                l[g] *= al;
#pragma unroll
                for (int e = 0; e < kEpc; ++e) o[g][e] *= al;
#pragma unroll
                for (int j = 0; j < kSub; ++j) {
                    sc[j][g] = fast_exp2(sc[j][g] - mn);
                    l[g] += sc[j][g];
                }
            }
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                const int row = (sub * kSub + j) * kRpp + rr;
                if (row < valid) {
                    float vv[kEpc];
                    E::unpack(lds128(swizzled(vbox, row, cc)), vv);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < kEpc; ++e) o[g][e] = fmaf(sc[j][g], vv[e], o[g][e]);
                }
            }
        }
    }

    __device__ __forceinline__ void write_state(float* st, int lane) {
#pragma unroll
        for (int off = kLpr; off < 32; off <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
                for (int e = 0; e < kEpc; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], off);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) { st[g] = m[g]; st[G + g] = l[g]; }
        }
        if (rr == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < kEpc; ++e) st[2 * G + g * D + ch * kEpc + e] = o[g][e];
        }
    }
};

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int W, int STAGES, typename Geom, int G, int D>
struct DecodeSmem {
    static constexpr int kRing = STAGES * Geom::kStageBytes;
    static constexpr int kState = 2 * G + G * D;
    static_assert(W * kState * 4 <= kRing, "the merge scratch reuses the ring");
    // align slack + ring + full/empty barriers + flags + block ids
    static size_t bytes(int partition_size) {
        return 1024 + kRing + 16 * STAGES + 4 * 4 + 4 * (partition_size / kTileRows + 2);
    }
};

template <typename T>
__device__ __forceinline__ void write_zero_rows(const DecodeParams& p, int s, int h, int G, int D) {
    T* out = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.num_heads + h * G) * D;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) ElemTraits<T>::store(out + i, 0.f);
}

// Stage ownership: tile t lives in stage t % STAGES and is consumed by warp
// t % W. With STAGES a multiple of W every stage belongs to one warp, which
// waits on its uses in order, so a waiter is never more than one phase ahead
// of the barrier it polls. (A parity wait cannot tell phase u from phase u+2:
// if a stage were shared between warps, a fast warp could see the stage's
// previous phase as its own and consume a tile that has not landed.)
template <class Math, int D, int G, int W, int STAGES>
__global__ void __launch_bounds__((W + 1) * 32)
decode_tma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    static_assert(STAGES % W == 0, "each ring stage must belong to exactly one consumer warp");
    using T = typename Math::T;
    using Geom = typename Math::Geom;
    using Smem = DecodeSmem<W, STAGES, Geom, G, D>;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + Smem::kRing);
    uint64_t* empty = full + STAGES;
    volatile int32_t* flags = reinterpret_cast<volatile int32_t*>(empty + STAGES);
    // flags[0]: bad block id seen; flags[1]: producer gave up; flags[2]: a consumer gave up
    int32_t* s_blk = reinterpret_cast<int32_t*>(empty + STAGES) + 4;

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
    const int P = p.partition_size;
    const int lo = part * P;
    if (n == 0) {
        if (part == 0) write_zero_rows<T>(p, s, h, G, D);
        return;
    }
    if (lo >= n) return;
    const int hi = min(n, lo + P);
    const int ntiles = (hi - lo + kTileRows - 1) / kTileRows;
    const int nparts = (n + P - 1) / P;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bs = p.block_size;
    const int b0 = lo / bs;
    const int nblk = (hi - 1) / bs - b0 + 1;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), 1);
        }
        flags[1] = 0;
        flags[2] = 0;
        mbar_init_fence();
    }
    Math math;
    if (warp == W) {
        bool bad = false;
        const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks_per_seq + b0;
        for (int j = lane; j < nblk; j += 32) {
            const int id = __ldg(bt + j);
            bad |= (id < 0) | (id >= p.num_blocks);
            s_blk[j] = id;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            flags[0] = bad ? 1 : 0;
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
    } else {
        math.init(p, s, h, lane);
    }
    __syncthreads();
    if (flags[0]) {
        if (threadIdx.x == 0) raise_error(p.error_word, PA_DEVERR_BLOCK_ID);
        return;
    }

    const uint32_t ring_addr = smem_addr(ring);
    if (warp == W) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const int stage = t % STAGES;
                if (t >= STAGES && !mbar_wait(smem_addr(&empty[stage]), ((t / STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (flags[2]) break;
                const int tok = lo + kTileRows * t;
                const int id = s_blk[tok / bs - b0];
                const int row = (id * p.num_kv_heads + h) * bs + (tok % bs);
                const uint32_t fb = smem_addr(&full[stage]);
                const uint32_t dst = ring_addr + stage * Geom::kStageBytes;
                mbar_arrive_expect_tx(fb, Geom::kStageBytes);
#pragma unroll
                for (int b = 0; b < Geom::kBoxes; ++b)
                    tma_load_2d(dst + b * kBoxBytes, &tmap_k, fb, b * Geom::kBoxElems, row);
#pragma unroll
                for (int b = 0; b < Geom::kBoxes; ++b)
                    tma_load_2d(dst + Geom::kTileBytes + b * kBoxBytes, &tmap_v, fb,
                                b * Geom::kBoxElems, row);
                issued = t + 1;
            }
            if (!ok) {
                raise_error(p.error_word, PA_DEVERR_TIMEOUT);
                flags[1] = 1;
            }
            // Copies still in flight must land before this CTA's shared memory
            // can be released: wait (bounded) for the last issued stages.
            for (int t = issued > STAGES ? issued - STAGES : 0; t < issued; ++t)
                (void)mbar_wait(smem_addr(&full[t % STAGES]), (t / STAGES) & 1);
        }
        return;
    }

    // ---------------- consumers ----------------
    bool ok = true;
    for (int t = warp; t < ntiles; t += W) {
        const int stage = t % STAGES;
        const bool got = mbar_wait(smem_addr(&full[stage]), (t / STAGES) & 1);
        if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
        }
        const int valid = min(kTileRows, hi - (lo + kTileRows * t));
        const uint32_t kb = ring_addr + stage * Geom::kStageBytes;
        math.tile(kb, kb + Geom::kTileBytes, valid, p.scale_log2, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[stage]));
    }
    if (!ok && lane == 0) {
        raise_error(p.error_word, PA_DEVERR_TIMEOUT);
        flags[2] = 1;
    }
    named_barrier(1, W * 32);
    if (flags[2]) return;   // copies may still land in the ring: no merge

    float* state = reinterpret_cast<float*>(ring);
    math.write_state(state + warp * Smem::kState, lane);
    named_barrier(1, W * 32);

    const int qh0 = h * G;
    for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
        const int g = idx / D;
        const int d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, state[w * Smem::kState + g]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float* sw = state + w * Smem::kState;
            const float cw = fast_exp2(sw[g] - M);
            L = fmaf(cw, sw[G + g], L);
            O = fmaf(cw, sw[2 * G + g * D + d], O);
        }
        const size_t row = static_cast<size_t>(s) * p.num_heads + qh0 + g;
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
}

// Host-side launch of one instance.
template <class Math, int D, int G, int W, int STAGES>
cudaError_t launch_tma_instance(const CUtensorMap& tk, const CUtensorMap& tv,
                                const DecodeParams& p, cudaStream_t stream) {
    using Smem = DecodeSmem<W, STAGES, typename Math::Geom, G, D>;
    auto kernel = decode_tma_kernel<Math, D, G, W, STAGES>;
    const size_t smem = Smem::bytes(p.partition_size);
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const long long grid = static_cast<long long>(p.max_parts) * p.num_seqs * p.num_kv_heads;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kernel<<<static_cast<unsigned>(grid), (W + 1) * 32, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace pa
