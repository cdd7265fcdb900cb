// pa_tile_math.cuh -- the per-tile math of the paged decode kernels.
//
// A tile is 16 consecutive rows of one sequence's K (and V) for one KV head:
// 16 rows x head_dim of one physical block, staged in shared memory by TMA as
// 128-byte-wide boxes with the 128-byte swizzle. A consumer warp folds tiles
// into an online-softmax state per query head of its group (running max m,
// running sum l, unnormalised output o, rescaled by 2^(m_old - m_new) when the
// max grows: the online softmax of "MLSys Engineer -- Inference Systems Q&A",
// Q4 "How would you write a fused attention kernel?"), accumulating in fp32.
// Scores are kept in base 2: the score scale is scale * log2(e).
//
//   MmaMath   bf16: S^T = K_tile . Q^T and O^T += V_tile^T . P^T as m16n8k16
//             tensor-core MMAs (tokens, then head-dim rows, as M; the G <= 8
//             query heads of the group as N), softmax on the accumulators;
//   SimtMath  fp32 or bf16: CUDA-core dot products and warp-shuffle sums.
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

// The query columns of one work item (sequence s, KV head h): with Q query
// tokens per sequence and G query heads per KV head, column c is query token
// j = c / G of head h * G + c % G, i.e. row (s * Q + j) * num_heads + h * G +
// c % G of q and out. One query per sequence: the G heads of the group.
__device__ __forceinline__ size_t query_row(const DecodeParams& p, int s, int h, int c, int grp) {
    const int j = c / grp;
    return (static_cast<size_t>(s) * p.num_queries + j) * p.num_heads + h * grp + (c - j * grp);
}

// One warp copies the ncols q rows (D bf16 each) of (sequence s, KV head h)
// into a staging buffer whose rows are ROW_BYTES apart, with cp.async.
template <int D, int ROW_BYTES>
__device__ __forceinline__ void stage_q_rows(const DecodeParams& p, int s, int h, int ncols,
                                             int grp, uint32_t qbuf, int lane) {
    constexpr int kChunksPerRow = D * 2 / 16;
    const uint8_t* q = reinterpret_cast<const uint8_t*>(p.q);
    for (int c = lane; c < ncols * kChunksPerRow; c += 32) {
        const int col = c / kChunksPerRow, ch = c - col * kChunksPerRow;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         qbuf + static_cast<uint32_t>(col * ROW_BYTES + ch * 16)),
                     "l"(q + query_row(p, s, h, col, grp) * D * 2 + ch * 16)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Tensor-core tile math (bf16). Fragment layouts are those of mma.m16n8k16:
// lane = 4 * gid + t4; accumulator c0,c1 = (row gid, cols 2t4, 2t4+1),
// c2,c3 = (row gid + 8, same cols).
//   QK:  C = S^T [16 tokens][8 columns], A = K tile [16 tokens][16 dims] per
//        k-step (ldmatrix), B = Q^T [16 dims][8 columns] (registers). The
//        columns are the item's query columns (query_row): the G <= 8 heads of
//        the group, or G heads x Q query tokens when several tokens per
//        sequence are verified together; columns past them are zero.
//   PV:  C = O^T [16 dims][8 heads] per m-tile of 16 dims, A = V^T [16 dims]
//        [16 tokens] (ldmatrix.trans of the V tile), B = P^T [16 tokens]
//        [8 heads], built from the QK accumulators with four shuffles.
// ---------------------------------------------------------------------------
// CAUSAL: items may carry several query tokens per sequence, each seeing
// rows up to its own (masks per column, max -inf guards); otherwise one query
// per sequence and rows past the sequence are the only masked ones.
template <int D, int G, bool CAUSAL = false>
struct MmaMath {
    using T = __nv_bfloat16;
    static constexpr bool kCausal = CAUSAL;
    static constexpr bool kQuantAppend = false;   // a fused append copies rows as they are
    static constexpr int kExtraStageBytes = 0;
    using Geom = TileGeom<T, D>;
    static constexpr int kSteps = D / 16;
    // G: query columns the state holds (a capacity: an item uses ncols <= G).
    static_assert(G >= 1 && G <= 8, "the MMA N dimension holds at most 8 query columns");

    // q of the next item is staged in shared memory ([G][D] bf16 rows padded
    // to D * 2 + 16 bytes, so that the fragment reads below hit 32 different
    // banks) by one warp with cp.async, instead of being held in registers.
    static constexpr bool kQInSmem = true;
    static constexpr int kQRowBytes = D * 2 + 16;
    static constexpr int kQBufBytes = ((G * kQRowBytes + 127) / 128) * 128;
    struct QRegs {};

    uint32_t qb[kSteps][2];
    float o[kSteps][4];
    float m[2], l[2];
    int gid, t4;

    __device__ __forceinline__ void setup(int lane, const DecodeParams&) {
        gid = lane >> 2;
        t4 = lane & 3;
    }

    // One warp copies q of (sequence s, KV head h) into the staging buffer.
    __device__ __forceinline__ void stage_q(const DecodeParams& p, int s, int h, int ncols,
                                            int grp, uint32_t qbuf, int lane) const {
        stage_q_rows<D, kQRowBytes>(p, s, h, ncols, grp, qbuf, lane);
    }

    // Start an item: read q's B fragments from the staging buffer and clear
    // the softmax state.
    __device__ __forceinline__ void begin_staged(const uint8_t* qbuf, int ncols) {
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const uint8_t* r = qbuf + gid * kQRowBytes + (16 * kk + 2 * t4) * 2;
            qb[kk][0] = 0u;
            qb[kk][1] = 0u;
            if (gid < ncols) {
                qb[kk][0] = *reinterpret_cast<const uint32_t*>(r);
                qb[kk][1] = *reinterpret_cast<const uint32_t*>(r + 16);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) o[kk][i] = 0.f;
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    // valid: rows of the tile before the end of the sequence (V rows past it
    // are zeroed). Row row0 + i is visible to query column c when row0 + i <=
    // limit0 + c / grp (limit0: the last row query token 0 sees) and i >= skip
    // (rows before a sliding window; skip <= 0 without one). A tile always
    // holds a visible row for one query per sequence.
    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float scale_log2, int lane, int row0, int limit0,
                                         int grp, int skip, uint32_t /*xb: none*/) {
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
        if constexpr (CAUSAL) {
            if (row0 + kTileRows - 1 > limit0) {
                // Rows past the query token's own row.
                const int j0 = (2 * t4) / grp, j1 = (2 * t4 + 1) / grp;
                const int r = row0 + gid;
                if (r > limit0 + j0) c[0] = -INFINITY;
                if (r > limit0 + j1) c[1] = -INFINITY;
                if (r + 8 > limit0 + j0) c[2] = -INFINITY;
                if (r + 8 > limit0 + j1) c[3] = -INFINITY;
            }
        } else {
            if (valid < kTileRows) {
                // Rows past the sequence.
                if (gid >= valid) c[0] = c[1] = -INFINITY;
                if (gid + 8 >= valid) c[2] = c[3] = -INFINITY;
            }
            if (skip > 0) {
                // Rows before a sliding window.
                if (gid < skip) c[0] = c[1] = -INFINITY;
                if (gid + 8 < skip) c[2] = c[3] = -INFINITY;
            }
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
        // With several query tokens, a column with no visible row yet keeps
        // max -inf: exponentiate against 0 then, so that its weights are 0
        // rather than NaN. (One query per sequence: every tile has a row.)
        const float ref0 = (CAUSAL && mn0 == -INFINITY) ? 0.f : mn0;
        const float ref1 = (CAUSAL && mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = fast_exp2(m[0] - ref0);
        const float al1 = fast_exp2(m[1] - ref1);
        const float p0 = fast_exp2(c[0] - ref0);
        const float p1 = fast_exp2(c[1] - ref1);
        const float p2 = fast_exp2(c[2] - ref0);
        const float p3 = fast_exp2(c[3] - ref1);
        l[0] = l[0] * al0 + (p0 + p2);
        l[1] = l[1] * al1 + (p1 + p3);
        // The rescale factor is exactly 1 where the max did not grow: skip the
        // multiply when that holds for the whole warp.
        const bool grew = __any_sync(0xffffffffu, (mn0 != m[0]) | (mn1 != m[1]));
        m[0] = mn0;
        m[1] = mn1;
        if (grew) {
#pragma unroll
            for (int mt = 0; mt < kSteps; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
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

    // State layout: m[G], l[G], o[G][D] (fp32, base-2 max); columns < ncols.
    __device__ __forceinline__ void write_state(float* st, int lane, int ncols) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
        (void)lane;
        const int h0 = 2 * t4, h1 = 2 * t4 + 1;
        if (gid == 0) {
            if (h0 < ncols) { st[h0] = m[0]; st[G + h0] = l[0]; }
            if (h1 < ncols) { st[h1] = m[1]; st[G + h1] = l[1]; }
        }
        float* so = st + 2 * G;
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            const int d0 = 16 * mt + gid;
            if (h0 < ncols) { so[h0 * D + d0] = o[mt][0]; so[h0 * D + d0 + 8] = o[mt][2]; }
            if (h1 < ncols) { so[h1 * D + d0] = o[mt][1]; so[h1 * D + d0 + 8] = o[mt][3]; }
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
    static constexpr bool kCausal = false;
    static constexpr bool kQuantAppend = false;   // a fused append copies rows as they are
    static constexpr int kExtraStageBytes = 0;
    using Geom = TileGeom<T, D>;
    using E = ElemTraits<T>;
    static constexpr int kEpc = E::kPerChunk;               // elements per 16-byte chunk
    static constexpr int kCpr = Geom::kRowBytes / 16;       // chunks per row
    static constexpr int kLpr = kCpr < 32 ? kCpr : 32;      // lanes per row
    static_assert(kCpr == kLpr, "one chunk per lane per row");
    static constexpr int kRpp = 32 / kLpr;                  // rows per pass
    static constexpr int kPasses = kTileRows / kRpp;
    static constexpr int kSub = kPasses < 8 ? kPasses : 8;  // passes per softmax sub-step

    // This lane's chunk of q for every head of the group, scaled to base 2.
    // It is prefetched one item ahead only when small; otherwise begin()
    // loads it (the extra registers would spill).
    static constexpr bool kPrefetch = G * kEpc <= 32;
    static constexpr bool kQInSmem = false;
    static constexpr int kQBufBytes = 0;
    struct QRegs {
        float f[kPrefetch ? G : 1][kPrefetch ? kEpc : 1];
        int s, h;
    };

    float qf[G][kEpc];
    float o[G][kEpc];
    float m[G], l[G];
    int rr, ch;

    __device__ __forceinline__ void setup(int lane, const DecodeParams&) {
        rr = lane / kLpr;
        ch = lane % kLpr;
    }

    __device__ __forceinline__ void load_rows(const DecodeParams& p, int s, int h,
                                              float (&dst)[G][kEpc]) const {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const T* qrow = static_cast<const T*>(p.q) +
                            (static_cast<size_t>(s) * p.num_heads + h * G + g) * D;
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow) + ch);
            E::unpack(raw, dst[g]);
#pragma unroll
            for (int e = 0; e < kEpc; ++e) dst[g][e] *= p.scale_log2;
        }
    }

    __device__ __forceinline__ void load_q(const DecodeParams& p, int s, int h, QRegs& r) const {
        r.s = s;
        r.h = h;
        if constexpr (kPrefetch) load_rows(p, s, h, r.f);
    }

    __device__ __forceinline__ void begin(const DecodeParams& p, const QRegs& r) {
        if constexpr (kPrefetch) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < kEpc; ++e) qf[g][e] = r.f[g][e];
        } else {
            load_rows(p, r.s, r.h, qf);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < kEpc; ++e) o[g][e] = 0.f;
            m[g] = -INFINITY;
            l[g] = 0.f;
        }
    }

    // One query per sequence: rows past `valid` are masked (limit0 and grp
    // describe the same boundary and are not needed), and the first `skip`
    // rows (a sliding window starting inside this tile).
    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float /*scale_log2*/, int /*lane*/, int /*row0*/,
                                         int /*limit0*/, int /*grp*/, int skip,
                                         uint32_t /*xb: none*/) {
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
            if (valid < kTileRows || skip > 0) {
#pragma unroll
                for (int j = 0; j < kSub; ++j) {
                    const int row = (sub * kSub + j) * kRpp + rr;
                    if (row >= valid || row < skip)
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
                // Rows before a window can mask a whole sub-step while the
                // max is still -inf: exponentiate against 0 then (weights 0).
                const float ref = mn == -INFINITY ? 0.f : mn;
                const float al = fast_exp2(m[g] - ref);
                m[g] = mn;
                l[g] *= al;
#pragma unroll
                for (int e = 0; e < kEpc; ++e) o[g][e] *= al;
#pragma unroll
                for (int j = 0; j < kSub; ++j) {
                    sc[j][g] = fast_exp2(sc[j][g] - ref);
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

    __device__ __forceinline__ void write_state(float* st, int lane, int /*ncols: G*/) {
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

}  // namespace pa
