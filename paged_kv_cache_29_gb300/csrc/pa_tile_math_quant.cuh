// pa_tile_math_quant.cuh -- per-tile math for quantised KV caches (8-bit codes)
// with bf16 q and output: FP8 (e4m3) with one scale per tensor, and INT8 with
// one scale per (row, KV head).
//
//   FP8   value = k_scale * e4m3(code) (V: v_scale); an FP8 cache halves the
//         bytes per token, scales per tensor ("Forward Deployed Engineering
//         Interview", Chapter 2 "Batching and the KV Cache").
//   INT8  value = scale_row * code with scale_row = max|row| / 127
//         ("MLSys Engineer -- Inference Systems Q&A", Q3: INT8 KV with
//         per-token scaling, dequantised before the softmax).
//
// The codes are widened to f16 in registers (exact for both formats: every
// e4m3 value and every int8 is an f16 value) and multiplied with m16n8k16 f16
// MMAs accumulating in fp32; the online softmax is that of MmaMath. The
// scales never touch the products:
//   FP8   S = (q * scale * log2(e) * k_scale) . code(K): q is scaled and
//         rounded to f16 once per item, so the accumulators are base-2
//         scores; O = v_scale * sum_i p_i code(V_i), v_scale applied when the
//         warp state is written.
//   INT8  S_row = k_scale_row * (q * scale * log2(e)) . code(K_row): each
//         accumulator row is multiplied by its K scale; O = sum_row (p_row *
//         v_scale_row) code(V_row): the V scale folds into the probability
//         before it becomes an MMA operand, while the softmax sum keeps p_row.
//         The 16 K and 16 V scales of a tile arrive with it, in a small
//         per-stage array (extra stage bytes).
//
// Widening: e4m3 with cvt.rn.f16x2.e4m3x2; int8 code c as the f16 bit pattern
// 0x6400 | (c ^ 0x80), the value 1024 + 128 + c, minus 1152.
//
// Fragment assignment (lane = 4 * gid + t4; the dot products and the output
// rows are sums and rows, so any fixed assignment of dims works when A, B and
// the output agree on it):
//   QK  k-step j (0..7) covers, for lane t4, dims 16 c + 4 (j % 4) .. + 3 of
//       chunk c = 2 t4 + j / 4: the A registers of row gid are that 4-byte
//       word of K row gid (two codes per register), q' is dealt the same way.
//       Each lane reads whole 16-byte chunks 2 t4 and 2 t4 + 1 of rows gid
//       and gid + 8; with the 128-byte swizzle the 8 lanes of a phase hit 8
//       different chunks (no bank conflicts).
//   PV  m-tile mt covers dims 16 mt + gid (row gid) and 16 mt + gid + 8 (row
//       gid + 8): the 16-byte chunk mt of the tile's 16 token rows, read with
//       a transposing 8-bit ldmatrix (m16n16.trans.b8). That load gives lane
//       (gid, t4) column gid (first word) and column gid + 8 (second word) of
//       matrix rows 4 t4 .. 4 t4 + 3; matrix row 4 t + j is pointed at token
//       row 2 t + (j & 1) + 8 (j >> 1), so each word holds the codes of tokens
//       2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9: the A registers' token pairs,
//       widened with no byte shuffling.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_tile_math.cuh"

namespace pa {

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// D (16x8, fp32) += A (16x16, f16, row) . B (16x8, f16, col)
__device__ __forceinline__ void mma_16816_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two 16 x 16 byte matrices (threads 0-15 give matrix 0's row addresses,
// threads 16-31 matrix 1's), transposed: lane (gid, t4) receives column gid
// (w0 / w2) and column gid + 8 (w1 / w3) of rows 4 t4 .. 4 t4 + 3, the lowest
// row in the lowest byte.
__device__ __forceinline__ void ldsm_x2_trans_b8(uint32_t addr, uint32_t& w0, uint32_t& w1,
                                                 uint32_t& w2, uint32_t& w3) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(addr));
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// e4m3 codes with one scale per tensor.
struct E4m3Codes {
    static constexpr bool kRowScales = false;
    // One new bf16 row of K and of V (D = 128; kx, vx: this lane's 4 values)
    // quantised into cache row `row`: code = e4m3(x / scale), the division in fp32
    // (IEEE), round to nearest even, saturating (the append kernel's rule).
    __device__ static __forceinline__ void append_row(const DecodeParams& p, uint2 kx, uint2 vx,
                                                      size_t row, int lane) {
        auto enc = [](uint2 x, float sc) -> uint32_t {
            const float2 a = make_float2(__fdiv_rn(bf16_lo(x.x), sc), __fdiv_rn(bf16_hi(x.x), sc));
            const float2 b = make_float2(__fdiv_rn(bf16_lo(x.y), sc), __fdiv_rn(bf16_hi(x.y), sc));
            return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3)) |
                   (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3)) << 16);
        };
        static_cast<uint32_t*>(const_cast<void*>(p.k_cache))[row * 32 + lane] = enc(kx, p.k_scale);
        static_cast<uint32_t*>(const_cast<void*>(p.v_cache))[row * 32 + lane] = enc(vx, p.v_scale);
    }
    // Four codes -> two f16x2 registers (the low byte of each pair becomes
    // the low half).
    __device__ static __forceinline__ void widen(uint32_t w, uint32_t& lo, uint32_t& hi) {
        asm("{\n\t.reg .b16 l, h;\n\t"
            "mov.b32 {l, h}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
            "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    }
};

// int8 codes with one scale per (row, KV head).
struct S8Codes {
    static constexpr bool kRowScales = true;
    // One new bf16 row of K and of V (D = 128; kx, vx: this lane's 4 values)
    // quantised into cache row `row` with its scale: scale = max|x| / 127, code = x /
    // scale rounded to nearest even, clamped to [-127, 127], both divisions
    // in fp32 (IEEE); an all-zero row gets scale 0 and codes 0 (the append
    // kernel's rule).
    __device__ static __forceinline__ void append_row(const DecodeParams& p, uint2 kx, uint2 vx,
                                                      size_t row, int lane) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint2 w = which ? vx : kx;
            const float x[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float scale = __fdiv_rn(amax, 127.0f);
            uint32_t codes = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int c = 0;
                if (scale != 0.f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(x[i], scale))));
                codes |= (static_cast<uint32_t>(c) & 0xffu) << (8 * i);
            }
            static_cast<uint32_t*>(const_cast<void*>(which ? p.v_cache : p.k_cache))[row * 32 + lane] = codes;
            if (lane == 0) const_cast<float*>(which ? p.v_row_scales : p.k_row_scales)[row] = scale;
        }
    }
    __device__ static __forceinline__ void widen(uint32_t w, uint32_t& lo, uint32_t& hi) {
        const uint32_t t = w ^ 0x80808080u;
        const uint32_t a = prmt(t, 0x64646464u, 0x4140u);   // (t.b0, 0x64, t.b1, 0x64)
        const uint32_t b = prmt(t, 0x64646464u, 0x4342u);   // (t.b2, 0x64, t.b3, 0x64)
        const uint32_t bias = 0x64806480u;                  // f16x2 {1152, 1152}
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
    }
};

template <int D, int G, class CodesT>
struct QuantMmaMath {
    using T = __nv_bfloat16;                    // q and out
    using Geom = TileGeom<uint8_t, D>;
    using Codes = CodesT;
    static constexpr bool kCausal = false;
    // The fused append quantises new rows with Codes::append_row.
    static constexpr bool kQuantAppend = true;
    static_assert(D == 128, "one 128-byte row of codes per token");
    static_assert(G >= 1 && G <= 8, "the MMA N dimension holds at most 8 query heads");
    static constexpr int kSteps = D / 16;
    // Row scales: 16 K then 16 V scales (fp32) beside each stage.
    static constexpr int kExtraStageBytes = Codes::kRowScales ? 2 * kTileRows * 4 : 0;

    static constexpr bool kQInSmem = true;
    static constexpr int kQRowBytes = D * 2 + 16;
    static constexpr int kQBufBytes = ((G * kQRowBytes + 127) / 128) * 128;
    struct QRegs {};

    uint32_t qb[kSteps][2];
    float o[kSteps][4];
    float m[2], l[2];
    float qscale, vscale;
    int gid, t4;

    __device__ __forceinline__ void setup(int lane, const DecodeParams& p) {
        gid = lane >> 2;
        t4 = lane & 3;
        qscale = Codes::kRowScales ? p.scale_log2 : p.scale_log2 * p.k_scale;
        vscale = Codes::kRowScales ? 1.f : p.v_scale;
    }

    __device__ __forceinline__ void stage_q(const DecodeParams& p, int s, int h, int ncols,
                                            int grp, uint32_t qbuf, int lane) const {
        stage_q_rows<D, kQRowBytes>(p, s, h, ncols, grp, qbuf, lane);
    }

    // q' = q * qscale in f16, dealt as the k-steps deal the dims; the softmax
    // state is cleared. Lanes of heads gid >= G read nothing (the buffer holds
    // G rows) and hold zeros.
    __device__ __forceinline__ void begin_staged(const uint8_t* qbuf, int /*ncols: G*/) {
        const uint8_t* row = qbuf + gid * kQRowBytes;
#pragma unroll
        for (int j = 0; j < kSteps; ++j) {
            const int d0 = 16 * (2 * t4 + (j >> 2)) + 4 * (j & 3);
            qb[j][0] = 0u;
            qb[j][1] = 0u;
            if (gid < G) {
                const uint2 w = *reinterpret_cast<const uint2*>(row + d0 * 2);
                qb[j][0] = pack_f16x2(bf16_lo(w.x) * qscale, bf16_hi(w.x) * qscale);
                qb[j][1] = pack_f16x2(bf16_lo(w.y) * qscale, bf16_hi(w.y) * qscale);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) o[j][i] = 0.f;
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    // c += code(K tile) . q'^T: c = S^T[token gid, gid + 8][heads 2 t4, 2 t4 + 1].
    __device__ __forceinline__ void qk(uint32_t kbase, float* c) const {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 r0 = lds128(swizzled(kbase, gid, 2 * t4 + half));
            const uint4 r1 = lds128(swizzled(kbase, gid + 8, 2 * t4 + half));
            const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w};
            const uint32_t w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int j = 4 * half + jj;
                uint32_t a0, a1, a2, a3;
                Codes::widen(w0[jj], a0, a2);
                Codes::widen(w1[jj], a1, a3);
                mma_16816_f16(c, a0, a1, a2, a3, qb[j][0], qb[j][1]);
            }
        }
    }

    // P^T B fragments from this lane's probabilities (as in MmaMath): lane
    // (gid, t4) gets P[tokens 2t4, 2t4+1][head gid] and P[tokens 2t4+8,
    // 2t4+9][head gid].
    __device__ __forceinline__ void p_fragments(float p0, float p1, float p2, float p3,
                                                uint32_t& b0, uint32_t& b1) const {
        const uint32_t p01 = pack_f16x2(p0, p1);
        const uint32_t p23 = pack_f16x2(p2, p3);
        const int src_a = 8 * t4 + (gid >> 1);
        const uint32_t v0 = __shfl_sync(0xffffffffu, p01, src_a);
        const uint32_t v1 = __shfl_sync(0xffffffffu, p01, src_a + 4);
        const uint32_t u0 = __shfl_sync(0xffffffffu, p23, src_a);
        const uint32_t u1 = __shfl_sync(0xffffffffu, p23, src_a + 4);
        const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
        b0 = prmt(v0, v1, sel);
        b1 = prmt(u0, u1, sel);
    }

    // O^T += code(V)^T . P^T over one 16-row tile (two 16-dim chunks per
    // ldmatrix). MASK zeroes the V values of rows past `valid`, whose codes may
    // be NaN (e4m3) so that 0 * V stays 0; int8 codes are finite.
    template <bool MASK>
    __device__ __forceinline__ void pv(uint32_t vbase, int valid, uint32_t b0, uint32_t b1) {
        const int r = (4 * gid + t4) & 15;                 // matrix row this lane points at
        const int tok = 2 * (r >> 2) + (r & 1) + 8 * ((r >> 1) & 1);
        const uint32_t row = vbase + static_cast<uint32_t>(tok * 128);
        const int sw = tok & 7;                            // 128-byte swizzle of that row
        const int second = gid >> 2;                       // lanes 16-31: the second chunk
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if constexpr (MASK) {
            const int tk = 2 * t4;
            mlo = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
            mhi = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < kSteps / 2; ++i) {
            uint32_t w[4];
            ldsm_x2_trans_b8(row + static_cast<uint32_t>(((2 * i + second) ^ sw) << 4), w[0], w[1],
                             w[2], w[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int mt = 2 * i + h;
                uint32_t a0, a1, a2, a3;
                Codes::widen(w[2 * h], a0, a2);            // dim 16 mt + gid
                Codes::widen(w[2 * h + 1], a1, a3);        // dim 16 mt + gid + 8
                if constexpr (MASK) {
                    a0 &= mlo;
                    a1 &= mlo;
                    a2 &= mhi;
                    a3 &= mhi;
                }
                mma_16816_f16(o[mt], a0, a1, a2, a3, b0, b1);
            }
        }
    }

    // One query per sequence: rows past `valid` and the first `skip` rows (a
    // sliding window) are masked; a tile always holds a visible row. xb: the
    // stage's row scales (INT8).
    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float /*scale_log2: folded into q'*/, int /*lane*/,
                                         int /*row0*/, int /*limit0*/, int /*grp*/, int skip,
                                         uint32_t xb) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        qk(kbase, c);
        float vs0 = 1.f, vs1 = 1.f;
        if constexpr (Codes::kRowScales) {
            const bool ok0 = gid < valid && gid >= skip;
            const bool ok1 = gid + 8 < valid && gid + 8 >= skip;
            // Scales of rows past the sequence are whatever memory holds: only
            // visible rows read theirs.
            const float ks0 = ok0 ? lds_f32(xb + 4 * gid) : 0.f;
            const float ks1 = ok1 ? lds_f32(xb + 4 * (gid + 8)) : 0.f;
            vs0 = ok0 ? lds_f32(xb + 4 * (kTileRows + gid)) : 0.f;
            vs1 = ok1 ? lds_f32(xb + 4 * (kTileRows + gid + 8)) : 0.f;
            c[0] = ok0 ? c[0] * ks0 : -INFINITY;
            c[1] = ok0 ? c[1] * ks0 : -INFINITY;
            c[2] = ok1 ? c[2] * ks1 : -INFINITY;
            c[3] = ok1 ? c[3] * ks1 : -INFINITY;
        } else {
            (void)xb;
            if (valid < kTileRows) {
                if (gid >= valid) c[0] = c[1] = -INFINITY;
                if (gid + 8 >= valid) c[2] = c[3] = -INFINITY;
            }
            if (skip > 0) {
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
        const float al0 = fast_exp2(m[0] - mn0);
        const float al1 = fast_exp2(m[1] - mn1);
        const float p0 = fast_exp2(c[0] - mn0);
        const float p1 = fast_exp2(c[1] - mn1);
        const float p2 = fast_exp2(c[2] - mn0);
        const float p3 = fast_exp2(c[3] - mn1);
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
        uint32_t b0, b1;
        if constexpr (Codes::kRowScales) {
            p_fragments(p0 * vs0, p1 * vs0, p2 * vs1, p3 * vs1, b0, b1);
            pv<false>(vbase, valid, b0, b1);
        } else {
            p_fragments(p0, p1, p2, p3, b0, b1);
            if (valid == kTileRows)
                pv<false>(vbase, valid, b0, b1);
            else
                pv<true>(vbase, valid, b0, b1);
        }
    }

    // State layout: m[G], l[G], o[G][D] (fp32, base-2 max), o times vscale.
    __device__ __forceinline__ void write_state(float* st, int /*lane*/, int /*ncols: G*/) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
        }
        const int h0 = 2 * t4, h1 = 2 * t4 + 1;
        if (gid == 0) {
            if (h0 < G) { st[h0] = m[0]; st[G + h0] = l[0]; }
            if (h1 < G) { st[h1] = m[1]; st[G + h1] = l[1]; }
        }
        float* so = st + 2 * G;
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            const int d0 = 16 * mt + gid;
            if (h0 < G) { so[h0 * D + d0] = o[mt][0] * vscale; so[h0 * D + d0 + 8] = o[mt][2] * vscale; }
            if (h1 < G) { so[h1 * D + d0] = o[mt][1] * vscale; so[h1 * D + d0 + 8] = o[mt][3] * vscale; }
        }
    }
};

template <int D, int G>
using Fp8MmaMath = QuantMmaMath<D, G, E4m3Codes>;
template <int D, int G>
using Int8MmaMath = QuantMmaMath<D, G, S8Codes>;

}  // namespace pa
