// pa_tile_math_int8.cuh -- per-tile math for an INT8 KV cache with one fp32
// scale per (row, KV head) and bf16 q and output.
//
// Each cached row is int8 codes with its own scale: value = scale_row * code
// ("MLSys Engineer -- Inference Systems Q&A", Q3: INT8 KV with per-token
// scaling, scale = max(|row|) / 127, dequantised before the softmax). The
// codes are widened to f16 in registers (exact: |code| <= 127) and multiplied
// with m16n8k16 f16 MMAs accumulating in fp32. The row scales never touch the
// products:
//   scores  S_row = k_scale_row * (q * scale * log2(e)) . code(K_row): each
//           accumulator row is multiplied by its K scale;
//   output  O = sum_row (p_row * v_scale_row) code(V_row): the V scale folds
//           into the probability before it becomes an MMA operand, while the
//           softmax sum keeps p_row.
// The 16 K and 16 V scales of a tile arrive with it, in a small per-stage
// array (extra stage bytes). Fragment assignment as in Fp8MmaMath.
//
// int8 -> f16: a code c becomes the f16 bit pattern 0x6400 | (c ^ 0x80), the
// value 1024 + 128 + c; subtracting 1152 leaves c exactly.
#pragma once

#include <cuda_fp16.h>

#include "pa_tile_math_fp8.cuh"

namespace pa {

// Four int8 codes -> two f16x2 registers (the low byte of each pair becomes
// the low half).
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = w ^ 0x80808080u;
    const uint32_t a = prmt(t, 0x64646464u, 0x4140u);   // (t.b0, 0x64, t.b1, 0x64)
    const uint32_t b = prmt(t, 0x64646464u, 0x4342u);   // (t.b2, 0x64, t.b3, 0x64)
    const uint32_t bias = 0x64806480u;                  // f16x2 {1152, 1152}
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

template <int D, int G>
struct Int8MmaMath {
    using T = __nv_bfloat16;                    // q and out
    using Geom = TileGeom<uint8_t, D>;
    static constexpr bool kCausal = false;
    static_assert(D == 128, "one 128-byte row of codes per token");
    static_assert(G >= 1 && G <= 8, "the MMA N dimension holds at most 8 query heads");
    static constexpr int kSteps = D / 16;
    // Per stage: 16 K scales then 16 V scales (fp32).
    static constexpr int kExtraStageBytes = 2 * kTileRows * 4;

    static constexpr bool kQInSmem = true;
    static constexpr int kQRowBytes = D * 2 + 16;
    static constexpr int kQBufBytes = ((G * kQRowBytes + 127) / 128) * 128;
    struct QRegs {};

    uint32_t qb[kSteps][2];
    float o[kSteps][4];
    float m[2], l[2];
    float qscale;
    int gid, t4;

    __device__ __forceinline__ void setup(int lane, const DecodeParams& p) {
        gid = lane >> 2;
        t4 = lane & 3;
        qscale = p.scale_log2;
    }

    __device__ __forceinline__ void stage_q(const DecodeParams& p, int s, int h, int ncols,
                                            int grp, uint32_t qbuf, int lane) const {
        stage_q_rows<D, kQRowBytes>(p, s, h, ncols, grp, qbuf, lane);
    }

    // q' = q * scale * log2(e) in f16, dealt as Fp8MmaMath deals the dims.
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

    // One query per sequence: rows past `valid` and the first `skip` rows (a
    // sliding window) are masked. xb: the stage's 16 K then 16 V scales.
    __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int valid,
                                         float /*scale_log2: folded into q'*/, int /*lane*/,
                                         int /*row0*/, int /*limit0*/, int /*grp*/, int skip,
                                         uint32_t xb) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
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
                s8x4_to_f16x2x2(w0[jj], a0, a2);
                s8x4_to_f16x2x2(w1[jj], a1, a3);
                mma_16816_f16(c, a0, a1, a2, a3, qb[j][0], qb[j][1]);
            }
        }
        const bool ok0 = gid < valid && gid >= skip;
        const bool ok1 = gid + 8 < valid && gid + 8 >= skip;
        // Scales of rows past the sequence are whatever memory holds: only
        // visible rows read theirs.
        const float ks0 = ok0 ? lds_f32(xb + 4 * gid) : 0.f;
        const float ks1 = ok1 ? lds_f32(xb + 4 * (gid + 8)) : 0.f;
        const float vs0 = ok0 ? lds_f32(xb + 4 * (kTileRows + gid)) : 0.f;
        const float vs1 = ok1 ? lds_f32(xb + 4 * (kTileRows + gid + 8)) : 0.f;
        c[0] = ok0 ? c[0] * ks0 : -INFINITY;
        c[1] = ok0 ? c[1] * ks0 : -INFINITY;
        c[2] = ok1 ? c[2] * ks1 : -INFINITY;
        c[3] = ok1 ? c[3] * ks1 : -INFINITY;
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
        // P' = P * v_scale as the f16 B operand (gathered as in MmaMath).
        const uint32_t p01 = pack_f16x2(p0 * vs0, p1 * vs0);
        const uint32_t p23 = pack_f16x2(p2 * vs1, p3 * vs1);
        const int src_a = 8 * t4 + (gid >> 1);
        const uint32_t v0 = __shfl_sync(0xffffffffu, p01, src_a);
        const uint32_t v1 = __shfl_sync(0xffffffffu, p01, src_a + 4);
        const uint32_t u0 = __shfl_sync(0xffffffffu, p23, src_a);
        const uint32_t u1 = __shfl_sync(0xffffffffu, p23, src_a + 4);
        const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = prmt(v0, v1, sel);
        const uint32_t b1 = prmt(u0, u1, sel);
        // V rows 2t4, 2t4+1, 2t4+8, 2t4+9, chunk gid. Codes of invalid rows
        // are finite and meet a zero probability.
        const uint4 x0 = lds128(swizzled(vbase, 2 * t4, gid));
        const uint4 x1 = lds128(swizzled(vbase, 2 * t4 + 1, gid));
        const uint4 x2 = lds128(swizzled(vbase, 2 * t4 + 8, gid));
        const uint4 x3 = lds128(swizzled(vbase, 2 * t4 + 9, gid));
        const uint32_t e0[4] = {x0.x, x0.y, x0.z, x0.w};
        const uint32_t e1[4] = {x1.x, x1.y, x1.z, x1.w};
        const uint32_t e2[4] = {x2.x, x2.y, x2.z, x2.w};
        const uint32_t e3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
            const uint32_t sel_v = (mt & 1) ? 0x7362u : 0x5140u;
            const uint32_t lo = prmt(e0[mt >> 1], e1[mt >> 1], sel_v);
            const uint32_t hi = prmt(e2[mt >> 1], e3[mt >> 1], sel_v);
            uint32_t a0, a1, a2, a3;
            s8x4_to_f16x2x2(lo, a0, a1);
            s8x4_to_f16x2x2(hi, a2, a3);
            mma_16816_f16(o[mt], a0, a1, a2, a3, b0, b1);
        }
    }

    // State layout: m[G], l[G], o[G][D] (fp32, base-2 max).
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
            const int d0 = 16 * gid + 2 * mt;
            if (h0 < G) { so[h0 * D + d0] = o[mt][0]; so[h0 * D + d0 + 1] = o[mt][2]; }
            if (h1 < G) { so[h1 * D + d0] = o[mt][1]; so[h1 * D + d0 + 1] = o[mt][3]; }
        }
    }
};

}  // namespace pa
