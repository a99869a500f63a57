// The int4 tensor-core block product shared by the GEMV and the attention kernel's
// fused O projection ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07 int4 sidecar quantization: w = (q - 8) s + z, group 128 along K).
//
// One (16-row tile, 128-input group) block of the KMR4 layout (include/kmr.h) against
// up to 8 staged rows of x: x is held in fp16, scaled per (row, group) by a power of
// two sigma, in B-fragment order; each lane's 32-bit weight word is its A fragment of
// a 16x16 block, turned into fp16 (1024 + q) or (1024 + 16 q) by OR-ing the nibble
// into the mantissa of 1024.0; the offset, the -8 and the zero point are folded in
// once per group with the group sum X' of the staged halves:
//     y += (s (D - 1024 X') / c + (z - 8 s) X') / sigma,   c = 1 (rows 0..7) or 16 (rows 8..15).
#pragma once

#include <cuda_fp16.h>

#include "kmr_internal.cuh"

namespace kmr {

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position (in halves) of group-local input kk (0..127) in B-fragment order: two blocks
// of 64; inside a block, lane slot t (16 halves) holds for each of its 4 k-steps
// (k0 = 16 step) the inputs (k0+2t, k0+2t+1, k0+2t+8, k0+2t+9).
__device__ __forceinline__ int bpos(int kk) {
    const int j = kk & 15;
    return (kk >> 6) * 64 + ((j & 7) >> 1) * 16 + ((kk >> 4) & 3) * 4 + (j >> 3) * 2 + (j & 1);
}

// sigma = 2^(13 - floor(log2 a)) (so a * sigma lies in [2^13, 2^14)) and 1 / sigma, from the
// bits of a = the group's largest |u|; 1 for a group of zeros, denormals or non-finite values.
// Both are powers of two built from the exponent field: exact, and no division.
__device__ __forceinline__ void pow2_scale(uint32_t abits, float& sig, float& isig) {
    const int e = int(abits >> 23);                        // biased exponent (abits has no sign bit)
    if (e == 0 || e >= 255) {
        sig = isig = 1.f;
        return;
    }
    const int se = max(1, min(253, 267 - e));              // 127 + 13 - (e - 127), clamped
    sig = __uint_as_float(uint32_t(se) << 23);
    isig = __uint_as_float(uint32_t(254 - se) << 23);
}

// The B fragments of one staged group for this lane (batch row g, both 64-input blocks)
// and the fold constants (X'_{2t}, 1/sigma_{2t}, X'_{2t+1}, 1/sigma_{2t+1}); loaded once
// per group and reused for every tile.
struct XFrag {
    uint32_t b[16];
    float4 X;
};
__device__ __forceinline__ void load_xfrag(XFrag& f, const __half* xb, bool bload, int lane, const float* st) {
    const int t = lane & 3;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint4 xa = make_uint4(0, 0, 0, 0), xc = make_uint4(0, 0, 0, 0);
        if (bload) {
            const uint4* xp = reinterpret_cast<const uint4*>(xb + blk * 64 + t * 16);
            xa = xp[0];
            xc = xp[1];
        }
        f.b[blk * 8 + 0] = xa.x; f.b[blk * 8 + 1] = xa.y; f.b[blk * 8 + 2] = xa.z; f.b[blk * 8 + 3] = xa.w;
        f.b[blk * 8 + 4] = xc.x; f.b[blk * 8 + 5] = xc.y; f.b[blk * 8 + 6] = xc.z; f.b[blk * 8 + 7] = xc.w;
    }
    f.X = *reinterpret_cast<const float4*>(st + 4 * t);
}

// Sum of the four k-step chains, then the fold of the group's offset, -8 and zero point for
// rows g (x1) and g+8 (x16) and batch columns 2t, 2t+1 (ODD = false: column 2t only).
template <bool ODD>
__device__ __forceinline__ void fold_group(const uint8_t* gb, int g, const float (&d)[4][4], const float4 X,
                                           float (&acc)[4]) {
    float D[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (ODD || (i & 1) == 0) D[i] = __fadd_rn(__fadd_rn(d[0][i], d[1][i]), __fadd_rn(d[2][i], d[3][i]));
    const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(gb + 1024 + g * 4);
    const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(gb + 1024 + (g + 8) * 4);
    // X = (X'_{2t}, is_{2t}, X'_{2t+1}, is_{2t+1})
    const float s0 = bf16_lo(sz0), z0 = bf16_hi(sz0), s1 = bf16_lo(sz1), z1 = bf16_hi(sz1);
    const float s1c = __fmul_rn(s1, 0.0625f);
    const float zz0 = __fmaf_rn(-8.f, s0, z0), zz1 = __fmaf_rn(-8.f, s1, z1);
    const float x0 = 1024.f * X.x, x1 = ODD ? 1024.f * X.z : 0.f;
    acc[0] = __fmaf_rn(__fmaf_rn(s0, __fsub_rn(D[0], x0), __fmul_rn(zz0, X.x)), X.y, acc[0]);
    acc[2] = __fmaf_rn(__fmaf_rn(s1c, __fsub_rn(D[2], x0), __fmul_rn(zz1, X.x)), X.y, acc[2]);
    if (ODD) {
        acc[1] = __fmaf_rn(__fmaf_rn(s0, __fsub_rn(D[1], x1), __fmul_rn(zz0, X.z)), X.w, acc[1]);
        acc[3] = __fmaf_rn(__fmaf_rn(s1c, __fsub_rn(D[3], x1), __fmul_rn(zz1, X.z)), X.w, acc[3]);
    }
}

// One (16-row tile, 128-input group) block: 8 tensor-core k-steps on four independent
// accumulator chains, then the fold for rows g (x1) and g+8 (x16) and batch columns
// 2t, 2t+1.  ODD = false skips the odd columns (one row of x: column 2t+1 never exists).
template <bool ODD = true>
__device__ __forceinline__ void group_product(const uint8_t* gb, const XFrag& xf, int lane, float (&acc)[4]) {
    const int g = lane >> 2;
    float d[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c][0] = d[c][1] = d[c][2] = d[c][3] = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const uint4 wq = *reinterpret_cast<const uint4*>(gb + blk * 512 + lane * 16);
        const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t w = w4[ks], w2 = w >> 8;
            mma16816(d[ks], and_or(w, 0x000F000Fu, 0x64006400u), and_or(w, 0x00F000F0u, 0x64006400u),
                     and_or(w2, 0x000F000Fu, 0x64006400u), and_or(w2, 0x00F000F0u, 0x64006400u),
                     xf.b[blk * 8 + 2 * ks], xf.b[blk * 8 + 2 * ks + 1]);
        }
    }
    fold_group<ODD>(gb, g, d, xf.X, acc);
}

// The same block against two staged halves of up to 8 rows each (batch rows 0..7 in xa,
// 8..15 in xb): every weight word is unpacked once and feeds two mma, one per half.  Each
// half's chains, sums and fold are those of group_product, so each row gets the same bits.
__device__ __forceinline__ void group_product2(const uint8_t* gb, const XFrag& xa, const XFrag& xb, int lane,
                                               float (&acca)[4], float (&accb)[4]) {
    const int g = lane >> 2;
    float da[4][4], db[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) da[c][i] = db[c][i] = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const uint4 wq = *reinterpret_cast<const uint4*>(gb + blk * 512 + lane * 16);
        const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint32_t w = w4[ks], w2 = w >> 8;
            const uint32_t a0 = and_or(w, 0x000F000Fu, 0x64006400u), a1 = and_or(w, 0x00F000F0u, 0x64006400u);
            const uint32_t a2 = and_or(w2, 0x000F000Fu, 0x64006400u), a3 = and_or(w2, 0x00F000F0u, 0x64006400u);
            mma16816(da[ks], a0, a1, a2, a3, xa.b[blk * 8 + 2 * ks], xa.b[blk * 8 + 2 * ks + 1]);
            mma16816(db[ks], a0, a1, a2, a3, xb.b[blk * 8 + 2 * ks], xb.b[blk * 8 + 2 * ks + 1]);
        }
    }
    fold_group<true>(gb, g, da, xa.X, acca);
    fold_group<true>(gb, g, db, xb.X, accb);
}

}  // namespace kmr
