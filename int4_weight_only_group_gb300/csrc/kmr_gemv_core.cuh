// The int4 GEMV's per-CTA building blocks, shared by the one-projection GEMV kernel
// (kmr_gemv.cu) and the persistent decode-step kernel (kmr_step.cu), so that a row's
// projection is the same bits on either path ("kaminari — a single-GPU Qwen3-VL inference
// engine, explained", §07 int4 sidecar quantization: w = (q - 8) s + z, group 128 along K).
//
//   * stage_x: a warp stages the x of its own 128-input groups as fp16 scaled by a
//     per-(row, group) power of two, with the group sums X' and each row's sum of squares
//     (for the RMSNorm factor) from one reduce-scatter;
//   * store_part / warp16_sum / tile_epilogue: each warp leaves its partial of a 16-row tile,
//     the 16 partials are summed as a fixed pairwise tree, the RMSNorm factor applied, then a
//     store, a residual add or SiLU(gate) * up.
// Activations and the residual are read with ld.global.cg: inside one persistent kernel
// they are written by other CTAs, so they must come from L2, never from a stale L1 line.
#pragma once

#include <cuda_fp16.h>

#include "kmr_int4_mma.cuh"
#include "kmr_internal.cuh"

namespace kmr {

constexpr int kGemvThreads = 512;              // 16 warps: latency hiding for the unpack + mma chains
constexpr int kGemvWarps = kGemvThreads / 32;

// The warp's partial of one tile: rows g, g+8 and batch columns 2t, 2t+1 (< MB kept).
template <int MB>
__device__ __forceinline__ void store_part(float* wp, int lane, const float (&acc)[4]) {
    const int g = lane >> 2, t = lane & 3, c0 = 2 * t, c1 = 2 * t + 1;
    if (c0 < MB) {
        wp[g * MB + c0] = acc[0];
        wp[(g + 8) * MB + c0] = acc[2];
    }
    if (c1 < MB) {
        wp[g * MB + c1] = acc[1];
        wp[(g + 8) * MB + c1] = acc[3];
    }
}

// Sum of the 16 per-warp values v[w * stride] as a fixed pairwise tree (depth 4).
__device__ __forceinline__ float warp16_sum(const float* v, int stride) {
    float a[kGemvWarps];
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) a[w] = v[w * stride];
#pragma unroll
    for (int n = kGemvWarps / 2; n > 0; n >>= 1)
#pragma unroll
        for (int i = 0; i < n; ++i) a[i] = __fadd_rn(a[2 * i], a[2 * i + 1]);
    return a[0];
}

// RMSNorm factor of row m from the per-warp sums of squares.
__device__ __forceinline__ float norm_factor(const GemvParams& p, const float* ssw, int m) {
    if (p.in_kind == IN_F32) return 1.f;
    return rsqrtf(warp16_sum(ssw + m, 8) / float(p.K) + p.eps);
}

// Epilogue of one tile: fixed-order sum of the warp partials, RMSNorm factor, store / add / SiLU-mul.
template <int MB, int WS = 16 * MB>                // WS: floats from one warp's partial to the next
__device__ __forceinline__ void tile_epilogue(const GemvParams& p, const float* ps, int tile, int idx,
                                              const float* ssw, bool have_res = false, float res = 0.f) {
    if (p.epi == EPI_SILU) {
        if (idx >= 8 * MB) return;
        const int j = idx / MB, m = idx % MB;
        const int jj = tile * 8 + j;
        if (m >= p.M || jj >= p.N / 2) return;
        float gv = warp16_sum(ps + j * MB + m, WS), uv = warp16_sum(ps + (j + 8) * MB + m, WS);
        const float r = norm_factor(p, ssw, m);
        gv = __fmul_rn(gv, r);
        uv = __fmul_rn(uv, r);
        p.y[size_t(m) * p.ldy + jj] = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.f, expf(-gv))), uv);
    } else {
        if (idx >= 16 * MB) return;
        const int rr = idx / MB, m = idx % MB;
        const int n = tile * 16 + rr;
        if (m >= p.M || n >= p.N) return;
        float v = __fmul_rn(warp16_sum(ps + rr * MB + m, WS), norm_factor(p, ssw, m));
        float* yp = p.y + size_t(m) * p.ldy + n;
        *yp = (p.epi == EPI_RESID) ? __fadd_rn(have_res ? res : __ldcg(yp), v) : v;
    }
}

// Stage x for this warp's groups: lane l holds inputs 4l..4l+3 of each group.  Loads
// first, then `pre` (a caller's early global load), then every (group, row)'s arithmetic,
// then all warp reductions together (independent, so their latencies overlap), then the
// stores: fp16 halves in B-fragment order (xw), (X', 1/sigma) per (group, row) (xst) and
// each row's sum of squares (ssw, for the RMSNorm factor).
template <int MB, int GPW, typename Pre>
__device__ __forceinline__ void stage_x(const GemvParams& p, __half* xw, float* xst, float* ssw,
                                        const uint2 (&nwv)[GPW], int c, Pre&& pre) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K = p.K, G = K >> 7;
    const bool norm = p.in_kind != IN_F32;
    float4 xv[GPW][MB];
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
        const int grp = warp + j * kGemvWarps;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            xv[j][m] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (grp >= G || m >= p.M) continue;
            const size_t k = size_t(grp) * 128 + lane * 4;
            if (p.in_kind == IN_EMBED_NORM) {
                int tok = p.tokens[m];
                if (tok < 0 || tok >= p.vocab) {
                    if (lane == 0 && grp == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
                    tok = 0;
                }
                const uint2 raw = *reinterpret_cast<const uint2*>(p.embed + size_t(tok) * K + k);
                xv[j][m] = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
                if (c == 0 && p.x_out) *reinterpret_cast<float4*>(p.x_out + size_t(m) * K + k) = xv[j][m];
            } else {
                xv[j][m] = __ldcg(reinterpret_cast<const float4*>(p.x + size_t(m) * K + k));
            }
        }
    }
    pre();
    float ss[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) ss[m] = 0.f;
    __half2 h01[GPW][MB], h23[GPW][MB];
    float gs[GPW][MB], isg[GPW][MB];
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
        const float w0 = bf16_lo(nwv[j].x), w1 = bf16_hi(nwv[j].x), w2 = bf16_lo(nwv[j].y), w3 = bf16_hi(nwv[j].y);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            float u[4] = {xv[j][m].x, xv[j][m].y, xv[j][m].z, xv[j][m].w};
            if (norm) {
#pragma unroll
                for (int e = 0; e < 4; ++e) ss[m] = __fmaf_rn(u[e], u[e], ss[m]);
                u[0] = __fmul_rn(u[0], w0);
                u[1] = __fmul_rn(u[1], w1);
                u[2] = __fmul_rn(u[2], w2);
                u[3] = __fmul_rn(u[3], w3);
            }
            // per-(row, group) power-of-two scale from the group's largest |u| (one redux:
            // the bits of non-negative floats order like unsigned integers)
            const float la = fmaxf(fmaxf(fabsf(u[0]), fabsf(u[1])), fmaxf(fabsf(u[2]), fabsf(u[3])));
            float sig;
            pow2_scale(__reduce_max_sync(0xffffffffu, __float_as_uint(la)), sig, isg[j][m]);
            h01[j][m] = __floats2half2_rn(__fmul_rn(u[0], sig), __fmul_rn(u[1], sig));
            h23[j][m] = __floats2half2_rn(__fmul_rn(u[2], sig), __fmul_rn(u[3], sig));
            const float2 f01 = __half22float2(h01[j][m]), f23 = __half22float2(h23[j][m]);
            gs[j][m] = __fadd_rn(__fadd_rn(f01.x, f01.y), __fadd_rn(f23.x, f23.y));
        }
    }
    // the warp sums of every (group, row) X' and every row's sum of squares in one
    // reduce-scatter (the butterfly's bits, fewer shuffles); value i lands on lanes
    // [i * LPV, (i + 1) * LPV)
    // (up to 40 values: the first 32 in one pass, the rest in a second)
    constexpr int NVAL = GPW * MB + MB;
    constexpr int NA = NVAL < 32 ? NVAL : 32, NB = NVAL - NA;
    static_assert(NB <= 32, "two passes at most");
    constexpr int NVA = pow2_at_least(NA), NVB = pow2_at_least(NB);
    auto value = [&](int i) { return i < GPW * MB ? gs[i / MB][i % MB] : ss[i - GPW * MB]; };
    auto put = [&](int vi, float tot) {
        if (vi < GPW * MB) {
            if (warp + (vi / MB) * kGemvWarps < G) xst[(vi / MB) * 16 + (vi % MB) * 2] = tot;
        } else if (vi < NVAL) {
            ssw[warp * 8 + vi - GPW * MB] = tot;
        }
    };
    float va[NVA];
#pragma unroll
    for (int i = 0; i < NVA; ++i) va[i] = i < NA ? value(i) : 0.f;
    const float tota = reduce_scatter<NVA>(va, lane);
    float totb = 0.f;
    if constexpr (NB > 0) {
        float vb[NVB];
#pragma unroll
        for (int i = 0; i < NVB; ++i) vb[i] = i < NB ? value(32 + i) : 0.f;
        totb = reduce_scatter<NVB>(vb, lane);
    }
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
        const int grp = warp + j * kGemvWarps;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            __half* blk = xw + size_t(j * MB + m) * 128;
            *reinterpret_cast<__half2*>(blk + bpos(lane * 4)) = h01[j][m];
            *reinterpret_cast<__half2*>(blk + bpos(lane * 4 + 2)) = h23[j][m];
            if (lane == 0 && grp < G) xst[j * 16 + m * 2 + 1] = isg[j][m];
        }
        if (lane == 0) {
#pragma unroll
            for (int m = MB; m < 8; ++m) xst[j * 16 + m * 2] = xst[j * 16 + m * 2 + 1] = 0.f;
        }
    }
    if (lane % (32 / NVA) == 0) put(lane / (32 / NVA), tota);
    if constexpr (NB > 0)
        if (lane % (32 / NVB) == 0) put(32 + lane / (32 / NVB), totb);
    if (lane == 0) {
#pragma unroll
        for (int m = MB; m < 8; ++m) ssw[warp * 8 + m] = 0.f;
    }
    __syncwarp();
}

}  // namespace kmr
