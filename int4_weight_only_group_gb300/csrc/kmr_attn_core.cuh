// Per-warp building blocks of the split-KV decode attention, shared by the attention kernel
// (kmr_attn.cu) and the persistent decode-step kernel (kmr_step.cu), so that a row's
// attention is the same bits on either path ("The Ghost in the Batch: How vLLM Silently
// Switches Algorithms", What Attention Does: out = softmax(q K^T / sqrt(d)) V and the
// LSE-weighted merge of partial results; "kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §03 Mrope / TextAttention and §04 per-step positions (3, B)).
//
//   * attn_rope_constants / attn_prologue_warp: per-head RMSNorm of a q or k head, the
//     3-section M-RoPE (frequency f turns the pair (f, f + D/2)), the query scaled into base 2;
//   * attn_score_chunk: one warp's online-softmax update over CH positions for every query head
//     of the KV head (reduce-scatter scoring, base-2 exponentials);
//   * attn_warp_merge: the fixed-order merge of the 8 warps' states for one output element;
//   * attn_split_merge: the fixed-order merge of up to kAttnClusterSplits split states.
#pragma once

#include <math.h>

#include "kmr_internal.cuh"

namespace kmr {

constexpr float kAttnLog2e = 1.4426950408889634f;
constexpr int kAttnMaxRep = 4;          // query heads per KV head supported

// RMSNorm weight of this lane's dims and the rotation of this row's positions, for a warp
// handling one q or k head (EPL = D / 32 contiguous dims per lane).
template <int D>
__device__ __forceinline__ void attn_rope_constants(const uint16_t* nrm, const int32_t* positions, int pos_ld, int b,
                                                    const float* inv_freq, int sec0, int sec1, int lane,
                                                    float (&nw)[D / 32], float (&cs)[D / 32], float (&sn)[D / 32]) {
    constexpr int EPL = D / 32;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int dim = lane * EPL + e, f = dim % (D / 2);
        nw[e] = nrm ? bf16_to_f32(nrm[dim]) : 1.f;
        const int axis = f < sec0 ? 0 : (f < sec0 + sec1 ? 1 : 2);
        const float pos = float(positions[size_t(axis) * pos_ld + b]);
        sincosf(pos * inv_freq[f], &sn[e], &cs[e]);
    }
}

// One head of the new token: x (this lane's EPL dims) normalised over D when `norm`, then
// rotated; the partner dim of frequency f sits 16 lanes away.
template <int D>
__device__ __forceinline__ void attn_norm_rope(float (&x)[D / 32], bool norm, float eps, const float (&nw)[D / 32],
                                               const float (&cs)[D / 32], const float (&sn)[D / 32], int lane) {
    constexpr int EPL = D / 32;
    if (norm) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) ss = __fmaf_rn(x[e], x[e], ss);
        const float r = rsqrtf(warp_sum(ss) / float(D) + eps);
#pragma unroll
        for (int e = 0; e < EPL; ++e) x[e] = __fmul_rn(__fmul_rn(x[e], r), nw[e]);
    }
    const bool lo = lane < 16;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
        x[e] = lo ? __fsub_rn(__fmul_rn(x[e], cs[e]), __fmul_rn(other, sn[e]))
                  : __fadd_rn(__fmul_rn(x[e], cs[e]), __fmul_rn(other, sn[e]));
    }
}

template <int D>
__device__ __forceinline__ void attn_load_row(const uint16_t* row, float (&v)[D / 32], int lane) {
    if constexpr (D / 32 == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
        v[0] = bf16_lo(u); v[1] = bf16_hi(u);
    }
}

// One warp's online-softmax update over nv (<= CH) positions: krow(j) / vrow(j) give the
// shared-memory rows of position j (rows j >= nv re-read row 0 and get weight 0).  Scores for
// all REP heads x CH positions are formed per lane and completed by one reduce-scatter;
// m, l, o are the warp's running state per query head (scores in base 2).
template <int D, int REP, int CH, typename KRow, typename VRow>
__device__ __forceinline__ void attn_score_chunk(int nv, KRow&& krow, VRow&& vrow, const float (&qreg)[REP][D / 32],
                                                 float (&m)[REP], float (&l)[REP], float (&o)[REP][D / 32], int lane) {
    constexpr int EPL = D / 32;
    constexpr int NV = REP * CH;
    constexpr int JS = 32 / NV;
    static_assert(REP * CH <= 32, "one score per lane after the reduce-scatter");
    const int myidx = lane / JS;
    const int myhh = myidx / CH, myj = myidx % CH;
    float sc[NV];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        float kv[EPL];
        attn_load_row<D>(krow(j < nv ? j : 0), kv, lane);
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) a = __fmaf_rn(qreg[hh][e], kv[e], a);
            sc[hh * CH + j] = a;
        }
    }
    const float mine = reduce_scatter<NV>(sc, lane);
    const bool valid = myj < nv;
    const float sv = valid ? mine : -INFINITY;
    // chunk maximum per head: butterfly over the lanes of the same head
    float cm = sv;
#pragma unroll
    for (int off = JS; off < JS * CH; off <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    float mn[REP], cf[REP], mymn = 0.f;
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        const float cmh = __shfl_sync(0xffffffffu, cm, hh * CH * JS);
        mn[hh] = fmaxf(m[hh], cmh);
        cf[hh] = (m[hh] == -INFINITY) ? 0.f : exp2f(__fsub_rn(m[hh], mn[hh]));
        if (hh == myhh) mymn = mn[hh];
    }
    const float pme = valid ? exp2f(__fsub_rn(sv, mymn)) : 0.f;
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        l[hh] = __fmul_rn(l[hh], cf[hh]);
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[hh][e] = __fmul_rn(o[hh][e], cf[hh]);
        m[hh] = mn[hh];
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        float vv[EPL];
        attn_load_row<D>(vrow(j < nv ? j : 0), vv, lane);
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
            const float pj = __shfl_sync(0xffffffffu, pme, (hh * CH + j) * JS);
            l[hh] = __fadd_rn(l[hh], pj);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[hh][e] = __fmaf_rn(pj, vv[e], o[hh][e]);
        }
    }
}

// Merge of the 8 warps' states for output element i = hh * D + dim, in warp order:
// wml[(w * kAttnMaxRep + hh) * 2 + {0, 1}] = (m, l), wo[(w * REP + hh) * D + dim] = o.
template <int D, int REP>
__device__ __forceinline__ void attn_warp_merge(const float* wml, const float* wo, int hh, int dim, float& mx,
                                                float& num, float& den) {
    mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wml[(w * kAttnMaxRep + hh) * 2]);
    num = 0.f;
    den = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float mw = wml[(w * kAttnMaxRep + hh) * 2];
            const float wt = (mw == -INFINITY) ? 0.f : exp2f(__fsub_rn(mw, mx));
            den = __fmaf_rn(wt, wml[(w * kAttnMaxRep + hh) * 2 + 1], den);
            num = __fmaf_rn(wt, wo[(size_t(w) * REP + hh) * D + dim], num);
        }
    }
}

// Merge of the splits' states (m_r, l_r, num_r) of one output element in split order; splits
// r >= ns (empty) count as m = -inf.  out = sum_r w_r num_r / sum_r w_r l_r, w_r = 2^(m_r - max m).
__device__ __forceinline__ float attn_split_merge(const float (&mr)[kAttnClusterSplits],
                                                  const float (&lr)[kAttnClusterSplits],
                                                  const float (&nr)[kAttnClusterSplits]) {
    float mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < kAttnClusterSplits; ++r) mx = fmaxf(mx, mr[r]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int r = 0; r < kAttnClusterSplits; ++r) {
        const float wt = (mr[r] == -INFINITY) ? 0.f : exp2f(__fsub_rn(mr[r], mx));
        den = __fmaf_rn(wt, lr[r], den);
        num = __fmaf_rn(wt, nr[r], num);
    }
    return __fdiv_rn(num, den);
}

// Split plan of a row: L = cache_position + 1 positions over `nsplit` splits of
// ceil(L / nsplit) rounded up to 16 (depends only on the row's own length).
__host__ __device__ __forceinline__ void attn_split_plan(int cp, int nsplit, int& chunk, int& ns) {
    const int Lq = cp + 1;
    chunk = (((Lq + nsplit - 1) / nsplit) + 15) & ~15;
    ns = (Lq + chunk - 1) / chunk;
}

}  // namespace kmr
