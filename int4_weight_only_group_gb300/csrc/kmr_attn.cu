// Split-KV GQA decode attention over the static, slot-addressable bf16 cache.
//
// What it computes ("The Ghost in the Batch: How vLLM Silently Switches
// Algorithms", What Attention Does: out = softmax(q K^T / sqrt(d)) V over the
// row's cached positions, and the LSE-weighted merge of partial results;
// "kaminari — a single-GPU Qwen3-VL inference engine, explained", §03:
// StaticKVCache rows per slot, mutated in place; §04: per-step positions
// (3, B) and cache_position).
//
// Fused mode (inside the decode step) also finishes the QKV projection for
// its KV head: per-head q/k RMSNorm, 3-section M-RoPE on q and k, bf16
// rounding of the new k and v, and their write into the cache at
// cache_position — done by the CTA whose split owns that position, which uses
// the new values straight from shared memory.
//
// GB300 design: grid (split, kv head, row).  The split length is
// ceil(L / splits) rounded up to 16, where L = cache_position + 1 and splits is
// fixed per call site — it depends only on the row's own length, never on the
// batch, so a row's result is the same at any batch size.  Each CTA streams its
// K and V positions with cp.async.bulk (contiguous in the [slot][head][pos][d]
// layout) into a ring of shared-memory stages whose first fill is issued,
// together with the RoPE angles, before griddepcontrol.wait.
//   * Scoring: a warp takes 8 positions at a time.  Every lane holds d/32
//     dimensions of each query head and forms partial dot products for all 8
//     positions and all heads of the group; one reduce-scatter over the warp
//     (halving the values held at each shuffle level) leaves each lane one
//     complete score, so 8 x heads scores cost about as many shuffles as full
//     butterflies would for one or two.  Online softmax in base 2 (log2(e)
//     folded into the query scale), no block barrier inside the loop.
//   * Merge: the 8 warp states merge in shared memory; then the splits merge
//     in split order:
//       - cluster mode: the splits of one (row, KV head) are one thread-block
//         cluster; every split pushes its state for output slice r into CTA
//         r's shared memory (distributed shared memory stores), one cluster
//         barrier, and each CTA merges its slice from local memory — no
//         global memory, no atomics, no remote loads on the critical path;
//       - global mode: each split writes its state to a caller workspace and
//         the last CTA to arrive (atomic counter) merges — for any number of
//         splits.
#include <cooperative_groups.h>
#include <math.h>

#include "kmr_attn_core.cuh"
#include "kmr_int4_mma.cuh"
#include "kmr_internal.cuh"

namespace cg = cooperative_groups;

namespace kmr {

namespace {

// A warp scores CH positions at a time (8, or 16 when a split can exceed 64 positions and a
// KV head serves at most 2 query heads, so that NV = heads x CH stays <= 32); a ring stage
// holds the 8 scoring warps x CH positions.  The batch-1 kernel that also computes the QKV
// projection runs 16 warps (one 128-input group each, as the int4 GEMV does); warps 8..15 take
// no part in the scoring, so every path scores and merges in the same order.
constexpr int kScoreWarps = 8;
constexpr int kAttnThreadsPlain = kScoreWarps * 32;
constexpr int kAttnThreadsQkv = 16 * 32;
constexpr int kMaxStages = 4;
constexpr int kMaxRep = kAttnMaxRep;
constexpr float kLog2e = kAttnLog2e;

__host__ __device__ inline size_t al16a(size_t v) { return (v + 15) & ~size_t(15); }

struct AttnSmem {
    size_t bar, kst, vst, knew, vnew, qs, wml, wo, co, cml, recv, flag;
    size_t qbar, qw, qxw, qxst, qss, qpart, qkvh;              // fused QKV projection
    size_t total;
};
// QKV tiles (16 rows) of a head group per cluster rank: (rep q heads + k + v) x D rows / 16 / 8.
__host__ __device__ inline int qkv_tiles_per_rank(int D, int rep) { return (rep + 2) * D / 128; }
__host__ __device__ inline AttnSmem attn_layout(int D, int rep, int nstage, int sub, int qkv_tb) {
    AttnSmem L;
    const int per = rep * D / 8;                                // output slice merged by each cluster rank
    const int tpr = qkv_tiles_per_rank(D, rep);
    size_t o = 0;
    L.bar = o;   o += al16a(kMaxStages * 8);
    L.qbar = o;  o += 16;
    o = (o + 127) & ~size_t(127);
    L.qw = o;    o += qkv_tb ? size_t(tpr) * qkv_tb : 0;        // this rank's QKV weight tiles
    L.qxw = o;   o += qkv_tb ? size_t(16) * 128 * 2 : 0;          // per warp: its staged group of x
    L.qxst = o;  o += qkv_tb ? size_t(16) * 16 * 4 : 0;         // per group: (X', 1/sigma) x 8 rows
    L.qss = o;   o += qkv_tb ? 16 * 4 : 0;                       // per group: sum of x^2
    L.qpart = o; o += qkv_tb ? size_t(tpr) * 16 * 16 * 4 : 0;   // per tile, per group: 16 rows
    L.qkvh = o;  o += qkv_tb ? al16a(size_t(rep + 2) * D * 4) : 0;   // the head group's q, k, v
    o = (o + 127) & ~size_t(127);
    L.kst = o;   o += size_t(nstage) * sub * D * 2;
    L.vst = o;   o += size_t(nstage) * sub * D * 2;
    L.knew = o;  o += al16a(size_t(D) * 2);
    L.vnew = o;  o += al16a(size_t(D) * 2);
    L.qs = o;    o += al16a(size_t(rep) * D * 4);
    L.wml = o;   o += al16a(size_t(kScoreWarps) * kMaxRep * 2 * 4);   // per scoring warp: (m, l) per head
    L.wo = o;    o += al16a(size_t(kScoreWarps) * rep * D * 4);       // per scoring warp: o per head
    L.co = o;    o += al16a(size_t(rep) * D * 4);              // CTA state (global mode)
    L.cml = o;   o += al16a(size_t(kMaxRep) * 2 * 4);
    L.recv = o;  o += al16a(size_t(8) * (per + 2) * 4);        // per source rank: (m, l, slice)
    L.flag = o;  o += 16;
    L.total = o;
    return L;
}

// Fixed pairwise tree over 16 values v[i * stride] (the int4 GEMV's warp-partial order).
__device__ __forceinline__ float tree16(const float* v, int stride) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = v[i * stride];
#pragma unroll
    for (int n = 8; n > 0; n >>= 1)
#pragma unroll
        for (int i = 0; i < n; ++i) a[i] = __fadd_rn(a[2 * i], a[2 * i + 1]);
    return a[0];
}

// Fused QKV projection of one cluster rank for one row (see AttnParams): stage the row's
// RMSNorm input (warp w: group w), multiply this rank's QKV tiles on the tensor cores, reduce
// each tile's 16 group partials in the one-row GEMV's fixed order, apply the RMSNorm factor
// and push the rank's rows into every rank's q/k/v buffer.  Every step mirrors the one-row
// int4 GEMV (kmr_gemv.cu: one group per warp at K = 2048), so a row's q, k, v are the same
// bits whether the step ran it fused (small batches) or through the GEMV (larger ones).
template <int D, int REP>
__device__ __forceinline__ void qkv_phase(const AttnParams& p, uint8_t* smem, const AttnSmem& L, int s, int h,
                                          int b, int lane, int warp, uint2 nwv) {
    constexpr int TPR = (REP + 2) * D / 128;
    const int K = p.hidden, G = K >> 7;
    const int tid = threadIdx.x;
    __half* xw = reinterpret_cast<__half*>(smem + L.qxw) + warp * 128;
    float* xst = reinterpret_cast<float*>(smem + L.qxst);
    float* ssg = reinterpret_cast<float*>(smem + L.qss);
    float* part = reinterpret_cast<float*>(smem + L.qpart);
    float* qkvh = reinterpret_cast<float*>(smem + L.qkvh);
    const uint8_t* qw = smem + L.qw;
    uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + L.qbar);
    const bool embed = p.x_kind == IN_EMBED_NORM;
    const int g = warp;
    float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g < G) {
        const size_t k = size_t(g) * 128 + lane * 4;
        if (embed) {
            int tok = p.tokens[b];
            if (tok < 0 || tok >= p.vocab) {
                if (lane == 0 && g == 0 && s == 0 && h == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
                tok = 0;
            }
            const uint2 raw = *reinterpret_cast<const uint2*>(p.embed + size_t(tok) * K + k);
            xv = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
            if (s == 0 && h == 0 && p.x_out) *reinterpret_cast<float4*>(p.x_out + size_t(b) * K + k) = xv;
        } else {
            xv = *reinterpret_cast<const float4*>(p.x + size_t(b) * K + k);
        }
    }
    // (X', sum of squares) of the group in one reduce-scatter: lanes 0..15 end with X',
    // 16..31 with the sum of squares (the butterfly's bits)
    float rv[2];
    {
        const float w0 = bf16_lo(nwv.x), w1 = bf16_hi(nwv.x), w2 = bf16_lo(nwv.y), w3 = bf16_hi(nwv.y);
        float u[4] = {xv.x, xv.y, xv.z, xv.w};
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = __fmaf_rn(u[e], u[e], ss);
        u[0] = __fmul_rn(u[0], w0);
        u[1] = __fmul_rn(u[1], w1);
        u[2] = __fmul_rn(u[2], w2);
        u[3] = __fmul_rn(u[3], w3);
        const float la = fmaxf(fmaxf(fabsf(u[0]), fabsf(u[1])), fmaxf(fabsf(u[2]), fabsf(u[3])));
        float sig, isg;
        pow2_scale(__reduce_max_sync(0xffffffffu, __float_as_uint(la)), sig, isg);
        const __half2 h01 = __floats2half2_rn(__fmul_rn(u[0], sig), __fmul_rn(u[1], sig));
        const __half2 h23 = __floats2half2_rn(__fmul_rn(u[2], sig), __fmul_rn(u[3], sig));
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        rv[0] = __fadd_rn(__fadd_rn(f01.x, f01.y), __fadd_rn(f23.x, f23.y));
        rv[1] = ss;
        *reinterpret_cast<__half2*>(xw + bpos(lane * 4)) = h01;
        *reinterpret_cast<__half2*>(xw + bpos(lane * 4 + 2)) = h23;
        if (lane >= 1 && lane < 16) xst[g * 16 + lane] = (g < G && lane == 1) ? isg : 0.f;
    }
    const float tot = reduce_scatter<2>(rv, lane);
    if (lane == 0) xst[g * 16] = g < G ? tot : 0.f;
    if (lane == 16) ssg[g] = g < G ? tot : 0.f;
    __syncwarp();
    const int gl = lane >> 2;
    // the group's fragments once, then all TPR block products unrolled: independent
    // accumulator chains the scheduler can interleave
    XFrag xf;
    load_xfrag(xf, xw, gl == 0, lane, xst + g * 16);
    mbar_wait(qbar, 0u, p.err);
    float acc[TPR][4];
#pragma unroll
    for (int t = 0; t < TPR; ++t) {
        acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        if (g < G) group_product<false>(qw + size_t(t) * p.qkv_tile_bytes + size_t(g) * kGroupBytes, xf, lane, acc[t]);
    }
    if ((lane & 3) == 0) {
#pragma unroll
        for (int t = 0; t < TPR; ++t) {
            part[(t * 16 + g) * 16 + gl] = acc[t][0];
            part[(t * 16 + g) * 16 + gl + 8] = acc[t][2];
        }
    }
    __syncthreads();
    if (tid < TPR * 16) {
        const int t = tid >> 4, rr = tid & 15;
        const float nf = rsqrtf(tree16(ssg, 1) / float(K) + p.eps);
        const float v = __fmul_rn(tree16(part + t * 256 + rr, 16), nf);
        const int hr = (s * TPR + t) * 16 + rr;              // row within the head group's q|k|v
#pragma unroll
        for (int r = 0; r < kAttnClusterSplits; ++r) cg::this_cluster().map_shared_rank(qkvh, r)[hr] = v;
    }
    cg::this_cluster().sync();
}

template <int D, int REP, bool CLUSTER, int CH, bool QKVF>
__global__ void __launch_bounds__(QKVF ? kAttnThreadsQkv : kAttnThreadsPlain, 1) attn_kernel(const AttnParams p) {
    constexpr int NT = QKVF ? kAttnThreadsQkv : kAttnThreadsPlain;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int EPL = D / 32;               // contiguous dims per lane
    constexpr int kChunk = CH;                // positions a warp scores at once
    constexpr int kSub = kScoreWarps * CH;    // positions per ring stage
    static_assert(REP * CH <= 32, "one score per lane after the reduce-scatter");
    constexpr int PER = REP * D / 8;          // output slice per cluster rank
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nst = p.nstage;
    const AttnSmem L = attn_layout(D, REP, nst, kSub, QKVF ? p.qkv_tile_bytes : 0);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint16_t* kst = reinterpret_cast<uint16_t*>(smem + L.kst);
    uint16_t* vst = reinterpret_cast<uint16_t*>(smem + L.vst);
    uint16_t* knew = reinterpret_cast<uint16_t*>(smem + L.knew);
    uint16_t* vnew = reinterpret_cast<uint16_t*>(smem + L.vnew);
    float* qs = reinterpret_cast<float*>(smem + L.qs);
    float* wml = reinterpret_cast<float*>(smem + L.wml);
    float* wo = reinterpret_cast<float*>(smem + L.wo);
    float* co = reinterpret_cast<float*>(smem + L.co);
    float* cml = reinterpret_cast<float*>(smem + L.cml);
    float* recv = reinterpret_cast<float*>(smem + L.recv);
    int* flag = reinterpret_cast<int*>(smem + L.flag);

    // Row state (and the positions) come from the previous step, complete before
    // this graph ran, not from the kernels of this step, so they may be read
    // before griddepcontrol.wait.
    const bool fin = p.finished != nullptr && p.finished[b] != 0;
    const int slot = p.slot_ids[b], cp = p.cpos[b];
    const bool bad_slot = slot < 0 || slot >= p.slots;
    const bool bad_pos = cp < 0 || cp >= p.S;
    float* outrow = p.out + size_t(b) * p.nq * D + size_t(h) * REP * D;
    if (fin || bad_slot || bad_pos) {            // uniform over the whole cluster / row
        if (s == 0) {
            pdl_wait();
            if (!fin && h == 0 && tid == 0) set_error(p.err, bad_slot ? KMR_ERR_SLOT_RANGE : KMR_ERR_CACHE_FULL);
            for (int i = tid; i < REP * D; i += NT) outrow[i] = 0.f;
            if constexpr (QKVF) {
                // the layer-0 embedding still lands in the residual, as the GEMV path stores it
                if (h == 0 && p.x_kind == IN_EMBED_NORM && p.x_out) {
                    int tok = p.tokens[b];
                    if (tok < 0 || tok >= p.vocab) {
                        if (tid == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
                        tok = 0;
                    }
                    for (int k = tid; k < p.hidden; k += NT)
                        p.x_out[size_t(b) * p.hidden + k] = bf16_to_f32(p.embed[size_t(tok) * p.hidden + k]);
                }
            }
        }
        return;
    }
    const int nsplit = gridDim.x;
    const int Lq = cp + 1;
    int chunk, ns;
    attn_split_plan(cp, nsplit, chunk, ns);
    if (!CLUSTER && s >= ns) return;             // (cluster mode: empty splits still merge a slice)
    const int t0 = s * chunk, t1 = min(Lq, t0 + chunk);      // t1 <= t0 for an empty split
    const int cached_end = p.fused ? min(t1, cp) : t1;
    const int nsub = t1 > t0 ? (t1 - t0 + kSub - 1) / kSub : 0;
    const size_t headoff = (size_t(slot) * p.nkv + h) * p.S * D;
    const uint16_t* kbase = p.kc + headoff;
    const uint16_t* vbase = p.vc + headoff;

    if (tid == 0) {
        for (int i = 0; i < nst; ++i) mbar_init(&bar[i], 1);
        if constexpr (QKVF) mbar_init(reinterpret_cast<uint64_t*>(smem + L.qbar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int st) {
        const int sb = st % nst;
        const int pa = t0 + st * kSub;
        const int pb = min(pa + kSub, cached_end);
        const int np = pb > pa ? pb - pa : 0;
        if (np > 0) {
            const uint32_t bytes = uint32_t(np) * D * 2;
            mbar_arrive_expect_tx(&bar[sb], 2 * bytes);
            bulk_g2s(kst + size_t(sb) * kSub * D, kbase + size_t(pa) * D, bytes, &bar[sb]);
            bulk_g2s(vst + size_t(sb) * kSub * D, vbase + size_t(pa) * D, bytes, &bar[sb]);
        } else {
            mbar_arrive(&bar[sb]);
        }
    };
    if (tid == 0) {
        const int n0 = nsub < nst ? nsub : nst;
        for (int i = 0; i < n0; ++i) issue(i);
    }
    uint2 qnw = make_uint2(0, 0);
    if constexpr (QKVF) {
        constexpr int TPR = (REP + 2) * D / 128, QT = REP * D / 16, KT = D / 16;
        if (tid == 0) {
            // this rank's tiles of the head group's rows [q heads | k | v], each one contiguous copy
            uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + L.qbar);      // initialised above
            const uint32_t tb = uint32_t(p.qkv_tile_bytes);
            mbar_arrive_expect_tx(qbar, tb * TPR);
            const uint64_t pol = policy_evict_first();
            for (int t = 0; t < TPR; ++t) {
                const int li = s * TPR + t;
                const int gt = li < QT ? h * QT + li
                                       : (li < QT + KT ? p.nq * D / 16 + h * KT + (li - QT)
                                                       : (p.nq + p.nkv) * D / 16 + h * KT + (li - QT - KT));
                bulk_g2s_stream(smem + L.qw + size_t(t) * tb, p.wqkv + size_t(gt) * tb, tb, qbar, pol);
            }
        }
        if (warp < (p.hidden >> 7)) qnw = *reinterpret_cast<const uint2*>(p.in_norm_w + size_t(warp) * 128 + lane * 4);
    }
    // constants of the prologue, and the RoPE angles of this row's positions, before the wait
    const bool qk_warp = p.fused && warp <= REP;
    float nw[EPL], cs[EPL], sn[EPL];
    if (qk_warp)
        attn_rope_constants<D>(warp < REP ? p.qn_w : p.kn_w, p.positions, p.pos_ld, b, p.inv_freq, p.sec0, p.sec1,
                               lane, nw, cs, sn);
    pdl_launch_dependents();
    pdl_wait();

    if constexpr (QKVF) qkv_phase<D, REP>(p, smem, L, s, h, b, lane, warp, qnw);

    // ---- prologue: q (and, fused, the new k / v) of this KV head
    const float qscale = __fmul_rn(p.scale, kLog2e);       // scores in base 2
    const float* in = p.in + size_t(b) * p.in_ld;
    if (p.fused) {
        if (warp <= REP + 1) {
            const bool isq = warp < REP, isk = warp == REP;
            const float* src;
            if constexpr (QKVF) {
                const float* qkvh = reinterpret_cast<const float*>(smem + L.qkvh);   // [q heads | k | v]
                src = qkvh + size_t(isq ? warp : (isk ? REP : REP + 1)) * D;
            } else {
                src = isq ? in + size_t(h * REP + warp) * D
                          : (isk ? in + size_t(p.nq) * D + size_t(h) * D : in + size_t(p.nq + p.nkv) * D + size_t(h) * D);
            }
            float x[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[e] = src[lane * EPL + e];
            if (qk_warp)
                attn_norm_rope<D>(x, isq ? p.qn_w != nullptr : p.kn_w != nullptr, p.eps, nw, cs, sn, lane);
            if (isq) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) qs[warp * D + lane * EPL + e] = __fmul_rn(x[e], qscale);
            } else {
                uint16_t* dst = isk ? knew : vnew;
                uint16_t* cache = isk ? p.kc : p.vc;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const uint16_t v = f32_to_bf16_rn(x[e]);
                    dst[lane * EPL + e] = v;
                    if (s == ns - 1) cache[headoff + size_t(cp) * D + lane * EPL + e] = v;
                }
            }
        }
    } else {
        for (int i = tid; i < REP * D; i += NT) qs[i] = __fmul_rn(in[size_t(h) * REP * D + i], qscale);
    }
    __syncthreads();

    // ---- per-warp online softmax, 8 positions at a time
    float qreg[REP][EPL];
#pragma unroll
    for (int hh = 0; hh < REP; ++hh)
#pragma unroll
        for (int e = 0; e < EPL; ++e) qreg[hh][e] = qs[hh * D + lane * EPL + e];
    float m[REP], l[REP], o[REP][EPL];
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[hh][e] = 0.f;
    }
    for (int st = 0; st < nsub; ++st) {
        const int sb = st % nst;
        mbar_wait(&bar[sb], uint32_t((st / nst) & 1), p.err);
        const int pa = t0 + st * kSub;
        const int np = min(kSub, t1 - pa);       // positions of this stage, the new one included
        const int c0 = warp * kChunk;
        if (c0 < np) {
            const int nv = min(kChunk, np - c0);
            const uint16_t* ks = kst + size_t(sb) * kSub * D;
            const uint16_t* vs = vst + size_t(sb) * kSub * D;
            // rows past the end of the chunk re-read its first row (weight 0 in the update)
            auto krow = [&](int j) -> const uint16_t* {
                const int i = c0 + j;
                return (p.fused && pa + i == cp) ? knew : ks + size_t(i) * D;
            };
            auto vrow = [&](int j) -> const uint16_t* {
                const int i = c0 + j;
                return (p.fused && pa + i == cp) ? vnew : vs + size_t(i) * D;
            };
            attn_score_chunk<D, REP, kChunk>(nv, krow, vrow, qreg, m, l, o, lane);
        }
        if (st + nst < nsub) {
            __syncthreads();                      // every warp is done with this stage
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(st + nst);
            }
        }
    }
    // ---- merge the 8 scoring warps (fixed order)
    if (warp < kScoreWarps) {
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
            if (lane == 0) {
                wml[(warp * kMaxRep + hh) * 2] = m[hh];
                wml[(warp * kMaxRep + hh) * 2 + 1] = l[hh];
            }
#pragma unroll
            for (int e = 0; e < EPL; ++e) wo[(size_t(warp) * REP + hh) * D + lane * EPL + e] = o[hh][e];
        }
    }
    __syncthreads();
    for (int i = tid; i < REP * D; i += NT) {
        const int hh = i / D, dim = i % D;
        float mx, num, den;
        attn_warp_merge<D, REP>(wml, wo, hh, dim, mx, num, den);
        if constexpr (CLUSTER) {
            // push this split's state for output i to the rank that merges i's slice
            if (s < ns) {
                const int dest = i / PER, k = i % PER;
                float* r = cg::this_cluster().map_shared_rank(recv, dest) + s * (PER + 2);
                r[2 + k] = num;
                if (k == 0) {
                    r[0] = mx;
                    r[1] = den;
                }
            }
        } else {
            co[i] = num;
            if (dim == 0) {
                cml[hh * 2] = mx;
                cml[hh * 2 + 1] = den;
            }
        }
    }
    if constexpr (CLUSTER) {
        // ---- every split's state for this rank's slice is now in local shared memory
        cg::this_cluster().sync();
        for (int k = tid; k < PER; k += NT) {
            // all sources' states first (independent loads), then the fixed-order sums
            float mr[kAttnClusterSplits], lr[kAttnClusterSplits], nr[kAttnClusterSplits];
#pragma unroll
            for (int r = 0; r < kAttnClusterSplits; ++r) {
                mr[r] = -INFINITY;
                lr[r] = nr[r] = 0.f;
                if (r < ns) {
                    mr[r] = recv[r * (PER + 2)];
                    lr[r] = recv[r * (PER + 2) + 1];
                    nr[r] = recv[r * (PER + 2) + 2 + k];
                }
            }
            outrow[s * PER + k] = attn_split_merge(mr, lr, nr);
        }
    } else {
        // ---- global mode: one split writes directly; otherwise the last CTA merges
        __syncthreads();
        if (ns == 1) {
            for (int i = tid; i < REP * D; i += NT) outrow[i] = __fdiv_rn(co[i], cml[(i / D) * 2 + 1]);
            return;
        }
        float* mypart = p.part + ((size_t(b) * p.nkv + h) * p.tsplit + s) * REP * (D + 2);
        for (int i = tid; i < REP * D; i += NT) mypart[(i / D) * (D + 2) + 2 + i % D] = co[i];
        if (tid < REP) {
            mypart[tid * (D + 2)] = cml[tid * 2];
            mypart[tid * (D + 2) + 1] = cml[tid * 2 + 1];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int* ctr = &p.counters[size_t(b) * p.nkv + h];
            const int old = atomicAdd(ctr, 1);
            flag[0] = old == ns - 1;
            if (old == ns - 1) {
                *ctr = 0;
                __threadfence();
            }
        }
        __syncthreads();
        if (!flag[0]) return;
        const float* parts = p.part + (size_t(b) * p.nkv + h) * p.tsplit * REP * (D + 2);
        // Every split's (m, l) in one round of independent loads and the merge weights once,
        // in shared memory (the warp states in wo are consumed); then each output sums its
        // splits with its own loads in flight together.  Same operations in the same order
        // as a per-output loop over the splits, so the same bits.
        float* mq = wo;                                   // [split][head]
        float* lq = wo + ns * REP;
        float* wq = wo + 2 * ns * REP;
        for (int i = tid; i < ns * REP; i += NT) {
            const float* pq = parts + size_t(i) * (D + 2);
            mq[i] = __ldcg(&pq[0]);
            lq[i] = __ldcg(&pq[1]);
        }
        __syncthreads();
        for (int i = tid; i < ns * REP; i += NT) {
            const int hh = i % REP;
            float mx = -INFINITY;
            for (int q = 0; q < ns; ++q) mx = fmaxf(mx, mq[q * REP + hh]);
            wq[i] = (mq[i] == -INFINITY) ? 0.f : exp2f(__fsub_rn(mq[i], mx));
        }
        __syncthreads();
        for (int i = tid; i < REP * D; i += NT) {
            const int hh = i / D, dim = i % D;
            float num = 0.f, den = 0.f;
#pragma unroll 8
            for (int q = 0; q < ns; ++q) {
                const float wt = wq[q * REP + hh];
                den = __fmaf_rn(wt, lq[q * REP + hh], den);
                num = __fmaf_rn(wt, __ldcg(&parts[(size_t(q) * REP + hh) * (D + 2) + 2 + dim]), num);
            }
            outrow[i] = __fdiv_rn(num, den);
        }
    }
}

template <bool CL, int CH, bool QF>
const void* attn_fn_ch(int d, int rep) {
    if (d == 64) {
        if (rep == 1) return (const void*)attn_kernel<64, 1, CL, CH, false>;   // (REP + 2) x 64 rows: no whole tiles per rank
        if (rep == 2) return (const void*)attn_kernel<64, 2, CL, CH, QF>;
        return (const void*)attn_kernel<64, 4, CL, 8, QF>;
    }
    if (rep == 1) return (const void*)attn_kernel<128, 1, CL, CH, QF>;
    if (rep == 2) return (const void*)attn_kernel<128, 2, CL, CH, QF>;
    return (const void*)attn_kernel<128, 4, CL, 8, QF>;
}
template <bool CL>
const void* attn_fn(int d, int rep, int ch, bool qkv = false) {
    if (CL && qkv) return ch == 16 ? attn_fn_ch<CL, 16, CL>(d, rep) : attn_fn_ch<CL, 8, CL>(d, rep);
    return ch == 16 ? attn_fn_ch<CL, 16, false>(d, rep) : attn_fn_ch<CL, 8, false>(d, rep);
}

}  // namespace

// Positions a warp scores at once for a launch (attn_chunk_for).
int attn_chunk(int max_len, int splits, int rep) {
    if (splits < 1) splits = 1;
    const int chunk = (((max_len + splits - 1) / splits) + 15) & ~15;
    return (chunk > 64 && rep <= 2) ? 16 : 8;
}
// Ring depth: enough stages (of 8 x ch positions) for the longest split, at most kMaxStages
// and at most 192 KB of K/V staging.
int attn_stages(int max_len, int splits, int ch, int d) {
    if (splits < 1) splits = 1;
    const int chunk = (((max_len + splits - 1) / splits) + 15) & ~15;
    int n = (chunk + kScoreWarps * ch - 1) / (kScoreWarps * ch);
    const int cap = int((192u * 1024u) / (unsigned(kScoreWarps * ch) * unsigned(d) * 4u));
    if (n > kMaxStages) n = kMaxStages;
    if (n > cap) n = cap;
    return n < 1 ? 1 : n;
}
size_t attn_smem_bytes(int d, int rep, int nstage, int ch, int qkv_tb) {
    return attn_layout(d, rep, nstage, kScoreWarps * ch, qkv_tb).total;
}
bool attn_can_fuse_qkv(int d, int rep, int hidden) {
    return ((rep + 2) * d) % 128 == 0 && hidden % 128 == 0 && hidden / 128 <= 16;
}
int attn_default_tsplit(int nkv) {
    int t = (num_sms() + nkv - 1) / nkv;
    return t < 1 ? 1 : (t > 32 ? 32 : t);
}
size_t attn_workspace_bytes(int B, int nq, int nkv, int d, int tsplit) {
    return al16a(size_t(B) * nq * size_t(tsplit) * (d + 2) * 4) + al16a(size_t(B) * nkv * 4);
}

cudaError_t launch_attn(const AttnParams& p, cudaStream_t st, bool pdl) {
    const int rep = p.nq / p.nkv;
    AttnParams q = p;
    if (p.cluster) q.tsplit = kAttnClusterSplits;
    const int ch = attn_chunk(p.S, q.tsplit, rep);
    q.nstage = attn_stages(p.S, q.tsplit, ch, p.d);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(q.tsplit, p.nkv, p.B);
    const bool qkv = p.cluster && p.wqkv != nullptr && attn_can_fuse_qkv(p.d, rep, p.hidden);
    cfg.blockDim = dim3(qkv ? kAttnThreadsQkv : kAttnThreadsPlain);
    if (!qkv) q.wqkv = nullptr;
    cfg.dynamicSmemBytes = attn_smem_bytes(p.d, rep, q.nstage, ch, qkv ? p.qkv_tile_bytes : 0);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (p.cluster) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = kAttnClusterSplits;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const void* fn = p.cluster ? attn_fn<true>(p.d, rep, ch, qkv) : attn_fn<false>(p.d, rep, ch);
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t attn_set_attributes() {
    const int mx = 227 * 1024;
    const int reps[3] = {1, 2, 4}, ds[2] = {64, 128};
    for (int d : ds)
        for (int r : reps)
            for (int cl = 0; cl < 8; ++cl) {
                const int ch = (cl & 2) ? 16 : 8;
                const void* k = (cl & 1) ? attn_fn<true>(d, r, ch, (cl & 4) != 0) : attn_fn<false>(d, r, ch);
                cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
                if (e != cudaSuccess) return e;
                e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

}  // namespace kmr
