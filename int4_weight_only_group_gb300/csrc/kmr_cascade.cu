// Shared-prefix (cascade) decode attention ("The Ghost in the Batch: How vLLM Silently
// Switches Algorithms", The Optimization That Changes Everything: when many requests share a
// prompt prefix, attend over the prefix once for all of their queries, over each request's
// own suffix separately, and merge the two partial results with their log-sum-exp weights;
// What Attention Does: out = softmax(q K^T / sqrt(d)) V).
//
// Row b's context is positions [0, P) of the prefix cache row (one per call) followed by
// positions [P, cache_position[b]] of its own cache row.  Two launches on one stream:
//   1. prefix: grid (prefix split, KV head).  A CTA stages its split of the prefix K and V
//      once (cp.async.bulk) and runs every row's query heads of that KV head over it, one
//      warp per row at a time; each (row, query head, split) leaves an unnormalised state
//      (m, l, o) in base 2 in the workspace.  The prefix is read from HBM once per call,
//      not once per row.
//   2. suffix + merge: grid (KV head, row), launched as a programmatic dependent of the prefix
//      pass so that the two run together.  A CTA streams the row's own positions through
//      a two-stage ring (8 warps x 8 positions per stage), waits for the prefix pass
//      (griddepcontrol.wait), then merges, for each output,
//      the prefix split states in split order followed by its 8 warp states in warp order,
//      and divides.  The prefix split plan depends only on P and the KV head count, so a
//      row's result does not depend on which other rows share the call.
#include <math.h>

#include "kmr_internal.cuh"

namespace kmr {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCasThreads = 256;            // 8 warps
constexpr int kSufCh = 8;                   // positions a warp scores at once
constexpr int kSufSub = 8 * kSufCh;         // positions per suffix stage

// One warp's online softmax (base 2) over n staged positions for REP query heads whose
// scaled queries the lane holds for dims [lane * D/32, (lane + 1) * D/32).  State (m, l, o)
// accumulates across calls.
template <int D, int REP>
__device__ __forceinline__ void warp_attend(const float (&qreg)[REP][D / 32], const uint16_t* ks, const uint16_t* vs,
                                            int n, int lane, float (&m)[REP], float (&l)[REP],
                                            float (&o)[REP][D / 32]) {
    constexpr int EPL = D / 32, CH = kSufCh, NV = REP * CH, JS = 32 / NV;
    static_assert(NV <= 32, "one score per lane after the reduce-scatter");
    auto load_row = [&](const uint16_t* row, float (&v)[EPL]) {
        if constexpr (EPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
            v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
            v[0] = bf16_lo(u); v[1] = bf16_hi(u);
        }
    };
    const int myidx = lane / JS, myhh = myidx / CH, myj = myidx % CH;
    for (int c0 = 0; c0 < n; c0 += CH) {
        const int nv = min(CH, n - c0);
        float sc[NV];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            float kv[EPL];
            load_row(ks + size_t(c0 + (j < nv ? j : 0)) * D, kv);     // past the end: re-read (weight 0)
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
            load_row(vs + size_t(c0 + (j < nv ? j : 0)) * D, vv);
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                const float pj = __shfl_sync(0xffffffffu, pme, (hh * CH + j) * JS);
                l[hh] = __fadd_rn(l[hh], pj);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[hh][e] = __fmaf_rn(pj, vv[e], o[hh][e]);
            }
        }
    }
}

template <int D, int REP>
__device__ __forceinline__ void load_query(const CascadeParams& p, int b, int h, int lane, float (&qreg)[REP][D / 32]) {
    constexpr int EPL = D / 32;
    const float qscale = __fmul_rn(p.scale, kLog2e);
#pragma unroll
    for (int hh = 0; hh < REP; ++hh)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            qreg[hh][e] = __fmul_rn(p.q[(size_t(b) * p.nq + h * REP + hh) * D + lane * EPL + e], qscale);
}

template <int D, int REP>
__global__ void __launch_bounds__(kCasThreads) cascade_prefix_kernel(const CascadeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int EPL = D / 32;
    const int sp = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c0 = sp * p.pchunk, n = min(p.prefix_len, c0 + p.pchunk) - c0;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem + 128);
    uint16_t* vs = ks + size_t(p.pchunk) * D;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();                    // the suffix pass needs the states only at its merge
    if (tid == 0) {
        const size_t base = ((size_t(p.prefix_slot) * p.nkv + h) * p.S + c0) * D;
        const uint32_t bytes = uint32_t(n) * D * 2;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(ks, p.kc + base, bytes, bar);
        bulk_g2s(vs, p.vc + base, bytes, bar);
    }
    mbar_wait(bar, 0u, p.err);
    for (int b = warp; b < p.B; b += kCasThreads / 32) {
        float qreg[REP][EPL], m[REP], l[REP], o[REP][EPL];
        load_query<D, REP>(p, b, h, lane, qreg);
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
            m[hh] = -INFINITY;
            l[hh] = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[hh][e] = 0.f;
        }
        warp_attend<D, REP>(qreg, ks, vs, n, lane, m, l, o);
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
            float* st = p.part + ((size_t(b) * p.nq + h * REP + hh) * p.psplits + sp) * (D + 2);
            if (lane == 0) {
                st[0] = m[hh];
                st[1] = l[hh];
            }
#pragma unroll
            for (int e = 0; e < EPL; ++e) st[2 + lane * EPL + e] = o[hh][e];
        }
    }
}

template <int D, int REP>
__global__ void __launch_bounds__(kCasThreads) cascade_suffix_kernel(const CascadeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int EPL = D / 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                        // 2 stages
    float* wml = reinterpret_cast<float*>(smem + 16);                        // [8 warps][REP][2]
    float* wo = reinterpret_cast<float*>(smem + 16 + 8 * REP * 2 * 4);       // [8 warps][REP][D]
    uint16_t* kst = reinterpret_cast<uint16_t*>(smem + 16 + 8 * REP * 2 * 4 + 8 * REP * D * 4);
    uint16_t* vst = kst + 2 * size_t(kSufSub) * D;
    float* outrow = p.out + (size_t(b) * p.nq + h * REP) * D;

    const int slot = p.slot_ids[b], cp = p.cpos[b];
    if (slot < 0 || slot >= p.slots || cp < p.prefix_len || cp >= p.S) {
        if (tid == 0 && h == 0) set_error(p.err, (slot < 0 || slot >= p.slots) ? KMR_ERR_SLOT_RANGE : KMR_ERR_CACHE_FULL);
        for (int i = tid; i < REP * D; i += kCasThreads) outrow[i] = 0.f;
        return;
    }
    const int t0 = p.prefix_len, ns = cp + 1 - t0;                   // own positions [t0, cp]
    const int nstg = (ns + kSufSub - 1) / kSufSub;
    const size_t base = ((size_t(slot) * p.nkv + h) * p.S) * D;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int st) {
        const int pa = t0 + st * kSufSub, np = min(kSufSub, cp + 1 - pa);
        const uint32_t bytes = uint32_t(np) * D * 2;
        mbar_arrive_expect_tx(&bar[st & 1], 2 * bytes);
        bulk_g2s(kst + size_t(st & 1) * kSufSub * D, p.kc + base + size_t(pa) * D, bytes, &bar[st & 1]);
        bulk_g2s(vst + size_t(st & 1) * kSufSub * D, p.vc + base + size_t(pa) * D, bytes, &bar[st & 1]);
    };
    if (tid == 0) {
        issue(0);
        if (nstg > 1) issue(1);
    }
    float qreg[REP][EPL], m[REP], l[REP], o[REP][EPL];
    load_query<D, REP>(p, b, h, lane, qreg);
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[hh][e] = 0.f;
    }
    for (int st = 0; st < nstg; ++st) {
        mbar_wait(&bar[st & 1], uint32_t((st >> 1) & 1), p.err);
        const int pa = t0 + st * kSufSub, np = min(kSufSub, cp + 1 - pa);
        const int w0 = warp * kSufCh;
        if (w0 < np)
            warp_attend<D, REP>(qreg, kst + (size_t(st & 1) * kSufSub + w0) * D,
                                vst + (size_t(st & 1) * kSufSub + w0) * D, min(kSufCh, np - w0), lane, m, l, o);
        if (st + 2 < nstg) {
            __syncthreads();                                         // every warp is done with this stage
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(st + 2);
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        if (lane == 0) {
            wml[(warp * REP + hh) * 2] = m[hh];
            wml[(warp * REP + hh) * 2 + 1] = l[hh];
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) wo[(warp * REP + hh) * D + lane * EPL + e] = o[hh][e];
    }
    __syncthreads();
    pdl_wait();                                 // the prefix pass's states are complete from here
    // merge: prefix split states in split order, then the 8 warp states in warp order
    for (int i = tid; i < REP * D; i += kCasThreads) {
        const int hh = i / D, dim = i % D;
        const float* pst = p.part + (size_t(b) * p.nq + h * REP + hh) * p.psplits * (D + 2);
        float mx = -INFINITY;
        for (int s = 0; s < p.psplits; ++s) mx = fmaxf(mx, pst[size_t(s) * (D + 2)]);
#pragma unroll
        for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wml[(w * REP + hh) * 2]);
        float num = 0.f, den = 0.f;
        for (int s = 0; s < p.psplits; ++s) {
            const float ms = pst[size_t(s) * (D + 2)];
            const float wt = (ms == -INFINITY) ? 0.f : exp2f(__fsub_rn(ms, mx));
            den = __fmaf_rn(wt, pst[size_t(s) * (D + 2) + 1], den);
            num = __fmaf_rn(wt, pst[size_t(s) * (D + 2) + 2 + dim], num);
        }
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float mw = wml[(w * REP + hh) * 2];
            const float wt = (mw == -INFINITY) ? 0.f : exp2f(__fsub_rn(mw, mx));
            den = __fmaf_rn(wt, wml[(w * REP + hh) * 2 + 1], den);
            num = __fmaf_rn(wt, wo[(w * REP + hh) * D + dim], num);
        }
        outrow[i] = __fdiv_rn(num, den);
    }
}

template <int D, int REP>
size_t suffix_smem() { return 16 + 8 * REP * 2 * 4 + 8 * REP * D * 4 + 2 * 2 * size_t(kSufSub) * D * 2; }

template <int D, int REP>
cudaError_t launch_cascade_t(const CascadeParams& p, cudaStream_t st) {
    static bool attr = false;
    const size_t pre_smem = 128 + 2 * size_t(p.pchunk) * D * 2;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(cascade_prefix_kernel<D, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(128 + 2 * size_t(kCascadeMaxChunk) * D * 2));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(cascade_suffix_kernel<D, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(suffix_smem<D, REP>()));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (p.prefix_len > 0) {
        cascade_prefix_kernel<D, REP><<<dim3(p.psplits, p.nkv), kCasThreads, pre_smem, st>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // the suffix pass overlaps the prefix pass (programmatic dependent launch) and waits for it
    // only before its merge
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nkv, p.B);
    cfg.blockDim = dim3(kCasThreads);
    cfg.dynamicSmemBytes = suffix_smem<D, REP>();
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = p.prefix_len > 0 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, cascade_suffix_kernel<D, REP>, p);
}

}  // namespace

void cascade_plan(int prefix_len, int nkv, int sms, int* pchunk, int* psplits) {
    if (prefix_len <= 0) {
        *pchunk = 16;
        *psplits = 0;
        return;
    }
    const int target = sms / nkv > 1 ? sms / nkv : 1;
    int c = (prefix_len + target - 1) / target;
    c = (c + 15) & ~15;
    if (c > kCascadeMaxChunk) c = kCascadeMaxChunk;
    *pchunk = c;
    *psplits = (prefix_len + c - 1) / c;
}

size_t cascade_workspace_bytes(int B, int nq, int d, int psplits) {
    return size_t(B) * nq * (psplits > 0 ? psplits : 1) * (d + 2) * 4;
}

cudaError_t launch_cascade(const CascadeParams& p, cudaStream_t st) {
    const int rep = p.nq / p.nkv;
    if (p.d == 128) {
        if (rep == 1) return launch_cascade_t<128, 1>(p, st);
        if (rep == 2) return launch_cascade_t<128, 2>(p, st);
        return launch_cascade_t<128, 4>(p, st);
    }
    if (rep == 1) return launch_cascade_t<64, 1>(p, st);
    if (rep == 2) return launch_cascade_t<64, 2>(p, st);
    return launch_cascade_t<64, 4>(p, st);
}

}  // namespace kmr
