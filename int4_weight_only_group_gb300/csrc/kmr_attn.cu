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
// layout) into a 2-stage ring whose first fill is issued before
// griddepcontrol.wait.  Every warp runs its own online softmax over its
// positions (two at a time, no block barrier inside the loop); the 8 warp
// states merge in shared memory, then the splits merge in split order:
//   * cluster mode: the splits of one (row, KV head) are one thread-block
//     cluster; the merge reads the peers' shared memory (DSMEM) after a
//     cluster barrier — no global memory, no atomics;
//   * global mode: each split writes its state to a caller workspace and the
//     last CTA to arrive (atomic counter) merges — for any number of splits.
#include <cooperative_groups.h>
#include <math.h>

#include "kmr_internal.cuh"

namespace cg = cooperative_groups;

namespace kmr {

namespace {

constexpr int kSub = 64;       // positions per ring stage
constexpr int kStages = 2;
constexpr int kMaxRep = 4;     // query heads per KV head supported

__host__ __device__ inline size_t al16a(size_t v) { return (v + 15) & ~size_t(15); }

struct AttnSmem {
    size_t bar, kst, vst, knew, vnew, qs, wml, wo, cml, co, flag, total;
};
__host__ __device__ inline AttnSmem attn_layout(int D, int rep) {
    AttnSmem L;
    size_t o = 0;
    L.bar = o;   o += al16a(kStages * 8);
    o = (o + 127) & ~size_t(127);
    L.kst = o;   o += size_t(kStages) * kSub * D * 2;
    L.vst = o;   o += size_t(kStages) * kSub * D * 2;
    L.knew = o;  o += al16a(size_t(D) * 2);
    L.vnew = o;  o += al16a(size_t(D) * 2);
    L.qs = o;    o += al16a(size_t(rep) * D * 4);
    L.wml = o;   o += al16a(size_t(8) * kMaxRep * 2 * 4);     // per warp: (m, l) per head
    L.wo = o;    o += al16a(size_t(8) * rep * D * 4);         // per warp: o per head
    L.cml = o;   o += al16a(size_t(kMaxRep) * 2 * 4);         // CTA state: (m, l) per head
    L.co = o;    o += al16a(size_t(rep) * D * 4);             // CTA state: o per head
    L.flag = o;  o += 16;
    L.total = o;
    return L;
}

template <int D, int REP, bool CLUSTER>
__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int EPL = D / 32;          // contiguous dims per lane
    const AttnSmem L = attn_layout(D, REP);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint16_t* kst = reinterpret_cast<uint16_t*>(smem + L.kst);
    uint16_t* vst = reinterpret_cast<uint16_t*>(smem + L.vst);
    uint16_t* knew = reinterpret_cast<uint16_t*>(smem + L.knew);
    uint16_t* vnew = reinterpret_cast<uint16_t*>(smem + L.vnew);
    float* qs = reinterpret_cast<float*>(smem + L.qs);
    float* wml = reinterpret_cast<float*>(smem + L.wml);
    float* wo = reinterpret_cast<float*>(smem + L.wo);
    float* cml = reinterpret_cast<float*>(smem + L.cml);
    float* co = reinterpret_cast<float*>(smem + L.co);
    int* flag = reinterpret_cast<int*>(smem + L.flag);

    // Row state comes from the previous step (complete before this graph ran), not
    // from the kernels of this step, so it may be read before griddepcontrol.wait.
    const bool fin = p.finished != nullptr && p.finished[b] != 0;
    const int slot = p.slot_ids[b], cp = p.cpos[b];
    const bool bad_slot = slot < 0 || slot >= p.slots;
    const bool bad_pos = cp < 0 || cp >= p.S;
    float* outrow = p.out + size_t(b) * p.nq * D + size_t(h) * REP * D;
    if (fin || bad_slot || bad_pos) {            // uniform over the whole cluster / row
        if (s == 0) {
            pdl_wait();
            if (!fin && h == 0 && tid == 0) set_error(p.err, bad_slot ? KMR_ERR_SLOT_RANGE : KMR_ERR_CACHE_FULL);
            for (int i = tid; i < REP * D; i += kThreads) outrow[i] = 0.f;
        }
        return;
    }
    const int nsplit = gridDim.x;
    const int Lq = cp + 1;
    const int chunk = (((Lq + nsplit - 1) / nsplit) + 15) & ~15;
    const int ns = (Lq + chunk - 1) / chunk;
    if (!CLUSTER && s >= ns) return;             // (cluster mode: empty splits still join the barriers)
    const int t0 = s * chunk, t1 = min(Lq, t0 + chunk);      // t1 <= t0 for an empty split
    const int cached_end = p.fused ? min(t1, cp) : t1;
    const int nsub = t1 > t0 ? (t1 - t0 + kSub - 1) / kSub : 0;
    const size_t headoff = (size_t(slot) * p.nkv + h) * p.S * D;
    const uint16_t* kbase = p.kc + headoff;
    const uint16_t* vbase = p.vc + headoff;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int st) {
        const int sb = st % kStages;
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
        const int n0 = nsub < kStages ? nsub : kStages;
        for (int i = 0; i < n0; ++i) issue(i);
    }
    // constants of the prologue, fetched before the wait as well
    const bool qk_warp = p.fused && warp <= REP;
    float nw[EPL], invf[EPL];
    int axis[EPL];
    if (qk_warp) {
        const uint16_t* nrm = warp < REP ? p.qn_w : p.kn_w;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int dim = lane * EPL + e, f = dim % (D / 2);
            nw[e] = nrm ? bf16_to_f32(nrm[dim]) : 1.f;
            invf[e] = p.inv_freq[f];
            axis[e] = f < p.sec0 ? 0 : (f < p.sec0 + p.sec1 ? 1 : 2);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // ---- prologue: q (and, fused, the new k / v) of this KV head
    const float* in = p.in + size_t(b) * p.in_ld;
    if (p.fused) {
        if (warp <= REP + 1) {
            const bool isq = warp < REP, isk = warp == REP;
            const float* src = isq ? in + size_t(h * REP + warp) * D
                                   : (isk ? in + size_t(p.nq) * D + size_t(h) * D
                                          : in + size_t(p.nq + p.nkv) * D + size_t(h) * D);
            float x[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[e] = src[lane * EPL + e];
            if (qk_warp) {
                if (isq ? p.qn_w != nullptr : p.kn_w != nullptr) {
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) ss = __fmaf_rn(x[e], x[e], ss);
                    const float r = rsqrtf(warp_sum(ss) / float(D) + p.eps);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) x[e] = __fmul_rn(__fmul_rn(x[e], r), nw[e]);
                }
                // 3-section M-RoPE: frequency f turns the pair (f, f + D/2); the partner
                // dim sits 16 lanes away
                const bool lo = lane < 16;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
                    const float pos = float(p.positions[size_t(axis[e]) * p.pos_ld + b]);
                    float sn, cs;
                    sincosf(pos * invf[e], &sn, &cs);
                    x[e] = lo ? __fsub_rn(__fmul_rn(x[e], cs), __fmul_rn(other, sn))
                              : __fadd_rn(__fmul_rn(x[e], cs), __fmul_rn(other, sn));
                }
            }
            if (isq) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) qs[warp * D + lane * EPL + e] = __fmul_rn(x[e], p.scale);
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
        for (int i = tid; i < REP * D; i += kThreads) qs[i] = __fmul_rn(in[size_t(h) * REP * D + i], p.scale);
    }
    __syncthreads();

    // ---- per-warp online softmax over positions t0 + warp + 8 i, two at a time
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
    auto load_row = [&](const uint16_t* row, float (&v)[EPL]) {
        if constexpr (EPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
            v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
            v[0] = bf16_lo(u); v[1] = bf16_hi(u);
        }
    };
    for (int st = 0; st < nsub; ++st) {
        const int sb = st % kStages;
        mbar_wait(&bar[sb], uint32_t((st / kStages) & 1), p.err);
        const int pa = t0 + st * kSub;
        const int np = min(kSub, t1 - pa);
        const uint16_t* ks = kst + size_t(sb) * kSub * D;
        const uint16_t* vs = vst + size_t(sb) * kSub * D;
        for (int i = warp; i < np; i += 16) {
            const bool two = i + 8 < np;
            const int i1 = two ? i + 8 : i;       // a lone last position pairs with itself (weight 0)
            const uint16_t* k0 = (p.fused && pa + i == cp) ? knew : ks + size_t(i) * D;
            const uint16_t* k1 = (p.fused && pa + i1 == cp) ? knew : ks + size_t(i1) * D;
            float ka[EPL], kb[EPL];
            load_row(k0, ka);
            load_row(k1, kb);
            float s0[REP], s1[REP];
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                float a = 0.f, c = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    a = __fmaf_rn(qreg[hh][e], ka[e], a);
                    c = __fmaf_rn(qreg[hh][e], kb[e], c);
                }
                s0[hh] = a;
                s1[hh] = c;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int hh = 0; hh < REP; ++hh) {
                    s0[hh] += __shfl_xor_sync(0xffffffffu, s0[hh], off);
                    s1[hh] += __shfl_xor_sync(0xffffffffu, s1[hh], off);
                }
            const uint16_t* v0 = (p.fused && pa + i == cp) ? vnew : vs + size_t(i) * D;
            const uint16_t* v1 = (p.fused && pa + i1 == cp) ? vnew : vs + size_t(i1) * D;
            float va[EPL], vb[EPL];
            load_row(v0, va);
            load_row(v1, vb);
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                const float mn = fmaxf(m[hh], two ? fmaxf(s0[hh], s1[hh]) : s0[hh]);
                const float cf = (m[hh] == -INFINITY) ? 0.f : expf(m[hh] - mn);
                const float p0 = expf(s0[hh] - mn);
                const float p1 = two ? expf(s1[hh] - mn) : 0.f;
                l[hh] = __fadd_rn(__fmaf_rn(l[hh], cf, p0), p1);
#pragma unroll
                for (int e = 0; e < EPL; ++e)
                    o[hh][e] = __fmaf_rn(p1, vb[e], __fmaf_rn(p0, va[e], __fmul_rn(o[hh][e], cf)));
                m[hh] = mn;
            }
        }
        if (st + kStages < nsub) {
            __syncthreads();                      // every warp is done with this stage
            if (tid == 0) {
                fence_proxy_async_smem();
                issue(st + kStages);
            }
        }
    }
    // ---- merge the 8 warps (fixed order) into the CTA state
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        if (lane == 0) {
            wml[(warp * kMaxRep + hh) * 2] = m[hh];
            wml[(warp * kMaxRep + hh) * 2 + 1] = l[hh];
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) wo[(size_t(warp) * REP + hh) * D + lane * EPL + e] = o[hh][e];
    }
    __syncthreads();
    for (int i = tid; i < REP * D; i += kThreads) {
        const int hh = i / D, dim = i % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wml[(w * kMaxRep + hh) * 2]);
        float num = 0.f, den = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float mw = wml[(w * kMaxRep + hh) * 2];
                const float wt = (mw == -INFINITY) ? 0.f : expf(mw - mx);
                den = __fmaf_rn(wt, wml[(w * kMaxRep + hh) * 2 + 1], den);
                num = __fmaf_rn(wt, wo[(size_t(w) * REP + hh) * D + dim], num);
            }
        }
        co[hh * D + dim] = num;
        if (dim == 0) {
            cml[hh * 2] = mx;
            cml[hh * 2 + 1] = den;
        }
    }
    if constexpr (CLUSTER) {
        // ---- merge the splits of this (row, KV head) through distributed shared memory
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int per = (REP * D + nsplit - 1) / nsplit;       // outputs merged by each rank
        for (int i = tid; i < per; i += kThreads) {
            const int oi = s * per + i;
            if (oi >= REP * D) break;
            const int hh = oi / D, dim = oi % D;
            float mx = -INFINITY;
            for (int r = 0; r < ns; ++r) mx = fmaxf(mx, cluster.map_shared_rank(cml, r)[hh * 2]);
            float num = 0.f, den = 0.f;
            for (int r = 0; r < ns; ++r) {
                const float* rml = cluster.map_shared_rank(cml, r);
                const float mr = rml[hh * 2];
                const float wt = (mr == -INFINITY) ? 0.f : expf(mr - mx);
                den = __fmaf_rn(wt, rml[hh * 2 + 1], den);
                num = __fmaf_rn(wt, cluster.map_shared_rank(co, r)[hh * D + dim], num);
            }
            outrow[oi] = __fdiv_rn(num, den);
        }
        cluster.sync();                           // peers' shared memory stays alive until read
    } else {
        // ---- global mode: one split writes directly; otherwise the last CTA merges
        __syncthreads();
        if (ns == 1) {
            for (int i = tid; i < REP * D; i += kThreads) outrow[i] = __fdiv_rn(co[i], cml[(i / D) * 2 + 1]);
            return;
        }
        float* mypart = p.part + ((size_t(b) * p.nkv + h) * p.tsplit + s) * REP * (D + 2);
        for (int i = tid; i < REP * D; i += kThreads) mypart[(i / D) * (D + 2) + 2 + i % D] = co[i];
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
        for (int i = tid; i < REP * D; i += kThreads) {
            const int hh = i / D, dim = i % D;
            float mx = -INFINITY;
            for (int q = 0; q < ns; ++q) mx = fmaxf(mx, __ldcg(&parts[(size_t(q) * REP + hh) * (D + 2)]));
            float num = 0.f, den = 0.f;
            for (int q = 0; q < ns; ++q) {
                const float* pq = parts + (size_t(q) * REP + hh) * (D + 2);
                const float mq = __ldcg(&pq[0]);
                const float wt = (mq == -INFINITY) ? 0.f : expf(mq - mx);
                den = __fmaf_rn(wt, __ldcg(&pq[1]), den);
                num = __fmaf_rn(wt, __ldcg(&pq[2 + dim]), num);
            }
            outrow[i] = __fdiv_rn(num, den);
        }
    }
}

template <bool CL>
const void* attn_fn(int d, int rep) {
    if (d == 64) {
        if (rep == 1) return (const void*)attn_kernel<64, 1, CL>;
        if (rep == 2) return (const void*)attn_kernel<64, 2, CL>;
        return (const void*)attn_kernel<64, 4, CL>;
    }
    if (rep == 1) return (const void*)attn_kernel<128, 1, CL>;
    if (rep == 2) return (const void*)attn_kernel<128, 2, CL>;
    return (const void*)attn_kernel<128, 4, CL>;
}

}  // namespace

size_t attn_smem_bytes(int d, int rep) { return attn_layout(d, rep).total; }
int attn_default_tsplit(int nkv) {
    int t = (num_sms() + nkv - 1) / nkv;
    return t < 1 ? 1 : (t > 32 ? 32 : t);
}
size_t attn_workspace_bytes(int B, int nq, int nkv, int d, int tsplit) {
    return al16a(size_t(B) * nq * size_t(tsplit) * (d + 2) * 4) + al16a(size_t(B) * nkv * 4);
}

cudaError_t launch_attn(const AttnParams& p, cudaStream_t st, bool pdl) {
    const int rep = p.nq / p.nkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.cluster ? kAttnClusterSplits : p.tsplit, p.nkv, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attn_smem_bytes(p.d, rep);
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
    AttnParams q = p;
    if (p.cluster) q.tsplit = kAttnClusterSplits;
    const void* fn = p.cluster ? attn_fn<true>(p.d, rep) : attn_fn<false>(p.d, rep);
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t attn_set_attributes() {
    const int mx = 227 * 1024;
    const int reps[3] = {1, 2, 4}, ds[2] = {64, 128};
    for (int d : ds)
        for (int r : reps)
            for (int cl = 0; cl < 2; ++cl) {
                const void* k = cl ? attn_fn<true>(d, r) : attn_fn<false>(d, r);
                cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
                if (e != cudaSuccess) return e;
                e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

}  // namespace kmr
