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
// GB300 design: grid (split, kv head, row); the split length depends only on
// the row's own length (ceil(L / tsplit) rounded up to 16), never on the batch,
// so a row's result is the same at any batch size.  Each CTA streams its K and
// V positions with cp.async.bulk (contiguous in the [slot][head][pos][d]
// layout) into a 4-stage ring; the first fill is issued before
// griddepcontrol.wait.  Online softmax over 32-position sub-tiles; partial
// (max, sum, unnormalised o) per split are merged in split order by the last
// CTA of the (row, kv head) to arrive — no float atomics.
#include <math.h>

#include "kmr_internal.cuh"

namespace kmr {

namespace {

constexpr int kSub = 32;       // positions per sub-tile
constexpr int kStages = 4;
constexpr int kMaxRep = 4;     // query heads per KV head supported

__host__ __device__ inline size_t al16a(size_t v) { return (v + 15) & ~size_t(15); }

struct AttnSmem {
    size_t bar, kst, vst, knew, vnew, qs, sc, st, opart, flag, total;
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
    L.sc = o;    o += al16a(size_t(rep) * kSub * 4);
    L.st = o;    o += al16a(size_t(3) * kMaxRep * 4);   // running max, running sum, correction
    L.opart = o; o += al16a(size_t(kThreads) * 2 * kMaxRep * 4);
    L.flag = o;  o += 16;
    L.total = o;
    return L;
}

template <int D, int REP>
__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int rep = REP;
    const AttnSmem L = attn_layout(D, rep);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint16_t* kst = reinterpret_cast<uint16_t*>(smem + L.kst);
    uint16_t* vst = reinterpret_cast<uint16_t*>(smem + L.vst);
    uint16_t* knew = reinterpret_cast<uint16_t*>(smem + L.knew);
    uint16_t* vnew = reinterpret_cast<uint16_t*>(smem + L.vnew);
    float* qs = reinterpret_cast<float*>(smem + L.qs);
    float* sc = reinterpret_cast<float*>(smem + L.sc);
    float* runm = reinterpret_cast<float*>(smem + L.st);
    float* runl = runm + kMaxRep;
    float* corr = runl + kMaxRep;
    float* opart = reinterpret_cast<float*>(smem + L.opart);
    int* flag = reinterpret_cast<int*>(smem + L.flag);

    const bool fin = p.finished != nullptr && p.finished[b] != 0;
    const int slot = p.slot_ids[b], cp = p.cpos[b];
    const bool bad_slot = slot < 0 || slot >= p.slots;
    const bool bad_pos = cp < 0 || cp >= p.S;
    float* outrow = p.out + size_t(b) * p.nq * D + size_t(h) * rep * D;
    if (fin || bad_slot || bad_pos) {
        if (s == 0) {
            pdl_wait();
            if (!fin && h == 0 && tid == 0) set_error(p.err, bad_slot ? KMR_ERR_SLOT_RANGE : KMR_ERR_CACHE_FULL);
            for (int i = tid; i < rep * D; i += kThreads) outrow[i] = 0.f;
        }
        return;
    }
    const int Lq = cp + 1;
    const int chunk = (((Lq + p.tsplit - 1) / p.tsplit) + 15) & ~15;
    const int ns = (Lq + chunk - 1) / chunk;
    if (s >= ns) return;
    const int t0 = s * chunk, t1 = min(Lq, t0 + chunk);
    const int cached_end = p.fused ? min(t1, cp) : t1;
    const int nsub = (t1 - t0 + kSub - 1) / kSub;
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
    pdl_launch_dependents();
    pdl_wait();

    // ---- prologue: q (and, fused, the new k / v) for this KV head
    constexpr int EPL = D / 32;          // elements per lane
    const float* in = p.in + size_t(b) * p.in_ld;
    if (p.fused) {
        if (warp <= rep + 1) {
            const bool isq = warp < rep, isk = warp == rep;
            const float* src = isq ? in + size_t(h * rep + warp) * D
                                   : (isk ? in + size_t(p.nq) * D + size_t(h) * D
                                          : in + size_t(p.nq + p.nkv) * D + size_t(h) * D);
            float x[EPL];
#pragma unroll
            for (int j = 0; j < EPL; ++j) x[j] = src[lane + 32 * j];
            if (warp <= rep) {
                const uint16_t* nw = isq ? p.qn_w : p.kn_w;
                if (nw) {
                    float ss = 0.f;
#pragma unroll
                    for (int j = 0; j < EPL; ++j) ss += x[j] * x[j];
                    const float r = rsqrtf(warp_sum(ss) / float(D) + p.eps);
#pragma unroll
                    for (int j = 0; j < EPL; ++j) x[j] = x[j] * r * bf16_to_f32(nw[lane + 32 * j]);
                }
                // 3-section M-RoPE: frequency i turns the pair (i, i + D/2)
#pragma unroll
                for (int j = 0; j < EPL / 2; ++j) {
                    const int i = lane + 32 * j;
                    const int axis = i < p.sec0 ? 0 : (i < p.sec0 + p.sec1 ? 1 : 2);
                    const float pos = float(p.positions[size_t(axis) * p.pos_ld + b]);
                    float sn, cs;
                    sincosf(pos * p.inv_freq[i], &sn, &cs);
                    const float x1 = x[j], x2 = x[j + EPL / 2];
                    x[j] = x1 * cs - x2 * sn;
                    x[j + EPL / 2] = x2 * cs + x1 * sn;
                }
            }
            if (isq) {
#pragma unroll
                for (int j = 0; j < EPL; ++j) qs[warp * D + lane + 32 * j] = x[j] * p.scale;
            } else {
                uint16_t* dst = isk ? knew : vnew;
                uint16_t* cache = isk ? p.kc : p.vc;
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const uint16_t v = f32_to_bf16_rn(x[j]);
                    dst[lane + 32 * j] = v;
                    if (s == ns - 1) cache[headoff + size_t(cp) * D + lane + 32 * j] = v;
                }
            }
        }
    } else {
        for (int i = tid; i < rep * D; i += kThreads) qs[i] = in[size_t(h) * rep * D + i] * p.scale;
    }
    if (tid < rep) {
        runm[tid] = -INFINITY;
        runl[tid] = 0.f;
    }
    __syncthreads();

    // score mapping: 8 lanes per position, 4 positions per warp, D/8 dims per lane
    constexpr int DPL = D / 8;
    const int g = lane >> 3, dj = lane & 7;
    const int pi_s = warp * 4 + g;
    float qreg[REP][DPL];
#pragma unroll
    for (int hh = 0; hh < REP; ++hh)
#pragma unroll
        for (int e = 0; e < DPL; ++e) qreg[hh][e] = hh < rep ? qs[hh * D + dj * DPL + e] : 0.f;
    // PV mapping: one dim pair per thread, positions split in quarters
    constexpr int NDP = D / 2;
    constexpr int NQ4 = kThreads / NDP;
    constexpr int PPQ = kSub / NQ4;
    const int dp = tid % NDP, q4 = tid / NDP;
    float oacc[REP][2];
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) oacc[hh][0] = oacc[hh][1] = 0.f;

    for (int st = 0; st < nsub; ++st) {
        const int sb = st % kStages;
        mbar_wait(&bar[sb], uint32_t((st / kStages) & 1), p.err);
        const int pa = t0 + st * kSub;
        const int np = min(kSub, t1 - pa);
        const uint16_t* ks = kst + size_t(sb) * kSub * D;
        const uint16_t* vs = vst + size_t(sb) * kSub * D;
        // scores
        {
            float dot[REP];
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) dot[hh] = 0.f;
            if (pi_s < np) {
                const int pos = pa + pi_s;
                const uint16_t* krow = (p.fused && pos == cp) ? knew : ks + size_t(pi_s) * D;
                const uint4* kp = reinterpret_cast<const uint4*>(krow + dj * DPL);
#pragma unroll
                for (int v4 = 0; v4 < DPL / 8; ++v4) {
                    const uint4 kv = kp[v4];
                    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float k0 = bf16_lo(kw[e]), k1 = bf16_hi(kw[e]);
#pragma unroll
                        for (int hh = 0; hh < REP; ++hh) {
                            dot[hh] = fmaf(qreg[hh][v4 * 8 + 2 * e], k0, dot[hh]);
                            dot[hh] = fmaf(qreg[hh][v4 * 8 + 2 * e + 1], k1, dot[hh]);
                        }
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                dot[hh] += __shfl_xor_sync(0xffffffffu, dot[hh], 4);
                dot[hh] += __shfl_xor_sync(0xffffffffu, dot[hh], 2);
                dot[hh] += __shfl_xor_sync(0xffffffffu, dot[hh], 1);
            }
            if (dj == 0) {
                for (int hh = 0; hh < rep; ++hh) sc[hh * kSub + pi_s] = pi_s < np ? dot[hh] : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax update (warp 0: lane = position)
        if (warp == 0) {
            for (int hh = 0; hh < rep; ++hh) {
                const float v = sc[hh * kSub + lane];
                const float mo = runm[hh];
                const float mn = fmaxf(mo, warp_max(v));
                const float pr = (v == -INFINITY) ? 0.f : expf(v - mn);
                const float ps = warp_sum(pr);
                sc[hh * kSub + lane] = pr;
                __syncwarp();
                if (lane == 0) {
                    const float cf = (mo == -INFINITY) ? 0.f : expf(mo - mn);
                    corr[hh] = cf;
                    runm[hh] = mn;
                    runl[hh] = runl[hh] * cf + ps;
                }
                __syncwarp();
            }
        }
        __syncthreads();
        // P V
        {
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                if (hh < rep) {
                    oacc[hh][0] *= corr[hh];
                    oacc[hh][1] *= corr[hh];
                }
            }
            for (int pi = q4 * PPQ; pi < q4 * PPQ + PPQ && pi < np; ++pi) {
                const int pos = pa + pi;
                const uint16_t* vrow = (p.fused && pos == cp) ? vnew : vs + size_t(pi) * D;
                const uint32_t v2 = *reinterpret_cast<const uint32_t*>(vrow + 2 * dp);
                const float v0 = bf16_lo(v2), v1 = bf16_hi(v2);
#pragma unroll
                for (int hh = 0; hh < REP; ++hh) {
                    if (hh < rep) {
                        const float pr = sc[hh * kSub + pi];
                        oacc[hh][0] = fmaf(pr, v0, oacc[hh][0]);
                        oacc[hh][1] = fmaf(pr, v1, oacc[hh][1]);
                    }
                }
            }
        }
        __syncthreads();
        if (tid == 0 && st + kStages < nsub) {
            fence_proxy_async_smem();
            issue(st + kStages);
        }
    }

    // ---- combine the position quarters, then the splits
#pragma unroll
    for (int hh = 0; hh < REP; ++hh) {
        if (hh < rep) {
            opart[(size_t(q4) * kMaxRep + hh) * D + 2 * dp] = oacc[hh][0];
            opart[(size_t(q4) * kMaxRep + hh) * D + 2 * dp + 1] = oacc[hh][1];
        }
    }
    __syncthreads();
    const int rd = rep * D;
    if (ns == 1) {
        for (int i = tid; i < rd; i += kThreads) {
            const int hh = i / D, dim = i % D;
            float o = 0.f;
            for (int q = 0; q < NQ4; ++q) o += opart[(size_t(q) * kMaxRep + hh) * D + dim];
            outrow[i] = o / runl[hh];
        }
        return;
    }
    float* mypart = p.part + ((size_t(b) * p.nkv + h) * p.tsplit + s) * rep * (D + 2);
    for (int i = tid; i < rd; i += kThreads) {
        const int hh = i / D, dim = i % D;
        float o = 0.f;
        for (int q = 0; q < NQ4; ++q) o += opart[(size_t(q) * kMaxRep + hh) * D + dim];
        mypart[hh * (D + 2) + 2 + dim] = o;
    }
    if (tid < rep) {
        mypart[tid * (D + 2)] = runm[tid];
        mypart[tid * (D + 2) + 1] = runl[tid];
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
    const float* parts = p.part + (size_t(b) * p.nkv + h) * p.tsplit * rep * (D + 2);
    for (int i = tid; i < rd; i += kThreads) {
        const int hh = i / D, dim = i % D;
        float mx = -INFINITY;
        for (int q = 0; q < ns; ++q) mx = fmaxf(mx, __ldcg(&parts[(size_t(q) * rep + hh) * (D + 2)]));
        float num = 0.f, den = 0.f;
        for (int q = 0; q < ns; ++q) {
            const float* pq = parts + (size_t(q) * rep + hh) * (D + 2);
            const float w = expf(__ldcg(&pq[0]) - mx);
            den = fmaf(w, __ldcg(&pq[1]), den);
            num = fmaf(w, __ldcg(&pq[2 + dim]), num);
        }
        outrow[i] = num / den;
    }
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
    cfg.gridDim = dim3(p.tsplit, p.nkv, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attn_smem_bytes(p.d, rep);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.d == 64) {
        if (rep == 1) return cudaLaunchKernelEx(&cfg, attn_kernel<64, 1>, p);
        if (rep == 2) return cudaLaunchKernelEx(&cfg, attn_kernel<64, 2>, p);
        return cudaLaunchKernelEx(&cfg, attn_kernel<64, 4>, p);
    }
    if (rep == 1) return cudaLaunchKernelEx(&cfg, attn_kernel<128, 1>, p);
    if (rep == 2) return cudaLaunchKernelEx(&cfg, attn_kernel<128, 2>, p);
    return cudaLaunchKernelEx(&cfg, attn_kernel<128, 4>, p);
}

cudaError_t attn_set_attributes() {
    const int mx = 227 * 1024;
    cudaError_t e;
    const void* ks[6] = {(const void*)attn_kernel<64, 1>, (const void*)attn_kernel<64, 2>,
                         (const void*)attn_kernel<64, 4>, (const void*)attn_kernel<128, 1>,
                         (const void*)attn_kernel<128, 2>, (const void*)attn_kernel<128, 4>};
    for (const void* k : ks) {
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kmr
