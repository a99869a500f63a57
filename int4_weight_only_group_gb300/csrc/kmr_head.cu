// Tied bf16 LM head with the final RMSNorm, greedy argmax and the decode-step
// finalize fused in ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07: lm_head and norms stay bf16; §04 decode: greedy argmax
// stays on the device, per-row EOS flips a finished flag, finished rows are
// padded).
//
// logits[m, v] = sum_k rmsnorm(x[m])[k] * E[v, k]; next[m] = argmax_v (lowest
// index on ties, NaN never wins).  The 622 MB table at vocab 151936 is 43% of
// the step's bytes, so it is streamed once at full bandwidth: a persistent
// grid, each CTA a contiguous range of 8-row tiles moved by cp.async.bulk into
// a ring of shared-memory stages by a dedicated producer warp that never waits
// on the previous kernel.  Eight consumer warps split each tile along K; the
// last warp to finish a tile (shared-memory counter) sums the eight partials
// in a fixed order.  The logits are never re-read: each warp keeps a running
// (value, index) best, CTAs publish theirs, and the last CTA to finish
// (global counter) picks the winner and advances the step state.
#include "kmr_internal.cuh"

namespace kmr {

namespace {

constexpr int kHeadThreads = kThreads + 32;   // 8 consumer warps + 1 producer warp

__host__ __device__ inline size_t al16h(size_t v) { return (v + 15) & ~size_t(15); }

struct HeadSmem {
    size_t full, empty, xb, red, tsum, cnt, wbv, wbi, red2, flag, stage, total;
};
__host__ __device__ inline HeadSmem head_layout(int MB, int K, int nst) {
    HeadSmem L;
    size_t o = 0;
    L.full = o;  o += al16h(size_t(nst) * 8);
    L.empty = o; o += al16h(size_t(nst) * 8);
    L.xb = o;    o += al16h(size_t(MB) * K * 2);
    L.red = o;   o += al16h(size_t(nst) * 8 * 8 * MB * 4);
    L.tsum = o;  o += al16h(size_t(nst) * 8 * MB * 4);
    L.cnt = o;   o += al16h(size_t(nst) * 4);
    L.wbv = o;   o += al16h(size_t(8) * MB * 4);
    L.wbi = o;   o += al16h(size_t(8) * MB * 4);
    L.red2 = o;  o += al16h(size_t(8) * 4);
    L.flag = o;  o += 16;
    o = (o + 127) & ~size_t(127);
    L.stage = o; o += size_t(nst) * 8 * K * 2;
    L.total = o;
    return L;
}

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int MB>
__global__ void __launch_bounds__(kHeadThreads, 1) head_kernel(const HeadParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = gridDim.x, c = blockIdx.x, K = p.K, nst = p.nstage;
    const int t0 = int((long long)c * p.tiles / P), t1 = int((long long)(c + 1) * p.tiles / P);
    const int nt = t1 - t0;
    const HeadSmem L = head_layout(MB, K, nst);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.xb);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* tsum = reinterpret_cast<float*>(smem + L.tsum);
    int* cnt = reinterpret_cast<int*>(smem + L.cnt);
    float* wbv = reinterpret_cast<float*>(smem + L.wbv);
    int* wbi = reinterpret_cast<int*>(smem + L.wbi);
    float* red2 = reinterpret_cast<float*>(smem + L.red2);
    int* flag = reinterpret_cast<int*>(smem + L.flag);
    uint8_t* stages = smem + L.stage;
    const size_t tile_bytes = size_t(8) * K * 2;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 8);
            cnt[s] = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int i) {
        const int s = i % nst, t = t0 + i;
        const int rows = min(8, p.V - t * 8);
        const uint32_t bytes = uint32_t(rows) * K * 2;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_stream(stages + size_t(s) * tile_bytes, p.E + size_t(t) * 8 * K, bytes, &full[s],
                        policy_evict_first());
    };

    if (warp == 8) {
        // ---- producer: needs nothing from the previous kernel, so it never waits on it
        if (lane == 0) {
            const int n0 = nt < nst ? nt : nst;
            for (int i = 0; i < n0; ++i) issue(i);
        }
        pdl_launch_dependents();
        if (lane == 0) {
            for (int i = nst; i < nt; ++i) {
                mbar_wait(&empty[i % nst], uint32_t(((i / nst) - 1) & 1), p.err);
                issue(i);
            }
        }
    } else {
        pdl_launch_dependents();
        pdl_wait();
        // ---- prologue: final RMSNorm of the residual rows, rounded to bf16
        for (int m = 0; m < MB; ++m) {
            const bool real = m < p.M;
            float ss = 0.f;
            for (int k = tid; k < K; k += kThreads) {
                const float v = real ? p.x[size_t(m) * K + k] : 0.f;
                ss = __fmaf_rn(v, v, ss);
            }
            ss = warp_sum(ss);
            consumers_sync();
            if (lane == 0) red2[warp] = ss;
            consumers_sync();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) tot += red2[w];
            const float r = rsqrtf(tot / float(K) + p.eps);
            for (int k = tid; k < K; k += kThreads) {
                const float v = real ? __fmul_rn(__fmul_rn(p.x[size_t(m) * K + k], r), bf16_to_f32(p.norm_w[k])) : 0.f;
                xb[size_t(m) * K + k] = f32_to_bf16_rn(v);
            }
        }
        consumers_sync();

        float bv = -INFINITY;
        int bi = 0x7fffffff;
        const int cpw = K >> 6;   // 8-element chunks per warp per row
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
        const int row = (lane >> 2) & 7;
        for (int i = 0; i < nt; ++i) {
            const int s = i % nst;
            mbar_wait(&full[s], uint32_t((i / nst) & 1), p.err);
            const uint16_t* tile = reinterpret_cast<const uint16_t*>(stages + size_t(s) * tile_bytes);
            float acc[8][MB];
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int m = 0; m < MB; ++m) acc[r][m] = 0.f;
            for (int cc = lane; cc < cpw; cc += 32) {
                const int k0 = warp * (K >> 3) + cc * 8;
                uint4 xv[MB];
#pragma unroll
                for (int m = 0; m < MB; ++m) xv[m] = *reinterpret_cast<const uint4*>(xb + size_t(m) * K + k0);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(tile + size_t(r) * K + k0);
#pragma unroll
                    for (int m = 0; m < MB; ++m) {
                        fma_bf16x2_f32(acc[r][m], wv.x, xv[m].x);
                        fma_bf16x2_f32(acc[r][m], wv.y, xv[m].y);
                        fma_bf16x2_f32(acc[r][m], wv.z, xv[m].z);
                        fma_bf16x2_f32(acc[r][m], wv.w, xv[m].w);
                    }
                }
            }
            // reduce-scatter over lanes: lane l keeps row (l >> 2) & 7
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                float a[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float keep = b4 ? acc[q + 4][m] : acc[q][m];
                    const float send = b4 ? acc[q][m] : acc[q + 4][m];
                    a[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
                float cc2[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float keep = b3 ? a[q + 2] : a[q];
                    const float send = b3 ? a[q] : a[q + 2];
                    cc2[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                float e = (b2 ? cc2[1] : cc2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? cc2[0] : cc2[1], 4);
                e += __shfl_xor_sync(0xffffffffu, e, 2);
                e += __shfl_xor_sync(0xffffffffu, e, 1);
                if ((lane & 3) == 0) red[((size_t(s) * 8 + warp) * 8 + row) * MB + m] = e;
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&cnt[s], 1) == 7;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence_block();
                const int tbase = (t0 + i) * 8;
                for (int idx = lane; idx < 8 * MB; idx += 32) {
                    const int r = idx / MB, m = idx % MB;
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) v += red[((size_t(s) * 8 + w) * 8 + r) * MB + m];
                    tsum[(size_t(s) * 8 + r) * MB + m] = v;
                    const int n = tbase + r;
                    if (p.logits && m < p.M && n < p.V) p.logits[size_t(m) * p.ldl + n] = v;
                }
                __syncwarp();
                if (lane < MB) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int n = tbase + r;
                        if (n >= p.V) break;
                        float v = tsum[(size_t(s) * 8 + r) * MB + lane];
                        if (v != v) v = -INFINITY;
                        if (better(v, n, bv, bi)) { bv = v; bi = n; }
                    }
                }
                if (lane == 0) cnt[s] = 0;
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (lane < MB) {
            wbv[warp * MB + lane] = bv;
            wbi[warp * MB + lane] = bi;
        }
    }
    __syncthreads();
    // ---- CTA winner per row, then the grid winner by the last CTA to finish
    if (tid < MB) {
        float v = wbv[tid];
        int ix = wbi[tid];
        for (int w = 1; w < 8; ++w)
            if (better(wbv[w * MB + tid], wbi[w * MB + tid], v, ix)) { v = wbv[w * MB + tid]; ix = wbi[w * MB + tid]; }
        p.gbest_val[size_t(c) * MB + tid] = v;
        p.gbest_idx[size_t(c) * MB + tid] = ix;
        __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(p.counter, 1);
        flag[0] = (old == P - 1);
        if (old == P - 1) {
            *p.counter = 0;
            __threadfence();
        }
    }
    __syncthreads();
    if (!flag[0] || tid >= p.M) return;
    float v = -INFINITY;
    int ix = 0x7fffffff;
    for (int cc = 0; cc < P; ++cc) {
        const float cv = __ldcg(&p.gbest_val[size_t(cc) * MB + tid]);
        const int ci = __ldcg(&p.gbest_idx[size_t(cc) * MB + tid]);
        if (better(cv, ci, v, ix)) { v = cv; ix = ci; }
    }
    if (ix == 0x7fffffff) ix = 0;
    // ---- finalize: emit, pad, advance ("kaminari", §04 decode)
    const int m = tid;
    if (p.finished[m]) {
        p.tokens[m] = p.pad;
    } else {
        p.tokens[m] = ix;
        const int cp = p.cpos[m] + 1;
        p.cpos[m] = cp;
        p.positions[m] += 1;
        p.positions[p.pos_ld + m] += 1;
        p.positions[2 * p.pos_ld + m] += 1;
        if (ix == p.eos || cp >= p.max_len) p.finished[m] = 1;
    }
}

}  // namespace

size_t head_smem_bytes(int MB, int K, int nstage) { return head_layout(MB, K, nstage).total; }

template <int MB>
static cudaError_t launch_head_mb(const HeadParams& p, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kHeadThreads);
    cfg.dynamicSmemBytes = head_smem_bytes(MB, p.K, p.nstage);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, head_kernel<MB>, p);
}

cudaError_t launch_head(const HeadParams& p, int MB, int grid, cudaStream_t st, bool pdl) {
    switch (MB) {
        case 1: return launch_head_mb<1>(p, grid, st, pdl);
        case 2: return launch_head_mb<2>(p, grid, st, pdl);
        case 4: return launch_head_mb<4>(p, grid, st, pdl);
        default: return launch_head_mb<8>(p, grid, st, pdl);
    }
}

cudaError_t head_set_attributes() {
    const int mx = 227 * 1024;
    const void* ks[4] = {(const void*)head_kernel<1>, (const void*)head_kernel<2>, (const void*)head_kernel<4>,
                         (const void*)head_kernel<8>};
    for (const void* k : ks) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kmr
