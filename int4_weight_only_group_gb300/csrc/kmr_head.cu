// Tied bf16 LM head with the final RMSNorm, greedy argmax and the decode-step
// finalize fused in ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07: lm_head and norms stay bf16; §04 decode: greedy argmax
// stays on the device, per-row EOS flips a finished flag, finished rows are
// padded).
//
// logits[m, v] = sum_k rmsnorm(x[m])[k] * E[v, k]; next[m] = argmax_v (lowest
// index on ties, NaN never wins).  The 622 MB table at vocab 151936 is 43% of
// the step's bytes, so it is streamed once at full bandwidth: a persistent
// grid, each CTA a contiguous range of 8-row tiles moved by cp.async.bulk
// (one copy per row, into rows padded by 16 bytes) into a ring of shared-memory
// stages by a dedicated producer warp that never waits on the previous kernel.
// Eight consumer warps split each tile along K and multiply on the tensor
// cores (mma.m16n8k16, bf16 in, f32 accumulate): the normalised x rows are the
// A operand (up to 16 rows, the rest zero), the tile's 8 vocabulary rows the B
// operand, so a warp spends three instructions per 128 weights at any batch
// size up to 16 and the kernel stays bandwidth-bound; the 16-byte row padding
// makes the fragment loads conflict-free.  The last warp to finish a tile
// (shared-memory counter) sums the eight partials in a fixed order.  The
// logits are never re-read: each warp keeps a running (value, index) best,
// CTAs publish theirs, and the last CTA to finish (global counter) picks the
// winner and advances the step state.
#include "kmr_internal.cuh"

namespace kmr {

namespace {

constexpr int kHeadThreads = kThreads + 32;   // 8 consumer warps + 1 producer warp

__host__ __device__ inline size_t al16h(size_t v) { return (v + 15) & ~size_t(15); }

struct HeadSmem {
    size_t full, empty, xb, red, tsum, cnt, wbv, wbi, red2, flag, stage, total;
};
// Shared-memory row strides (bytes): vocabulary rows and x rows are padded by 16 bytes
// so that the eight rows of a fragment load fall in different banks.
__host__ __device__ inline size_t head_row_bytes(int K) { return size_t(K) * 2 + 16; }
__host__ __device__ inline HeadSmem head_layout(int MB, int K, int nst) {
    HeadSmem L;
    size_t o = 0;
    L.full = o;  o += al16h(size_t(nst) * 8);
    L.empty = o; o += al16h(size_t(nst) * 8);
    L.xb = o;    o += al16h(size_t(MB) * head_row_bytes(K));
    L.red = o;   o += al16h(size_t(nst) * 8 * MB * 8 * 4);      // per stage, per warp: [MB][8] partials
    L.tsum = o;  o += al16h(size_t(nst) * MB * 8 * 4);
    L.cnt = o;   o += al16h(size_t(nst) * 4);
    L.wbv = o;   o += al16h(size_t(8) * MB * 4);
    L.wbi = o;   o += al16h(size_t(8) * MB * 4);
    L.red2 = o;  o += al16h(size_t(MB) * 8 * 4);
    L.flag = o;  o += 16;
    o = (o + 127) & ~size_t(127);
    L.stage = o; o += size_t(nst) * 8 * head_row_bytes(K);
    L.total = o;
    return L;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
    const size_t rs = head_row_bytes(K), tile_bytes = size_t(8) * rs;
    const int xs = int(rs / 2);                  // x row stride in bf16 elements

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
        mbar_arrive_expect_tx(&full[s], uint32_t(rows) * K * 2);
        const uint64_t pol = policy_evict_first();
        for (int r = 0; r < rows; ++r)
            bulk_g2s_stream(stages + size_t(s) * tile_bytes + size_t(r) * rs, p.E + (size_t(t) * 8 + r) * K,
                            uint32_t(K) * 2, &full[s], pol);
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
        // ---- prologue: final RMSNorm of the residual rows, rounded to bf16.  Every row's
        // sum of squares in one pass and one reduce-scatter (the butterfly's bits), so
        // two barriers in all rather than two per row.
        float ss[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) ss[m] = 0.f;
        for (int k = tid; k < K; k += kThreads) {
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                const float v = m < p.M ? p.x[size_t(m) * K + k] : 0.f;
                ss[m] = __fmaf_rn(v, v, ss[m]);
            }
        }
        const float wsum = reduce_scatter<MB>(ss, lane);
        if (lane % (32 / MB) == 0) red2[(lane / (32 / MB)) * 8 + warp] = wsum;
        consumers_sync();
        for (int m = 0; m < MB; ++m) {
            const bool real = m < p.M;
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) tot += red2[m * 8 + w];
            const float r = rsqrtf(tot / float(K) + p.eps);
            for (int k = tid; k < K; k += kThreads) {
                const float v = real ? __fmul_rn(__fmul_rn(p.x[size_t(m) * K + k], r), bf16_to_f32(p.norm_w[k])) : 0.f;
                xb[size_t(m) * xs + k] = f32_to_bf16_rn(v);
            }
        }
        consumers_sync();

        float bv = -INFINITY;
        int bi = 0x7fffffff;
        const int g = lane >> 2, t = lane & 3;
        const int ks_n = K >> 7;                 // 16-wide k-steps in this warp's eighth of K
        const int kbeg = warp * (K >> 3);
        const uint16_t* xg = xb + size_t(g) * xs;
        const uint16_t* xg8 = xb + size_t(g + 8) * xs;
        for (int i = 0; i < nt; ++i) {
            const int s = i % nst;
            mbar_wait(&full[s], uint32_t((i / nst) & 1), p.err);
            const uint8_t* tile = stages + size_t(s) * tile_bytes;
            const uint8_t* brow = tile + size_t(g) * rs;       // vocabulary row g of the tile (B column g)
            float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            auto kstep = [&](float (&dd)[4], int ks) {
                const int k0 = kbeg + ks * 16 + 2 * t;
                uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
                if (g < MB) {
                    a0 = *reinterpret_cast<const uint32_t*>(xg + k0);
                    a2 = *reinterpret_cast<const uint32_t*>(xg + k0 + 8);
                }
                if (MB > 8 && g + 8 < MB) {
                    a1 = *reinterpret_cast<const uint32_t*>(xg8 + k0);
                    a3 = *reinterpret_cast<const uint32_t*>(xg8 + k0 + 8);
                }
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(brow + size_t(k0) * 2);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(brow + size_t(k0 + 8) * 2);
                mma_bf16_16816(dd, a0, a1, a2, a3, b0, b1);
            };
            int ks = 0;
            for (; ks + 1 < ks_n; ks += 2) {     // two accumulator chains
                kstep(d[0], ks);
                kstep(d[1], ks + 1);
            }
            if (ks < ks_n) kstep(d[0], ks);
            // this warp's partials: rows g, g+8 of x, vocabulary rows 2t, 2t+1 of the tile
            float* rp = red + (size_t(s) * 8 + warp) * MB * 8;
            if (g < MB) {
                rp[g * 8 + 2 * t] = __fadd_rn(d[0][0], d[1][0]);
                rp[g * 8 + 2 * t + 1] = __fadd_rn(d[0][1], d[1][1]);
            }
            if (MB > 8 && g + 8 < MB) {
                rp[(g + 8) * 8 + 2 * t] = __fadd_rn(d[0][2], d[1][2]);
                rp[(g + 8) * 8 + 2 * t + 1] = __fadd_rn(d[0][3], d[1][3]);
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
                    const int m = idx >> 3, r = idx & 7;
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) v = __fadd_rn(v, red[((size_t(s) * 8 + w) * MB + m) * 8 + r]);
                    tsum[(size_t(s) * MB + m) * 8 + r] = v;
                    const int n = tbase + r;
                    if (p.logits && m < p.M && n < p.V) p.logits[size_t(m) * p.ldl + n] = v;
                }
                __syncwarp();
                if (lane < MB) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int n = tbase + r;
                        if (n >= p.V) break;
                        float v = tsum[(size_t(s) * MB + lane) * 8 + r];
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
        case 8: return launch_head_mb<8>(p, grid, st, pdl);
        default: return launch_head_mb<16>(p, grid, st, pdl);
    }
}
int head_pick_mb(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

cudaError_t head_set_attributes() {
    const int mx = 227 * 1024;
    const void* ks[5] = {(const void*)head_kernel<1>, (const void*)head_kernel<2>, (const void*)head_kernel<4>,
                         (const void*)head_kernel<8>, (const void*)head_kernel<16>};
    for (const void* k : ks) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kmr
