// Dequant-fused int4 weight-only GEMV / skinny GEMM (up to 8 rows of x per pass).
//
// What it computes ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07 int4 sidecar quantization; group 128 along K):
//     y[m, n] = sum_k x[m, k] * ((q[n, k] - 8) * s[n, k/128] + z[n, k/128])
// optionally after an RMSNorm of x (prologue) and followed by a store, a
// residual add or SiLU(gate) * up (epilogue).
//
// GB300 design
//   * HBM-bound: every packed byte is read once.  A CTA owns whole 16-row
//     tiles (no cross-CTA reduction, no global scratch) and pulls them with
//     cp.async.bulk into a shared-memory ring whose first fill is issued
//     BEFORE griddepcontrol.wait: under programmatic dependent launch a kernel
//     streams its weights while the previous kernel of the step finishes.
//   * Issue-rate bound on CUDA cores: at GB300's ~47 int4 weights per SM-clock
//     a float FMA per weight plus the unpacking would exceed the SM's issue
//     rate (2+ instructions per weight at batch 1, 4+ at batch 4).  The
//     multiply-adds therefore go to the tensor cores (mma.m16n8k16, f16 in,
//     f32 accumulate, the 16 rows of a tile as M and the batch rows as N) and
//     the threads only unpack: the KMR4 layout stores each lane's A fragment
//     of one 16x16 block in one 32-bit word, so 8 weights cost one shift and
//     four LOP3s.  OR-ing a nibble into the mantissa of fp16 1024.0 gives
//     1024 + q exactly (1024 + 16q for rows 8..15, whose nibble sits one
//     position higher); the offset, the -8 and the zero point are folded in
//     once per group with the group sums X of x:
//         y = s * (D - 1024 X) / c + (z - 8 s) X,   c = 1 or 16 per row.
//   * x is staged once per CTA in shared memory as fp16, scaled per row by a
//     power of two (exact) so its largest magnitude sits below 2^13, in the
//     order of the B fragments.
//   * Deterministic and batch invariant: fixed k order inside the mma, fixed
//     group order per warp, fixed warp order in the tile sum; a row's result
//     never depends on the other rows or on M.
#include <cuda_fp16.h>

#include "kmr_internal.cuh"

namespace kmr {

namespace {

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

struct GemvSmem {
    size_t bar, xh, xs, isig, red, part, stage, total;
};
// xh: MB rows of (K + 8) halves; xs: [groups][8] group sums; part: [nst][8 warps][16 rows][8 cols]
__host__ __device__ inline GemvSmem gemv_layout(int MB, int K, int tile_bytes, int nst) {
    GemvSmem L;
    size_t o = 0;
    L.bar = o;   o += al16(size_t(nst) * 8);
    L.xh = o;    o += al16(size_t(MB) * (K + 8) * 2);
    L.xs = o;    o += al16(size_t(K / 128) * 8 * 4);
    L.isig = o;  o += al16(size_t(8) * 4);
    L.red = o;   o += al16(size_t(2) * 8 * 4);
    L.part = o;  o += al16(size_t(nst) * 8 * 128 * 4);
    o = (o + 127) & ~size_t(127);
    L.stage = o; o += size_t(nst) * tile_bytes;
    L.total = o;
    return L;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position (in halves, within a row of x') of input k in B-fragment order: blocks of
// 64 inputs; inside a block, lane slot t (16 halves) holds, for each of the 4 k-steps
// k0 = 64*block + 16*step, the inputs (k0+2t, k0+2t+1, k0+2t+8, k0+2t+9).
__device__ __forceinline__ int xpos(int k) {
    const int kk = k & 15;
    return (k >> 6) * 64 + ((kk & 7) >> 1) * 16 + ((k >> 4) & 3) * 4 + (kk >> 3) * 2 + (kk & 1);
}

template <int MB>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = gridDim.x, c = blockIdx.x;
    const int t0 = int((long long)c * p.tiles / P), t1 = int((long long)(c + 1) * p.tiles / P);
    const int nt = t1 - t0;
    const int K = p.K, G = K >> 7, tb = p.tile_bytes, nst = p.nstage;
    const GemvSmem L = gemv_layout(MB, K, tb, nst);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    __half* xh = reinterpret_cast<__half*>(smem + L.xh);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* isig = reinterpret_cast<float*>(smem + L.isig);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint8_t* stages = smem + L.stage;

    // ---- weight ring: first fill before waiting on the previous kernel
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = policy_evict_first();
        const int n0 = nt < nst ? nt : nst;
        for (int i = 0; i < n0; ++i) {
            mbar_arrive_expect_tx(&bar[i], tb);
            bulk_g2s_stream(stages + size_t(i) * tb, p.w + size_t(t0 + i) * tb, tb, &bar[i], pol);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // ---- prologue: x rows -> (RMSNorm) -> fp16 (scaled) in B-fragment order, group sums
    const int segs = K >> 3;
    const int nit = (segs + kThreads - 1) / kThreads;   // <= 4 (K <= 8192)
    const bool norm = p.in_kind != IN_F32;
    for (int i = tid; i < G * (8 - MB); i += kThreads) xs[(i / (8 - MB)) * 8 + MB + i % (8 - MB)] = 0.f;
    for (int m = 0; m < MB; ++m) {
        if (m >= p.M) {
            for (int i = tid; i < G; i += kThreads) xs[i * 8 + m] = 0.f;
            continue;
        }
        float v[4][8];
        float ss = 0.f, amax = 0.f;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int sg = it * kThreads + tid;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[it][e] = 0.f;
            if (it < nit && sg < segs) {
                if (p.in_kind == IN_EMBED_NORM) {
                    int tok = p.tokens[m];
                    if (tok < 0 || tok >= p.vocab) {
                        if (sg == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
                        tok = 0;
                    }
                    const uint4 raw = *reinterpret_cast<const uint4*>(p.embed + size_t(tok) * K + size_t(sg) * 8);
                    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[it][2 * e] = bf16_lo(rw[e]);
                        v[it][2 * e + 1] = bf16_hi(rw[e]);
                    }
                    if (c == 0 && p.x_out) {
                        float4* xo = reinterpret_cast<float4*>(p.x_out + size_t(m) * K + size_t(sg) * 8);
                        xo[0] = make_float4(v[it][0], v[it][1], v[it][2], v[it][3]);
                        xo[1] = make_float4(v[it][4], v[it][5], v[it][6], v[it][7]);
                    }
                } else {
                    const float4* xp = reinterpret_cast<const float4*>(p.x + size_t(m) * K + size_t(sg) * 8);
                    const float4 a = xp[0], b = xp[1];
                    v[it][0] = a.x; v[it][1] = a.y; v[it][2] = a.z; v[it][3] = a.w;
                    v[it][4] = b.x; v[it][5] = b.y; v[it][6] = b.z; v[it][7] = b.w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ss = __fmaf_rn(v[it][e], v[it][e], ss);
                    if (norm) v[it][e] = __fmul_rn(v[it][e], bf16_to_f32(p.norm_w[sg * 8 + e]));
                    amax = fmaxf(amax, fabsf(v[it][e]));
                }
            }
        }
        // one block reduction for both the sum of squares and the largest |x * w|
        ss = warp_sum(ss);
        amax = warp_max(amax);
        if (lane == 0) {
            red[warp] = ss;
            red[8 + warp] = amax;
        }
        __syncthreads();
        float tot = 0.f, mx = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            tot += red[i];
            mx = fmaxf(mx, red[8 + i]);
        }
        __syncthreads();
        const float r = norm ? rsqrtf(tot / float(K) + p.eps) : 1.f;
        if (norm) mx = __fmul_rn(mx, r);
        float sigma = 1.f;
        if (mx > 0.f && mx < 3.0e38f) {
            int ex;
            frexpf(mx, &ex);                       // mx < 2^ex
            sigma = ldexpf(1.f, max(-100, min(100, 13 - ex)));
        }
        __half* xrow = xh + size_t(m) * (K + 8);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            if (it >= nit) break;
            const int sg = it * kThreads + tid;
            float gs = 0.f;
            if (sg < segs) {
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    // (x * r) * w, then the exact power-of-two scale
                    const float f0 = norm ? __fmul_rn(v[it][e], r) : v[it][e];
                    const float f1 = norm ? __fmul_rn(v[it][e + 1], r) : v[it][e + 1];
                    const __half a = __float2half_rn(__fmul_rn(f0, sigma));
                    const __half b = __float2half_rn(__fmul_rn(f1, sigma));
                    gs = __fadd_rn(gs, __fadd_rn(__half2float(a), __half2float(b)));
                    *reinterpret_cast<__half2*>(xrow + xpos(sg * 8 + e)) = __halves2half2(a, b);
                }
            }
            // 16 consecutive threads cover one group of 128 inputs
            gs += __shfl_xor_sync(0xffffffffu, gs, 1);
            gs += __shfl_xor_sync(0xffffffffu, gs, 2);
            gs += __shfl_xor_sync(0xffffffffu, gs, 4);
            gs += __shfl_xor_sync(0xffffffffu, gs, 8);
            if ((tid & 15) == 0 && sg < segs) xs[(sg >> 4) * 8 + m] = gs;
        }
        if (tid == 0) isig[m] = 1.f / sigma;
    }
    __syncthreads();

    // ---- main loop: all warps on one tile at a time; warp w takes groups w, w+8, ...
    const int g = lane >> 2, t = lane & 3;
    const bool bload = g < p.M;
    const __half* xrow = xh + size_t(bload ? g : 0) * (K + 8);
    for (int i = 0; i < nt; ++i) {
        const int s = i % nst;
        mbar_wait(&bar[s], uint32_t((i / nst) & 1), p.err);
        const uint8_t* st = stages + size_t(s) * tb;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int grp = warp; grp < G; grp += 8) {
            const uint8_t* gb = st + size_t(grp) * 1088;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                const uint4 wq = *reinterpret_cast<const uint4*>(gb + blk * 512 + lane * 16);
                uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
                if (bload) {
                    const uint4* xp = reinterpret_cast<const uint4*>(xrow + (grp * 2 + blk) * 64 + t * 16);
                    xa = xp[0];
                    xb = xp[1];
                }
                const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
                const uint32_t bx[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t w = w4[ks], w2 = w >> 8;
                    mma16816(d, and_or(w, 0x000F000Fu, 0x64006400u), and_or(w, 0x00F000F0u, 0x64006400u),
                             and_or(w2, 0x000F000Fu, 0x64006400u), and_or(w2, 0x00F000F0u, 0x64006400u),
                             bx[2 * ks], bx[2 * ks + 1]);
                }
            }
            // fold offset, -8 and zero point: rows g (x1) and g+8 (x16), batch cols 2t, 2t+1
            const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(gb + 1024 + g * 4);
            const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(gb + 1024 + (g + 8) * 4);
            const float2 X = *reinterpret_cast<const float2*>(xs + grp * 8 + 2 * t);
            const float s0 = bf16_lo(sz0), z0 = bf16_hi(sz0), s1 = bf16_lo(sz1), z1 = bf16_hi(sz1);
            const float s1c = __fmul_rn(s1, 0.0625f);
            const float zz0 = __fmaf_rn(-8.f, s0, z0), zz1 = __fmaf_rn(-8.f, s1, z1);
            const float x0 = 1024.f * X.x, x1 = 1024.f * X.y;
            acc[0] = __fadd_rn(acc[0], __fmaf_rn(s0, __fsub_rn(d[0], x0), __fmul_rn(zz0, X.x)));
            acc[1] = __fadd_rn(acc[1], __fmaf_rn(s0, __fsub_rn(d[1], x1), __fmul_rn(zz0, X.y)));
            acc[2] = __fadd_rn(acc[2], __fmaf_rn(s1c, __fsub_rn(d[2], x0), __fmul_rn(zz1, X.x)));
            acc[3] = __fadd_rn(acc[3], __fmaf_rn(s1c, __fsub_rn(d[3], x1), __fmul_rn(zz1, X.y)));
        }
        float* wp = part + (size_t(s) * 8 + warp) * 128;
        wp[g * 8 + 2 * t] = acc[0];
        wp[g * 8 + 2 * t + 1] = acc[1];
        wp[(g + 8) * 8 + 2 * t] = acc[2];
        wp[(g + 8) * 8 + 2 * t + 1] = acc[3];
        __syncthreads();
        // stage s is free again: refill it with tile i + nst while the epilogue runs
        if (tid == 0 && i + nst < nt) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[s], tb);
            bulk_g2s_stream(stages + size_t(s) * tb, p.w + size_t(t0 + i + nst) * tb, tb, &bar[s],
                            policy_evict_first());
        }
        // ---- epilogue: fixed-order sum over the 8 warps
        const int tile = t0 + i;
        const float* ps = part + size_t(s) * 8 * 128;
        if (p.epi == EPI_SILU) {
            if (tid < 8 * MB) {
                const int j = tid / MB, m = tid % MB;
                const int jj = tile * 8 + j;
                if (m < p.M && jj < p.N / 2) {
                    float gv = 0.f, uv = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        gv = __fadd_rn(gv, ps[w * 128 + j * 8 + m]);
                        uv = __fadd_rn(uv, ps[w * 128 + (j + 8) * 8 + m]);
                    }
                    gv = __fmul_rn(gv, isig[m]);
                    uv = __fmul_rn(uv, isig[m]);
                    p.y[size_t(m) * p.ldy + jj] = __fmul_rn(__fdiv_rn(gv, __fadd_rn(1.f, expf(-gv))), uv);
                }
            }
        } else if (tid < 16 * MB) {
            const int r = tid / MB, m = tid % MB;
            const int n = tile * 16 + r;
            if (m < p.M && n < p.N) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) v = __fadd_rn(v, ps[w * 128 + r * 8 + m]);
                v = __fmul_rn(v, isig[m]);
                float* yp = p.y + size_t(m) * p.ldy + n;
                *yp = (p.epi == EPI_RESID) ? __fadd_rn(*yp, v) : v;
            }
        }
    }
}

}  // namespace

int gemv_pick_mb(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// At most one CTA per SM, each owning ceil(tiles / SMs) whole tiles (the last
// CTA may own fewer), never more CTAs than tiles.
int gemv_grid(int tiles, int sms) {
    if (sms < 1) sms = 1;
    const int tpc = (tiles + sms - 1) / sms;
    const int g = (tiles + tpc - 1) / tpc;
    return g < 1 ? 1 : g;
}
int gemv_nstage(int tiles, int grid, int tile_bytes) {
    const int tpc = (tiles + grid - 1) / grid;
    int cap = (104 * 1024) / tile_bytes;
    if (cap < 2) cap = 2;
    const int n = tpc < cap ? tpc : cap;
    return n < 1 ? 1 : n;
}
size_t gemv_smem_bytes(int MB, int K, int tile_bytes, int nstage) {
    return gemv_layout(MB, K, tile_bytes, nstage).total;
}

template <int MB>
static cudaError_t launch_mb(const GemvParams& p, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes(MB, p.K, p.tile_bytes, p.nstage);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MB>, p);
}

cudaError_t launch_gemv(const GemvParams& p, int MB, int grid, cudaStream_t st, bool pdl) {
    switch (MB) {
        case 1: return launch_mb<1>(p, grid, st, pdl);
        case 2: return launch_mb<2>(p, grid, st, pdl);
        case 4: return launch_mb<4>(p, grid, st, pdl);
        default: return launch_mb<8>(p, grid, st, pdl);
    }
}

cudaError_t gemv_set_attributes() {
    const int mx = 227 * 1024;
    const void* ks[4] = {(const void*)gemv_kernel<1>, (const void*)gemv_kernel<2>, (const void*)gemv_kernel<4>,
                         (const void*)gemv_kernel<8>};
    for (const void* k : ks) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kmr
