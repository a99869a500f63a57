// Dequant-fused int4 weight-only GEMV / skinny GEMM (M <= 8 rows per pass).
//
// What it computes ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07 int4 sidecar quantization; group 128 along K):
//     y[m, n] = sum_k x[m, k] * ((q[n, k] - 8) * s[n, k/128] + z[n, k/128])
// optionally after an RMSNorm of x (prologue) and followed by a store, a
// residual add or SiLU(gate) * up (epilogue).
//
// GB300 design
//   * HBM-bound: every packed byte is read exactly once.  The matrix is a
//     sequence of equal units (8 rows x one K-slice, KMR4 layout); a
//     persistent grid of one CTA per SM takes an equal, contiguous unit range
//     (stream-K), so small-N matrices still spread over all 152 SMs.
//   * Weights move with cp.async.bulk into a shared-memory ring.  The first
//     ring fill is issued BEFORE griddepcontrol.wait, so with programmatic
//     dependent launch a kernel streams its weights while the previous kernel
//     of the decode step is still finishing.
//   * Dequantisation is magic-number based: a nibble OR'd into the mantissa of
//     fp16 1024.0 gives 1024 + q exactly (or 1024 + 16q for the nibble one
//     position higher, compensated by pre-scaling that x by 1/16).  The f16
//     products accumulate in f32 (fma.rn.f32.f16); the 1024 offset, the -8
//     and the zero point are folded in once per 32-input chunk using the
//     chunk sums of x:  y = s * (D - 1024 * X') + (z - 8 s) * X.
//   * x is staged once per CTA in shared memory as fp16 scaled by a per-row
//     power of two (exact) so its largest magnitude sits below 2^14.
//   * Deterministic: fixed-order warp reduce-scatter, fixed-order sums over
//     units, and a last-arriver (atomic counter, no float atomics) combine for
//     tiles split between CTAs.  No result depends on M or on other rows.
#include <cuda_fp16.h>

#include "kmr_internal.cuh"

namespace kmr {

namespace {

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

struct GemvSmem {
    size_t bar, xh, xs1, xs2, isig, red, upart, tval, flags, stage, total;
};
__host__ __device__ inline GemvSmem gemv_layout(int MB, int K, int ub, int nst, int upc) {
    GemvSmem L;
    size_t o = 0;
    L.bar = o;   o += al16(size_t(nst) * 8);
    L.xh = o;    o += al16(size_t(MB) * K * 2);
    L.xs1 = o;   o += al16(size_t(MB) * (K / 32) * 4);
    L.xs2 = o;   o += al16(size_t(MB) * (K / 32) * 4);
    L.isig = o;  o += al16(size_t(MB) * 4);
    L.red = o;   o += al16(size_t(2) * 8 * 4);
    L.upart = o; o += al16(size_t(upc) * 8 * MB * 4);
    L.tval = o;  o += al16(size_t(upc + 2) * 8 * MB * 4);
    L.flags = o; o += 16;
    o = (o + 127) & ~size_t(127);
    L.stage = o; o += size_t(nst) * ub;
    L.total = o;
    return L;
}

__device__ __forceinline__ long long unit_start(int c, int U, int P) { return (long long)c * U / P; }
__device__ __forceinline__ int unit_owner(long long u, int U, int P) {
    return int(((u + 1) * (long long)P - 1) / U);
}

// Block-wide sum / max over 256 threads through `red` (8 floats); all threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) r += red[i];
    return r;
}
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[8 + w] = v;
    __syncthreads();
    float r = red[8];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[8 + i]);
    return r;
}

// One 32-bit word of 8 nibbles (KMR4 bit order) against 4 fp16 pairs of x.
template <int MB>
__device__ __forceinline__ void dot_word(float (&D)[MB], uint32_t w, const uint32_t (*xr)[16], int j) {
    const uint32_t w2 = w >> 8;
    const uint32_t h0 = and_or(w, 0x000F000Fu, 0x64006400u);    // 1024 + q  (k+0, k+1)
    const uint32_t h1 = and_or(w, 0x00F000F0u, 0x64006400u);    // 1024 + 16q (k+2, k+3)
    const uint32_t h2 = and_or(w2, 0x000F000Fu, 0x64006400u);   // 1024 + q  (k+4, k+5)
    const uint32_t h3 = and_or(w2, 0x00F000F0u, 0x64006400u);   // 1024 + 16q (k+6, k+7)
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        fma_f16x2_f32(D[m], h0, xr[m][4 * j + 0]);
        fma_f16x2_f32(D[m], h1, xr[m][4 * j + 1]);
        fma_f16x2_f32(D[m], h2, xr[m][4 * j + 2]);
        fma_f16x2_f32(D[m], h3, xr[m][4 * j + 3]);
    }
}

template <int MB>
__global__ void __launch_bounds__(kThreads, (MB <= 4 ? 2 : 1)) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int U = p.units, P = gridDim.x, c = blockIdx.x;
    const int u0 = int(unit_start(c, U, P)), u1 = int(unit_start(c + 1, U, P));
    const int nu = u1 - u0;
    const int ub = p.unit_bytes, nst = p.nstage, K = p.K, ksl = p.ksl;
    const int upc = (U + P - 1) / P;
    const GemvSmem L = gemv_layout(MB, K, ub, nst, upc);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    __half* xh = reinterpret_cast<__half*>(smem + L.xh);
    float* xs1 = reinterpret_cast<float*>(smem + L.xs1);
    float* xs2 = reinterpret_cast<float*>(smem + L.xs2);
    float* isig = reinterpret_cast<float*>(smem + L.isig);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* upart = reinterpret_cast<float*>(smem + L.upart);
    float* tval = reinterpret_cast<float*>(smem + L.tval);
    int* flags = reinterpret_cast<int*>(smem + L.flags);
    uint8_t* stages = smem + L.stage;

    // ---- weight ring: first fill before waiting on the previous kernel
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = policy_evict_first();
        const int n0 = nu < nst ? nu : nst;
        for (int i = 0; i < n0; ++i) {
            mbar_arrive_expect_tx(&bar[i], ub);
            bulk_g2s_stream(stages + size_t(i) * ub, p.w + size_t(u0 + i) * ub, ub, &bar[i], pol);
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // ---- prologue: x rows -> (RMSNorm) -> fp16, scaled, with chunk sums
    const int segs = K >> 3;
    const int nit = (segs + kThreads - 1) / kThreads;   // <= 4 (K <= 8192)
    const bool norm = p.in_kind != IN_F32;
    for (int m = 0; m < MB; ++m) {
        const bool real = m < p.M;
        float v[4][8];
        float ss = 0.f;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int sg = it * kThreads + tid;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[it][e] = 0.f;
            if (it < nit && sg < segs && real) {
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
                for (int e = 0; e < 8; ++e) ss = __fmaf_rn(v[it][e], v[it][e], ss);
            }
        }
        float r = 1.f;
        if (norm) r = rsqrtf(block_sum(ss, red) / float(K) + p.eps);
        float amax = 0.f;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int sg = it * kThreads + tid;
            if (it < nit && sg < segs) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float h = v[it][e];
                    if (norm) h = __fmul_rn(__fmul_rn(h, r), bf16_to_f32(p.norm_w[sg * 8 + e]));
                    v[it][e] = h;
                    amax = fmaxf(amax, fabsf(h));
                }
            }
        }
        amax = block_max(amax, red);
        float sigma = 1.f;
        if (amax > 0.f && amax < 3.0e38f) {
            int ex;
            frexpf(amax, &ex);            // amax < 2^ex
            sigma = ldexpf(1.f, max(-100, min(100, 14 - ex)));
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            if (it >= nit) break;
            const int sg = it * kThreads + tid;
            float s1 = 0.f, s2 = 0.f;
            if (sg < segs) {
                uint32_t hp[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float f0 = __fmul_rn(__fmul_rn(v[it][e], sigma), (e & 2) ? 0.0625f : 1.f);
                    const float f1 = __fmul_rn(__fmul_rn(v[it][e + 1], sigma), (e & 2) ? 0.0625f : 1.f);
                    const __half a = __float2half_rn(f0), b = __float2half_rn(f1);
                    const float ra = __half2float(a), rb = __half2float(b);
                    const float pr = __fadd_rn(ra, rb);
                    s1 = __fadd_rn(s1, pr);
                    s2 = __fadd_rn(s2, (e & 2) ? __fmul_rn(16.f, pr) : pr);
                    hp[e >> 1] = uint32_t(__half_as_ushort(a)) | (uint32_t(__half_as_ushort(b)) << 16);
                }
                *reinterpret_cast<uint4*>(xh + size_t(m) * K + size_t(sg) * 8) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
            }
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
            if ((tid & 3) == 0 && sg < segs) {
                xs1[m * (K / 32) + (sg >> 2)] = s1;
                xs2[m * (K / 32) + (sg >> 2)] = s2;
            }
        }
        if (tid == 0) isig[m] = 1.f / sigma;
    }
    __syncthreads();

    // ---- main loop: warp w takes local units w, w+8, ...
    const int wks = p.wks;
    const int lanes_act = wks >> 5;
    const int rstride = wks >> 1, szstride = (wks >> 7) * 4;
    for (int i = warp; i < nu; i += 8) {
        const int s = i % nst;
        mbar_wait(&bar[s], uint32_t((i / nst) & 1), p.err);
        const uint8_t* st = stages + size_t(s) * ub;
        const int u = u0 + i;
        const int j = u % ksl;
        float acc[8][MB];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int m = 0; m < MB; ++m) acc[r][m] = 0.f;
        if (lane < lanes_act) {
            const int ch = j * lanes_act + lane;             // 32-input chunk index along K
            uint32_t xr[MB][16];
            float c1[MB], c2[MB], is[MB];
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                const uint4* xp = reinterpret_cast<const uint4*>(xh + size_t(m) * K + size_t(ch) * 32);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint4 t = xp[q4];
                    xr[m][4 * q4 + 0] = t.x; xr[m][4 * q4 + 1] = t.y;
                    xr[m][4 * q4 + 2] = t.z; xr[m][4 * q4 + 3] = t.w;
                }
                c1[m] = 1024.f * xs1[m * (K / 32) + ch];
                c2[m] = xs2[m * (K / 32) + ch];
                is[m] = isig[m];
            }
            const uint8_t* wrow = st + lane * 16;
            const uint8_t* szp = st + 4 * wks + (lane >> 2) * 4;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint4 wq = *reinterpret_cast<const uint4*>(wrow + r * rstride);
                const uint32_t sz = *reinterpret_cast<const uint32_t*>(szp + r * szstride);
                float D[MB];
#pragma unroll
                for (int m = 0; m < MB; ++m) D[m] = 0.f;
                dot_word<MB>(D, wq.x, xr, 0);
                dot_word<MB>(D, wq.y, xr, 1);
                dot_word<MB>(D, wq.z, xr, 2);
                dot_word<MB>(D, wq.w, xr, 3);
                const float sc = bf16_lo(sz), zc = bf16_hi(sz);
                const float z8 = __fmaf_rn(-8.f, sc, zc);
#pragma unroll
                for (int m = 0; m < MB; ++m)
                    acc[r][m] = __fmul_rn(__fmaf_rn(sc, __fsub_rn(D[m], c1[m]), __fmul_rn(z8, c2[m])), is[m]);
            }
        }
        // reduce-scatter the 8 row sums over the 32 lanes: lane l ends with row (l>>2)&7
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
        const int row = (lane >> 2) & 7;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            float a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float keep = b4 ? acc[q + 4][m] : acc[q][m];
                const float send = b4 ? acc[q][m] : acc[q + 4][m];
                a[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            float cc[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float keep = b3 ? a[q + 2] : a[q];
                const float send = b3 ? a[q] : a[q + 2];
                cc[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            float e = (b2 ? cc[1] : cc[0]) + __shfl_xor_sync(0xffffffffu, b2 ? cc[0] : cc[1], 4);
            e += __shfl_xor_sync(0xffffffffu, e, 2);
            e += __shfl_xor_sync(0xffffffffu, e, 1);
            if ((lane & 3) == 0) upart[(size_t(i) * 8 + row) * MB + m] = e;
        }
        __syncwarp();
        if (lane == 0 && i + nst < nu) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[s], ub);
            bulk_g2s_stream(stages + size_t(s) * ub, p.w + size_t(u0 + i + nst) * ub, ub, &bar[s],
                            policy_evict_first());
        }
    }
    __syncthreads();
    if (nu <= 0) return;

    // ---- per-tile sums (fixed order over the CTA's units of each tile)
    const int t_first = u0 / ksl, t_last = (u1 - 1) / ksl, ntl = t_last - t_first + 1;
    const int RM = 8 * MB;
    auto tile_full = [&](int tl) {
        const int t = t_first + tl;
        return u0 <= t * ksl && u1 >= t * ksl + ksl;
    };
    for (int idx = tid; idx < ntl * RM; idx += kThreads) {
        const int tl = idx / RM, rm = idx % RM, t = t_first + tl;
        const int ua = max(u0, t * ksl), ue = min(u1, t * ksl + ksl);
        float v = 0.f;
        for (int uu = ua; uu < ue; ++uu) v += upart[size_t(uu - u0) * RM + rm];
        if (tile_full(tl)) tval[size_t(tl) * RM + rm] = v;
        else p.gpart[(size_t(c) * 2 + (tl == 0 ? 0 : 1)) * RM + rm] = v;
    }
    __threadfence();
    __syncthreads();
    // ---- tiles shared with neighbouring CTAs: the last to arrive combines them
    if (tid < 2) {
        int last = 0;
        const int tl = tid == 0 ? 0 : ntl - 1;
        if ((tid == 0 || ntl > 1) && !tile_full(tl)) {
            const int t = t_first + tl;
            const int c_lo = unit_owner((long long)t * ksl, U, P), c_hi = unit_owner((long long)t * ksl + ksl - 1, U, P);
            __threadfence();
            const int old = atomicAdd(&p.counters[t], 1);
            if (old == c_hi - c_lo) {
                last = 1;
                p.counters[t] = 0;
                __threadfence();
            }
        }
        flags[tid] = last;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        if (!flags[b]) continue;
        const int tl = b == 0 ? 0 : ntl - 1, t = t_first + tl;
        const int c_lo = unit_owner((long long)t * ksl, U, P), c_hi = unit_owner((long long)t * ksl + ksl - 1, U, P);
        for (int rm = tid; rm < RM; rm += kThreads) {
            float v = 0.f;
            for (int cc = c_lo; cc <= c_hi; ++cc) {
                const int slot = (int(unit_start(cc, U, P)) / ksl == t) ? 0 : 1;
                v += __ldcg(&p.gpart[(size_t(cc) * 2 + slot) * RM + rm]);
            }
            tval[size_t(tl) * RM + rm] = v;
        }
    }
    __syncthreads();
    // ---- epilogue on every tile this CTA completed
    for (int idx = tid; idx < ntl * RM; idx += kThreads) {
        const int tl = idx / RM, rm = idx % RM, r = rm / MB, m = rm % MB, t = t_first + tl;
        const bool ready = tile_full(tl) || (tl == 0 && flags[0]) || (tl == ntl - 1 && ntl > 1 && flags[1]);
        if (!ready || m >= p.M) continue;
        const float v = tval[size_t(tl) * RM + rm];
        if (p.epi == EPI_SILU) {
            if (r >= 4) continue;
            const int jj = t * 4 + r;
            if (jj >= p.N / 2) continue;
            const float up = tval[size_t(tl) * RM + (r + 4) * MB + m];
            p.y[size_t(m) * p.ldy + jj] = __fmul_rn(__fdiv_rn(v, __fadd_rn(1.f, expf(-v))), up);
        } else {
            const int n = t * 8 + r;
            if (n >= p.N) continue;
            float* yp = p.y + size_t(m) * p.ldy + n;
            if (p.epi == EPI_RESID) *yp = __fadd_rn(*yp, v);
            else *yp = v;
        }
    }
}

}  // namespace

int gemv_pick_mb(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }
int gemv_grid(int units, int sms) {
    constexpr int kMaxUnitsPerCta = 64;
    int g = sms < 1 ? 1 : sms;
    if ((units + g - 1) / g > kMaxUnitsPerCta) g = (units + kMaxUnitsPerCta - 1) / kMaxUnitsPerCta;
    if (g > units) g = units;
    return g < 1 ? 1 : g;
}
int gemv_units_per_cta(int units, int grid) { return (units + grid - 1) / grid; }
int gemv_nstage(int units, int grid, int unit_bytes) {
    const int upc = gemv_units_per_cta(units, grid);
    int cap = (96 * 1024) / unit_bytes;
    if (cap < 2) cap = 2;
    const int n = upc < cap ? upc : cap;
    return n < 1 ? 1 : n;
}
size_t gemv_smem_bytes(int MB, int K, int unit_bytes, int nstage, int upc) {
    return gemv_layout(MB, K, unit_bytes, nstage, upc).total;
}
size_t gemv_workspace_bytes(int grid, int tiles) {
    return al16(size_t(grid) * 2 * 8 * kMaxMB * sizeof(float)) + al16(size_t(tiles) * sizeof(int));
}

template <int MB>
static cudaError_t launch_mb(const GemvParams& p, int grid, cudaStream_t st, bool pdl) {
    const int upc = gemv_units_per_cta(p.units, grid);
    const size_t smem = gemv_smem_bytes(MB, p.K, p.unit_bytes, p.nstage, upc);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
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
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
    if ((e = cudaFuncSetAttribute(gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
    if ((e = cudaFuncSetAttribute(gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
    return cudaFuncSetAttribute(gemv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
}

}  // namespace kmr
