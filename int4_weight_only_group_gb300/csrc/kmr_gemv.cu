// Dequant-fused int4 weight-only GEMV / skinny GEMM (up to 8 rows of x per pass).
//
// What it computes ("kaminari — a single-GPU Qwen3-VL inference engine,
// explained", §07 int4 sidecar quantization; group 128 along K):
//     y[m, n] = sum_k x[m, k] * ((q[n, k] - 8) * s[n, k/128] + z[n, k/128])
// optionally on RMSNorm(x) (prologue) and followed by a store, a residual
// add or SiLU(gate) * up (epilogue).
//
// GB300 design
//   * HBM-bound: every packed byte is read once.  A CTA owns whole 16-row
//     tiles (no cross-CTA reduction, no global scratch) and pulls them with
//     cp.async.bulk into shared memory; the whole fill is issued BEFORE
//     griddepcontrol.wait, so under programmatic dependent launch a kernel
//     streams its weights while the previous kernel of the step finishes.
//   * Issue-rate bound on CUDA cores: at GB300's ~47 int4 weights per SM-clock
//     a float FMA per weight plus the unpacking would exceed the SM's issue
//     rate.  The multiply-adds therefore go to the tensor cores (mma.m16n8k16,
//     f16 in, f32 accumulate; 16 tile rows as M, batch rows as N) and the
//     threads only unpack: the KMR4 layout stores each lane's A fragment of a
//     16x16 block in one 32-bit word, so 8 weights cost one shift and four
//     LOP3s.  OR-ing a nibble into the mantissa of fp16 1024.0 gives 1024 + q
//     exactly (1024 + 16q for tile rows 8..15, whose nibble sits one position
//     higher); the offset, the -8 and the zero point are folded in once per
//     group with the group sum X' of the staged x:
//         y += (s (D - 1024 X') / c + (z - 8 s) X') / sigma,   c = 1 or 16.
//   * Latency: after griddepcontrol.wait nothing waits on a block barrier
//     until the products are done.  Each warp stages only the x of its own
//     groups (w, w + 16, ...): one coalesced load per lane, fp16 scaled by a
//     per-(row, group) power of two sigma taken from that group's largest
//     value (exact; undone in the fold), in B-fragment order in a warp-private
//     shared buffer.  RMSNorm is applied to the result instead of the input,
//     y = r * W (x * w) with r = rsqrt(mean(x^2) + eps), so its reduction
//     joins the one barrier before the epilogue.
//   * Deterministic and batch invariant: fixed k order inside the mma, fixed
//     group and warp orders in every sum; a row's result never depends on the
//     other rows or on M.
#include <cuda_fp16.h>

#include "kmr_gemv_core.cuh"

namespace kmr {

namespace {

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

// xw: per warp, GPW groups x MB rows of 128 staged halves (B-fragment order);
// xst: per warp, GPW groups x 8 rows x (X', 1/sigma); ssw: per warp, sum of x^2 per row;
// part: per tile in the ring, per warp, 16 rows x MB columns.
struct GemvSmem {
    size_t bar, xw, xst, ssw, part, stage, total;
};
__host__ __device__ inline GemvSmem gemv_layout(int MB, int GPW, int tile_bytes, int nst) {
    GemvSmem L;
    size_t o = 0;
    L.bar = o;   o += al16(size_t(nst) * 8);
    L.xw = o;    o += al16(size_t(kGemvWarps) * GPW * MB * 128 * 2);
    L.xst = o;   o += al16(size_t(kGemvWarps) * GPW * 8 * 2 * 4);
    L.ssw = o;   o += al16(size_t(kGemvWarps) * 8 * 4);
    L.part = o;  o += al16(size_t(nst) * kGemvWarps * 16 * MB * 4);
    o = (o + 127) & ~size_t(127);
    L.stage = o; o += size_t(nst) * tile_bytes;
    L.total = o;
    return L;
}

// Two CTAs per SM (so the next GEMV of the step can be resident and prefetching) where the
// staging registers allow it.
// Everything after griddepcontrol.wait for up to MB rows of x: stage x, run the tile products
// on the resident weight tiles, reduce and apply the epilogue.  Called once per group of MB
// rows (two calls let a CTA serve 16 rows from one weight fill).
template <int MB, int GPW>
__device__ __forceinline__ void gemv_rows(const GemvParams p, uint8_t* smem, const GemvSmem& L, const uint2 (&nwv)[GPW],
                                          int t0, int nt, int c) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, G = K >> 7, tb = p.tile_bytes, nst = p.nstage;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    __half* xw = reinterpret_cast<__half*>(smem + L.xw) + size_t(warp) * GPW * MB * 128;
    float* xst = reinterpret_cast<float*>(smem + L.xst) + size_t(warp) * GPW * 16;
    float* ssw = reinterpret_cast<float*>(smem + L.ssw);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint8_t* stages = smem + L.stage;

    // All tiles fit (the usual case): an EPI_RESID thread fetches its first residual value
    // (written by an earlier kernel of the step) while x is staged, so the epilogue does not
    // wait on L2.
    const bool fast = nt <= nst;
    const int per = (p.epi == EPI_SILU ? 8 : 16) * MB;
    float res0 = 0.f;
    bool have_res0 = false;
    stage_x<MB, GPW>(p, xw, xst, ssw, nwv, c, [&] {
        if (fast && p.epi == EPI_RESID && tid < nt * per) {
            const int tl = tid / per, e = tid - tl * per, rr = e / MB, m = e % MB, n = (t0 + tl) * 16 + rr;
            if (m < p.M && n < p.N) {
                res0 = p.y[size_t(m) * p.ldy + n];
                have_res0 = true;
            }
        }
    });

    // ---- products: every warp runs its groups of every tile, no block barrier until the end
    const int g = lane >> 2;
    const bool bload = g < p.M;
    constexpr int WS = 16 * MB;                    // floats per warp partial
    // One group per warp (K <= 2048): its x fragments stay in registers across tiles.
    // More groups per warp: reloaded from shared memory per tile (registers would
    // otherwise keep two CTAs from sharing an SM).
    XFrag xf1;
    if (GPW == 1 && warp < G) load_xfrag(xf1, xw + size_t(bload ? g : 0) * 128, bload, lane, xst);
    auto tile_products = [&](const uint8_t* st, float (&acc)[4]) {
        if constexpr (GPW == 1) {
            if (warp < G) group_product<(MB > 1)>(st + size_t(warp) * kGroupBytes, xf1, lane, acc);
        } else {
#pragma unroll
            for (int j = 0; j < GPW; ++j) {
                const int grp = warp + j * kGemvWarps;
                if (grp < G) {
                    XFrag xf;
                    load_xfrag(xf, xw + size_t(j * MB + (bload ? g : 0)) * 128, bload, lane, xst + j * 16);
                    group_product<(MB > 1)>(st + size_t(grp) * kGroupBytes, xf, lane, acc);
                }
            }
        }
    };
    if (fast) {
        // every tile was requested before griddepcontrol.wait; with all of them in, the
        // product loop has no wait between tiles
        mbar_wait(&bar[0], 0u, p.err);
#pragma unroll 1
        for (int tl = 0; tl < nt; ++tl) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            tile_products(stages + size_t(tl) * tb, acc);
            store_part<MB>(part + (size_t(tl) * kGemvWarps + warp) * WS, lane, acc);
        }
        __syncthreads();
        for (int idx = tid; idx < nt * per; idx += kGemvThreads) {
            const int tl = idx / per;
            tile_epilogue<MB>(p, part + size_t(tl) * kGemvWarps * WS, t0 + tl, idx - tl * per, ssw,
                              idx == tid && have_res0, res0);
        }
        return;
    }
    // ---- ring: one tile at a time, a barrier per tile frees its stage
    for (int i = 0; i < nt; ++i) {
        const int s = i % nst;
        mbar_wait(&bar[s], uint32_t((i / nst) & 1), p.err);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        tile_products(stages + size_t(s) * tb, acc);
        store_part<MB>(part + (size_t(s) * kGemvWarps + warp) * WS, lane, acc);
        __syncthreads();
        if (tid == 0 && i + nst < nt) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[s], tb);
            bulk_g2s_stream(stages + size_t(s) * tb, p.w + size_t(t0 + i + nst) * tb, tb, &bar[s],
                            policy_evict_first());
        }
        tile_epilogue<MB>(p, part + size_t(s) * kGemvWarps * WS, t0 + i, tid, ssw);
    }
}

// 16 rows (two halves of 8) on resident tiles when every warp owns exactly one group
// (K = 2048): both halves are staged and held as x fragments, every weight block is
// unpacked once for both (group_product2), and each warp leaves its two partials in the
// block it has just consumed (only that warp reads a block).  Per row the same operations
// in the same order as one half at a time, so the same bits.
__device__ __forceinline__ void gemv_rows16(const GemvParams p, uint8_t* smem, const GemvSmem& L,
                                            const uint2 (&nwv)[1], int t0, int nt, int c) {
    constexpr int MB = 8;
    constexpr int PWS = kGroupBytes / 4;           // floats from one warp's partials to the next
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, tb = p.tile_bytes;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    __half* xw = reinterpret_cast<__half*>(smem + L.xw) + size_t(warp) * MB * 128;
    float* xst = reinterpret_cast<float*>(smem + L.xst) + size_t(warp) * 16;
    float* ssw[2] = {reinterpret_cast<float*>(smem + L.ssw),
                     reinterpret_cast<float*>(smem + L.part)};     // the partial ring is unused here
    uint8_t* stages = smem + L.stage;
    GemvParams h[2] = {p, p};
    h[0].M = MB;
    h[1].M = p.M - MB;
    h[1].x = p.x ? p.x + size_t(MB) * K : nullptr;
    h[1].tokens = p.tokens ? p.tokens + MB : nullptr;
    h[1].x_out = p.x_out ? p.x_out + size_t(MB) * K : nullptr;
    h[1].y = p.y + size_t(MB) * p.ldy;
    const int per = (p.epi == EPI_SILU ? 8 : 16) * MB;
    float res0[2] = {0.f, 0.f};
    bool have_res0[2] = {false, false};
    const int g = lane >> 2;
    XFrag xf[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const GemvParams& q = h[hh];
        stage_x<MB, 1>(q, xw, xst, ssw[hh], nwv, c, [&] {
            if (q.epi == EPI_RESID && tid < nt * per) {
                const int tl = tid / per, e = tid - tl * per, rr = e / MB, m = e % MB, n = (t0 + tl) * 16 + rr;
                if (m < q.M && n < q.N) {
                    res0[hh] = q.y[size_t(m) * q.ldy + n];
                    have_res0[hh] = true;
                }
            }
        });
        const bool bload = g < q.M;
        load_xfrag(xf[hh], xw + size_t(bload ? g : 0) * 128, bload, lane, xst);
        __syncwarp();                              // xw / xst are restaged for the second half
    }
    mbar_wait(&bar[0], 0u, p.err);
#pragma unroll 1
    for (int tl = 0; tl < nt; ++tl) {
        float acca[4] = {0.f, 0.f, 0.f, 0.f}, accb[4] = {0.f, 0.f, 0.f, 0.f};
        uint8_t* blk = stages + size_t(tl) * tb + size_t(warp) * kGroupBytes;
        group_product2(blk, xf[0], xf[1], lane, acca, accb);
        __syncwarp();                              // every lane's reads of the block are done
        float* wp = reinterpret_cast<float*>(blk);
        store_part<MB>(wp, lane, acca);
        store_part<MB>(wp + 16 * MB, lane, accb);
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
        for (int idx = tid; idx < nt * per; idx += kGemvThreads) {
            const int tl = idx / per;
            tile_epilogue<MB, PWS>(h[hh], reinterpret_cast<const float*>(stages + size_t(tl) * tb) + hh * 16 * MB,
                                   t0 + tl, idx - tl * per, ssw[hh], idx == tid && have_res0[hh], res0[hh]);
        }
}

template <int MB, int GPW, int NH>
__global__ void __launch_bounds__(kGemvThreads, (MB * GPW * NH <= 8) ? 2 : 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = gridDim.x, c = blockIdx.x;
    const int t0 = int((long long)c * p.tiles / P), t1 = int((long long)(c + 1) * p.tiles / P);
    const int nt = t1 - t0;
    const int K = p.K, G = K >> 7, tb = p.tile_bytes, nst = p.nstage;
    const GemvSmem L = gemv_layout(MB, GPW, tb, nst);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint8_t* stages = smem + L.stage;

    // ---- weight ring: whole fill issued before waiting on the previous kernel
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = policy_evict_first();
        if (nt <= nst) {
            // every tile fits: one barrier counts all of them (nt * tb < 2^20 bytes)
            mbar_arrive_expect_tx(&bar[0], uint32_t(nt) * tb);
            for (int i = 0; i < nt; ++i)
                bulk_g2s_stream(stages + size_t(i) * tb, p.w + size_t(t0 + i) * tb, tb, &bar[0], pol);
        } else {
            for (int i = 0; i < nst; ++i) {
                mbar_arrive_expect_tx(&bar[i], tb);
                bulk_g2s_stream(stages + size_t(i) * tb, p.w + size_t(t0 + i) * tb, tb, &bar[i], pol);
            }
        }
    }
    const bool norm = p.in_kind != IN_F32;
    // norm weights of this warp's groups (constants): fetched before the wait
    uint2 nwv[GPW];
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
        const int grp = warp + j * kGemvWarps;
        nwv[j] = (norm && grp < G) ? *reinterpret_cast<const uint2*>(p.norm_w + size_t(grp) * 128 + lane * 4)
                                   : make_uint2(0, 0);
    }
    pdl_launch_dependents();
    pdl_wait();

    if constexpr (NH == 1) {
        gemv_rows<MB, GPW>(p, smem, L, nwv, t0, nt, c);
    } else if (GPW == 1 && (K >> 7) == kGemvWarps) {
        if constexpr (GPW == 1) gemv_rows16(p, smem, L, nwv, t0, nt, c);
    } else {
        // rows [0, MB), then [MB, M) on the same resident weight tiles
        GemvParams q = p;
        q.M = MB;
        gemv_rows<MB, GPW>(q, smem, L, nwv, t0, nt, c);
        __syncthreads();                         // the first rows' staging and partials are consumed
        q.x = p.x ? p.x + size_t(MB) * K : nullptr;
        q.tokens = p.tokens ? p.tokens + MB : nullptr;
        q.x_out = p.x_out ? p.x_out + size_t(MB) * K : nullptr;
        q.y = p.y + size_t(MB) * p.ldy;
        q.M = p.M - MB;
        gemv_rows<MB, GPW>(q, smem, L, nwv, t0, nt, c);
    }

}

}  // namespace

int gemv_pick_mb(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }
// Two groups of 8 rows share one weight fill when every CTA's tiles stay resident (no ring).
bool gemv_two_halves_ok(int tiles, int grid, int tile_bytes) {
    const int tpc = (tiles + grid - 1) / grid;
    return tpc <= gemv_nstage(tiles, grid, tile_bytes);
}
static int gemv_gpw(int K) { return ((K >> 7) + kGemvWarps - 1) / kGemvWarps; }

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
    return gemv_layout(MB, gemv_gpw(K), tile_bytes, nstage).total;
}

template <int MB, int GPW>
static const void* gemv_fn() { return (const void*)gemv_kernel<MB, GPW, 1>; }

static const void* gemv_fn_for(int MB, int GPW, int NH = 1) {
    if (NH == 2) {
        switch (GPW) {
            case 1: return (const void*)gemv_kernel<8, 1, 2>;
            case 2: return (const void*)gemv_kernel<8, 2, 2>;
            case 3: return (const void*)gemv_kernel<8, 3, 2>;
            default: return (const void*)gemv_kernel<8, 4, 2>;
        }
    }
    switch (MB * 8 + GPW) {
        case 1 * 8 + 1: return gemv_fn<1, 1>();
        case 1 * 8 + 2: return gemv_fn<1, 2>();
        case 1 * 8 + 3: return gemv_fn<1, 3>();
        case 1 * 8 + 4: return gemv_fn<1, 4>();
        case 2 * 8 + 1: return gemv_fn<2, 1>();
        case 2 * 8 + 2: return gemv_fn<2, 2>();
        case 2 * 8 + 3: return gemv_fn<2, 3>();
        case 2 * 8 + 4: return gemv_fn<2, 4>();
        case 4 * 8 + 1: return gemv_fn<4, 1>();
        case 4 * 8 + 2: return gemv_fn<4, 2>();
        case 4 * 8 + 3: return gemv_fn<4, 3>();
        case 4 * 8 + 4: return gemv_fn<4, 4>();
        case 8 * 8 + 1: return gemv_fn<8, 1>();
        case 8 * 8 + 2: return gemv_fn<8, 2>();
        case 8 * 8 + 3: return gemv_fn<8, 3>();
        default: return gemv_fn<8, 4>();
    }
}

cudaError_t launch_gemv(const GemvParams& p, int MB, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes(MB, p.K, p.tile_bytes, p.nstage);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    GemvParams q = p;
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, gemv_fn_for(MB, gemv_gpw(p.K), p.halves), args);
}

cudaError_t gemv_set_attributes() {
    const int mx = 227 * 1024;
    const int mbs[5] = {1, 2, 4, 8, 16};         // 16: two groups of 8 rows per launch
    for (int mb : mbs)
        for (int gpw = 1; gpw <= 4; ++gpw) {
            const void* k = mb == 16 ? gemv_fn_for(8, gpw, 2) : gemv_fn_for(mb, gpw);
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

}  // namespace kmr
