// Prefill's int4 projections as a weight-stationary GEMM ("kaminari — a single-GPU Qwen3-VL
// inference engine, explained", §07 int4 sidecar quantization: w = (q - 8) s + z, group 128
// along K; §04: prefill runs every prompt position through the same linears).
//
// With hundreds of rows the contraction is dense, and the int4 unpack (integer ops, the
// limit of the one-row GEMV) can be shared by many rows: each unpacked A fragment feeds
// 8 row-blocks of 8 rows.  Two kernels:
//   stage_kernel  x [M][K] fp32 (or the embedding rows of the tokens), optionally times the
//                 RMSNorm weight, to fp16 halves in B-fragment order with a power-of-two scale
//                 per (row, group) — the GEMV's staging arithmetic, done once for the whole
//                 batch instead of once per CTA — plus (X', 1/sigma) per (row, group) and
//                 the row's RMSNorm factor.  Layout [group][row][...] so that a group's block
//                 of rows is one contiguous copy.
//   gemm_kernel   CTA tile: TW = 8 (or 4, when 8 would leave most SMs idle) weight tiles x
//                 128 rows.  A producer warp streams, per 128-input group, the tiles' 1088-byte
//                 blocks and the rows' staged block into a 4-stage ring (cp.async.bulk,
//                 mbarriers); each of 8 consumer warps owns a pair of tiles and TW row-blocks
//                 of 8 rows, unpacks the pair's A fragments once per group, and loads each
//                 row-block's B fragments once for both tiles (mma.sync m16n8k16), folding
//                 each group into fp32 accumulators (s (D - 1024 X') / c + (z - 8 s) X') / sigma.
//                 Groups are summed in order; a row's result depends on nothing but that row.
#include <cuda_fp16.h>

#include "kmr_int4_mma.cuh"
#include "kmr_internal.cuh"

namespace kmr {
namespace {

constexpr int kGemmRows = 128;              // rows per CTA
constexpr int kGemmStages = 4;
constexpr int kGemmConsumers = 8;           // warps (all compute; lane 0 of warp 0 also refills the ring)
constexpr int kGemmThreads = kGemmConsumers * 32;
constexpr int kStageX = kGemmRows * 128 * 2;                 // 32768
constexpr int kStageS = kGemmRows * 8;                       // 1024: (X', 1/sigma) per row
constexpr int stage_bytes(int tw) { return tw * kGroupBytes + kStageX + kStageS; }

// A staged row's 16-byte chunks are stored XOR-swizzled by the row's low 3 bits, so that the
// 8 rows of a row-block, read at the same chunk by the GEMM's B-fragment loads, fall in
// different shared-memory banks.
__device__ __forceinline__ int swz(int q, int row) { return (((q >> 3) ^ (row & 7)) << 3) | (q & 7); }

// ---- staging: one CTA per row, 8 warps; warp w takes groups w, w + 8, ...
__global__ void __launch_bounds__(256) stage_kernel(const StageParams p) {
    const int row = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K = p.K, G = K >> 7;
    __shared__ float red[8];
    __half* xs = reinterpret_cast<__half*>(p.xs);
    float2* xst = p.xst;
    if (row >= p.M) {                                       // padding rows: zeros, scale 1
        for (int g = warp; g < G; g += 8) {
            reinterpret_cast<uint2*>(xs + (size_t(g) * p.Mpad + row) * 128)[lane] = make_uint2(0, 0);
            if (lane == 0) xst[size_t(g) * p.Mpad + row] = make_float2(0.f, 1.f);
        }
        if (threadIdx.x == 0) p.rnorm[row] = 1.f;
        return;
    }
    int tok = 0;
    if (p.in_kind == IN_EMBED_NORM) {
        tok = p.tokens[row];
        if (tok < 0 || tok >= p.vocab) {
            if (threadIdx.x == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
            tok = 0;
        }
    }
    const bool norm = p.in_kind != IN_F32;
    float ss = 0.f;
    for (int g = warp; g < G; g += 8) {
        const size_t k = size_t(g) * 128 + lane * 4;
        float u[4];
        if (p.in_kind == IN_EMBED_NORM) {
            const uint2 raw = *reinterpret_cast<const uint2*>(p.embed + size_t(tok) * K + k);
            u[0] = bf16_lo(raw.x); u[1] = bf16_hi(raw.x); u[2] = bf16_lo(raw.y); u[3] = bf16_hi(raw.y);
            if (p.x_out) *reinterpret_cast<float4*>(p.x_out + size_t(row) * K + k) = make_float4(u[0], u[1], u[2], u[3]);
        } else {
            const float4 v = *reinterpret_cast<const float4*>(p.x + size_t(row) * K + k);
            u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
        }
        if (norm) {
            const uint2 nw = *reinterpret_cast<const uint2*>(p.norm_w + k);
#pragma unroll
            for (int e = 0; e < 4; ++e) ss = __fmaf_rn(u[e], u[e], ss);
            u[0] = __fmul_rn(u[0], bf16_lo(nw.x));
            u[1] = __fmul_rn(u[1], bf16_hi(nw.x));
            u[2] = __fmul_rn(u[2], bf16_lo(nw.y));
            u[3] = __fmul_rn(u[3], bf16_hi(nw.y));
        }
        const float la = fmaxf(fmaxf(fabsf(u[0]), fabsf(u[1])), fmaxf(fabsf(u[2]), fabsf(u[3])));
        float sig, isg;
        pow2_scale(__reduce_max_sync(0xffffffffu, __float_as_uint(la)), sig, isg);
        const __half2 h01 = __floats2half2_rn(__fmul_rn(u[0], sig), __fmul_rn(u[1], sig));
        const __half2 h23 = __floats2half2_rn(__fmul_rn(u[2], sig), __fmul_rn(u[3], sig));
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const float gs = warp_sum(__fadd_rn(__fadd_rn(f01.x, f01.y), __fadd_rn(f23.x, f23.y)));
        __half* blk = xs + (size_t(g) * p.Mpad + row) * 128;
        *reinterpret_cast<__half2*>(blk + swz(bpos(lane * 4), row)) = h01;
        *reinterpret_cast<__half2*>(blk + swz(bpos(lane * 4 + 2), row)) = h23;
        if (lane == 0) xst[size_t(g) * p.Mpad + row] = make_float2(gs, isg);
    }
    if (norm) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int w = 0; w < 8; ++w) tot += red[w];
            p.rnorm[row] = rsqrtf(tot / float(K) + p.eps);
        }
    } else if (threadIdx.x == 0) {
        p.rnorm[row] = 1.f;
    }
}

// ---- GEMM: TW weight tiles x 128 rows per CTA; warp w takes tile pair w % (TW / 2) and the
// TW row-blocks starting at TW * (w / (TW / 2)) (8 warps cover TW / 2 pairs x 16 row-blocks).
// Two warps per SM sub-partition leave up to 255 registers per thread: 64 accumulators and
// the pair's 64 A-fragment registers stay resident.
template <int TW>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const GemmParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int PAIRS = TW / 2, RBW = 2 * PAIRS;           // row-blocks per warp (16 in all)
    constexpr int SW = TW * kGroupBytes, SB = SW + kStageX + kStageS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.K >> 7;
    const int tile0 = blockIdx.x * TW, r0 = blockIdx.y * kGemmRows;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    int* released = reinterpret_cast<int*>(smem + 64);          // per stage: warps done with it
    uint8_t* stages = smem + 128;
    if (tid == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int ntl = min(TW, p.tiles - tile0);                 // tiles this CTA owns (>= 1)

    // the ring: groups 0..stages-1 are requested now; group g + stages by the last warp to
    // release group g's stage (no warp waits for another)
    auto issue = [&](int g) {
        const int s = g % kGemmStages;
        uint8_t* st = stages + size_t(s) * SB;
        mbar_arrive_expect_tx(&full[s], uint32_t(ntl * kGroupBytes + kStageX + kStageS));
        for (int t = 0; t < ntl; ++t)
            bulk_g2s(st + t * kGroupBytes, p.w + (size_t(tile0 + t) * G + g) * kGroupBytes, kGroupBytes, &full[s]);
        bulk_g2s(st + SW, p.xs + (size_t(g) * p.Mpad + r0) * 128, kStageX, &full[s]);
        bulk_g2s(st + SW + kStageX, p.xst + size_t(g) * p.Mpad + r0, kStageS, &full[s]);
    };
    if (tid == 0)
        for (int g = 0; g < G && g < kGemmStages; ++g) issue(g);
    const int pr = warp % PAIRS, rb0 = (warp / PAIRS) * RBW;
    const int ta = 2 * pr;                                   // tiles ta, ta + 1 of the CTA
    const bool act0 = ta < ntl, act1 = ta + 1 < ntl;
    const int g8 = lane >> 2, t4 = lane & 3;
    float acc[RBW][2][4];
#pragma unroll
    for (int rb = 0; rb < RBW; ++rb)
#pragma unroll
        for (int u = 0; u < 2; ++u) acc[rb][u][0] = acc[rb][u][1] = acc[rb][u][2] = acc[rb][u][3] = 0.f;
    for (int g = 0; g < G; ++g) {
        const int s = g % kGemmStages;
        mbar_wait(&full[s], uint32_t((g / kGemmStages) & 1), p.err);
        const uint8_t* st = stages + size_t(s) * SB;
        if (act0) {
            const __half* xb = reinterpret_cast<const __half*>(st + SW);
            const float2* xsc = reinterpret_cast<const float2*>(st + SW + kStageX);
            // both tiles' A fragments for the group's 8 k-steps, unpacked once (a missing second
            // tile repeats the first; its results are never stored)
            uint32_t a[2][8][4];
            float s0[2], s1c[2], zz0[2], zz1[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint8_t* gb = st + (act1 ? ta + u : ta) * kGroupBytes;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const uint4 wq = *reinterpret_cast<const uint4*>(gb + blk * 512 + lane * 16);
                    const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t w = w4[ks], w2 = w >> 8;
                        a[u][blk * 4 + ks][0] = and_or(w, 0x000F000Fu, 0x64006400u);
                        a[u][blk * 4 + ks][1] = and_or(w, 0x00F000F0u, 0x64006400u);
                        a[u][blk * 4 + ks][2] = and_or(w2, 0x000F000Fu, 0x64006400u);
                        a[u][blk * 4 + ks][3] = and_or(w2, 0x00F000F0u, 0x64006400u);
                    }
                }
                const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(gb + 1024 + g8 * 4);
                const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(gb + 1024 + (g8 + 8) * 4);
                s0[u] = bf16_lo(sz0);
                s1c[u] = __fmul_rn(bf16_lo(sz1), 0.0625f);
                zz0[u] = __fmaf_rn(-8.f, s0[u], bf16_hi(sz0));
                zz1[u] = __fmaf_rn(-8.f, bf16_lo(sz1), bf16_hi(sz1));
            }
#pragma unroll
            for (int rb = 0; rb < RBW; ++rb) {
                const int rbase = (rb0 + rb) * 8;
                const __half* xr = xb + size_t(rbase + g8) * 128;                // this lane's column
                float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    // chunks blk * 8 + 2 t4 and + 1 of the row, swizzled by the row's low bits (g8)
                    const uint4 xa = *reinterpret_cast<const uint4*>(xr + (((blk * 8 + 2 * t4) ^ g8) << 3));
                    const uint4 xc = *reinterpret_cast<const uint4*>(xr + (((blk * 8 + 2 * t4 + 1) ^ g8) << 3));
                    const uint32_t bb[8] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            mma16816(d[u], a[u][blk * 4 + ks][0], a[u][blk * 4 + ks][1], a[u][blk * 4 + ks][2],
                                     a[u][blk * 4 + ks][3], bb[2 * ks], bb[2 * ks + 1]);
                }
                const float2 X0 = xsc[rbase + 2 * t4], X1 = xsc[rbase + 2 * t4 + 1];   // (X', 1/sigma)
                const float x0 = 1024.f * X0.x, x1 = 1024.f * X1.x;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    acc[rb][u][0] = __fmaf_rn(__fmaf_rn(s0[u], __fsub_rn(d[u][0], x0), __fmul_rn(zz0[u], X0.x)), X0.y, acc[rb][u][0]);
                    acc[rb][u][1] = __fmaf_rn(__fmaf_rn(s0[u], __fsub_rn(d[u][1], x1), __fmul_rn(zz0[u], X1.x)), X1.y, acc[rb][u][1]);
                    acc[rb][u][2] = __fmaf_rn(__fmaf_rn(s1c[u], __fsub_rn(d[u][2], x0), __fmul_rn(zz1[u], X0.x)), X0.y, acc[rb][u][2]);
                    acc[rb][u][3] = __fmaf_rn(__fmaf_rn(s1c[u], __fsub_rn(d[u][3], x1), __fmul_rn(zz1[u], X1.x)), X1.y, acc[rb][u][3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && g + kGemmStages < G) {
            // this warp's reads of the stage are done (their values are in registers); the
            // counter only grows, so the warp that completes a multiple of 8 refills the stage
            __threadfence_block();
            if (atomicAdd(&released[s], 1) % kGemmConsumers == kGemmConsumers - 1) {
                __threadfence_block();
                fence_proxy_async_smem();
                issue(g + kGemmStages);
            }
        }
    }
    // ---- epilogue: tile rows g8 ([0..1]) and g8 + 8 ([2..3]) for x rows rbase + 2 t4 (+1)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        if (!(u == 0 ? act0 : act1)) continue;
        const int tile = tile0 + ta + u;
#pragma unroll
        for (int rb = 0; rb < RBW; ++rb) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int m = r0 + (rb0 + rb) * 8 + 2 * t4 + c;
                if (m >= p.M) continue;
                const float r = p.rnorm[m];
                const float v0 = __fmul_rn(acc[rb][u][c], r), v1 = __fmul_rn(acc[rb][u][2 + c], r);
                float* yr = p.y + size_t(m) * p.ldy;
                if (p.epi == EPI_SILU) {
                    // gate rows 8 tile .. + 7 are tile rows 0..7, the matching up rows tile rows 8..15
                    const int j = tile * 8 + g8;
                    if (j < p.N / 2) yr[j] = __fmul_rn(__fdiv_rn(v0, __fadd_rn(1.f, expf(-v0))), v1);
                } else {
                    const int n0 = tile * 16 + g8, n1 = n0 + 8;
                    if (n0 < p.N) yr[n0] = p.epi == EPI_RESID ? __fadd_rn(yr[n0], v0) : v0;
                    if (n1 < p.N) yr[n1] = p.epi == EPI_RESID ? __fadd_rn(yr[n1], v1) : v1;
                }
            }
        }
    }
}

}  // namespace

size_t gemm_smem_bytes(int tw) { return 128 + size_t(kGemmStages) * stage_bytes(tw); }
int gemm_rows_pad(int M) { return (M + kGemmRows - 1) / kGemmRows * kGemmRows; }

cudaError_t gemm_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(gemm_smem_bytes(8)));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(gemm_smem_bytes(4)));
}

cudaError_t launch_stage(const StageParams& p, cudaStream_t st) {
    stage_kernel<<<p.Mpad, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmParams& p, int sms, cudaStream_t st) {
    // 8 tiles per CTA unless that leaves more than half of the SMs without a CTA
    const int rows = p.Mpad / kGemmRows;
    const int tw = ((p.tiles + 7) / 8) * rows * 2 >= sms ? 8 : 4;
    const dim3 grid((p.tiles + tw - 1) / tw, rows);
    if (tw == 8)
        gemm_kernel<8><<<grid, kGemmThreads, gemm_smem_bytes(8), st>>>(p);
    else
        gemm_kernel<4><<<grid, kGemmThreads, gemm_smem_bytes(4), st>>>(p);
    return cudaGetLastError();
}

}  // namespace kmr
