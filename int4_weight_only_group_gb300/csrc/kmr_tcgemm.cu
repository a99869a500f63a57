// Prefill projections on the 5th-generation tensor cores: y = x W^T for one prompt chunk
// (M tokens) and an int4 weight-only group-wise linear ("kaminari — a single-GPU Qwen3-VL
// inference engine, explained", §07 int4 sidecar quantization: w = (q - 8) s + z, group 128
// along K; the prefill of §04 runs every prompt position through the same projections).
//
// At a few hundred tokens the projection is a dense contraction, so it goes to tcgen05.mma
// (kind::f16, fp32 accumulators in tensor memory) instead of the warp-level mma the decode
// GEMV uses:
//   * CTA tile: 128 packed weight rows (the MMA's M, one TMEM lane each) x nt tokens (the
//     MMA's N, 64 or 128 TMEM columns); 4 warps, one per TMEM lane quarter.
//   * Per 128-input group: the eight 1088-byte KMR4 blocks of the CTA's weight rows arrive
//     through a 4-deep cp.async.bulk ring; every warp turns two of them into fp16
//     w = (q - 8) s + z (the nibble OR-ed into the mantissa of 1024.0 gives 1024 + q, or
//     1024 + 16 q for tile rows 8..15, exactly; one HFMA2 applies s and z) and writes them
//     into the K-major core-matrix layout (8 rows x 16 bytes per core matrix) of a
//     double-buffered A operand; the staged tokens of the group are one bulk copy into the
//     matching B buffer.  One thread issues the group's 8 MMAs (K = 16 each) and commits
//     them to an mbarrier, which frees the A and B buffers two groups later.
//   * The accumulator stays in tensor memory across all K; the epilogue reads it once
//     (tcgen05.ld 32x32b), applies the row's RMSNorm factor / sigma and stores, adds to the
//     residual, or applies SiLU(gate) * up across the gate / up rows of a tile.
//   * Every wait is bounded (mbar_wait); a timeout records KMR_ERR_DEVICE_TIMEOUT, skips
//     the remaining work, drains the copies in flight and frees tensor memory.
#include <cuda_fp16.h>

#include "kmr_int4_mma.cuh"
#include "kmr_tcgemm.cuh"

namespace kmr {

namespace {

constexpr int kTcThreads = 128;
constexpr int kTcRows = 128;                      // packed weight rows per CTA (MMA M)
constexpr int kTcTiles = kTcRows / 16;            // KMR4 tiles per CTA
constexpr int kTcWStages = 4;                     // weight-group ring depth
constexpr uint32_t kTcWBytes = kTcTiles * kGroupBytes;      // one group of the CTA's tiles
constexpr uint32_t kTcABytes = kTcRows * 128 * 2;           // fp16 A operand of one group
constexpr uint32_t kCoreSBO = 2048;               // bytes between 8-row core-matrix groups (16 x 128 B)
constexpr uint32_t kCoreLBO = 128;                // bytes between core matrices along K

struct TcSmem {
    uint32_t a[2], b[2], w, bar, total;
};
__host__ __device__ inline TcSmem tc_layout(int nt) {
    TcSmem L;
    uint32_t o = 0;
    L.a[0] = o; o += kTcABytes;
    L.a[1] = o; o += kTcABytes;
    L.b[0] = o; o += uint32_t(nt) * 256;
    L.b[1] = o; o += uint32_t(nt) * 256;
    L.w = o;    o += kTcWStages * kTcWBytes;
    L.bar = o;  o += 128;                         // wfull[4], bfull[2], mdone[2], TMEM address
    L.total = o;
    return L;
}

// ---- tcgen05 wrappers (cta_group::1)
__device__ __forceinline__ void tc_alloc(uint32_t* slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Shared-memory matrix descriptor: K-major, no swizzle; start address, the byte distance
// between core matrices along K (leading) and along M / N (stride), fixed version bits 0b001.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr) {
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t((kCoreLBO >> 4) & 0x3FFFu) << 16) |
           (uint64_t((kCoreSBO >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46);
}
// Instruction descriptor of kind::f16: fp32 D, fp16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t taddr, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(taddr),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// ---- staging: one CTA (256 threads) per token row
constexpr int kTcStageThreads = 256;
constexpr int kTcStageMaxK = 8192;

__global__ void __launch_bounds__(kTcStageThreads) tc_stage_kernel(const TcStageParams p) {
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, G = K >> 7, K4 = K >> 2;
    __half* xs = reinterpret_cast<__half*>(p.xs);
    const int tile = row / p.nt, rin = row % p.nt;
    // half offset of input k in this row's staged layout
    auto at = [&](int k) {
        return (size_t(tile) * G + (k >> 7)) * size_t(p.nt) * 128 + (rin >> 3) * 1024 + ((k & 127) >> 3) * 64 +
               (rin & 7) * 8 + (k & 7);
    };
    if (row >= p.M) {                             // tile padding: zeros, scale 0
        for (int k4 = tid; k4 < K4; k4 += kTcStageThreads)
            *reinterpret_cast<uint2*>(xs + at(k4 * 4)) = make_uint2(0, 0);
        if (tid == 0) p.rs[row] = 0.f;
        return;
    }
    __shared__ float red[2][kTcStageThreads / 32];
    int tok = 0;
    if (p.in_kind == IN_EMBED_NORM) {
        tok = p.tokens[row];
        if (tok < 0 || tok >= p.vocab) {
            if (tid == 0) set_error(p.err, KMR_ERR_INVALID_ARG);
            tok = 0;
        }
    }
    const bool norm = p.in_kind != IN_F32;
    constexpr int kPer = kTcStageMaxK / 4 / kTcStageThreads;   // float4 per thread at most
    float4 u[kPer];
    float ss = 0.f, mx = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int k4 = tid + i * kTcStageThreads;
        u[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k4 >= K4) continue;
        const size_t k = size_t(k4) * 4;
        float4 v;
        if (p.in_kind == IN_EMBED_NORM) {
            const uint2 raw = *reinterpret_cast<const uint2*>(p.embed + size_t(tok) * K + k);
            v = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
            if (p.x_out) *reinterpret_cast<float4*>(p.x_out + size_t(row) * K + k) = v;
        } else {
            v = *reinterpret_cast<const float4*>(p.x + size_t(row) * K + k);
        }
        if (norm) {
            ss = __fmaf_rn(v.x, v.x, ss);
            ss = __fmaf_rn(v.y, v.y, ss);
            ss = __fmaf_rn(v.z, v.z, ss);
            ss = __fmaf_rn(v.w, v.w, ss);
            const uint2 nw = *reinterpret_cast<const uint2*>(p.norm_w + k);
            v.x = __fmul_rn(v.x, bf16_lo(nw.x));
            v.y = __fmul_rn(v.y, bf16_hi(nw.x));
            v.z = __fmul_rn(v.z, bf16_lo(nw.y));
            v.w = __fmul_rn(v.w, bf16_hi(nw.y));
        }
        u[i] = v;
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    ss = warp_sum(ss);
    mx = warp_max(mx);
    if (lane == 0) {
        red[0][warp] = ss;
        red[1][warp] = mx;
    }
    __syncthreads();
    float tot = 0.f, amax = 0.f;
#pragma unroll
    for (int w = 0; w < kTcStageThreads / 32; ++w) {
        tot = __fadd_rn(tot, red[0][w]);
        amax = fmaxf(amax, red[1][w]);
    }
    float sig, isg;
    pow2_scale(__float_as_uint(amax), sig, isg);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int k4 = tid + i * kTcStageThreads;
        if (k4 >= K4) continue;
        const __half2 h01 = __floats2half2_rn(__fmul_rn(u[i].x, sig), __fmul_rn(u[i].y, sig));
        const __half2 h23 = __floats2half2_rn(__fmul_rn(u[i].z, sig), __fmul_rn(u[i].w, sig));
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&h01);
        o.y = *reinterpret_cast<const uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(xs + at(k4 * 4)) = o;
    }
    if (tid == 0) {
        const float r = norm ? rsqrtf(tot / float(K) + p.eps) : 1.f;
        p.rs[row] = __fmul_rn(r, isg);
    }
}

// ---- GEMM
// Unpacks one KMR4 block (16 tile rows x 128 inputs of one group) into the fp16 A operand:
// lane (g, t) holds, per k-step ks, rows g and g + 8 at inputs 16 ks + 2t (+1) and + 8 (+9).
__device__ __forceinline__ void tc_unpack_block(const uint8_t* blk, __half* a, int tl, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(blk + 1024 + g * 4);
    const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(blk + 1024 + (g + 8) * 4);
    const __half2 s0 = __float2half2_rn(bf16_lo(sz0)), z0 = __float2half2_rn(bf16_hi(sz0));
    const __half2 s1 = __float2half2_rn(bf16_lo(sz1)), z1 = __float2half2_rn(bf16_hi(sz1));
    const __half2 off0 = __float2half2_rn(-1032.f);            // 1024 + q - 1032 = q - 8
    const __half2 sc1 = __float2half2_rn(0.0625f), off1 = __float2half2_rn(-72.f);   // (1024 + 16 q) / 16 - 72
    uint32_t* r0 = reinterpret_cast<uint32_t*>(a + (2 * tl) * 1024 + g * 8 + 2 * t);       // tile row g
    uint32_t* r1 = reinterpret_cast<uint32_t*>(a + (2 * tl + 1) * 1024 + g * 8 + 2 * t);   // tile row g + 8
    auto cvt = [](uint32_t v) { return *reinterpret_cast<const __half2*>(&v); };
    auto bits = [](__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); };
#pragma unroll
    for (int blk_i = 0; blk_i < 2; ++blk_i) {
        const uint4 wq = *reinterpret_cast<const uint4*>(blk + blk_i * 512 + lane * 16);
        const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int ks = blk_i * 4 + j;
            const uint32_t w = w4[j], w2 = w >> 8;
            const __half2 qa = __hadd2(cvt(and_or(w, 0x000F000Fu, 0x64006400u)), off0);
            const __half2 qb = __hfma2(cvt(and_or(w, 0x00F000F0u, 0x64006400u)), sc1, off1);
            const __half2 qc = __hadd2(cvt(and_or(w2, 0x000F000Fu, 0x64006400u)), off0);
            const __half2 qd = __hfma2(cvt(and_or(w2, 0x00F000F0u, 0x64006400u)), sc1, off1);
            // core matrix kc = 2 ks (inputs 16 ks .. + 7) and 2 ks + 1 (+ 8 .. + 15): 64 halves each
            r0[(2 * ks) * 32] = bits(__hfma2(qa, s0, z0));
            r1[(2 * ks) * 32] = bits(__hfma2(qb, s1, z1));
            r0[(2 * ks + 1) * 32] = bits(__hfma2(qc, s0, z0));
            r1[(2 * ks + 1) * 32] = bits(__hfma2(qd, s1, z1));
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const TcGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const TcSmem L = tc_layout(NT);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.K >> 7;
    const int tile0 = blockIdx.x * kTcTiles;                     // first KMR4 tile of the CTA
    const int ttile = blockIdx.y;                                 // token tile
    uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + L.bar);  // [kTcWStages]
    uint64_t* bfull = wfull + kTcWStages;                         // [2]
    uint64_t* mdone = bfull + 2;                                  // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mdone + 2);
    __shared__ int abort_flag;
    const uint32_t sbase = smem_u32(smem);
    constexpr uint32_t kBBytes = uint32_t(NT) * 256;

    auto issue_w = [&](int g) {                                   // the CTA's 8 blocks of group g
        uint8_t* dst = smem + L.w + (g % kTcWStages) * kTcWBytes;
        uint64_t* bar = &wfull[g % kTcWStages];
        mbar_arrive_expect_tx(bar, kTcWBytes);
        const uint64_t pol = policy_evict_first();
        for (int i = 0; i < kTcTiles; ++i)
            bulk_g2s_stream(dst + i * kGroupBytes, p.w + (size_t(tile0 + i) * G + g) * kGroupBytes, kGroupBytes, bar,
                            pol);
    };
    auto issue_b = [&](int g) {                                   // the staged tokens of group g
        mbar_arrive_expect_tx(&bfull[g & 1], kBBytes);
        bulk_g2s(smem + L.b[g & 1], p.xs + (size_t(ttile) * G + g) * NT * 128, kBBytes, &bfull[g & 1]);
    };

    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kTcWStages; ++s) mbar_init(&wfull[s], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bfull[s], 1);
            mbar_init(&mdone[s], 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(tslot, NT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tslot;
    if (tid == 0) {
        for (int g = 0; g < G && g < kTcWStages; ++g) issue_w(g);
        issue_b(0);
    }
    int issued_w = G < kTcWStages ? G : kTcWStages, issued_b = 1, committed = 0;   // thread 0's counts

    for (int g = 0; g < G; ++g) {
        const int slot = g & 1;
        bool ok = true;
        if (g >= 2) ok = mbar_wait(&mdone[slot], uint32_t(((g - 2) >> 1) & 1), p.err);   // A[slot] free
        if (ok) ok = mbar_wait(&wfull[g % kTcWStages], uint32_t((g / kTcWStages) & 1), p.err);
        if (ok) {
            tc_fence_after();
            const uint8_t* wst = smem + L.w + (g % kTcWStages) * kTcWBytes;
            __half* a = reinterpret_cast<__half*>(smem + L.a[slot]);
#pragma unroll
            for (int i = 0; i < 2; ++i) tc_unpack_block(wst + (warp * 2 + i) * kGroupBytes, a, warp * 2 + i, lane);
        } else {
            abort_flag = 1;
        }
        fence_proxy_async_smem();                  // the A operand's generic stores, before the MMA reads
        __syncthreads();
        if (abort_flag) break;
        if (tid == 0) {
            if (g + kTcWStages < G) {              // every warp is done with this weight stage
                issue_w(g + kTcWStages);
                ++issued_w;
            }
            bool okb = true;
            if (g + 1 < G) {                       // B[(g + 1) & 1] was read by the MMAs of group g - 1
                if (g >= 1) okb = mbar_wait(&mdone[(g + 1) & 1], uint32_t(((g - 1) >> 1) & 1), p.err);
                if (okb) {
                    issue_b(g + 1);
                    ++issued_b;
                }
            }
            if (okb) okb = mbar_wait(&bfull[slot], uint32_t((g >> 1) & 1), p.err);
            if (okb) {
                tc_fence_after();
                const uint32_t ab = sbase + L.a[slot], bb = sbase + L.b[slot];
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma(taddr, tc_desc(ab + ks * 256), tc_desc(bb + ks * 256), tc_idesc(kTcRows, NT),
                           (g > 0 || ks > 0) ? 1u : 0u);
                tc_commit(&mdone[slot]);
                ++committed;
            } else {
                abort_flag = 1;                    // seen by every thread at the next barrier
            }
        }
    }
    __syncthreads();
    const bool aborted = abort_flag != 0;
    if (!aborted) {
        // the last commit tracks every MMA issued before it
        if (mbar_wait(&mdone[(G - 1) & 1], uint32_t(((G - 1) >> 1) & 1), p.err)) {
            tc_fence_after();
            const int n = (tile0 * 16) + warp * 32 + lane;           // packed weight row of this lane
            const uint32_t lane_base = taddr + (uint32_t(warp * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < NT; c0 += 16) {
                float v[16];
                tc_ld16(lane_base + uint32_t(c0), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = ttile * NT + c0 + j;
                    const float x = t < p.M ? __fmul_rn(v[j], p.rs[t]) : 0.f;
                    if (p.epi == EPI_SILU) {
                        const float up = __shfl_down_sync(0xffffffffu, x, 8);
                        if ((lane & 15) < 8 && t < p.M) {
                            const int jj = (n >> 4) * 8 + (lane & 7);
                            if (jj < p.N / 2)
                                p.y[size_t(t) * p.ldy + jj] = __fmul_rn(__fdiv_rn(x, __fadd_rn(1.f, expf(-x))), up);
                        }
                    } else if (t < p.M && n < p.N) {
                        float* yp = p.y + size_t(t) * p.ldy + n;
                        *yp = p.epi == EPI_RESID ? __fadd_rn(*yp, x) : x;
                    }
                }
            }
        }
    } else if (tid == 0) {
        // drain what is still in flight before the CTA's shared memory is released
        for (int g = issued_w - kTcWStages < 0 ? 0 : issued_w - kTcWStages; g < issued_w; ++g)
            mbar_wait(&wfull[g % kTcWStages], uint32_t((g / kTcWStages) & 1), p.err, 100000000ull);
        for (int g = issued_b - 2 < 0 ? 0 : issued_b - 2; g < issued_b; ++g)
            mbar_wait(&bfull[g & 1], uint32_t((g >> 1) & 1), p.err, 100000000ull);
        if (committed > 0)
            mbar_wait(&mdone[(committed - 1) & 1], uint32_t(((committed - 1) >> 1) & 1), p.err, 100000000ull);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(taddr, NT);
}

}  // namespace

bool tc_gemm_supported(int N, int K) { return N > 0 && N % kTcRows == 0 && K > 0 && K % 128 == 0 && K <= kTcStageMaxK; }

// 128 tokens per CTA when that already gives every SM a tile, else 64 (twice the CTAs).
int tc_gemm_pick_nt(int N, int M, int sms) {
    const long long ctas = (long long)(N / kTcRows) * ((M + 127) / 128);
    return ctas >= sms ? 128 : 64;
}

cudaError_t tc_gemm_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(tc_layout(128).total));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tc_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(tc_layout(64).total));
}

cudaError_t launch_tc_stage(const TcStageParams& p, cudaStream_t st) {
    const int rows = (p.M + p.nt - 1) / p.nt * p.nt;
    tc_stage_kernel<<<rows, kTcStageThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const TcGemmParams& p, cudaStream_t st) {
    const dim3 grid(p.N / kTcRows, (p.M + p.nt - 1) / p.nt);
    if (p.nt == 128) {
        tc_gemm_kernel<128><<<grid, kTcThreads, tc_layout(128).total, st>>>(p);
    } else {
        tc_gemm_kernel<64><<<grid, kTcThreads, tc_layout(64).total, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kmr
