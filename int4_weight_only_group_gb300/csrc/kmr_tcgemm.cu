// Prefill projections on the 5th-generation tensor cores: y = x W^T for one prompt chunk
// (M tokens) and an int4 weight-only group-wise linear ("kaminari — a single-GPU Qwen3-VL
// inference engine, explained", §07 int4 sidecar quantization: w = (q - 8) s + z, group 128
// along K; the prefill of §04 runs every prompt position through the same projections).
//
// At a few hundred tokens the projection is a dense contraction, so it goes to tcgen05.mma
// (kind::f16, fp32 accumulators in tensor memory) instead of the warp-level mma the decode
// GEMV uses:
//   * CTA tile: 128 packed weight rows (the MMA's M, one TMEM lane each) x nt = 64, 128 or 256
//     tokens (the MMA's N, nt TMEM columns).
//   * Warp-specialised pipeline with a full and an empty mbarrier per stage and no block-wide
//     barrier inside the K loop: a weight producer warp and a token producer warp copy each
//     128-input group's eight 1088-byte KMR4 blocks and the group's staged tokens into their
//     rings (cp.async.bulk, all of a group's copies in one instruction); eight warps turn the
//     blocks into fp16 w = (q - 8) s + z (the nibble OR-ed into the mantissa of 1024.0 gives
//     1024 + q, or 1024 + 16 q for tile rows 8..15, exactly; one HFMA2 applies s and z) and store
//     them to tensor memory with tcgen05.st; one thread issues the group's 8 MMAs (A in TMEM, B
//     in shared memory) and commits them to the stages' empty barriers.
//   * The accumulator stays in tensor memory across the CTA's K range; the epilogue reads it
//     (tcgen05.ld 32x32b), applies the token's RMSNorm factor / sigma and stores, adds to the
//     residual, or applies SiLU(gate) * up across the gate / up rows of a tile.  A K split over
//     a thread-block cluster merges the CTAs' partials through distributed shared memory.
//   * Every wait is bounded; a timeout records KMR_ERR_DEVICE_TIMEOUT, skips the remaining work,
//     drains the copies in flight and frees tensor memory.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "kmr_int4_mma.cuh"
#include "kmr_tcgemm.cuh"

namespace kmr {

namespace cg = cooperative_groups;

// Diagnostic build (-DKMR_TC_TRACE): per 128-input group, %globaltimer of the copy issue
// (producer), the unpack start and end (warp 2) and the MMA issue (warp 1), for the CTAs of
// one launch at grid positions (0, 0, 0) and (0, 1, 0) (every launch, or those with N equal to
// the armed value); kmr_tc_trace copies the records out.
#ifdef KMR_TC_TRACE
__device__ unsigned long long g_tc_trace[2][64][5];
__device__ int g_tc_trace_armed;
#define TC_MARK(g, k) do { const int cs_ = (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) ? 0 : (blockIdx.x == 0 && blockIdx.y == 1 && blockIdx.z == 0) ? 1 : -1; \
    if (cs_ >= 0 && (g_tc_trace_armed == 1 || g_tc_trace_armed == p.N) && (g) < 64) g_tc_trace[cs_][(g)][(k)] = globaltimer_ns(); } while (0)
#else
#define TC_MARK(g, k) do { } while (0)
#endif

namespace {

// Bounded wait that spins on the non-blocking phase test (no suspension: the pipeline's
// hand-offs are short and a waiting warp has nothing else to do).
__device__ __forceinline__ bool spin_wait(uint64_t* b, uint32_t parity, int* err) {
    if (mbar_test_wait(b, parity)) return true;
    // bounded by the SM's cycle counter (about 2 s at 2 GHz; reading it is cheap, unlike the
    // global nanosecond timer)
    const long long c0 = clock64();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_test_wait(b, parity)) return true;
        if ((it & 1023u) == 0 && clock64() - c0 > 4000000000ll) break;
    }
    set_error(err, KMR_ERR_DEVICE_TIMEOUT);
    return false;
}

constexpr int kTcRows = 128;                      // packed weight rows per CTA (MMA M)
constexpr int kTcTiles = kTcRows / 16;            // KMR4 tiles per CTA
constexpr uint32_t kTcWBytes = kTcTiles * kGroupBytes;      // one group of the CTA's tiles
constexpr uint32_t kTcABytes = kTcRows * 128 * 2;           // fp16 A operand of one group
constexpr uint32_t kCoreLBO = 128;                // bytes between core matrices along K


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
// Instruction descriptor of kind::f16: fp32 D, fp16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}
// D (+)= A B^T for one K = 16 step, kind::f16: A (128 rows x 16 inputs, fp16 pairs, even input in
// the low half) in tensor memory, B in shared memory (descriptor), fp32 D in tensor memory.
__device__ __forceinline__ void tc_mma_ta(uint32_t taddr, uint32_t a_taddr, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(taddr),
        "r"(a_taddr), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// Issue of a 32x32b.x16 load (thread i: TMEM lane base + i, 16 consecutive columns); the
// registers are valid after tc_wait_ld16 on the same array.
__device__ __forceinline__ void tc_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// Waits for this thread's TMEM loads; the registers pass through so that no use of them can be
// scheduled before the wait.
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
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
    // launched as a programmatic dependent: the projection that consumes this staging may start
    // its set-up and weight stream now; every global access here waits for the previous kernel
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, G = K >> 7, K4 = K >> 2;
    __half* xs = reinterpret_cast<__half*>(p.xs);
    const int tile = row / p.nt, rin = row % p.nt;
    // half offset of input k in this row's staged layout
    // input k of the row sits at position p of its 16-input k-step, p = 2 (k % 8) - k % 2 + 2 ((k % 16) / 8)
    // (the column order of the dequantised weights in tensor memory); pairs (k, k + 1), k even, stay adjacent
    auto at = [&](int k) {
        const int i = k & 15, pos = 2 * (i & 7) - (i & 1) + ((i >> 3) << 1);
        return (size_t(tile) * G + (k >> 7)) * size_t(p.nt) * 128 + ((k & 127) >> 5) * size_t(p.nt) * 32 +
               (rin >> 3) * 256 + (((k & 31) >> 4) * 2 + (pos >> 3)) * 64 + (rin & 7) * 8 + (pos & 7);
    };
    if (row >= p.M) {                             // tile padding: zeros, scale 0
        for (int k4 = tid; k4 < K4; k4 += kTcStageThreads) {
            *reinterpret_cast<uint32_t*>(xs + at(k4 * 4)) = 0u;
            *reinterpret_cast<uint32_t*>(xs + at(k4 * 4 + 2)) = 0u;
        }
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
        *reinterpret_cast<uint32_t*>(xs + at(k4 * 4)) = *reinterpret_cast<const uint32_t*>(&h01);
        *reinterpret_cast<uint32_t*>(xs + at(k4 * 4 + 2)) = *reinterpret_cast<const uint32_t*>(&h23);
    }
    if (tid == 0) {
        const float r = norm ? rsqrtf(tot / float(K) + p.eps) : 1.f;
        p.rs[row] = __fmul_rn(r, isg);
    }
}

// ---- GEMM
// Operand staging unit: one quarter of a 128-input group (32 inputs, two K = 16 MMAs).  Token
// (B) stages hold 8-row x 16-byte core matrices, the 4 K chunks of a row group side by side
// (512 B per row group); the dequantised weights (A) go to tensor memory.
constexpr uint32_t kTcQSBO = 512;                  // bytes between 8-row core-matrix groups

// Dequantises k-step ks (inputs 16 ks .. 16 ks + 15) of one KMR4 block (16 tile rows) into tensor
// memory with tcgen05.st.16x256b: lane (g, t) of the warp holds, as the block stores them, rows g
// and g + 8 at inputs 2t, 2t + 1 and 2t + 8, 2t + 9, and the 16x256b shape puts its registers at
// (row g, column 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).  So column c of the k-step holds
// the fp16 pair of inputs (c, c + 1) for even c and (c + 7, c + 8) for odd c, and the staged
// tokens follow the same order (tc_stage_kernel).
__device__ __forceinline__ void tc_unpack_kstep_tmem(const uint8_t* blk, int ks, int lane, __half2 s0, __half2 z0,
                                                     __half2 s1, __half2 z1, uint32_t taddr) {
    const __half2 off0 = __float2half2_rn(-1032.f);            // 1024 + q - 1032 = q - 8
    const __half2 sc1 = __float2half2_rn(0.0625f), off1 = __float2half2_rn(-72.f);   // (1024 + 16 q) / 16 - 72
    auto cvt = [](uint32_t v) { return *reinterpret_cast<const __half2*>(&v); };
    auto bits = [](__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); };
    const uint32_t w = *reinterpret_cast<const uint32_t*>(blk + (ks >> 2) * 512 + lane * 16 + (ks & 3) * 4);
    const uint32_t wh = w >> 8;
    const __half2 qa = __hadd2(cvt(and_or(w, 0x000F000Fu, 0x64006400u)), off0);      // row g, inputs 2t, 2t + 1
    const __half2 qb = __hfma2(cvt(and_or(w, 0x00F000F0u, 0x64006400u)), sc1, off1); // row g + 8
    const __half2 qc = __hadd2(cvt(and_or(wh, 0x000F000Fu, 0x64006400u)), off0);     // row g, inputs 2t + 8, + 9
    const __half2 qd = __hfma2(cvt(and_or(wh, 0x00F000F0u, 0x64006400u)), sc1, off1);// row g + 8
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(bits(__hfma2(qa, s0, z0))), "r"(bits(__hfma2(qc, s0, z0))), "r"(bits(__hfma2(qb, s1, z1))),
                 "r"(bits(__hfma2(qd, s1, z1)))
                 : "memory");
}

// Warp-specialised pipeline over 128-input groups: a deep ring of the CTA's eight KMR4 blocks per
// group (warp 0 copies them), a ring of the tile's staged tokens, one group per stage (warp 10),
// and a ring of dequantised weight groups in tensor memory.  Each ring stage has a full and an
// empty mbarrier.  A producer issues a group's copies from several lanes in one instruction
// (copies a warp issues one instruction after another do not overlap).  Warp 1 issues the
// group's eight MMAs and commits them to the token and tensor-memory stages' empty barriers;
// warps 2..9 dequantise (warp w: the two tiles of TMEM lane quarter w % 4, half of the k-steps)
// and then run the epilogue (warp w: lane quarter w % 4, half of the token columns).
// With a K split (gridDim.z > 1, one thread-block cluster along z) each CTA accumulates its own
// contiguous group range, parks the fp32 partial in its shared memory, and after a cluster
// barrier every CTA sums one token slice over the cluster's partials in rank order (DSMEM),
// so the result does not depend on which CTA finishes first.
constexpr int kTcUnpackWarps = 8;
constexpr int kTcTokenWarp = 2 + kTcUnpackWarps;
constexpr int kTcWarps = 3 + kTcUnpackWarps;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcMaxSplit = 4;
constexpr int kTcAQ = 4;                           // groups of dequantised weights (64 TMEM columns each)
constexpr int kTcWS = 8;                           // weight groups in flight
constexpr uint32_t kTcBarBytes = 512;              // mbarriers, the TMEM address and the abort flag
// token stages: 2 x 64 KB (256 tokens per CTA), 4 x 32 KB, 6 x 16 KB
__host__ __device__ constexpr int tc_bstages(int nt) { return nt >= 256 ? 2 : nt >= 128 ? 4 : 6; }
__host__ __device__ constexpr uint32_t tc_tmem_cols(int nt) { return nt + kTcAQ * 64 <= 256 ? 256u : 512u; }
static_assert((2 * (6 + kTcWS + kTcAQ) + 1) * 8 + 8 <= int(kTcBarBytes), "barrier area");

struct TcSmem {
    uint32_t w, bar, rs, total;
};
// [token stages][weight stages][barriers][row factors of the tile's tokens]
__host__ __device__ constexpr TcSmem tc_layout(int nt) {
    return TcSmem{uint32_t(tc_bstages(nt)) * uint32_t(nt) * 256u,
                  uint32_t(tc_bstages(nt)) * uint32_t(nt) * 256u + kTcWS * kTcWBytes,
                  uint32_t(tc_bstages(nt)) * uint32_t(nt) * 256u + kTcWS * kTcWBytes + kTcBarBytes,
                  uint32_t(tc_bstages(nt)) * uint32_t(nt) * 256u + kTcWS * kTcWBytes + kTcBarBytes + uint32_t(nt) * 4u};
}
// the K-split partial (128 rows x nt fp32) reuses the rings
static_assert(tc_layout(256).bar >= 128u * 256u * 4u && tc_layout(128).bar >= 128u * 128u * 4u &&
                  tc_layout(64).bar >= 128u * 64u * 4u, "partial tile does not fit the rings");
static_assert(tc_layout(256).total <= 227u * 1024u && tc_layout(128).total <= 227u * 1024u &&
                  tc_layout(64).total <= 227u * 1024u, "shared memory");

// Shared-memory matrix descriptor: K-major, no swizzle; start address, the byte distance
// between core matrices along K (leading) and between 8-row groups (stride), version bits 0b001.
__device__ __forceinline__ uint64_t tc_qdesc(uint32_t addr) {
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t((kCoreLBO >> 4) & 0x3FFFu) << 16) |
           (uint64_t((kTcQSBO >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46);
}

__device__ __forceinline__ float tc_silu_mul(float x, float up) {
    return __fmul_rn(__fdiv_rn(x, __fadd_rn(1.f, expf(-x))), up);
}

// Barrier among the epilogue warps (2..9) only.
__device__ __forceinline__ void tc_epilogue_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kTcUnpackWarps * 32) : "memory"); }

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const TcGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr TcSmem L = tc_layout(NT);
    constexpr int kBS = tc_bstages(NT), kWS = kTcWS, kAQ = kTcAQ;
    constexpr uint32_t kBBytes = uint32_t(NT) * 256, kQBytes = uint32_t(NT) * 64;
    constexpr uint32_t kTmemCols = tc_tmem_cols(NT);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.K >> 7;
    const int nsplit = int(gridDim.z), split = int(blockIdx.z);
    const int g0 = split * G / nsplit, ng = (split + 1) * G / nsplit - g0;
    const int tile0 = blockIdx.x * kTcTiles, ttile = blockIdx.y;
    uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + L.bar);
    uint64_t* w_empty = w_full + kWS;
    uint64_t* b_full = w_empty + kWS;
    uint64_t* b_empty = b_full + kBS;
    uint64_t* a_full = b_empty + kBS;
    uint64_t* a_empty = a_full + kAQ;
    uint64_t* acc_done = a_empty + kAQ;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    float* rs_s = reinterpret_cast<float*>(smem + L.rs);
    const uint32_t sbase = smem_u32(smem);

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kWS; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kTcUnpackWarps);     // one arrival per unpack warp
        }
        for (int s = 0; s < kBS; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);                  // tcgen05.commit
        }
        for (int s = 0; s < kAQ; ++s) {
            mbar_init(&a_full[s], kTcUnpackWarps);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(acc_done, 1);
        fence_mbar_init();
    }
    if (tid == 0) TC_MARK(62, 0);
    if (warp == 0) tc_alloc(tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) TC_MARK(62, 1);
    const uint32_t taddr = *tslot;
    auto fail = [&]() { *abort_flag = 1; };
    int issued_w = 0, issued_b = 0;                    // the producer lanes' fills
    bool have_acc = false;                             // epilogue warps: the accumulator is complete

    if (warp == 0) {
        // ---- weight producer: lane 0 waits for the stage and counts its bytes, lanes 0..7 copy
        // the eight tiles' blocks
        const uint64_t pol = policy_evict_first();
        for (int gi = 0; gi < ng; ++gi) {
            const int g = g0 + gi, s = gi % kWS;
            int go = 0;
            if (lane == 0 && !*abort_flag) {
                go = gi < kWS || spin_wait(&w_empty[s], uint32_t((gi / kWS - 1) & 1), p.err);
                if (go) mbar_arrive_expect_tx(&w_full[s], kTcWBytes);
                else fail();
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            if (lane == 0 && gi < 62) TC_MARK(gi, 0);
            fence_proxy_async_smem();                  // the unpack warps' reads of the stage come first
            if (lane < kTcTiles)
                bulk_g2s_stream(smem + L.w + s * kTcWBytes + lane * kGroupBytes,
                                p.w + (size_t(tile0 + lane) * G + g) * kGroupBytes, kGroupBytes, &w_full[s], pol);
            ++issued_w;
        }
    } else if (warp == kTcTokenWarp) {
        // ---- token producer: lanes 0..3 copy the group's four quarter blocks, once the staging
        // kernel has finished (the weight producer does not wait: the weights are constant)
        pdl_wait();
        for (int gi = 0; gi < ng; ++gi) {
            const int g = g0 + gi, s = gi % kBS;
            int go = 0;
            if (lane == 0 && !*abort_flag) {
                go = gi < kBS || spin_wait(&b_empty[s], uint32_t((gi / kBS - 1) & 1), p.err);
                if (go) mbar_arrive_expect_tx(&b_full[s], kBBytes);
                else fail();
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            if (lane < 4)
                bulk_g2s(smem + s * kBBytes + lane * kQBytes, p.xs + (size_t(ttile) * G + g) * NT * 128 + lane * NT * 32,
                         kQBytes, &b_full[s]);
            ++issued_b;
        }
    } else if (warp == 1) {
        // ---- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc(kTcRows, NT);
            for (int gi = 0; gi < ng && !*abort_flag; ++gi) {
                const int s = gi % kBS, as = gi % kAQ;
                if (!spin_wait(&a_full[as], uint32_t((gi / kAQ) & 1), p.err) ||
                    !spin_wait(&b_full[s], uint32_t((gi / kBS) & 1), p.err)) {
                    fail();
                    break;
                }
                tc_fence_after();
                if (gi < 62) TC_MARK(gi, 3);
                const uint32_t at = taddr + NT + as * 64, bb = sbase + s * kBBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma_ta(taddr, at + ks * 8, tc_qdesc(bb + (ks >> 1) * kQBytes + (ks & 1) * 256), idesc,
                              (gi > 0 || ks > 0) ? 1u : 0u);
                tc_commit(&b_empty[s]);
                tc_commit(&a_empty[as]);
                if (gi < 62) TC_MARK(gi, 4);
            }
            tc_commit(acc_done);                       // every MMA issued above
        }
    } else {
        // ---- unpack: warp w dequantises the two tiles of its tensor-memory lane quarter
        // (rows 32 (w % 4) .. + 31), k-steps 4 (w - 2) / 4 .. + 3 of each group
        const int ut = warp - 2, lq = warp & 3, kj = ut >> 2;
        // the row factors of the tile's tokens, for the epilogue (published by tc_epilogue_bar);
        // they and the residuals come from the previous kernels (programmatic dependent launch)
        pdl_wait();
        for (int i = ut * 32 + lane; i < NT; i += kTcUnpackWarps * 32) {
            const int t = ttile * NT + i;
            rs_s[i] = t < p.M ? p.rs[t] : 0.f;
        }
        for (int gi = 0; gi < ng; ++gi) {
            // lane 0 polls the barriers and the warp follows its verdict
            const int s = gi % kWS, as = gi % kAQ;
            int ok = 0;
            if (lane == 0 && !*abort_flag) {
                ok = spin_wait(&w_full[s], uint32_t((gi / kWS) & 1), p.err);
                if (ok && gi >= kAQ) ok = spin_wait(&a_empty[as], uint32_t((gi / kAQ - 1) & 1), p.err);
                if (!ok) fail();
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            tc_fence_after();
            if (warp == 2 && lane == 0 && gi < 62) TC_MARK(gi, 1);
            const uint8_t* wst = smem + L.w + s * kTcWBytes + (2 * lq) * kGroupBytes;
            const int g = lane >> 2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t* blk = wst + h * kGroupBytes;
                const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(blk + 1024 + g * 4);
                const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(blk + 1024 + (g + 8) * 4);
                const __half2 s0 = __float2half2_rn(bf16_lo(sz0)), z0 = __float2half2_rn(bf16_hi(sz0));
                const __half2 s1 = __float2half2_rn(bf16_lo(sz1)), z1 = __float2half2_rn(bf16_hi(sz1));
                const uint32_t acol = taddr + NT + as * 64 + (uint32_t(32 * lq + 16 * h) << 16);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc_unpack_kstep_tmem(blk, 4 * kj + k, lane, s0, z0, s1, z1, acol + (4 * kj + k) * 8);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (warp == 2 && lane == 0 && gi < 62) TC_MARK(gi, 2);
            if (lane == 0) {
                mbar_arrive(&a_full[as]);
                mbar_arrive(&w_empty[s]);
            }
        }
        int acc_ok = 0;
        if (lane == 0) acc_ok = !*abort_flag && mbar_wait(acc_done, 0u, p.err);
        have_acc = __shfl_sync(0xffffffffu, acc_ok, 0) != 0;
        pdl_launch_dependents();                      // the next kernel may launch during the epilogue
        tc_fence_after();
        tc_epilogue_bar();                             // rs_s complete
        if (warp == 2 && lane == 0) TC_MARK(63, 0);
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its weight rows) and half of the
        // token columns
        const int q = lq, chalf = kj;
        const int n = tile0 * 16 + q * 32 + lane;
        const uint32_t lane_base = taddr + (uint32_t(q * 32) << 16);
        const int cbeg = chalf * (NT / 2), cend = cbeg + NT / 2;
        if (have_acc && nsplit == 1) {
            // chunks of 16 token columns: the TMEM load and the residual rows of chunk c + 1 are in
            // flight while chunk c is processed
            constexpr int kChunks = NT / 32;
            static_assert(kChunks % 2 == 0, "chunk pairs");
            const bool resid = p.epi == EPI_RESID && n < p.N;
            auto load_res = [&](int c0, float (&r)[16]) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = ttile * NT + c0 + j;
                    r[j] = (resid && t < p.M) ? p.y[size_t(t) * p.ldy + n] : 0.f;
                }
            };
            auto process = [&](int c0, const uint32_t (&v)[16], const float (&res)[16]) {
                if (p.epi == EPI_SILU) {
                    // tokens in pairs: the gate lanes (tile rows 0..7) finish token j, the up lanes
                    // (rows 8..15) token j + 1, each with the partner row's value by shuffle
                    const bool lo = (lane & 15) < 8;
                    const int jj = (n >> 4) * 8 + (lane & 7);
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float xa = __fmul_rn(__uint_as_float(v[j]), rs_s[c0 + j]);
                        const float xb = __fmul_rn(__uint_as_float(v[j + 1]), rs_s[c0 + j + 1]);
                        const float dn = __shfl_down_sync(0xffffffffu, xa, 8);
                        const float upb = __shfl_up_sync(0xffffffffu, xb, 8);
                        const float gate = lo ? xa : upb, up = lo ? dn : xb;
                        const int t = ttile * NT + c0 + j + (lo ? 0 : 1);
                        if (t < p.M && jj < p.N / 2) p.y[size_t(t) * p.ldy + jj] = tc_silu_mul(gate, up);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = ttile * NT + c0 + j;
                        const float x = __fmul_rn(__uint_as_float(v[j]), rs_s[c0 + j]);
                        if (t < p.M && n < p.N) p.y[size_t(t) * p.ldy + n] = p.epi == EPI_RESID ? __fadd_rn(res[j], x) : x;
                    }
                }
            };
            uint32_t va[16], vb[16];
            float ra[16], rb[16];
            tc_ld16_issue(lane_base + uint32_t(cbeg), va);
            load_res(cbeg, ra);
            tc_wait_ld16(va);
            // chunk pairs (kChunks is even): va / ra hold the even chunk, vb / rb the odd one
#pragma unroll 1
            for (int ci = 0; ci < kChunks; ci += 2) {
                const int c0 = cbeg + ci * 16;
                tc_ld16_issue(lane_base + uint32_t(c0 + 16), vb);
                load_res(c0 + 16, rb);
                process(c0, va, ra);
                tc_wait_ld16(vb);
                const bool more = ci + 2 < kChunks;
                if (more) {
                    tc_ld16_issue(lane_base + uint32_t(c0 + 32), va);
                    load_res(c0 + 32, ra);
                }
                process(c0 + 16, vb, rb);
                if (more) tc_wait_ld16(va);
                if (warp == 2 && lane == 0) TC_MARK(40 + ci / 2, 1);
            }
        } else if (nsplit > 1) {
            // park the partial: part[c][r] = accumulator of weight row r, token column c (the
            // rings are idle once every MMA has completed)
            float* part = reinterpret_cast<float*>(smem);
#pragma unroll 1
            for (int c0 = cbeg; c0 < cend; c0 += 16) {
                float v[16];
                if (have_acc) {
                    tc_ld16(lane_base + uint32_t(c0), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(c0 + j) * kTcRows + q * 32 + lane] = v[j];
            }
            if (warp == 2 && lane == 0) TC_MARK(63, 1);
        }
    }
    if (nsplit > 1) {
        // ---- K-split merge over the cluster: CTA rank r finishes token columns
        // [r nt / nsplit, (r + 1) nt / nsplit), summing the partials in rank order
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (tid == 64) TC_MARK(63, 2);
        if (warp >= 2 && warp < 2 + kTcUnpackWarps) {
            const int rank = int(cluster.block_rank());
            const int cols = NT / nsplit, cbeg = rank * cols;
            const int et = tid - 64;
            const float* parts[kTcMaxSplit];
#pragma unroll
            for (int s = 0; s < kTcMaxSplit; ++s)
                parts[s] = s < nsplit ? cluster.map_shared_rank(reinterpret_cast<const float*>(smem), s) : nullptr;
            auto sum_at = [&](int idx) {
                float v = parts[0][idx];
#pragma unroll
                for (int s = 1; s < kTcMaxSplit; ++s)
                    if (s < nsplit) v = __fadd_rn(v, parts[s][idx]);
                return v;
            };
            constexpr int kStep = kTcUnpackWarps * 32, kB = 8;
            if (p.epi == EPI_SILU) {
                // output j of the tile pairs gate row (j / 8) 16 + j % 8 with the up row 8 below
                const int total = cols * 64;
                for (int e0 = et; e0 < total; e0 += kStep * kB) {
                    float x[kB], up[kB];
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int e = e0 + b * kStep;
                        const int c = cbeg + ((e < total ? e : 0) >> 6), jl = e & 63;
                        const int rg = (jl >> 3) * 16 + (jl & 7);
                        x[b] = sum_at(c * kTcRows + rg);
                        up[b] = sum_at(c * kTcRows + rg + 8);
                    }
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int e = e0 + b * kStep;
                        if (e >= total) continue;
                        const int c = cbeg + (e >> 6), jl = e & 63;
                        const int t = ttile * NT + c, jj = blockIdx.x * 64 + jl;
                        if (t < p.M && jj < p.N / 2)
                            p.y[size_t(t) * p.ldy + jj] = tc_silu_mul(__fmul_rn(x[b], rs_s[c]), __fmul_rn(up[b], rs_s[c]));
                    }
                }
            } else {
                const int total = cols * kTcRows;
                for (int e0 = et; e0 < total; e0 += kStep * kB) {
                    float x[kB], res[kB];
                    // all loads of the batch (partials and residuals) before its stores
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int e = e0 + b * kStep;
                        const int ee = e < total ? e : 0;
                        const int c = cbeg + (ee >> 7), r = ee & 127;
                        const int t = ttile * NT + c, nn = tile0 * 16 + r;
                        x[b] = sum_at(c * kTcRows + r);
                        res[b] = (p.epi == EPI_RESID && e < total && t < p.M && nn < p.N) ? p.y[size_t(t) * p.ldy + nn] : 0.f;
                    }
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int e = e0 + b * kStep;
                        if (e >= total) continue;
                        const int c = cbeg + (e >> 7), r = e & 127;
                        const int t = ttile * NT + c, nn = tile0 * 16 + r;
                        if (t >= p.M || nn >= p.N) continue;
                        const float xv = __fmul_rn(x[b], rs_s[c]);
                        p.y[size_t(t) * p.ldy + nn] = p.epi == EPI_RESID ? __fadd_rn(res[b], xv) : xv;
                    }
                }
            }
        }
        if (tid == 64) TC_MARK(63, 3);
        cluster.sync();                                // the peers' reads of this CTA's partial are done
    }
    if (*abort_flag && lane == 0) {
        // drain the fills still in flight before the CTA's shared memory is released: the
        // latest issued phase of every stage (earlier phases of a stage have completed)
        if (warp == 0)
            for (int i = issued_w - kWS < 0 ? 0 : issued_w - kWS; i < issued_w; ++i)
                mbar_wait(&w_full[i % kWS], uint32_t((i / kWS) & 1), p.err, 50000000ull);
        if (warp == kTcTokenWarp)
            for (int i = issued_b - kBS < 0 ? 0 : issued_b - kBS; i < issued_b; ++i)
                mbar_wait(&b_full[i % kBS], uint32_t((i / kBS) & 1), p.err, 50000000ull);
    }
    if (tid == 64) TC_MARK(63, 4);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(taddr, kTmemCols);
}

template <int NT>
cudaError_t tc_gemm_set_attr() {
    return cudaFuncSetAttribute(tc_gemm_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(tc_layout(NT).total));
}

template <int NT>
cudaError_t tc_gemm_launch(const TcGemmParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.N / kTcRows, (p.M + NT - 1) / NT, p.ksplit);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_layout(NT).total;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = p.ksplit;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<NT>, p);
}

}  // namespace

bool tc_gemm_supported(int N, int K) { return N > 0 && N % kTcRows == 0 && K > 0 && K % 128 == 0 && K <= kTcStageMaxK; }

int tc_rows_pad(int M) { return (M + 255) / 256 * 256; }

// Tile width (tokens per CTA) and K split for an N x K projection of M tokens.  The modelled time
// of a choice is waves x (groups per CTA x group time + fixed cost), with group times measured for
// M = 128 MMAs (a 128 x N x 16 MMA costs about the same for any N <= 128; N = 256 runs at the full
// rate) and the fixed cost of a CTA (prologue, epilogue, and the split merge).  The K split fixes
// the order of each output's fp32 sums, so it depends on the projection's shape only (chosen for a
// 512-token chunk): a token's result is then the same whatever the prompt length or chunking.
// The tile width follows M; it does not change any output's arithmetic.
namespace {
double tc_model_us(int nt, int ks, int N, int K, int M, int sms) {
    const int G = K / 128, tiles = N / kTcRows;
    const long long ctas = (long long)tiles * ((M + nt - 1) / nt) * ks;
    const long long waves = (ctas + sms - 1) / sms;
    const double group_us = nt == 256 ? 0.55 : 0.33;
    const double fixed_us = 2.0 + (ks > 1 ? 0.5 + nt * 0.006 : 0.0);
    return double(waves) * (double((G + ks - 1) / ks) * group_us + fixed_us);
}
}  // namespace

TcPlan tc_gemm_plan(int N, int K, int M, int sms) {
    const int G = K / 128;
    const int nts[3] = {256, 128, 64};
    // the split: best at the reference chunk
    int ks_best = 1;
    double t_ref = 1e30;
    for (int nt : nts)
        for (int ks = 1; ks <= kTcMaxSplit && ks <= G; ks *= 2) {
            const double t = tc_model_us(nt, ks, N, K, 512, sms);
            if (t < t_ref * 0.999) {
                t_ref = t;
                ks_best = ks;
            }
        }
    // the tile width: best for this M with that split
    TcPlan best = {64, ks_best};
    double bt = 1e30;
    for (int nt : nts) {
        const double t = tc_model_us(nt, ks_best, N, K, M, sms);
        if (t < bt * 0.999) {
            bt = t;
            best.nt = nt;
        }
    }
    return best;
}

cudaError_t tc_gemm_set_attributes() {
    cudaError_t e = tc_gemm_set_attr<256>();
    if (e == cudaSuccess) e = tc_gemm_set_attr<128>();
    if (e == cudaSuccess) e = tc_gemm_set_attr<64>();
    return e;
}

cudaError_t launch_tc_stage(const TcStageParams& p, cudaStream_t st) {
    const int rows = (p.M + p.nt - 1) / p.nt * p.nt;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows);
    cfg.blockDim = dim3(kTcStageThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_stage_kernel, p);
}

cudaError_t launch_tc_gemm(const TcGemmParams& p, cudaStream_t st) {
    if (p.ksplit < 1 || p.ksplit > kTcMaxSplit || (p.ksplit & (p.ksplit - 1)) || p.ksplit > p.K / 128)
        return cudaErrorInvalidValue;
    switch (p.nt) {
        case 256: return tc_gemm_launch<256>(p, st);
        case 128: return tc_gemm_launch<128>(p, st);
        case 64: return tc_gemm_launch<64>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kmr

#ifdef KMR_TC_TRACE
extern "C" int kmr_tc_trace(int arm, unsigned long long* out) {
    if (arm >= 0) return cudaMemcpyToSymbol(kmr::g_tc_trace_armed, &arm, sizeof(int)) == cudaSuccess ? 0 : -1;
    return cudaMemcpyFromSymbol(out, kmr::g_tc_trace, sizeof(kmr::g_tc_trace)) == cudaSuccess ? 0 : -1;
}
#endif
