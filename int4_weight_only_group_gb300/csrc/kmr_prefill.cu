// Prefill's per-position attention prologue ("kaminari — a single-GPU Qwen3-VL inference
// engine, explained", §04 Request lifecycle: prefill runs the whole prompt through the
// decoder once, fills the static cache and yields the first token; §03: 3-section M-RoPE
// over (T, H, W) position ids, per-head q/k RMSNorm, the cache mutated in place).
//
// For every prompt position i of a chunk and KV head h, one CTA of (rep + 2) warps takes the
// QKV rows the GEMV produced: warps 0..rep-1 the query heads of the group, warp rep the key,
// warp rep+1 the value.  Queries and keys get the per-head RMSNorm and the rotary embedding
// at the position's (T, H, W) ids; the key and value are rounded to bf16 and stored in the
// cache row at start_pos + i; the queries go to a buffer the attention kernel reads.  The
// arithmetic is the decode attention prologue's, operation for operation, so a prompt
// position's q, k and v are the bits a decode step would give the same token.
#include <math.h>

#include "kmr_internal.cuh"

namespace kmr {
namespace {

template <int D>
__global__ void __launch_bounds__(192) prefill_rope_kernel(const PrefillRopeParams p) {
    // a programmatic dependent of the QKV projection: release the attention launch, then wait
    // for the projection's rows before reading anything
    pdl_launch_dependents();
    pdl_wait();
    constexpr int EPL = D / 32;
    const int i = blockIdx.x, h = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rep = p.nq / p.nkv;
    if (warp > rep + 1) return;
    const bool isq = warp < rep, isk = warp == rep;
    const float* row = p.qkv + size_t(i) * p.qkv_ld;
    const float* src = isq ? row + size_t(h * rep + warp) * D
                           : (isk ? row + size_t(p.nq) * D + size_t(h) * D : row + size_t(p.nq + p.nkv) * D + size_t(h) * D);
    float x[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[e] = src[lane * EPL + e];
    if (warp <= rep) {
        const uint16_t* nrm = isq ? p.qn_w : p.kn_w;
        if (nrm) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) ss = __fmaf_rn(x[e], x[e], ss);
            const float r = rsqrtf(warp_sum(ss) / float(D) + p.eps);
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[e] = __fmul_rn(__fmul_rn(x[e], r), bf16_to_f32(nrm[lane * EPL + e]));
        }
        // 3-section M-RoPE: frequency f turns the pair (f, f + D/2); the partner dim is 16 lanes away
        const bool lo = lane < 16;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int dim = lane * EPL + e, f = dim % (D / 2);
            const int axis = f < p.sec0 ? 0 : (f < p.sec0 + p.sec1 ? 1 : 2);
            const float pos = float(p.positions[size_t(axis) * p.T + i]);
            float sn, cs;
            sincosf(pos * p.inv_freq[f], &sn, &cs);
            const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
            x[e] = lo ? __fsub_rn(__fmul_rn(x[e], cs), __fmul_rn(other, sn))
                      : __fadd_rn(__fmul_rn(x[e], cs), __fmul_rn(other, sn));
        }
    }
    if (isq) {
        float* q = p.q_out + size_t(i) * p.nq * D + size_t(h * rep + warp) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) q[lane * EPL + e] = x[e];
    } else {
        uint16_t* cache = (isk ? p.kc : p.vc) + ((size_t(p.slot) * p.nkv + h) * p.S + p.start + i) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) cache[lane * EPL + e] = f32_to_bf16_rn(x[e]);
    }
    if (h == 0 && threadIdx.x == 0) {
        // the attention kernel's per-row view of the chunk: one cache row, position start + i
        p.slot_ids[i] = p.slot;
        p.cpos[i] = p.start + i;
        if (i == p.T - 1 && p.state_pos) {
            // the LM head advances this state to the first decode step's
            for (int a = 0; a < 3; ++a) p.state_pos[a] = p.positions[size_t(a) * p.T + i];
            *p.state_cpos = p.start + i;
            *p.state_fin = 0;
        }
    }
}

}  // namespace

cudaError_t launch_prefill_rope(const PrefillRopeParams& p, cudaStream_t st) {
    const int threads = (p.nq / p.nkv + 2) * 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.T, p.nkv);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.d == 128) return cudaLaunchKernelEx(&cfg, prefill_rope_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, prefill_rope_kernel<64>, p);
}

}  // namespace kmr

// ---------------------------------------------------------------------------------------------
// Causal attention of a prefill chunk on the tensor cores ("The Ghost in the Batch", What
// Attention Does: out = softmax(q K^T / sqrt(d)) V; prompt position i attends cache positions
// 0..start + i).  Grid (position blocks, KV head): a CTA of 4 warps takes BQ = 4 * 16 / rep
// consecutive positions and the rep query heads of its KV head; warp w owns 16 query rows
// (row r: position w * 16 / rep + r / rep, head r % rep).  K and V blocks of 64 positions are
// double-buffered in shared memory (cp.async, rows padded to d + 8 halves so that ldmatrix is
// conflict-free); per block a warp forms S = Q K^T (mma.sync bf16, queries rounded to bf16
// after the scale), applies the causal mask, updates its base-2 online softmax, and adds P V
// with P rounded to bf16 straight from the S accumulators.
namespace kmr {
namespace {

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(fill ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kPaBK = 64;                   // key positions per block
constexpr float kLog2eP = 1.4426950408889634f;

template <int D>
__host__ __device__ constexpr int pa_pitch() { return D + 8; }  // halves per staged row

template <int D, int REP>
__global__ void __launch_bounds__(128) prefill_attn_kernel(const PrefillAttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    // a programmatic dependent of the q/k norm + RoPE kernel: release the next launch, then wait
    // for the rotated queries and the cache rows before reading anything
    pdl_launch_dependents();
    pdl_wait();
    constexpr int PPT = 16 / REP, BQ = 4 * PPT, KT = D / 16, NT = D / 8, P = pa_pitch<D>();
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem);                       // [2][64][P]
    uint16_t* vs = ks + 2 * kPaBK * P;                                        // [2][64][P]
    const int qb = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int q0 = qb * BQ;
    const int qlast = min(p.T, q0 + BQ) - 1;                                  // last chunk position here
    const int kv_end = p.start + qlast + 1;                                   // positions [0, kv_end)
    const int nkb = (kv_end + kPaBK - 1) / kPaBK;
    const size_t base = (size_t(p.slot) * p.nkv + h) * p.S * D;
    const uint16_t* kg = p.kc + base;
    const uint16_t* vg = p.vc + base;

    auto load_block = [&](int kb, int buf) {
        constexpr int CPR = D / 8;                                            // 16-byte chunks per row
        for (int c = tid; c < kPaBK * CPR; c += 128) {
            const int r = c / CPR, ch = c % CPR, pos = kb * kPaBK + r;
            const bool ok = pos < kv_end;
            const size_t src = size_t(ok ? pos : 0) * D + ch * 8;
            cp_async16(ks + (size_t(buf) * kPaBK + r) * P + ch * 8, kg + src, ok);
            cp_async16(vs + (size_t(buf) * kPaBK + r) * P + ch * 8, vg + src, ok);
        }
        cp_async_commit();
    };
    load_block(0, 0);

    // the warp's 16 query rows (g and g + 8 for this lane), scaled to base 2 and rounded to bf16
    const float qscale = __fmul_rn(p.scale, kLog2eP);
    int pl[2], hd[2];
    bool live[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = g + 8 * i;
        pl[i] = q0 + warp * PPT + r / REP;
        hd[i] = h * REP + r % REP;
        live[i] = pl[i] < p.T;
    }
    uint32_t qf[KT][4];
#pragma unroll
    for (int ks_ = 0; ks_ < KT; ++ks_) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float* src = p.q + (size_t(live[i] ? pl[i] : 0) * p.nq + hd[i]) * D + ks_ * 16 + 2 * t;
            const float2 lo = live[i] ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
            const float2 hi = live[i] ? *reinterpret_cast<const float2*>(src + 8) : make_float2(0.f, 0.f);
            qf[ks_][i] = pack_bf16x2(__fmul_rn(lo.x, qscale), __fmul_rn(lo.y, qscale));
            qf[ks_][2 + i] = pack_bf16x2(__fmul_rn(hi.x, qscale), __fmul_rn(hi.y, qscale));
        }
    }
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const int qabs0 = p.start + pl[0], qabs1 = p.start + pl[1];
    const int lm = lane >> 3, lr = lane & 7;                                  // ldmatrix: matrix, row

    for (int kb = 0; kb < nkb; ++kb) {
        const int buf = kb & 1;
        if (kb + 1 < nkb) {
            load_block(kb + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t* kb_s = ks + size_t(buf) * kPaBK * P;
        const uint16_t* vb_s = vs + size_t(buf) * kPaBK * P;
        // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int ks_ = 0; ks_ < KT; ++ks_) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4(b, kb_s + size_t(np * 16 + (lm >> 1) * 8 + lr) * P + ks_ * 16 + (lm & 1) * 8);
                mma_bf16(s[2 * np], qf[ks_], b[0], b[1]);
                mma_bf16(s[2 * np + 1], qf[ks_], b[2], b[3]);
            }
        }
        // ---- causal mask, online softmax (rows g: elements 0, 1; rows g + 8: elements 2, 3)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kpos = kb * kPaBK + n * 8 + 2 * t + (e & 1);
                const int i = e >> 1;
                if (kpos > (i ? qabs1 : qabs0) || !live[i]) s[n][e] = -INFINITY;
                mx[i] = fmaxf(mx[i], s[n][e]);
            }
        float alpha[2], mref[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
            const float mn = fmaxf(m[i], mx[i]);
            mref[i] = mn == -INFINITY ? 0.f : mn;
            alpha[i] = m[i] == -INFINITY ? 0.f : exp2f(__fsub_rn(m[i], mref[i]));
            m[i] = mn;
            l[i] = __fmul_rn(l[i], alpha[i]);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            o[n][0] = __fmul_rn(o[n][0], alpha[0]);
            o[n][1] = __fmul_rn(o[n][1], alpha[0]);
            o[n][2] = __fmul_rn(o[n][2], alpha[1]);
            o[n][3] = __fmul_rn(o[n][3], alpha[1]);
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = e >> 1;
                const float pe = s[n][e] == -INFINITY ? 0.f : exp2f(__fsub_rn(s[n][e], mref[i]));
                s[n][e] = pe;
                l[i] = __fadd_rn(l[i], pe);
            }
        // ---- O += P V: 4 k-steps of 16 keys; P's A fragment comes from two S tiles
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {pack_bf16x2(s[2 * j][0], s[2 * j][1]), pack_bf16x2(s[2 * j][2], s[2 * j][3]),
                                   pack_bf16x2(s[2 * j + 1][0], s[2 * j + 1][1]),
                                   pack_bf16x2(s[2 * j + 1][2], s[2 * j + 1][3])};
#pragma unroll
            for (int dp = 0; dp < NT / 2; ++dp) {
                uint32_t b[4];
                ldsm_x4_t(b, vb_s + size_t(j * 16 + (lm & 1) * 8 + lr) * P + dp * 16 + (lm >> 1) * 8);
                mma_bf16(o[2 * dp], a, b[0], b[1]);
                mma_bf16(o[2 * dp + 1], a, b[2], b[3]);
            }
        }
        __syncthreads();                                                      // the buffer is refilled next
    }
    // ---- normalise and store: lane holds dims n * 8 + 2t, +1 of rows g and g + 8
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float lt = l[i];
        lt = __fadd_rn(lt, __shfl_xor_sync(0xffffffffu, lt, 1));
        lt = __fadd_rn(lt, __shfl_xor_sync(0xffffffffu, lt, 2));
        if (!live[i]) continue;
        float* dst = p.out + (size_t(pl[i]) * p.nq + hd[i]) * D;
#pragma unroll
        for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(dst + n * 8 + 2 * t) =
                make_float2(__fdiv_rn(o[n][2 * i], lt), __fdiv_rn(o[n][2 * i + 1], lt));
    }
}

template <int D, int REP>
cudaError_t launch_pa(const PrefillAttnParams& p, cudaStream_t st) {
    constexpr int BQ = 4 * (16 / REP);
    const size_t smem = size_t(4) * kPaBK * pa_pitch<D>() * 2;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel<D, REP>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.T + BQ - 1) / BQ, p.nkv);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_attn_kernel<D, REP>, p);
}

}  // namespace

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t st) {
    const int rep = p.nq / p.nkv;
    if (p.d == 128) {
        if (rep == 1) return launch_pa<128, 1>(p, st);
        if (rep == 2) return launch_pa<128, 2>(p, st);
        return launch_pa<128, 4>(p, st);
    }
    if (rep == 1) return launch_pa<64, 1>(p, st);
    if (rep == 2) return launch_pa<64, 2>(p, st);
    return launch_pa<64, 4>(p, st);
}

}  // namespace kmr
