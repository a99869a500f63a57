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
    if (p.d == 128)
        prefill_rope_kernel<128><<<dim3(p.T, p.nkv), threads, 0, st>>>(p);
    else
        prefill_rope_kernel<64><<<dim3(p.T, p.nkv), threads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kmr
