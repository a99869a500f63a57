// Internal declarations shared by the library's translation units: device
// helpers (mbarrier, bulk async copies, programmatic dependent launch, int4
// magic-number dequantisation) and the kernel parameter blocks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kmr.h"

namespace kmr {

constexpr int kThreads = 256;        // every compute kernel uses 8 warps
constexpr int kTileRows = 8;         // rows per packed int4 tile / LM-head tile
constexpr int kMaxMB = 8;            // rows of x per GEMV staging group (a launch serves up to 2 groups)
constexpr int kMaxBatch = 16;

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Programmatic dependent launch: release the next kernel in the stream early,
// and wait for the previous kernel's completion (and memory) before touching
// anything it writes.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
// Bulk (non-tensor) async copy global -> shared, completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(b))
        : "memory");
}
// Same, with an L2 evict-first hint for data streamed exactly once (weights).
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* b,
                                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(b)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok;
}
// Non-blocking test of an mbarrier phase (try_wait may suspend the thread for a while).
__device__ __forceinline__ uint32_t mbar_test_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait on an mbarrier phase.  Gives up after ~`limit_ns` (or 2^26
// polls), records KMR_ERR_DEVICE_TIMEOUT and returns false; never traps.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, int* err,
                                          uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
        if (mbar_try_wait(b, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
    }
    atomicCAS(err, 0, KMR_ERR_DEVICE_TIMEOUT);
    return false;
}

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// (a & mask) | bits — one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
    return d;
}
// acc += w.lo * x.lo + w.hi * x.hi with f16 products accumulated in f32.
__device__ __forceinline__ void fma_f16x2_f32(float& acc, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n}"
        : "+f"(acc)
        : "r"(w), "r"(x));
}
// acc += w.lo * x.lo + w.hi * x.hi with bf16 products accumulated in f32.
__device__ __forceinline__ void fma_bf16x2_f32(float& acc, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %0, a1, b1, %0;\n}"
        : "+f"(acc)
        : "r"(w), "r"(x));
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;   // NaN
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// bf16 tensor-core helpers: packing, m16n8k16 with fp32 accumulation, 8x8 matrix loads.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return uint32_t(f32_to_bf16_rn(lo)) | (uint32_t(f32_to_bf16_rn(hi)) << 16);
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
// Smallest power of two >= n (1 for n <= 1).
__host__ __device__ constexpr int pow2_at_least(int n) { return n <= 1 ? 1 : 2 * pow2_at_least((n + 1) / 2); }

// Sum of NV per-lane values over the warp, scattered: value i's total ends on the
// lanes l with l / (32 / NV) == i.  Each level pairs lane l with l ^ off (off = 16 .. 1)
// exactly as the xor butterfly of warp_sum does, and a sum is commutative, so every
// value gets the same bits the butterfly gives it, with NV - 1 + log2(32 / NV)
// shuffles instead of 5 NV.
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
    int n = NV;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const int half = n / 2;
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) {
                if (i < half) {
                    const float keep = up ? v[i + half] : v[i];
                    const float send = up ? v[i] : v[i + half];
                    v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, off));
                }
            }
            n = half;
        } else {
            v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], off));
        }
    }
    return v[0];
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------------ packed layout
struct PackGeom {
    int N, K, groups, tiles, tile_bytes;   // 16-row tiles, groups of 128 inputs
    long long bytes;
};
constexpr int kGroupBytes = 1088;          // one (tile, group): 1024 B of nibbles + 16 x (s, z)
// Returns false for unsupported shapes (group != 128, K not a multiple of 128).
bool pack_geom(int N, int K, int group, PackGeom* g);

// ------------------------------------------------------------------ GEMV
enum InKind { IN_F32 = 0, IN_F32_NORM = 1, IN_EMBED_NORM = 2 };
enum EpiKind { EPI_STORE = 0, EPI_RESID = 1, EPI_SILU = 2 };

struct GemvParams {
    const uint8_t* w;            // packed KMR4 tiles
    int N, K, tiles, tile_bytes;
    int M;                       // rows of x in this pass (<= MB <= 8)
    int in_kind;
    const float* x;              // [M][K] fp32, row stride K (IN_F32*)
    const uint16_t* embed;       // IN_EMBED_NORM: bf16 [V][K]
    const int32_t* tokens;       //   token per row (ids outside [0, vocab) read row 0 and set KMR_ERR_INVALID_ARG)
    int vocab;
    float* x_out;                //   CTA 0 stores the embedded rows (fp32 [M][K]) here
    const uint16_t* norm_w;      // bf16 [K] (IN_*_NORM)
    float eps;
    int epi;
    float* y;                    // output, row stride ldy
    int ldy;
    int* err;
    int nstage;                  // weight ring depth (tiles)
    int halves;                  // 1, or 2: rows [0, MB) then [MB, 2 MB) from one weight fill (needs all tiles resident)
};
size_t gemv_smem_bytes(int MB, int K, int tile_bytes, int nstage);
cudaError_t launch_gemv(const GemvParams& p, int MB, int grid, cudaStream_t st, bool pdl);
int gemv_pick_mb(int M);
bool gemv_two_halves_ok(int tiles, int grid, int tile_bytes);
// At most one CTA per SM, each owning an equal count of whole 16-row tiles.
int gemv_grid(int tiles, int sms);
int gemv_nstage(int tiles, int grid, int tile_bytes);

// ------------------------------------------------------------------ LM head
struct HeadParams {
    const uint16_t* E;           // bf16 [V][K]
    int V, K, tiles;
    int M;                       // rows in this pass (<= MB)
    const float* x;              // residual rows fp32 [M][K]
    const uint16_t* norm_w;
    float eps;
    float* logits;               // fp32 [M][ldl] or nullptr
    int ldl;
    float* gbest_val;            // [grid][MB]
    int* gbest_idx;              // [grid][MB]
    int* counter;                // one int (zero between launches)
    // step state of these rows (finalize)
    int32_t* tokens;
    int32_t* positions;          // [3][pos_ld]
    int pos_ld;
    int32_t* cpos;
    uint8_t* finished;
    int eos, pad, max_len;
    int* err;
    int nstage;
};
size_t head_smem_bytes(int MB, int K, int nstage);
cudaError_t launch_head(const HeadParams& p, int MB, int grid, cudaStream_t st, bool pdl);
constexpr int kMaxHeadRows = 16;     // rows of x per LM-head pass
int head_pick_mb(int M);

// ------------------------------------------------------------------ attention
struct AttnParams {
    const float* in;             // fused: raw qkv rows [B][in_ld]; plain: q rows [B][in_ld]
    int in_ld;
    int fused;
    uint16_t* kc;                // bf16 [slots][nkv][S][d] (one layer)
    uint16_t* vc;
    const int32_t* slot_ids;
    const int32_t* cpos;
    const int32_t* positions;    // [3][pos_ld] (fused)
    int pos_ld;
    const uint8_t* finished;     // may be null (plain)
    const uint16_t* qn_w;        // bf16 [d] or null (no q/k norm)
    const uint16_t* kn_w;
    float eps;
    const float* inv_freq;       // [d/2]
    int sec0, sec1;              // frequencies [0,sec0) follow T, [sec0, sec0+sec1) follow H, rest W
    int B, nq, nkv, d, S, slots;
    float scale;
    int tsplit;                  // grid.x (global merge): largest number of splits per (row, kv head)
    int nstage;                  // K/V ring stages (set by launch_attn from S and the split count)
    int cluster;                 // 1: splits of a (row, kv head) form one cluster, merged through DSMEM
    float* out;                  // [B][nq*d]
    float* part;                 // [B][nkv][tsplit][rep][d+2]
    int* counters;               // [B][nkv]
    int* err;
    // Fused QKV projection (cluster mode; wqkv == null: off).  Rank s of the cluster of
    // (KV head h, row b) computes the head group's QKV rows [s, s+1) * tpr tiles of row b itself, with the
    // one-row int4 GEMV's arithmetic, and the cluster all-gathers them through distributed
    // shared memory; the attention prologue then reads q, k, v from shared memory.
    const uint8_t* wqkv;         // packed QKV weights (KMR4; N = (nq + 2 nkv) d, K = hidden)
    int qkv_tile_bytes;          // (hidden / 128) * 1088
    int hidden;
    int x_kind;                  // IN_F32_NORM (x = residual row) or IN_EMBED_NORM (x = E[token])
    const float* x;              // residual rows fp32 [B][hidden]
    const uint16_t* embed;       // bf16 [vocab][hidden]
    const int32_t* tokens;       // token of each row (IN_EMBED_NORM)
    int vocab;
    float* x_out;                // IN_EMBED_NORM: the embedded rows are stored here (one CTA per row)
    const uint16_t* in_norm_w;   // bf16 [hidden]: input RMSNorm weight
};
// Shared-memory poisoning diagnostic (kmr_poison.cu).
// Shared-prefix (cascade) decode attention (kmr_cascade.cu): row b attends positions
// [0, prefix_len) of cache row prefix_slot, then [prefix_len, cpos[b]] of its own row.
constexpr int kCascadeMaxChunk = 256;       // prefix positions staged per CTA
struct CascadeParams {
    const float* q;                         // [B, nq, d]
    const uint16_t* kc;                     // one layer [slots][nkv][S][d]
    const uint16_t* vc;
    const int32_t* slot_ids;
    const int32_t* cpos;
    float* out;                             // [B, nq, d]
    float* part;                            // [B][nq][psplits][d + 2] prefix split states
    int* err;
    int B, nq, nkv, d, S, slots;
    int prefix_slot, prefix_len, pchunk, psplits;
    float scale;
};
void cascade_plan(int prefix_len, int nkv, int sms, int* pchunk, int* psplits);
size_t cascade_workspace_bytes(int B, int nq, int d, int psplits);
cudaError_t launch_cascade(const CascadeParams& p, cudaStream_t st);

// Prefill's int4 projections (kmr_gemm.cu): rows staged once, then a weight-stationary GEMM.
struct StageParams {
    int in_kind;                            // IN_F32, IN_F32_NORM or IN_EMBED_NORM
    const float* x;                         // [M][K]
    const uint16_t* embed;                  // bf16 [vocab][K] (IN_EMBED_NORM)
    const int32_t* tokens;
    int vocab;
    float* x_out;                           // IN_EMBED_NORM: embedded rows [M][K] (or null)
    const uint16_t* norm_w;                 // bf16 [K] (IN_*_NORM)
    float eps;
    int M, Mpad, K;
    uint16_t* xs;                           // fp16 [K/128][Mpad][128] in B-fragment order
    float2* xst;                            // [K/128][Mpad]: (X', 1/sigma)
    float* rnorm;                           // [Mpad]: RMSNorm factor (1 without norm)
    int* err;
};
struct GemmParams {
    const uint8_t* w;                       // packed KMR4
    int N, K, tiles;
    const uint16_t* xs;
    const float2* xst;
    const float* rnorm;
    int M, Mpad, epi;
    float* y;
    int ldy;
    int* err;
};
size_t gemm_smem_bytes(int tiles_per_cta);
int gemm_rows_pad(int M);
cudaError_t gemm_set_attributes();
cudaError_t launch_stage(const StageParams& p, cudaStream_t st);
cudaError_t launch_gemm(const GemmParams& p, int sms, cudaStream_t st);

// Prefill's per-position attention prologue (kmr_prefill.cu): q/k RMSNorm + M-RoPE of T
// prompt positions, K/V into cache row `slot` at [start, start + T), queries to q_out.
struct PrefillRopeParams {
    const float* qkv;                       // [T][qkv_ld] rows [q heads | k | v] from the QKV GEMV
    int qkv_ld;
    float* q_out;                           // [T][nq * d]
    uint16_t* kc;                           // one layer [slots][nkv][S][d]
    uint16_t* vc;
    const int32_t* positions;               // [3][T] (T, H, W) ids
    const uint16_t* qn_w;                   // bf16 [d] or null
    const uint16_t* kn_w;
    const float* inv_freq;                  // [d/2]
    int sec0, sec1;
    float eps;
    int T, start, slot, nq, nkv, d, S;
    int32_t* slot_ids;                      // [T] out: slot, for the attention kernel
    int32_t* cpos;                          // [T] out: start + i
    int32_t* state_pos;                     // [3] out: ids of the last position (or null)
    int32_t* state_cpos;                    // out: start + T - 1
    uint8_t* state_fin;                     // out: 0
};
cudaError_t launch_prefill_rope(const PrefillRopeParams& p, cudaStream_t st);
// Causal attention of a prefill chunk on the tensor cores (kmr_prefill.cu): prompt position i
// of the chunk attends cache positions [0, start + i] of row `slot`.
struct PrefillAttnParams {
    const float* q;                         // [T][nq * d] normalised, rotated queries
    const uint16_t* kc;                     // one layer [slots][nkv][S][d]
    const uint16_t* vc;
    int slot, start, T, nq, nkv, d, S;
    float scale;
    float* out;                             // [T][nq * d]
};
cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t st);

// KV row migration (kmr_slots.cu): positions [0, length) of one cache row, every layer,
// K and V, from a source cache to a destination cache of the same L, n_kv and d.
struct KvCopyParams {
    const uint16_t* src_k;
    const uint16_t* src_v;
    uint16_t* dst_k;
    uint16_t* dst_v;
    int L, nkv, d;
    int src_slots, src_max_len, src_row;
    int dst_slots, dst_max_len, dst_row;
    long long units;                        // 16-byte units per (layer, K/V, head) segment
};
cudaError_t launch_kv_row_copy(const KvCopyParams& p, int sms, cudaStream_t st);

cudaError_t poison_set_attributes();
cudaError_t launch_smem_poison(uint32_t pattern, int sms, cudaStream_t st);

constexpr int kAttnClusterSplits = 8;     // cluster size of the DSMEM-merged attention (portable)
size_t attn_smem_bytes(int d, int rep, int nstage, int ch, int qkv_tb);
int attn_stages(int max_len, int splits, int ch, int d);
int attn_chunk(int max_len, int splits, int rep);
// The attention kernel can take over the one-row QKV projection when a cluster rank gets whole
// 16-row tiles of the head group's QKV rows and K fits 16 groups of 128.
bool attn_can_fuse_qkv(int d, int rep, int hidden);
cudaError_t launch_attn(const AttnParams& p, cudaStream_t st, bool pdl);
size_t attn_workspace_bytes(int B, int nq, int nkv, int d, int tsplit);
int attn_default_tsplit(int nkv);

// ------------------------------------------------------------------ misc
int num_sms();
int* standalone_error_word();          // device address of the standalone-kernel error word
cudaError_t ensure_kernel_attributes();

}  // namespace kmr
