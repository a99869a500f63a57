// C ABI of the library (declared in kmr.h): argument checking, the model
// object (packed weights, static KV cache, step scratch), the decode step as
// a cached CUDA graph of programmatically-dependent kernel launches, and the
// standalone GEMV / attention entry points.
#include <math.h>
#include <stdio.h>

#include <cmath>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <tuple>
#include <vector>

#include "kmr_internal.cuh"
#include "kmr_step.cuh"
#include "kmr_tcgemm.cuh"

namespace kmr {
int pack_run(const uint8_t* q, const uint16_t* s, const uint16_t* z, int N, int K, int group, int flags,
             void* packed, size_t packed_bytes, int on_device, cudaStream_t st);
int unpack_run(const void* packed, size_t packed_bytes, int N, int K, int group, int flags, uint8_t* q, uint16_t* s,
               uint16_t* z, int on_device, cudaStream_t st);
cudaError_t gemv_set_attributes();
cudaError_t head_set_attributes();
cudaError_t attn_set_attributes();

__device__ int g_standalone_err;

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int* standalone_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_standalone_err) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

cudaError_t ensure_kernel_attributes() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev]) return cudaSuccess;
    if ((e = gemv_set_attributes()) != cudaSuccess) return e;
    if ((e = head_set_attributes()) != cudaSuccess) return e;
    if ((e = attn_set_attributes()) != cudaSuccess) return e;
    if ((e = poison_set_attributes()) != cudaSuccess) return e;
    if ((e = gemm_set_attributes()) != cudaSuccess) return e;
    if ((e = tc_gemm_set_attributes()) != cudaSuccess) return e;
    if ((e = step_set_attributes()) != cudaSuccess) return e;
    done[dev] = true;
    return cudaSuccess;
}

// ------------------------------------------------------------------ GEMV launch helper
struct GemvLaunch {
    const uint8_t* w;
    PackGeom g;
    int in_kind;
    const float* x;
    const uint16_t* embed;
    const int32_t* tokens;
    int vocab;
    float* x_out;
    const uint16_t* norm_w;
    float eps;
    int epi;
    float* y;
    int ldy;
};

// Rows in passes of at most 8; returns the number of launches or a negative KMR code.
// With `poison`, every pass is preceded by the shared-memory poisoning diagnostic.
static int enqueue_gemv(const GemvLaunch& a, int M, int* err, cudaStream_t st, bool pdl, int sms,
                        bool poison = false, uint32_t pattern = 0) {
    int launches = 0;
    const int grid = gemv_grid(a.g.tiles, sms);
    // rows per launch: 16 (two groups of 8 from one weight fill) when the CTA's tiles stay resident
    const int rows = gemv_two_halves_ok(a.g.tiles, grid, a.g.tile_bytes) ? 2 * kMaxMB : kMaxMB;
    for (int r0 = 0; r0 < M; r0 += rows) {
        const int mr = (M - r0) < rows ? (M - r0) : rows;
        const int MB = gemv_pick_mb(mr);
        GemvParams p = {};
        p.w = a.w;
        p.N = a.g.N;
        p.K = a.g.K;
        p.tiles = a.g.tiles;
        p.tile_bytes = a.g.tile_bytes;
        p.M = mr;
        p.in_kind = a.in_kind;
        p.x = a.x ? a.x + size_t(r0) * a.g.K : nullptr;
        p.embed = a.embed;
        p.tokens = a.tokens ? a.tokens + r0 : nullptr;
        p.vocab = a.vocab;
        p.x_out = a.x_out ? a.x_out + size_t(r0) * a.g.K : nullptr;
        p.norm_w = a.norm_w;
        p.eps = a.eps;
        p.epi = a.epi;
        p.y = a.y + size_t(r0) * a.ldy;
        p.ldy = a.ldy;
        p.err = err;
        p.nstage = gemv_nstage(a.g.tiles, grid, a.g.tile_bytes);
        p.halves = mr > kMaxMB ? 2 : 1;
        if (poison && launch_smem_poison(pattern, sms, st) != cudaSuccess) return KMR_ERR_CUDA;
        if (launch_gemv(p, MB, grid, st, pdl || launches > 0) != cudaSuccess) return KMR_ERR_CUDA;
        ++launches;
    }
    return launches;
}

}  // namespace kmr

using namespace kmr;

// ====================================================================== status / packing
extern "C" const char* kmr_status_string(int s) {
    switch (s) {
        case KMR_OK: return "ok";
        case KMR_ERR_INVALID_ARG: return "invalid argument";
        case KMR_ERR_SHAPE: return "unsupported or inconsistent shape";
        case KMR_ERR_SLOT_RANGE: return "slot id out of range";
        case KMR_ERR_CACHE_FULL: return "cache position out of range for an unfinished row";
        case KMR_ERR_NO_PACK: return "int4 weights not loaded";
        case KMR_ERR_CUDA: return "CUDA runtime error";
        case KMR_ERR_DEVICE_TIMEOUT: return "bounded device wait timed out";
        case KMR_ERR_BUFFER_SIZE: return "buffer too small";
        case KMR_ERR_BATCH: return "batch size out of range";
        default: return "unknown status";
    }
}

extern "C" int kmr_layout_version(void) { return 2; }

extern "C" size_t kmr_packed_size(int N, int K, int group) {
    PackGeom g;
    if (!pack_geom(N, K, group, &g)) return 0;
    return (size_t)g.bytes;
}

extern "C" int kmr_pack_int4(const uint8_t* q, const uint16_t* s, const uint16_t* z, int N, int K, int group,
                             int flags, void* packed, size_t packed_bytes, int on_device, void* stream) {
    return pack_run(q, s, z, N, K, group, flags, packed, packed_bytes, on_device,
                    static_cast<cudaStream_t>(stream));
}

extern "C" int kmr_unpack_int4(const void* packed, size_t packed_bytes, int N, int K, int group, int flags,
                               uint8_t* q, uint16_t* s, uint16_t* z, int on_device, void* stream) {
    return unpack_run(packed, packed_bytes, N, K, group, flags, q, s, z, on_device,
                      static_cast<cudaStream_t>(stream));
}

// ====================================================================== standalone GEMV
extern "C" int kmr_int4_gemv(const void* packed, int N, int K, int group, int flags, const float* x, int M,
                             float* y, int epilogue, void* stream) {
    PackGeom g;
    if (!packed || !x || !y) return KMR_ERR_INVALID_ARG;
    if (flags & ~KMR_PACK_GATE_UP) return KMR_ERR_INVALID_ARG;
    if (!pack_geom(N, K, group, &g) || K > 8192) return KMR_ERR_SHAPE;
    if (M < 1 || M > kMaxBatch) return KMR_ERR_BATCH;
    if (epilogue == KMR_EPI_SILU_MUL) {
        if (!(flags & KMR_PACK_GATE_UP) || N % 16 != 0) return KMR_ERR_INVALID_ARG;
    } else if (epilogue != KMR_EPI_NONE && epilogue != KMR_EPI_RESIDUAL) {
        return KMR_ERR_INVALID_ARG;
    }
    if (ensure_kernel_attributes() != cudaSuccess) return KMR_ERR_CUDA;
    int* err = standalone_error_word();
    if (!err) return KMR_ERR_CUDA;
    GemvLaunch a = {};
    a.w = static_cast<const uint8_t*>(packed);
    a.g = g;
    a.in_kind = IN_F32;
    a.x = x;
    a.epi = epilogue == KMR_EPI_NONE ? EPI_STORE : (epilogue == KMR_EPI_RESIDUAL ? EPI_RESID : EPI_SILU);
    a.y = y;
    a.ldy = epilogue == KMR_EPI_SILU_MUL ? N / 2 : N;
    const int r = enqueue_gemv(a, M, err, static_cast<cudaStream_t>(stream), true, num_sms());
    return r < 0 ? r : KMR_OK;
}

// ====================================================================== standalone attention
extern "C" size_t kmr_decode_attn_workspace_size(int B, int nq, int nkv, int d) {
    if (B < 1 || nq < 1 || nkv < 1 || nq % nkv) return 0;
    return attn_workspace_bytes(B, nq, nkv, d, 32);
}

extern "C" int kmr_decode_attn(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                               const int32_t* slot_ids, const int32_t* cache_position, int B, int nq, int nkv,
                               int d, int max_len, int slots, float scale, float* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !slot_ids || !cache_position || !out || !workspace) return KMR_ERR_INVALID_ARG;
    if (B < 1 || B > 65535) return KMR_ERR_BATCH;
    if (nq < 1 || nkv < 1 || nq % nkv || (nq / nkv) > 4 || (nq / nkv) == 3) return KMR_ERR_SHAPE;
    if ((d != 64 && d != 128) || max_len < 1 || slots < 1) return KMR_ERR_SHAPE;
    if (!(scale == scale)) return KMR_ERR_INVALID_ARG;
    if (workspace_bytes < attn_workspace_bytes(B, nq, nkv, d, 32)) return KMR_ERR_BUFFER_SIZE;
    if (ensure_kernel_attributes() != cudaSuccess) return KMR_ERR_CUDA;
    int* err = standalone_error_word();
    if (!err) return KMR_ERR_CUDA;
    AttnParams p = {};
    p.in = q;
    p.in_ld = nq * d;
    p.fused = 0;
    p.kc = const_cast<uint16_t*>(k_cache);
    p.vc = const_cast<uint16_t*>(v_cache);
    p.slot_ids = slot_ids;
    p.cpos = cache_position;
    p.B = B;
    p.nq = nq;
    p.nkv = nkv;
    p.d = d;
    p.S = max_len;
    p.slots = slots;
    p.scale = scale;
    p.tsplit = attn_default_tsplit(nkv);
    // The 8-CTA cluster form (splits merged through distributed shared memory, no global
    // partials) unless one row's grid would leave most SMs idle on long rows, where the
    // wider split (one CTA per SM) streams the cache faster.  Chosen from n_kv and max_len
    // only, never from B, so a row's result does not depend on the batch it is in.
    p.cluster = (nkv * kAttnClusterSplits >= num_sms() / 2 || max_len <= 4096) ? 1 : 0;
    p.out = out;
    p.part = static_cast<float*>(workspace);
    p.counters = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                        attn_workspace_bytes(B, nq, nkv, d, 32) - ((size_t(B) * nkv * 4 + 15) & ~size_t(15)));
    p.err = err;
    return launch_attn(p, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

extern "C" size_t kmr_decode_attn_cascade_workspace_size(int B, int nq, int nkv, int d, int prefix_len) {
    if (B < 1 || nq < 1 || nkv < 1 || (d != 64 && d != 128) || prefix_len < 0) return 0;
    int pchunk = 0, psplits = 0;
    cascade_plan(prefix_len, nkv, num_sms(), &pchunk, &psplits);
    return cascade_workspace_bytes(B, nq, d, psplits);
}

extern "C" int kmr_decode_attn_cascade(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                       const int32_t* slot_ids, const int32_t* cache_position, int prefix_slot,
                                       int prefix_len, int B, int nq, int nkv, int d, int max_len, int slots,
                                       float scale, float* out, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (!q || !k_cache || !v_cache || !slot_ids || !cache_position || !out) return KMR_ERR_INVALID_ARG;
    if (B < 1 || B > 65535) return KMR_ERR_BATCH;
    if (nq < 1 || nkv < 1 || nq % nkv || (nq / nkv) > 4 || (nq / nkv) == 3) return KMR_ERR_SHAPE;
    if ((d != 64 && d != 128) || max_len < 1 || slots < 1 || nkv > 65535) return KMR_ERR_SHAPE;
    if (!(scale == scale)) return KMR_ERR_INVALID_ARG;
    if (prefix_slot < 0 || prefix_slot >= slots) return KMR_ERR_SLOT_RANGE;
    if (prefix_len < 0) return KMR_ERR_INVALID_ARG;
    if (prefix_len >= max_len) return KMR_ERR_CACHE_FULL;         // the current token lies past the prefix
    CascadeParams p = {};
    cascade_plan(prefix_len, nkv, num_sms(), &p.pchunk, &p.psplits);
    if (prefix_len > 0) {
        if (!workspace) return KMR_ERR_INVALID_ARG;
        if (workspace_bytes < cascade_workspace_bytes(B, nq, d, p.psplits)) return KMR_ERR_BUFFER_SIZE;
    }
    int* err = standalone_error_word();
    if (!err) return KMR_ERR_CUDA;
    p.q = q;
    p.kc = k_cache;
    p.vc = v_cache;
    p.slot_ids = slot_ids;
    p.cpos = cache_position;
    p.out = out;
    p.part = static_cast<float*>(workspace);
    p.err = err;
    p.B = B;
    p.nq = nq;
    p.nkv = nkv;
    p.d = d;
    p.S = max_len;
    p.slots = slots;
    p.prefix_slot = prefix_slot;
    p.prefix_len = prefix_len;
    p.scale = scale;
    return launch_cascade(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

extern "C" int kmr_last_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return KMR_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_standalone_err, sizeof(int)) != cudaSuccess) return KMR_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_standalone_err, &zero, sizeof(int)) != cudaSuccess) return KMR_ERR_CUDA;
    return v;
}

// ====================================================================== model
namespace {

struct LayerW {
    uint8_t* w[4] = {nullptr, nullptr, nullptr, nullptr};
    PackGeom g[4];
    uint16_t* norm[4] = {nullptr, nullptr, nullptr, nullptr};
    bool wl[4] = {false, false, false, false};
    bool nl[4] = {false, false, false, false};
};

struct GraphKey {
    int B;
    const void* p[6];
    bool operator==(const GraphKey& o) const {
        if (B != o.B) return false;
        for (int i = 0; i < 6; ++i)
            if (p[i] != o.p[i]) return false;
        return true;
    }
};
struct GraphEntry {
    GraphKey key;
    cudaGraphExec_t exec;
    unsigned long long used;
};

}  // namespace

struct kmr_model {
    kmr_model_config cfg;
    int device = 0;
    int sms = 0;
    int tsplit = 1;
    std::vector<LayerW> layers;
    uint16_t* embed = nullptr;
    bool embed_loaded = false;
    uint16_t* final_norm = nullptr;
    bool final_loaded = false;
    uint16_t* kc = nullptr;
    uint16_t* vc = nullptr;
    size_t kv_layer_elems = 0;
    float* inv_freq = nullptr;
    float* x_resid = nullptr;
    float* qkv = nullptr;
    float* attn_out = nullptr;
    float* act = nullptr;
    float* apart = nullptr;
    int* acount = nullptr;
    float* hbest_v = nullptr;
    int* hbest_i = nullptr;
    int* hcount = nullptr;
    int* err = nullptr;
    // host-state staging for kmr_decode_step_host
    uint8_t* d_state = nullptr;
    uint8_t* h_state = nullptr;
    float* d_logits = nullptr;
    cudaStream_t cap = nullptr;
    std::vector<GraphEntry> graphs;
    unsigned long long tick = 0;
    bool poison = false;           // diagnostic: fill shared memory before every kernel of the step
    bool prefill_tc = true;        // prefill projections on tcgen05 (kmr_model_set_prefill_tcgen05)
    int pf_nt = 0, pf_ks = 0;      // forced tcgen05 tile width / K split (0: planned per projection)
    // persistent step (kmr_step.cu): every layer in one kernel for batches it serves
    bool persistent = false;       // kmr_model_set_persistent_step (opt-in: slower than the PDL-chained step, see header)
    bool persistent_failed = false;    // a capture of it failed: this model uses the multi-kernel step
    StepLayer* step_layers = nullptr;  // [L] device table
    float* step_part = nullptr;        // split states [max rows][nkv][8][rep][d + 2]
    unsigned* step_sync = nullptr;     // phase counters [L][5] | merge counters [rows][nkv] | done | abort
    // prefill scratch for chunks of up to prefill_cap positions (kmr_model_reserve_prefill)
    int prefill_cap = 0;
    float* px = nullptr;           // residual rows [cap][H]
    float* pqkv = nullptr;         // [cap][(nq + 2 nkv) d]
    float* pq = nullptr;           // [cap][nq d] normalised, rotated queries
    float* pattn = nullptr;        // [cap][nq d]
    float* pact = nullptr;         // [cap][I]
    int32_t* pslot = nullptr;      // [cap]
    int32_t* pcpos = nullptr;      // [cap]
    uint16_t* pxs = nullptr;       // staged rows fp16 [Gmax][Mpad][128] (Gmax = largest K / 128)
    float2* pxst = nullptr;        // [Gmax][Mpad] (X', 1/sigma)
    float* prn = nullptr;          // [Mpad] RMSNorm factors
    uint32_t poison_pattern = 0;
    std::vector<void*> allocs;
    std::vector<size_t> alloc_bytes;   // device bytes of allocs[i]
    std::mutex mu;
};

namespace {

template <typename T>
cudaError_t dalloc(kmr_model* m, T** p, size_t bytes) {
    void* q = nullptr;
    cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
    if (e != cudaSuccess) return e;
    m->allocs.push_back(q);
    m->alloc_bytes.push_back(bytes ? bytes : 16);
    *p = static_cast<T*>(q);
    return cudaMemset(q, 0, bytes ? bytes : 16);
}

bool cfg_ok(const kmr_model_config& c) {
    if (c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 || c.intermediate <= 0 ||
        c.vocab <= 0 || c.n_layers <= 0)
        return false;
    if (c.group != 128) return false;
    if (c.head_dim != 64 && c.head_dim != 128) return false;
    if (c.n_q_heads % c.n_kv_heads) return false;
    const int rep = c.n_q_heads / c.n_kv_heads;
    if (rep != 1 && rep != 2 && rep != 4) return false;
    if (c.hidden % 128 || c.intermediate % 128 || (c.n_q_heads * c.head_dim) % 128) return false;
    if (c.hidden > 8192 || c.intermediate > 8192 || c.n_q_heads * c.head_dim > 8192) return false;
    if (c.mrope_sections[0] < 0 || c.mrope_sections[1] < 0 || c.mrope_sections[2] < 0 ||
        c.mrope_sections[0] + c.mrope_sections[1] + c.mrope_sections[2] != c.head_dim / 2)
        return false;
    if (!(c.eps >= 0.f) || !(c.rope_theta > 0.f)) return false;
    if (c.max_len < 1 || c.slots < 1 || c.max_batch < 1 || c.max_batch > kMaxBatch) return false;
    if (c.pad_id < 0 || c.pad_id >= c.vocab || c.eos_id < -1 || c.eos_id >= c.vocab) return false;
    return true;
}

int linear_shape(const kmr_model_config& c, int which, int* N, int* K) {
    switch (which) {
        case KMR_W_QKV: *N = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim; *K = c.hidden; return 0;
        case KMR_W_O: *N = c.hidden; *K = c.n_q_heads * c.head_dim; return 0;
        case KMR_W_GATE_UP: *N = 2 * c.intermediate; *K = c.hidden; return 0;
        case KMR_W_DOWN: *N = c.hidden; *K = c.intermediate; return 0;
        default: return -1;
    }
}

bool all_loaded(const kmr_model* m) {
    if (!m->embed_loaded || !m->final_loaded) return false;
    for (const LayerW& l : m->layers) {
        for (int i = 0; i < 4; ++i)
            if (!l.wl[i]) return false;
        if (!l.nl[KMR_N_INPUT] || !l.nl[KMR_N_POST]) return false;
        if (m->cfg.qk_norm && (!l.nl[KMR_N_Q] || !l.nl[KMR_N_K])) return false;
    }
    return true;
}

struct StepArgs {
    int32_t* tok;
    int32_t* pos;
    int32_t* cpos;
    const int32_t* slot;
    uint8_t* fin;
    float* logits;
    int B;
};

// Queue the whole decode step (5 kernels per layer + the LM head) on `st`.
// At small batches the attention kernel can take over the QKV projection (whole QKV tiles per
// cluster rank, K <= 16 groups).
// Rows up to which the attention kernel computes the QKV projection itself: every (row, KV
// head) cluster multiplies its own row, so each row repeats the whole int4 unpack (the
// integer-pipe-bound part); from two rows on the batched GEMV, which unpacks each weight
// once for all rows, wins (measured: 4 rows fused 1.042 ms per step against 0.810 ms).
constexpr int kFuseQkvMaxRows = 1;
bool fused_qkv(const kmr_model_config& c, int B) {
    return B <= kFuseQkvMaxRows && attn_can_fuse_qkv(c.head_dim, c.n_q_heads / c.n_kv_heads, c.hidden);
}

// Whether this model runs the layers of a B-row step as the persistent kernel (kmr_step.cu),
// and its launch plan: every CTA must be resident at once (one per SM).
bool persistent_plan(const kmr_model* m, int B, StepPlan* plan) {
    if (!m->persistent || m->persistent_failed) return false;
    const kmr_model_config& c = m->cfg;
    if (!step_supported(B, c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.intermediate, c.max_len,
                        m->sms, plan))
        return false;
    return step_max_active_ctas(*plan, c.head_dim) >= 1;
}

// The layers of the step as one persistent kernel; the LM head follows.
int enqueue_persistent(kmr_model* m, const StepArgs& a, const StepPlan& plan, cudaStream_t st) {
    const kmr_model_config& c = m->cfg;
    const int rows = std::min(c.max_batch, kStepMaxRows);
    StepParams p = {};
    p.layers = m->step_layers;
    p.L = c.n_layers;
    p.H = c.hidden;
    p.nq = c.n_q_heads;
    p.nkv = c.n_kv_heads;
    p.I = c.intermediate;
    p.vocab = c.vocab;
    p.S = c.max_len;
    p.slots = c.slots;
    p.B = a.B;
    p.eps = c.eps;
    p.scale = 1.0f / sqrtf(float(c.head_dim));
    p.qk_norm = c.qk_norm;
    p.embed = m->embed;
    p.inv_freq = m->inv_freq;
    p.sec0 = c.mrope_sections[0];
    p.sec1 = c.mrope_sections[1];
    p.tok = a.tok;
    p.pos = a.pos;
    p.cpos = a.cpos;
    p.slot = a.slot;
    p.fin = a.fin;
    p.x = m->x_resid;
    p.qkv = m->qkv;
    p.attn = m->attn_out;
    p.act = m->act;
    p.part = m->step_part;
    p.phase_cnt = m->step_sync;
    p.merge_cnt = m->step_sync + size_t(c.n_layers) * 5;
    p.done_cnt = p.merge_cnt + size_t(rows) * c.n_kv_heads;
    p.abort_flag = p.done_cnt + 1;
    p.err = m->err;
    p.nslots = plan.nslots;
    p.slot_bytes = plan.slot_bytes;
    p.gpw_max = plan.gpw_max;
    p.max_tiles = plan.max_tiles;
    if (m->poison && launch_smem_poison(m->poison_pattern, m->sms, st) != cudaSuccess) return KMR_ERR_CUDA;
    return launch_step(p, plan, c.head_dim, st) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

int enqueue_step(kmr_model* m, const StepArgs& a, cudaStream_t st) {
    const kmr_model_config& c = m->cfg;
    const int B = a.B;
    const int qd = c.n_q_heads * c.head_dim;
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    const int grid = m->sms;
    bool pdl = false;   // the first kernel of the step has no kernel predecessor inside the graph
    // Small batches: the attention kernel computes each head group's QKV rows itself (no QKV launch).
    const bool fuse_qkv = fused_qkv(c, B);
    StepPlan plan;
    const bool persistent = persistent_plan(m, B, &plan);
    if (persistent) {
        const int rc = enqueue_persistent(m, a, plan, st);
        if (rc != KMR_OK) return rc;
    }
    for (int l = 0; l < c.n_layers && !persistent; ++l) {
        LayerW& L = m->layers[l];
        GemvLaunch g = {};
        if (!fuse_qkv) {
            // fused QKV (+ input RMSNorm; layer 0 embeds the tokens)
            g.w = L.w[KMR_W_QKV];
            g.g = L.g[KMR_W_QKV];
            g.in_kind = l == 0 ? IN_EMBED_NORM : IN_F32_NORM;
            g.x = m->x_resid;
            g.embed = m->embed;
            g.tokens = a.tok;
            g.vocab = c.vocab;
            g.x_out = l == 0 ? m->x_resid : nullptr;
            g.norm_w = L.norm[KMR_N_INPUT];
            g.eps = c.eps;
            g.epi = EPI_STORE;
            g.y = m->qkv;
            g.ldy = nqkv;
            if (enqueue_gemv(g, B, m->err, st, pdl, grid, m->poison, m->poison_pattern) < 0) return KMR_ERR_CUDA;
            pdl = true;
        }
        // attention (+ q/k norm, M-RoPE, KV write)
        AttnParams ap = {};
        if (fuse_qkv) {
            ap.wqkv = L.w[KMR_W_QKV];
            ap.qkv_tile_bytes = L.g[KMR_W_QKV].tile_bytes;
            ap.hidden = c.hidden;
            ap.x_kind = l == 0 ? IN_EMBED_NORM : IN_F32_NORM;
            ap.x = m->x_resid;
            ap.embed = m->embed;
            ap.tokens = a.tok;
            ap.vocab = c.vocab;
            ap.x_out = l == 0 ? m->x_resid : nullptr;
            ap.in_norm_w = L.norm[KMR_N_INPUT];
        }
        ap.in = m->qkv;
        ap.in_ld = nqkv;
        ap.fused = 1;
        ap.kc = m->kc + size_t(l) * m->kv_layer_elems;
        ap.vc = m->vc + size_t(l) * m->kv_layer_elems;
        ap.slot_ids = a.slot;
        ap.cpos = a.cpos;
        ap.positions = a.pos;
        ap.pos_ld = B;
        ap.finished = a.fin;
        ap.qn_w = c.qk_norm ? L.norm[KMR_N_Q] : nullptr;
        ap.kn_w = c.qk_norm ? L.norm[KMR_N_K] : nullptr;
        ap.eps = c.eps;
        ap.inv_freq = m->inv_freq;
        ap.sec0 = c.mrope_sections[0];
        ap.sec1 = c.mrope_sections[1];
        ap.B = B;
        ap.nq = c.n_q_heads;
        ap.nkv = c.n_kv_heads;
        ap.d = c.head_dim;
        ap.S = c.max_len;
        ap.slots = c.slots;
        ap.scale = 1.0f / sqrtf(float(c.head_dim));
        ap.tsplit = kAttnClusterSplits;
        ap.cluster = 1;
        ap.out = m->attn_out;
        ap.part = m->apart;
        ap.counters = m->acount;
        ap.err = m->err;
        if (m->poison && launch_smem_poison(m->poison_pattern, grid, st) != cudaSuccess) return KMR_ERR_CUDA;
        if (launch_attn(ap, st, pdl) != cudaSuccess) return KMR_ERR_CUDA;
        pdl = true;
        // O projection + residual
        g = GemvLaunch{};
        g.w = L.w[KMR_W_O];
        g.g = L.g[KMR_W_O];
        g.in_kind = IN_F32;
        g.x = m->attn_out;
        g.epi = EPI_RESID;
        g.y = m->x_resid;
        g.ldy = c.hidden;
        if (enqueue_gemv(g, B, m->err, st, pdl, grid, m->poison, m->poison_pattern) < 0) return KMR_ERR_CUDA;
        // gate_up (+ post-attention RMSNorm) -> SiLU(gate) * up
        g = GemvLaunch{};
        g.w = L.w[KMR_W_GATE_UP];
        g.g = L.g[KMR_W_GATE_UP];
        g.in_kind = IN_F32_NORM;
        g.x = m->x_resid;
        g.norm_w = L.norm[KMR_N_POST];
        g.eps = c.eps;
        g.epi = EPI_SILU;
        g.y = m->act;
        g.ldy = c.intermediate;
        if (enqueue_gemv(g, B, m->err, st, pdl, grid, m->poison, m->poison_pattern) < 0) return KMR_ERR_CUDA;
        // down + residual
        g = GemvLaunch{};
        g.w = L.w[KMR_W_DOWN];
        g.g = L.g[KMR_W_DOWN];
        g.in_kind = IN_F32;
        g.x = m->act;
        g.epi = EPI_RESID;
        g.y = m->x_resid;
        g.ldy = c.hidden;
        if (enqueue_gemv(g, B, m->err, st, pdl, grid, m->poison, m->poison_pattern) < 0) return KMR_ERR_CUDA;
        (void)qd;
    }
    // final norm + LM head + argmax + finalize, in passes of at most 8 rows
    for (int r0 = 0; r0 < B; r0 += kMaxHeadRows) {
        const int mr = (B - r0) < kMaxHeadRows ? (B - r0) : kMaxHeadRows;
        const int MB = head_pick_mb(mr);
        HeadParams hp = {};
        hp.E = m->embed;
        hp.V = c.vocab;
        hp.K = c.hidden;
        hp.tiles = (c.vocab + 7) / 8;
        hp.M = mr;
        hp.x = m->x_resid + size_t(r0) * c.hidden;
        hp.norm_w = m->final_norm;
        hp.eps = c.eps;
        hp.logits = a.logits ? a.logits + size_t(r0) * c.vocab : nullptr;
        hp.ldl = c.vocab;
        hp.gbest_val = m->hbest_v;
        hp.gbest_idx = m->hbest_i;
        hp.counter = m->hcount;
        hp.tokens = a.tok + r0;
        hp.positions = a.pos + r0;
        hp.pos_ld = B;
        hp.cpos = a.cpos + r0;
        hp.finished = a.fin + r0;
        hp.eos = c.eos_id;
        hp.pad = c.pad_id;
        hp.max_len = c.max_len;
        hp.err = m->err;
        const int hgrid = grid < hp.tiles ? grid : hp.tiles;
        const int tpc = (hp.tiles + hgrid - 1) / hgrid;
        int nst = int((128 * 1024) / (size_t(8) * c.hidden * 2));
        if (nst < 2) nst = 2;
        if (nst > tpc) nst = tpc;
        hp.nstage = nst;
        if (m->poison && launch_smem_poison(m->poison_pattern, grid, st) != cudaSuccess) return KMR_ERR_CUDA;
        if (launch_head(hp, MB, hgrid, st, true) != cudaSuccess) return KMR_ERR_CUDA;
    }
    return KMR_OK;
}

struct PrefillArgs {
    const int32_t* tok;        // [T]
    const int32_t* pos;        // [3][T]
    int T, slot, start;
    int32_t* st_tok;           // first decode step's state of the row (outputs)
    int32_t* st_pos;           // [3]
    int32_t* st_cpos;
    uint8_t* st_fin;
    float* logits;             // [V] or null
};

// One int4 projection of all T rows of a prefill chunk: stage the rows once, then the
// weight-stationary GEMM (each unpacked weight fragment serves 64 rows).
int enqueue_projection(kmr_model* m, const GemvLaunch& g, int T, cudaStream_t st) {
    if (m->prefill_tc && tc_gemm_supported(g.g.N, g.g.K)) {
        // 5th-generation tensor cores: staged tokens (fp16, per-row power of two) x dequantised
        // fp16 weights, fp32 accumulators in tensor memory
        TcStageParams tp = {};
        tp.in_kind = g.in_kind;
        tp.x = g.x;
        tp.embed = g.embed;
        tp.tokens = g.tokens;
        tp.vocab = g.vocab;
        tp.x_out = g.x_out;
        tp.norm_w = g.norm_w;
        tp.eps = g.eps;
        tp.M = T;
        tp.K = g.g.K;
        TcPlan plan = tc_gemm_plan(g.g.N, g.g.K, T, m->sms);
        if (m->pf_nt) {
            plan.nt = m->pf_nt;
            plan.ksplit = m->pf_ks;
            while (plan.ksplit > g.g.K / 128) plan.ksplit >>= 1;
        }
        tp.nt = plan.nt;
        tp.xs = m->pxs;
        tp.rs = m->prn;
        tp.err = m->err;
        if (launch_tc_stage(tp, st) != cudaSuccess) return KMR_ERR_CUDA;
        TcGemmParams tg = {};
        tg.w = g.w;
        tg.N = g.g.N;
        tg.K = g.g.K;
        tg.xs = m->pxs;
        tg.rs = m->prn;
        tg.M = T;
        tg.nt = tp.nt;
        tg.ksplit = plan.ksplit;
        tg.epi = g.epi;
        tg.y = g.y;
        tg.ldy = g.ldy;
        tg.err = m->err;
        return launch_tc_gemm(tg, st) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
    }
    StageParams sp = {};
    sp.in_kind = g.in_kind;
    sp.x = g.x;
    sp.embed = g.embed;
    sp.tokens = g.tokens;
    sp.vocab = g.vocab;
    sp.x_out = g.x_out;
    sp.norm_w = g.norm_w;
    sp.eps = g.eps;
    sp.M = T;
    sp.Mpad = gemm_rows_pad(T);
    sp.K = g.g.K;
    sp.xs = m->pxs;
    sp.xst = m->pxst;
    sp.rnorm = m->prn;
    sp.err = m->err;
    if (launch_stage(sp, st) != cudaSuccess) return KMR_ERR_CUDA;
    GemmParams gp = {};
    gp.w = g.w;
    gp.N = g.g.N;
    gp.K = g.g.K;
    gp.tiles = g.g.tiles;
    gp.xs = m->pxs;
    gp.xst = m->pxst;
    gp.rnorm = m->prn;
    gp.M = T;
    gp.Mpad = sp.Mpad;
    gp.epi = g.epi;
    gp.y = g.y;
    gp.ldy = g.ldy;
    gp.err = m->err;
    return launch_gemm(gp, m->sms, st) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

// Queue one prefill chunk: per layer the QKV projection of all T positions, the q/k norm +
// M-RoPE + KV write of every position, causal attention (position i attends 0..start + i of
// the same cache row), then O, gate_up and down over all positions; the LM head runs on the
// last position only.
int enqueue_prefill(kmr_model* m, const PrefillArgs& a, cudaStream_t st) {
    const kmr_model_config& c = m->cfg;
    const int T = a.T;
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    const int grid = m->sms;
    for (int l = 0; l < c.n_layers; ++l) {
        LayerW& L = m->layers[l];
        GemvLaunch g = {};
        g.w = L.w[KMR_W_QKV];
        g.g = L.g[KMR_W_QKV];
        g.in_kind = l == 0 ? IN_EMBED_NORM : IN_F32_NORM;
        g.x = m->px;
        g.embed = m->embed;
        g.tokens = a.tok;
        g.vocab = c.vocab;
        g.x_out = l == 0 ? m->px : nullptr;
        g.norm_w = L.norm[KMR_N_INPUT];
        g.eps = c.eps;
        g.epi = EPI_STORE;
        g.y = m->pqkv;
        g.ldy = nqkv;
        if (enqueue_projection(m, g, T, st) != KMR_OK) return KMR_ERR_CUDA;
        PrefillRopeParams rp = {};
        rp.qkv = m->pqkv;
        rp.qkv_ld = nqkv;
        rp.q_out = m->pq;
        rp.kc = m->kc + size_t(l) * m->kv_layer_elems;
        rp.vc = m->vc + size_t(l) * m->kv_layer_elems;
        rp.positions = a.pos;
        rp.qn_w = c.qk_norm ? L.norm[KMR_N_Q] : nullptr;
        rp.kn_w = c.qk_norm ? L.norm[KMR_N_K] : nullptr;
        rp.inv_freq = m->inv_freq;
        rp.sec0 = c.mrope_sections[0];
        rp.sec1 = c.mrope_sections[1];
        rp.eps = c.eps;
        rp.T = T;
        rp.start = a.start;
        rp.slot = a.slot;
        rp.nq = c.n_q_heads;
        rp.nkv = c.n_kv_heads;
        rp.d = c.head_dim;
        rp.S = c.max_len;
        rp.slot_ids = m->pslot;
        rp.cpos = m->pcpos;
        if (l == c.n_layers - 1) {
            rp.state_pos = a.st_pos;
            rp.state_cpos = a.st_cpos;
            rp.state_fin = a.st_fin;
        }
        if (launch_prefill_rope(rp, st) != cudaSuccess) return KMR_ERR_CUDA;
        // causal attention of every position on the tensor cores
        PrefillAttnParams pa = {};
        pa.q = m->pq;
        pa.kc = rp.kc;
        pa.vc = rp.vc;
        pa.slot = a.slot;
        pa.start = a.start;
        pa.T = T;
        pa.nq = c.n_q_heads;
        pa.nkv = c.n_kv_heads;
        pa.d = c.head_dim;
        pa.S = c.max_len;
        pa.scale = 1.0f / sqrtf(float(c.head_dim));
        pa.out = m->pattn;
        if (launch_prefill_attn(pa, st) != cudaSuccess) return KMR_ERR_CUDA;
        g = GemvLaunch{};
        g.w = L.w[KMR_W_O];
        g.g = L.g[KMR_W_O];
        g.in_kind = IN_F32;
        g.x = m->pattn;
        g.epi = EPI_RESID;
        g.y = m->px;
        g.ldy = c.hidden;
        if (enqueue_projection(m, g, T, st) != KMR_OK) return KMR_ERR_CUDA;
        g = GemvLaunch{};
        g.w = L.w[KMR_W_GATE_UP];
        g.g = L.g[KMR_W_GATE_UP];
        g.in_kind = IN_F32_NORM;
        g.x = m->px;
        g.norm_w = L.norm[KMR_N_POST];
        g.eps = c.eps;
        g.epi = EPI_SILU;
        g.y = m->pact;
        g.ldy = c.intermediate;
        if (enqueue_projection(m, g, T, st) != KMR_OK) return KMR_ERR_CUDA;
        g = GemvLaunch{};
        g.w = L.w[KMR_W_DOWN];
        g.g = L.g[KMR_W_DOWN];
        g.in_kind = IN_F32;
        g.x = m->pact;
        g.epi = EPI_RESID;
        g.y = m->px;
        g.ldy = c.hidden;
        if (enqueue_projection(m, g, T, st) != KMR_OK) return KMR_ERR_CUDA;
    }
    HeadParams hp = {};
    hp.E = m->embed;
    hp.V = c.vocab;
    hp.K = c.hidden;
    hp.tiles = (c.vocab + 7) / 8;
    hp.M = 1;
    hp.x = m->px + size_t(T - 1) * c.hidden;
    hp.norm_w = m->final_norm;
    hp.eps = c.eps;
    hp.logits = a.logits;
    hp.ldl = c.vocab;
    hp.gbest_val = m->hbest_v;
    hp.gbest_idx = m->hbest_i;
    hp.counter = m->hcount;
    hp.tokens = a.st_tok;
    hp.positions = a.st_pos;
    hp.pos_ld = 1;
    hp.cpos = a.st_cpos;
    hp.finished = a.st_fin;
    hp.eos = c.eos_id;
    hp.pad = c.pad_id;
    hp.max_len = c.max_len;
    hp.err = m->err;
    const int hgrid = grid < hp.tiles ? grid : hp.tiles;
    const int tpc = (hp.tiles + hgrid - 1) / hgrid;
    int nst = int((128 * 1024) / (size_t(8) * c.hidden * 2));
    if (nst < 2) nst = 2;
    if (nst > tpc) nst = tpc;
    hp.nstage = nst;
    if (launch_head(hp, 1, hgrid, st, false) != cudaSuccess) return KMR_ERR_CUDA;
    return KMR_OK;
}

int get_graph(kmr_model* m, const StepArgs& a, cudaGraphExec_t* out) {
    GraphKey key;
    key.B = a.B;
    key.p[0] = a.tok;
    key.p[1] = a.pos;
    key.p[2] = a.cpos;
    key.p[3] = a.slot;
    key.p[4] = a.fin;
    key.p[5] = a.logits;
    for (GraphEntry& e : m->graphs) {
        if (e.key == key) {
            e.used = ++m->tick;
            *out = e.exec;
            return KMR_OK;
        }
    }
    cudaGraphExec_t exec = nullptr;
    for (int attempt = 0;; ++attempt) {
        StepPlan plan;
        const bool persistent = persistent_plan(m, a.B, &plan);
        cudaGraph_t graph = nullptr;
        if (cudaStreamBeginCapture(m->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return KMR_ERR_CUDA;
        const int rc = enqueue_step(m, a, m->cap);
        const cudaError_t ec = cudaStreamEndCapture(m->cap, &graph);
        cudaError_t ei = cudaErrorUnknown;
        if (rc == KMR_OK && ec == cudaSuccess) ei = cudaGraphInstantiate(&exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (rc == KMR_OK && ec == cudaSuccess && ei == cudaSuccess) break;
        cudaGetLastError();
        // A persistent step that cannot be captured or instantiated here: this model falls back to
        // the multi-kernel step (kmr_model_kernels_per_step reports which one runs).
        if (persistent && attempt == 0) {
            m->persistent_failed = true;
            continue;
        }
        return rc != KMR_OK ? rc : KMR_ERR_CUDA;
    }
    if (m->graphs.size() >= 8) {
        size_t lru = 0;
        for (size_t i = 1; i < m->graphs.size(); ++i)
            if (m->graphs[i].used < m->graphs[lru].used) lru = i;
        cudaGraphExecDestroy(m->graphs[lru].exec);
        m->graphs.erase(m->graphs.begin() + lru);
    }
    m->graphs.push_back(GraphEntry{key, exec, ++m->tick});
    *out = exec;
    return KMR_OK;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" int kmr_model_create(const kmr_model_config* cfg, kmr_model** out) {
    if (!cfg || !out) return KMR_ERR_INVALID_ARG;
    *out = nullptr;
    if (!cfg_ok(*cfg)) return KMR_ERR_SHAPE;
    kmr_model* m = new kmr_model();
    m->cfg = *cfg;
    const kmr_model_config& c = m->cfg;
    auto fail = [&](int code) {
        kmr_model_destroy(m);
        return code;
    };
    if (cudaGetDevice(&m->device) != cudaSuccess) return fail(KMR_ERR_CUDA);
    if (ensure_kernel_attributes() != cudaSuccess) return fail(KMR_ERR_CUDA);
    m->sms = num_sms();
    m->tsplit = attn_default_tsplit(c.n_kv_heads);
    m->layers.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        for (int w = 0; w < 4; ++w) {
            int N, K;
            linear_shape(c, w, &N, &K);
            if (!pack_geom(N, K, c.group, &m->layers[l].g[w])) return fail(KMR_ERR_SHAPE);
            if (dalloc(m, &m->layers[l].w[w], (size_t)m->layers[l].g[w].bytes)) return fail(KMR_ERR_CUDA);
        }
        for (int n = 0; n < 4; ++n) {
            const int len = n < 2 ? c.hidden : c.head_dim;
            if (dalloc(m, &m->layers[l].norm[n], size_t(len) * 2)) return fail(KMR_ERR_CUDA);
        }
    }
    const int B = c.max_batch;
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    m->kv_layer_elems = size_t(c.slots) * c.n_kv_heads * c.max_len * c.head_dim;
    if (dalloc(m, &m->embed, size_t(c.vocab) * c.hidden * 2) || dalloc(m, &m->final_norm, size_t(c.hidden) * 2) ||
        dalloc(m, &m->kc, m->kv_layer_elems * c.n_layers * 2) || dalloc(m, &m->vc, m->kv_layer_elems * c.n_layers * 2) ||
        dalloc(m, &m->inv_freq, size_t(c.head_dim / 2) * 4) || dalloc(m, &m->x_resid, size_t(B) * c.hidden * 4) ||
        dalloc(m, &m->qkv, size_t(B) * nqkv * 4) || dalloc(m, &m->attn_out, size_t(B) * c.n_q_heads * c.head_dim * 4) ||
        dalloc(m, &m->act, size_t(B) * c.intermediate * 4) ||
        dalloc(m, &m->apart, size_t(B) * c.n_q_heads * m->tsplit * (c.head_dim + 2) * 4) ||
        dalloc(m, &m->acount, size_t(B) * c.n_kv_heads * 4) || dalloc(m, &m->hbest_v, size_t(m->sms) * kMaxHeadRows * 4) ||
        dalloc(m, &m->hbest_i, size_t(m->sms) * kMaxHeadRows * 4) || dalloc(m, &m->hcount, 16) || dalloc(m, &m->err, 16) ||
        dalloc(m, &m->d_state, size_t(B) * 32))
        return fail(KMR_ERR_CUDA);
    std::vector<float> inv(c.head_dim / 2);
    for (int i = 0; i < c.head_dim / 2; ++i)
        inv[i] = float(pow(double(c.rope_theta), -2.0 * double(i) / double(c.head_dim)));
    if (cudaMemcpy(m->inv_freq, inv.data(), inv.size() * 4, cudaMemcpyHostToDevice)) return fail(KMR_ERR_CUDA);
    {
        const int rows = std::min(B, kStepMaxRows), rep = c.n_q_heads / c.n_kv_heads;
        const size_t nsync = size_t(c.n_layers) * 5 + size_t(rows) * c.n_kv_heads + 2;
        if (dalloc(m, &m->step_layers, sizeof(StepLayer) * c.n_layers) ||
            dalloc(m, &m->step_part, size_t(rows) * c.n_kv_heads * kAttnClusterSplits * rep * (c.head_dim + 2) * 4) ||
            dalloc(m, &m->step_sync, nsync * 4))
            return fail(KMR_ERR_CUDA);
        std::vector<StepLayer> t(c.n_layers);
        for (int l = 0; l < c.n_layers; ++l) {
            for (int w = 0; w < 4; ++w) {
                t[l].w[w] = m->layers[l].w[w];
                t[l].norm[w] = m->layers[l].norm[w];
            }
            t[l].kc = m->kc + size_t(l) * m->kv_layer_elems;
            t[l].vc = m->vc + size_t(l) * m->kv_layer_elems;
        }
        if (cudaMemcpy(m->step_layers, t.data(), sizeof(StepLayer) * c.n_layers, cudaMemcpyHostToDevice))
            return fail(KMR_ERR_CUDA);
    }
    if (cudaMallocHost(&m->h_state, size_t(B) * 32) != cudaSuccess) return fail(KMR_ERR_CUDA);
    if (cudaStreamCreateWithFlags(&m->cap, cudaStreamNonBlocking) != cudaSuccess) return fail(KMR_ERR_CUDA);
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(KMR_ERR_CUDA);
    *out = m;
    return KMR_OK;
}

extern "C" int kmr_model_destroy(kmr_model* m) {
    if (!m) return KMR_ERR_INVALID_ARG;
    DeviceGuard dg(m->device);
    cudaDeviceSynchronize();
    for (GraphEntry& e : m->graphs) cudaGraphExecDestroy(e.exec);
    for (void* p : m->allocs) cudaFree(p);
    if (m->d_logits) cudaFree(m->d_logits);
    if (m->h_state) cudaFreeHost(m->h_state);
    if (m->cap) cudaStreamDestroy(m->cap);
    delete m;
    return KMR_OK;
}

extern "C" int kmr_model_set_linear(kmr_model* m, int layer, int which, const uint8_t* q, const uint16_t* s,
                                    const uint16_t* z) {
    if (!m || !q || !s || !z) return KMR_ERR_INVALID_ARG;
    if (layer < 0 || layer >= m->cfg.n_layers) return KMR_ERR_INVALID_ARG;
    int N, K;
    if (linear_shape(m->cfg, which, &N, &K)) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    LayerW& L = m->layers[layer];
    const size_t nq = size_t(N) * K, ns = size_t(N) * (K / 128);
    for (size_t i = 0; i < nq; ++i)
        if (q[i] > 15) return KMR_ERR_INVALID_ARG;
    uint8_t* dq = nullptr;
    uint16_t* ds = nullptr;
    uint16_t* dz = nullptr;
    int rc = KMR_OK;
    if (cudaMalloc(&dq, nq) || cudaMalloc(&ds, ns * 2) || cudaMalloc(&dz, ns * 2)) rc = KMR_ERR_CUDA;
    if (rc == KMR_OK && (cudaMemcpy(dq, q, nq, cudaMemcpyHostToDevice) ||
                         cudaMemcpy(ds, s, ns * 2, cudaMemcpyHostToDevice) ||
                         cudaMemcpy(dz, z, ns * 2, cudaMemcpyHostToDevice)))
        rc = KMR_ERR_CUDA;
    if (rc == KMR_OK)
        rc = pack_run(dq, ds, dz, N, K, 128, which == KMR_W_GATE_UP ? KMR_PACK_GATE_UP : 0, L.w[which],
                      (size_t)L.g[which].bytes, 1, nullptr);
    if (rc == KMR_OK && cudaDeviceSynchronize() != cudaSuccess) rc = KMR_ERR_CUDA;
    cudaFree(dq);
    cudaFree(ds);
    cudaFree(dz);
    if (rc == KMR_OK) L.wl[which] = true;
    return rc;
}

extern "C" int kmr_model_set_norm(kmr_model* m, int layer, int which, const uint16_t* w) {
    if (!m || !w) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    if (layer == -1) {
        if (which != KMR_N_INPUT) return KMR_ERR_INVALID_ARG;
        if (cudaMemcpy(m->final_norm, w, size_t(m->cfg.hidden) * 2, cudaMemcpyHostToDevice)) return KMR_ERR_CUDA;
        m->final_loaded = true;
        return KMR_OK;
    }
    if (layer < 0 || layer >= m->cfg.n_layers || which < 0 || which > 3) return KMR_ERR_INVALID_ARG;
    const int len = which < 2 ? m->cfg.hidden : m->cfg.head_dim;
    if (cudaMemcpy(m->layers[layer].norm[which], w, size_t(len) * 2, cudaMemcpyHostToDevice)) return KMR_ERR_CUDA;
    m->layers[layer].nl[which] = true;
    return KMR_OK;
}

extern "C" int kmr_model_set_embedding(kmr_model* m, const uint16_t* e) {
    if (!m || !e) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    if (cudaMemcpy(m->embed, e, size_t(m->cfg.vocab) * m->cfg.hidden * 2, cudaMemcpyHostToDevice))
        return KMR_ERR_CUDA;
    m->embed_loaded = true;
    return KMR_OK;
}

extern "C" int kmr_model_set_kv(kmr_model* m, int layer, int slot, int length, const uint16_t* k,
                                const uint16_t* v) {
    if (!m || (!k && length > 0) || (!v && length > 0)) return KMR_ERR_INVALID_ARG;
    const kmr_model_config& c = m->cfg;
    if (layer < 0 || layer >= c.n_layers) return KMR_ERR_INVALID_ARG;
    if (slot < 0 || slot >= c.slots) return KMR_ERR_SLOT_RANGE;
    if (length < 0 || length > c.max_len) return KMR_ERR_CACHE_FULL;
    if (length == 0) return KMR_OK;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    const size_t row = size_t(c.head_dim) * 2;
    for (int h = 0; h < c.n_kv_heads; ++h) {
        const size_t off = size_t(layer) * m->kv_layer_elems + ((size_t(slot) * c.n_kv_heads + h) * c.max_len) * c.head_dim;
        if (cudaMemcpy(m->kc + off, k + size_t(h) * length * c.head_dim, row * length, cudaMemcpyHostToDevice) ||
            cudaMemcpy(m->vc + off, v + size_t(h) * length * c.head_dim, row * length, cudaMemcpyHostToDevice))
            return KMR_ERR_CUDA;
    }
    return KMR_OK;
}

extern "C" int kmr_model_copy_row_from(kmr_model* m, int dst_slot, const uint16_t* src_k, const uint16_t* src_v,
                                       int src_slots, int src_max_len, int src_row, int length, void* stream) {
    if (!m) return KMR_ERR_INVALID_ARG;
    const kmr_model_config& c = m->cfg;
    if ((src_k == nullptr) != (src_v == nullptr)) return KMR_ERR_INVALID_ARG;
    const bool own = src_k == nullptr;
    if (own) {
        src_k = m->kc;
        src_v = m->vc;
        src_slots = c.slots;
        src_max_len = c.max_len;
    }
    if ((reinterpret_cast<uintptr_t>(src_k) | reinterpret_cast<uintptr_t>(src_v)) & 15) return KMR_ERR_INVALID_ARG;
    if (src_slots <= 0 || src_max_len <= 0) return KMR_ERR_INVALID_ARG;
    if (src_row < 0 || src_row >= src_slots) return own ? KMR_ERR_SLOT_RANGE : KMR_ERR_INVALID_ARG;
    if (dst_slot < 0 || dst_slot >= c.slots) return KMR_ERR_SLOT_RANGE;
    if (length < 0) return KMR_ERR_INVALID_ARG;
    if (length > c.max_len || length > src_max_len) return KMR_ERR_CACHE_FULL;
    if (length == 0 || (own && src_row == dst_slot)) return KMR_OK;
    DeviceGuard dg(m->device);
    KvCopyParams p;
    p.src_k = src_k;
    p.src_v = src_v;
    p.dst_k = m->kc;
    p.dst_v = m->vc;
    p.L = c.n_layers;
    p.nkv = c.n_kv_heads;
    p.d = c.head_dim;
    p.src_slots = src_slots;
    p.src_max_len = src_max_len;
    p.src_row = src_row;
    p.dst_slots = c.slots;
    p.dst_max_len = c.max_len;
    p.dst_row = dst_slot;
    p.units = (long long)length * c.head_dim / 8;
    return launch_kv_row_copy(p, m->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

extern "C" int kmr_model_reserve_prefill(kmr_model* m, int max_tokens) {
    if (!m || max_tokens < 1) return KMR_ERR_INVALID_ARG;
    const kmr_model_config& c = m->cfg;
    if (max_tokens > c.max_len) return KMR_ERR_CACHE_FULL;
    std::lock_guard<std::mutex> lk(m->mu);
    if (max_tokens <= m->prefill_cap) return KMR_OK;
    DeviceGuard dg(m->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return KMR_ERR_CUDA;
    void* old[10] = {m->px, m->pqkv, m->pq, m->pattn, m->pact, m->pslot, m->pcpos, m->pxs, m->pxst, m->prn};
    for (void* p : old) {
        if (!p) continue;
        for (size_t i = 0; i < m->allocs.size(); ++i)
            if (m->allocs[i] == p) {
                m->allocs.erase(m->allocs.begin() + i);
                m->alloc_bytes.erase(m->alloc_bytes.begin() + i);
                break;
            }
        cudaFree(p);
    }
    m->prefill_cap = 0;
    const size_t T = size_t(max_tokens);
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, qd = c.n_q_heads * c.head_dim;
    if (dalloc(m, &m->px, T * c.hidden * 4) || dalloc(m, &m->pqkv, T * nqkv * 4) || dalloc(m, &m->pq, T * qd * 4) ||
        dalloc(m, &m->pattn, T * qd * 4) || dalloc(m, &m->pact, T * c.intermediate * 4) ||
        dalloc(m, &m->pslot, T * 4) || dalloc(m, &m->pcpos, T * 4))
        return KMR_ERR_CUDA;
    const size_t Mpad = size_t(std::max(gemm_rows_pad(max_tokens), tc_rows_pad(max_tokens)));
    const size_t Gmax = size_t(std::max(std::max(c.hidden, qd), c.intermediate) / 128);
    if (dalloc(m, &m->pxs, Gmax * Mpad * 128 * 2) || dalloc(m, &m->pxst, Gmax * Mpad * 8) ||
        dalloc(m, &m->prn, Mpad * 4))
        return KMR_ERR_CUDA;
    m->prefill_cap = max_tokens;
    return KMR_OK;
}

extern "C" int kmr_prefill(kmr_model* m, const int32_t* token_ids, const int32_t* positions, int T, int slot,
                           int start_pos, int32_t* state_token, int32_t* state_positions,
                           int32_t* state_cache_position, uint8_t* state_finished, float* logits, void* stream) {
    if (!m || !token_ids || !positions || !state_token || !state_positions || !state_cache_position ||
        !state_finished)
        return KMR_ERR_INVALID_ARG;
    const kmr_model_config& c = m->cfg;
    if (T < 1) return KMR_ERR_INVALID_ARG;
    if (T > m->prefill_cap) return KMR_ERR_BUFFER_SIZE;
    if (slot < 0 || slot >= c.slots) return KMR_ERR_SLOT_RANGE;
    if (start_pos < 0 || start_pos + T > c.max_len) return KMR_ERR_CACHE_FULL;
    if (!all_loaded(m)) return KMR_ERR_NO_PACK;
    if (ensure_kernel_attributes() != cudaSuccess) return KMR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    PrefillArgs a;
    a.tok = token_ids;
    a.pos = positions;
    a.T = T;
    a.slot = slot;
    a.start = start_pos;
    a.st_tok = state_token;
    a.st_pos = state_positions;
    a.st_cpos = state_cache_position;
    a.st_fin = state_finished;
    a.logits = logits;
    return enqueue_prefill(m, a, static_cast<cudaStream_t>(stream));
}

extern "C" int kmr_model_kv_pointers(kmr_model* m, int layer, void** k, void** v) {
    if (!m || !k || !v || layer < 0 || layer >= m->cfg.n_layers) return KMR_ERR_INVALID_ARG;
    *k = m->kc + size_t(layer) * m->kv_layer_elems;
    *v = m->vc + size_t(layer) * m->kv_layer_elems;
    return KMR_OK;
}

extern "C" int kmr_smem_poison(uint32_t pattern, void* stream) {
    if (ensure_kernel_attributes() != cudaSuccess) return KMR_ERR_CUDA;
    return launch_smem_poison(pattern, num_sms(), static_cast<cudaStream_t>(stream)) == cudaSuccess ? KMR_OK
                                                                                                 : KMR_ERR_CUDA;
}

namespace kmr {
cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t st);   // kmr_poison.cu
}

extern "C" int kmr_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
    if (limit_ns < 1000ull || limit_ns > 2000000000ull) return KMR_ERR_INVALID_ARG;
    int* err = standalone_error_word();
    if (!err) return KMR_ERR_CUDA;
    return launch_wait_timeout(err, limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KMR_OK
                                                                                                : KMR_ERR_CUDA;
}

extern "C" int kmr_model_set_prefill_tcgen05(kmr_model* m, int enable) {
    if (!m) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    m->prefill_tc = enable != 0;
    return KMR_OK;
}

extern "C" int kmr_prefill_plan(int N, int K, int M, int sms, int* nt, int* ksplit) {
    if (!nt || !ksplit || M < 1 || sms < 1 || !tc_gemm_supported(N, K)) return KMR_ERR_INVALID_ARG;
    const TcPlan plan = tc_gemm_plan(N, K, M, sms);
    *nt = plan.nt;
    *ksplit = plan.ksplit;
    return KMR_OK;
}

extern "C" int kmr_model_set_prefill_plan(kmr_model* m, int nt, int ksplit) {
    if (!m) return KMR_ERR_INVALID_ARG;
    const bool automatic = nt == 0 && ksplit == 0;
    if (!automatic && !((nt == 64 || nt == 128 || nt == 256) && (ksplit == 1 || ksplit == 2 || ksplit == 4)))
        return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    m->pf_nt = nt;
    m->pf_ks = ksplit;
    return KMR_OK;
}

extern "C" int kmr_model_set_persistent_step(kmr_model* m, int enable) {
    if (!m) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return KMR_ERR_CUDA;
    m->persistent = enable != 0;
    for (GraphEntry& e : m->graphs) cudaGraphExecDestroy(e.exec);   // captured graphs follow the old setting
    m->graphs.clear();
    return KMR_OK;
}

extern "C" int kmr_model_set_smem_poison(kmr_model* m, int enable, uint32_t pattern) {
    if (!m) return KMR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return KMR_ERR_CUDA;
    m->poison = enable != 0;
    m->poison_pattern = pattern;
    for (GraphEntry& e : m->graphs) cudaGraphExecDestroy(e.exec);   // captured graphs follow the old setting
    m->graphs.clear();
    return KMR_OK;
}

extern "C" int kmr_decode_step(kmr_model* m, int32_t* tok, int32_t* pos, int32_t* cpos, const int32_t* slot,
                               uint8_t* fin, int B, float* logits, void* stream) {
    if (!m || !tok || !pos || !cpos || !slot || !fin) return KMR_ERR_INVALID_ARG;
    if (B < 1 || B > m->cfg.max_batch) return KMR_ERR_BATCH;
    if (!all_loaded(m)) return KMR_ERR_NO_PACK;
    std::lock_guard<std::mutex> lk(m->mu);
    DeviceGuard dg(m->device);
    StepArgs a = {tok, pos, cpos, slot, fin, logits, B};
    cudaGraphExec_t exec = nullptr;
    const int rc = get_graph(m, a, &exec);
    if (rc != KMR_OK) return rc;
    return cudaGraphLaunch(exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

extern "C" int kmr_decode_step_host(kmr_model* m, int32_t* tok, int32_t* pos, int32_t* cpos, const int32_t* slot,
                                    uint8_t* fin, int B, float* logits, void* stream) {
    if (!m || !tok || !pos || !cpos || !slot || !fin) return KMR_ERR_INVALID_ARG;
    const kmr_model_config& c = m->cfg;
    if (B < 1 || B > c.max_batch) return KMR_ERR_BATCH;
    if (!all_loaded(m)) return KMR_ERR_NO_PACK;
    for (int b = 0; b < B; ++b) {
        if (tok[b] < 0 || tok[b] >= c.vocab) return KMR_ERR_INVALID_ARG;
        if (fin[b]) continue;
        if (slot[b] < 0 || slot[b] >= c.slots) return KMR_ERR_SLOT_RANGE;
        if (cpos[b] < 0 || cpos[b] >= c.max_len) return KMR_ERR_CACHE_FULL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* d_tok;
    int32_t* d_pos;
    int32_t* d_cpos;
    int32_t* d_slot;
    uint8_t* d_fin;
    {
        std::lock_guard<std::mutex> lk(m->mu);
        DeviceGuard dg(m->device);
        if (logits && !m->d_logits) {
            void* p = nullptr;
            if (cudaMalloc(&p, size_t(c.max_batch) * c.vocab * 4) != cudaSuccess) return KMR_ERR_CUDA;
            m->d_logits = static_cast<float*>(p);
        }
        // state block: tok[Bmax] | pos[3][B] | cpos[Bmax] | slot[Bmax] | fin[Bmax]  (positions use row stride B)
        const int Bm = c.max_batch;
        uint8_t* h = m->h_state;
        const size_t o_tok = 0, o_pos = size_t(Bm) * 4, o_cpos = o_pos + size_t(3) * Bm * 4,
                     o_slot = o_cpos + size_t(Bm) * 4, o_fin = o_slot + size_t(Bm) * 4;
        memcpy(h + o_tok, tok, size_t(B) * 4);
        memcpy(h + o_pos, pos, size_t(3) * B * 4);
        memcpy(h + o_cpos, cpos, size_t(B) * 4);
        memcpy(h + o_slot, slot, size_t(B) * 4);
        memcpy(h + o_fin, fin, size_t(B));
        d_tok = reinterpret_cast<int32_t*>(m->d_state + o_tok);
        d_pos = reinterpret_cast<int32_t*>(m->d_state + o_pos);
        d_cpos = reinterpret_cast<int32_t*>(m->d_state + o_cpos);
        d_slot = reinterpret_cast<int32_t*>(m->d_state + o_slot);
        d_fin = m->d_state + o_fin;
        const size_t total = o_fin + size_t(Bm);
        if (cudaMemcpyAsync(m->d_state, h, total, cudaMemcpyHostToDevice, st) != cudaSuccess) return KMR_ERR_CUDA;
        StepArgs a = {d_tok, d_pos, d_cpos, d_slot, d_fin, logits ? m->d_logits : nullptr, B};
        cudaGraphExec_t exec = nullptr;
        const int rc = get_graph(m, a, &exec);
        if (rc != KMR_OK) return rc;
        if (cudaGraphLaunch(exec, st) != cudaSuccess) return KMR_ERR_CUDA;
        if (cudaMemcpyAsync(h, m->d_state, total, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KMR_ERR_CUDA;
        if (logits && cudaMemcpyAsync(logits, m->d_logits, size_t(B) * c.vocab * 4, cudaMemcpyDeviceToHost, st) !=
                          cudaSuccess)
            return KMR_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KMR_ERR_CUDA;
        memcpy(tok, h + o_tok, size_t(B) * 4);
        memcpy(pos, h + o_pos, size_t(3) * B * 4);
        memcpy(cpos, h + o_cpos, size_t(B) * 4);
        memcpy(fin, h + o_fin, size_t(B));
    }
    return KMR_OK;
}

extern "C" int kmr_model_sync_status(kmr_model* m, void* stream) {
    if (!m) return KMR_ERR_INVALID_ARG;
    DeviceGuard dg(m->device);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KMR_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, m->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KMR_ERR_CUDA;
    if (v != 0 && cudaMemset(m->err, 0, sizeof(int)) != cudaSuccess) return KMR_ERR_CUDA;
    return v;
}

extern "C" int kmr_model_kernels_per_step(const kmr_model* m, int B) {
    if (!m || B < 1) return 0;
    // GEMV launches per projection: one per 16 rows when the CTA's tiles stay resident, else per 8
    const kmr_model_config& c = m->cfg;
    const int grid = m->sms;
    int gemv_launches = 0;
    for (int w = 0; w < 4; ++w) {
        const PackGeom& g = m->layers[0].g[w];
        const int rows = gemv_two_halves_ok(g.tiles, gemv_grid(g.tiles, grid), g.tile_bytes) ? 2 * kMaxMB : kMaxMB;
        gemv_launches += (B + rows - 1) / rows;
    }
    if (fused_qkv(c, B)) gemv_launches -= 1;                 // QKV runs inside the attention kernel
    const int head_passes = (B + kMaxHeadRows - 1) / kMaxHeadRows;
    StepPlan plan;
    const int k = persistent_plan(m, B, &plan) ? 1 + head_passes : c.n_layers * (gemv_launches + 1) + head_passes;
    return m->poison ? 2 * k : k;                 // the diagnostic adds one fill per kernel
}

extern "C" size_t kmr_model_device_bytes(const kmr_model* m, size_t* weights, size_t* kv_cache, size_t* scratch) {
    if (!m) return 0;
    const kmr_model_config& c = m->cfg;
    size_t total = 0;
    for (size_t n : m->alloc_bytes) total += n;
    if (m->d_logits) total += size_t(c.max_batch) * c.vocab * 4;
    size_t w = size_t(c.vocab) * c.hidden * 2 + size_t(c.hidden) * 2;           // tied embedding, final norm
    for (const LayerW& l : m->layers) {
        for (int i = 0; i < 4; ++i) w += size_t(l.g[i].bytes);
        w += (size_t(2) * c.hidden + size_t(2) * c.head_dim) * 2;               // input, post, q, k norms
    }
    const size_t kv = size_t(2) * m->kv_layer_elems * c.n_layers * 2;
    if (weights) *weights = w;
    if (kv_cache) *kv_cache = kv;
    if (scratch) *scratch = total > w + kv ? total - w - kv : 0;
    return total;
}
