// The decode step's layers as one persistent kernel.
//
// What it computes: every decoder layer of the one-token greedy decode step ("kaminari — a
// single-GPU Qwen3-VL inference engine, explained", §03 Architecture overview: DecoderLayer =
// RMSNorm, TextAttention with fused QKV, q/k norm and Mrope over the StaticKVCache, O, RMSNorm,
// MLP with fused gate_up, SiLU * up and down; §04 Request lifecycle / decode: token ids (B, 1),
// positions (3, B, 1), per-row cache_position and finished flags; §07 int4 sidecar
// quantization: the linears are weight-only int4, group 128 along K), the attention as split-KV
// with the LSE-weighted merge ("The Ghost in the Batch: How vLLM Silently Switches
// Algorithms", What Attention Does).  The final norm, the LM head and the argmax follow in
// head_kernel (kmr_head.cu).
//
// Why one kernel: at batch 1 the step is a chain of five dependent phases per layer (QKV,
// attention, O, gate_up, down), each moving 2-13 MB; as separate launches every phase paid a
// launch hand-off and a fresh weight fill.  Here one CTA per SM lives for the whole step:
//   * the CTA's share of every layer's weights (and its attention splits' K/V rows) streams
//     through a ring of shared-memory slots with cp.async.bulk, in the order the CTA consumes
//     them, as far ahead as the ring allows — across phase and layer boundaries, since weights
//     and cached K/V never depend on this step's activations.  Thread 0 refills the ring from a
//     per-CTA copy list (the same for every layer but for the layer's base pointers) whenever
//     it waits — on a slot, on another CTA, or between tiles — so no warp is set aside for
//     copying and all 16 warps keep the registers of four warps per SM sub-partition;
//   * the 16 warps run the phases; a phase starts when every CTA has finished the one
//     before (a global counter per (layer, phase), released with a fence and read with
//     acquire loads; every wait is bounded and sets KMR_ERR_DEVICE_TIMEOUT and a global abort
//     flag rather than hang);
//   * the attention splits of a (row, KV head) write their partial states to global memory and
//     the last split to arrive merges them in split order.
// Arithmetic: the projections use the int4 GEMV's blocks (kmr_gemv_core.cuh: same staging,
// same warp-to-group map, same fixed-order sums) and the attention uses the attention kernel's
// blocks (kmr_attn_core.cuh) with the same 8-split plan, so every value is the same bits as
// the multi-kernel step; a row's result does not depend on the batch.
#include <cuda_fp16.h>

#include <algorithm>

#include "kmr_attn_core.cuh"
#include "kmr_gemv_core.cuh"
#include "kmr_step.cuh"

namespace kmr {

// Diagnostic build (-DKMR_STEP_TRACE): thread 0 of every CTA records %globaltimer at each
// phase's start (after its wait) and end, and at points inside the projection phases;
// kmr_step_trace copies the records out.  Compiled out otherwise.
#ifdef KMR_STEP_TRACE
__device__ unsigned long long g_step_trace[160][2 + 2 * 5 * 64];
__device__ unsigned long long g_step_sub[160][5 * 64][5];
#define STEP_MARK(i) do { if (threadIdx.x == 0 && blockIdx.x < 160) g_step_trace[blockIdx.x][(i)] = globaltimer_ns(); } while (0)
#define STEP_SUB(ph, k) do { if (threadIdx.x == 0 && blockIdx.x < 160 && (ph) < 5 * 64) g_step_sub[blockIdx.x][(ph)][(k)] = globaltimer_ns(); } while (0)
#else
#define STEP_MARK(i) do { } while (0)
#define STEP_SUB(ph, k) do { } while (0)
#endif

namespace {

constexpr int kStepWarps = 16;
constexpr int kStepThreads = kStepWarps * 32;
constexpr int kMaxSched = 64;                     // ring copies per CTA per layer
constexpr int kKvChunk = 64;                      // cached positions per ring slot
constexpr int kSplits = kAttnClusterSplits;
constexpr int kPhases = 5;                        // per layer: QKV, attention, O, gate_up, down

__host__ __device__ inline size_t al128(size_t v) { return (v + 127) & ~size_t(127); }

constexpr int kMaxLayersSmem = 64;                // layers whose base pointers are kept in shared memory

struct StepSmem {
    size_t full, empty, misc, rows, sched, bases, norms, gp, rope, ring, xw, xst, ssw, part, qs, knew, vnew, wml, wo, total;
};
__host__ __device__ inline StepSmem step_layout(int MB, int gpw_max, int max_tiles, int D, int REP, int nslots,
                                                int slot_bytes) {
    StepSmem L;
    size_t o = 0;
    L.full = o;  o += size_t(nslots) * 8;
    L.empty = o; o += size_t(nslots) * 8;
    L.misc = o;  o += 64;
    L.rows = o;  o += 256;                         // RowInfo[kStepMaxRows]
    L.sched = o; o += size_t(kMaxSched) * 8;       // SchedEntry[kMaxSched]
    L.bases = o; o += size_t(kMaxLayersSmem) * 6 * 8;   // per layer: the copy sources' base pointers
    L.norms = o; o += size_t(kMaxLayersSmem) * 4 * 8;   // per layer: the RMSNorm weights
    L.gp = o;    o += al128(sizeof(GemvParams));          // the running projection's descriptor
    L.rope = o;  o += al128(size_t(REP + 1) * 32 * 3 * (D / 32) * 4);   // first item's norm weight and rotation
    o = al128(o);
    // phase scratch: the GEMV buffers and the attention buffers are never live together
    const size_t scratch = o;
    L.xw = o;    o += al128(size_t(kStepWarps) * gpw_max * MB * 128 * 2);
    L.xst = o;   o += al128(size_t(kStepWarps) * gpw_max * 16 * 4);
    L.ssw = o;   o += al128(size_t(kStepWarps) * 8 * 4);
    L.part = o;  o += al128(size_t(max_tiles) * kStepWarps * 16 * MB * 4);
    const size_t gemv_end = o;
    o = scratch;
    L.qs = o;    o += al128(size_t(REP) * D * 4);
    L.knew = o;  o += al128(size_t(D) * 2);
    L.vnew = o;  o += al128(size_t(D) * 2);
    L.wml = o;   o += al128(size_t(8) * kAttnMaxRep * 2 * 4);
    L.wo = o;    o += al128(size_t(8) * REP * D * 4);
    o = o > gemv_end ? o : gemv_end;
    L.ring = o;  o += size_t(nslots) * slot_bytes;
    L.total = o;
    return L;
}

// ------------------------------------------------------------------ synchronisation
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kStepWarps * 32) : "memory"); }
__device__ __forceinline__ void attn_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// One thread: wait until *cnt >= target.  False if the step was aborted (by this wait running
// out, which records KMR_ERR_DEVICE_TIMEOUT, or by another CTA).
// The poll is a relaxed load, so a ring copy can be issued while it is in flight; once the
// count is reached, an acquire fence orders this CTA's later reads after the other CTAs' writes.
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ bool counter_wait(const unsigned* cnt, unsigned target, unsigned* abort_flag, int* err) {
    if (ld_relaxed(cnt) >= target) {
        fence_acquire_gpu();
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 28); ++it) {
        if (ld_relaxed(cnt) >= target) {
            fence_acquire_gpu();
            return true;
        }
        if ((it & 63u) == 0) {
            if (ld_relaxed(abort_flag)) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
    set_error(err, KMR_ERR_DEVICE_TIMEOUT);
    atomicExch(abort_flag, 1u);
    return false;
}

// mbarrier phase wait that also gives up when the step is aborted.
__device__ bool ring_wait(uint64_t* b, uint32_t parity, unsigned* abort_flag, int* err) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 28); ++it) {
        if (mbar_try_wait(b, parity)) return true;
        if ((it & 255u) == 0) {
            if (ld_relaxed(abort_flag)) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
    set_error(err, KMR_ERR_DEVICE_TIMEOUT);
    atomicExch(abort_flag, 1u);
    return false;
}

// ------------------------------------------------------------------ the CTA's share of each phase
__device__ __forceinline__ void share(int n, int c, int G, int& a, int& b) {
    a = int((long long)c * n / G);
    b = int((long long)(c + 1) * n / G);
}
__device__ __forceinline__ int tile_slots(int K) { return ((K >> 7) + kStepWarps - 1) / kStepWarps; }

struct RowInfo {
    int cp, slot;
    bool active;                                  // unfinished, slot and cache position in range
    bool bad_slot, bad_pos, fin;
};

// Positions a (row, head, split) item reads from the cache: [t0, cached_end), staged kSub at a time.
struct ItemPlan {
    int ns, t0, t1, cached_end, nsub;
};
__device__ __forceinline__ ItemPlan item_plan(const RowInfo& r, int s, int ksub) {
    ItemPlan q;
    int chunk;
    attn_split_plan(r.cp, kSplits, chunk, q.ns);
    q.t0 = s * chunk;
    q.t1 = min(r.cp + 1, q.t0 + chunk);
    q.cached_end = min(q.t1, r.cp);
    q.nsub = q.t1 > q.t0 ? (q.t1 - q.t0 + ksub - 1) / ksub : 0;
    return q;
}
// Ring slots of stage st: K chunks then V chunks of kKvChunk positions each.
__device__ __forceinline__ int stage_kv_chunks(const ItemPlan& q, int st, int ksub) {
    const int pa = q.t0 + st * ksub;
    const int pb = min(pa + ksub, q.cached_end);
    return pb > pa ? (pb - pa + kKvChunk - 1) / kKvChunk : 0;
}

// ------------------------------------------------------------------ ring copies
// One ring copy of a layer: `bytes` from base pointer `which` of the layer + `off`.
enum { SRC_QKV = 0, SRC_K = 1, SRC_V = 2, SRC_O = 3, SRC_GU = 4, SRC_DOWN = 5 };
struct SchedEntry {
    uint32_t off;
    uint32_t bytes_which;                          // bytes << 4 | which
};

// The CTA's copies of one layer, in the order its warps consume them: its QKV tiles, its
// attention items' K then V chunks stage by stage, its O, gate_up and down tiles (a tile of
// more than 16 groups spans several slots).  Returns the count (<= kMaxSched) or -1.
template <int D>
__device__ int build_schedule(const StepParams& p, const RowInfo* rows, int ksub, SchedEntry* out) {
    const int c = blockIdx.x, G = gridDim.x;
    int n = 0;
    auto put = [&](int which, size_t off, uint32_t bytes) {
        if (n < kMaxSched) out[n] = SchedEntry{uint32_t(off), (bytes << 4) | uint32_t(which)};
        ++n;
    };
    auto tiles = [&](int which, int N, int K) {
        int a, b;
        share(N / 16, c, G, a, b);
        const int groups = K >> 7, nsl = tile_slots(K);
        const size_t tb = size_t(groups) * kGroupBytes;
        for (int t = a; t < b; ++t)
            for (int j = 0; j < nsl; ++j) {
                const int g0 = j * kStepWarps, gn = min(kStepWarps, groups - g0);
                put(which, size_t(t) * tb + size_t(g0) * kGroupBytes, uint32_t(gn) * kGroupBytes);
            }
    };
    const int qd = p.nq * D, nqkv = (p.nq + 2 * p.nkv) * D;
    tiles(SRC_QKV, nqkv, p.H);
    int ia, ib;
    share(p.B * p.nkv * kSplits, c, G, ia, ib);
    for (int it = ia; it < ib; ++it) {
        const int b = it / (p.nkv * kSplits), h = (it / kSplits) % p.nkv, s = it % kSplits;
        const RowInfo& r = rows[b];
        if (!r.active) continue;
        const ItemPlan q = item_plan(r, s, ksub);
        const size_t headoff = ((size_t(r.slot) * p.nkv + h) * p.S) * D * 2;
        for (int st = 0; st < q.nsub; ++st) {
            const int pa = q.t0 + st * ksub, pb = min(pa + ksub, q.cached_end);
            const int nch = stage_kv_chunks(q, st, ksub);
            for (int kv = 0; kv < 2; ++kv)
                for (int j = 0; j < nch; ++j) {
                    const int c0 = pa + j * kKvChunk, c1 = min(pb, c0 + kKvChunk);
                    put(kv ? SRC_V : SRC_K, headoff + size_t(c0) * D * 2, uint32_t(c1 - c0) * D * 2);
                }
        }
    }
    tiles(SRC_O, p.H, qd);
    tiles(SRC_GU, 2 * p.I, p.H);
    tiles(SRC_DOWN, p.H, p.I);
    return n <= kMaxSched ? n : -1;
}

// The ring as every thread sees it (fixed for the kernel).
struct Ring {
    uint64_t* full;
    uint64_t* empty;
    uint8_t* base;
    int n, bytes;
    const SchedEntry* sched;
    const uint8_t* const* bases;                   // [layer][6]
};
// Copy progress, in shared memory, read and written by thread 0 only.
struct PumpState {
    uint32_t per_layer, total, issued, pad;
    uint64_t pol;
};

// The kernel's shared-memory views, rebuilt from the launch constants wherever needed (nothing
// is passed through local memory: with ~217 KB of shared memory the L1 is small, and local
// memory would go to L2).
extern __shared__ __align__(128) uint8_t step_smem[];
template <int MB, int D, int REP>
struct Ctx {
    StepSmem L;
    Ring R;
    PumpState* ps;
    RowInfo* rows;
    volatile int* misc;
    __device__ __forceinline__ explicit Ctx(const StepParams& p) {
        L = step_layout(MB, p.gpw_max, p.max_tiles, D, REP, p.nslots, p.slot_bytes);
        uint8_t* smem = step_smem;
        R = Ring{reinterpret_cast<uint64_t*>(smem + L.full), reinterpret_cast<uint64_t*>(smem + L.empty),
                 smem + L.ring, p.nslots, p.slot_bytes, reinterpret_cast<const SchedEntry*>(smem + L.sched),
                 reinterpret_cast<const uint8_t* const*>(smem + L.bases)};
        ps = reinterpret_cast<PumpState*>(smem + L.misc + 16);
        rows = reinterpret_cast<RowInfo*>(smem + L.rows);
        misc = reinterpret_cast<volatile int*>(smem + L.misc);
    }
};

// Thread 0: issue every copy whose slot is free, without waiting.
__device__ __forceinline__ void pump(const Ring& R, PumpState* ps, uint32_t max_copies = 0xffffffffu) {
    uint32_t q = ps->issued;
    const uint32_t total = ps->total, per = ps->per_layer;
    const uint32_t stop = total - q > max_copies ? q + max_copies : total;
    while (q < stop) {
        const int s = int(q % uint32_t(R.n));
        if (q >= uint32_t(R.n) && !mbar_test_wait(&R.empty[s], ((q / R.n) - 1) & 1)) break;
        const uint32_t l = q / per;
        const SchedEntry e = R.sched[q - l * per];
        const int which = int(e.bytes_which & 15u);
        const uint32_t bytes = e.bytes_which >> 4;
        const uint8_t* src = R.bases[l * 6 + which] + e.off;
        uint8_t* dst = R.base + size_t(s) * R.bytes;
        mbar_arrive_expect_tx(&R.full[s], bytes);
        if (which == SRC_K || which == SRC_V) bulk_g2s(dst, src, bytes, &R.full[s]);
        else bulk_g2s_stream(dst, src, bytes, &R.full[s], ps->pol);
        ++q;
    }
    ps->issued = q;
}

// Wait for ring slot `sq`; thread 0 keeps the ring filled meanwhile.
__device__ __forceinline__ bool ring_acquire(const Ring& R, PumpState* ps, uint32_t sq, unsigned* abort_flag,
                                             int* err) {
    const int s = int(sq % uint32_t(R.n));
    const uint32_t parity = (sq / R.n) & 1;
    if (threadIdx.x == 0) {
        // thread 0 refills the ring at phase boundaries; here only if this slot's copy is late
        if (mbar_test_wait(&R.full[s], parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1; it < (1u << 28); ++it) {
            pump(R, ps);
            if (mbar_test_wait(&R.full[s], parity)) return true;
            if ((it & 63u) == 0) {
                if (ld_relaxed(abort_flag)) return false;
                if (globaltimer_ns() - t0 > kWaitLimitNs) break;
            }
        }
        set_error(err, KMR_ERR_DEVICE_TIMEOUT);
        atomicExch(abort_flag, 1u);
        return false;
    }
    return ring_wait(&R.full[s], parity, abort_flag, err);
}

// ------------------------------------------------------------------ compute phases
// One int4 projection over the CTA's tiles [t0, t1): stage x, block products on the ring's
// tiles (slots released as soon as their products are done), fixed-order epilogue.
// Entry of phase `idx`: wait until every CTA has finished phase idx - 1 (thread 0 polls; lane 0
// of warp 1 refills the ring meanwhile, one copy at a time, until thread 0 raises misc[10]).
// misc[3] records a failed wait; it is read by all threads after the barrier, so every thread
// of the CTA takes the same path.  Returns false if the step was aborted.
template <int MB, int D, int REP>
__device__ __forceinline__ bool phase_enter(const StepParams& p, const Ctx<MB, D, REP>& cx, int idx) {
    const int tid = threadIdx.x;
    volatile int* misc = cx.misc;
    if (idx > 0) {
        if (tid == 0) {
            if (!misc[3] && !counter_wait(&p.phase_cnt[idx - 1], unsigned(gridDim.x), p.abort_flag, p.err))
                misc[3] = 1;
            misc[10] = 1;
        } else if (tid == 32) {
            while (!misc[10]) pump(cx.R, cx.ps, 1u);
        }
    }
    STEP_MARK(2 + 2 * idx);
    compute_sync();
    return misc[3] == 0;
}
// Exit of phase `idx`: once every thread is done (barrier), thread 0 counts this CTA finished
// with a release, which covers the CTA's writes.  Returns false if the CTA has failed.
template <int MB, int D, int REP>
__device__ __forceinline__ bool phase_leave(const StepParams& p, const Ctx<MB, D, REP>& cx, int idx, bool ok) {
    volatile int* misc = cx.misc;
    if (!ok) misc[3] = 1;
    if (threadIdx.x == 0) misc[10] = 0;
    compute_sync();
    STEP_MARK(3 + 2 * idx);
    ok = misc[3] == 0;
    if (threadIdx.x == 0 && ok) red_release_add(&p.phase_cnt[idx], 1u);
    return ok;
}

// What a projection phase can fetch before its grid wait: the RMSNorm weights of the warp's
// groups (constants) and, for a residual add, the first residual value this thread adds to
// (final since an earlier phase of this step, which every CTA has finished).
struct GemvPre {
    uint2 nwv[3];
    float res0;
    int have_res0;
};
template <int MB, int GPW>
__device__ __forceinline__ GemvPre gemv_prefetch(const GemvParams& gp, int t0, int t1) {
    GemvPre q;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, G = gp.K >> 7;
    const bool norm = gp.in_kind != IN_F32;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int grp = warp + j * kStepWarps;
        q.nwv[j] = (j < GPW && norm && grp < G)
                       ? *reinterpret_cast<const uint2*>(gp.norm_w + size_t(grp) * 128 + lane * 4)
                       : make_uint2(0, 0);
    }
    q.res0 = 0.f;
    q.have_res0 = 0;
    const int per = (gp.epi == EPI_SILU ? 8 : 16) * MB;
    if (gp.epi == EPI_RESID && tid < (t1 - t0) * per) {
        const int tl = tid / per, e = tid - tl * per, rr = e / MB, m = e % MB, n = (t0 + tl) * 16 + rr;
        if (m < gp.M && n < gp.N) {
            q.res0 = __ldcg(gp.y + size_t(m) * gp.ldy + n);
            q.have_res0 = 1;
        }
    }
    return q;
}

template <int MB, int GPW, int D, int REP>
__device__ __noinline__ bool gemv_phase(const StepParams& p, int t0, int t1, uint2 n0, uint2 n1, uint2 n2, float res0,
                                        int have_res0, uint32_t seq, int ph) {
    const Ctx<MB, D, REP> cx(p);
    const StepSmem& L = cx.L;
    const Ring& R = cx.R;
    PumpState* ps = cx.ps;
    uint8_t* smem = step_smem;
    unsigned* abort_flag = p.abort_flag;
    const GemvParams& gp = *reinterpret_cast<const GemvParams*>(smem + L.gp);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = t1 - t0;
    if (!phase_enter(p, cx, ph)) return false;
    if (nt <= 0) return phase_leave(p, cx, ph, true);
    STEP_SUB(ph, 0);
    const int K = gp.K, G = K >> 7;
    const int nsl = ((K >> 7) + kStepWarps - 1) / kStepWarps;
    __half* xw = reinterpret_cast<__half*>(smem + L.xw) + size_t(warp) * GPW * MB * 128;
    float* xst = reinterpret_cast<float*>(smem + L.xst) + size_t(warp) * GPW * 16;
    float* ssw = reinterpret_cast<float*>(smem + L.ssw);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint2 nwv[GPW];
    nwv[0] = n0;
    if constexpr (GPW > 1) nwv[1] = n1;
    if constexpr (GPW > 2) nwv[2] = n2;
    stage_x<MB, GPW>(gp, xw, xst, ssw, nwv, t0 == 0 ? 0 : 1, [] {});
    const int g = lane >> 2;
    const bool bload = g < gp.M;
    constexpr int WS = 16 * MB;
    XFrag xf1;
    if (GPW == 1 && warp < G) load_xfrag(xf1, xw + size_t(bload ? g : 0) * 128, bload, lane, xst);
    STEP_SUB(ph, 1);
    // every slot of the CTA's tiles was issued ahead (thread 0 refills only a late one); wait
    // for all of them, then run the products with no synchronisation between tiles
    bool ok = true;
    {
        bool all = true;                           // usually every slot has landed: one cheap sweep
        for (int k = 0; k < nt * nsl; ++k) {
            const uint32_t sq = seq + uint32_t(k);
            all = all && mbar_test_wait(&R.full[sq % uint32_t(R.n)], (sq / uint32_t(R.n)) & 1);
        }
        if (!all)
            for (int k = 0; k < nt * nsl; ++k)
                if (ok && !ring_acquire(R, ps, seq + uint32_t(k), abort_flag, gp.err)) ok = false;
    }
    STEP_SUB(ph, 2);
    const int n = R.n;
    int s = int(seq % uint32_t(n));                   // slot of the tile's first group block
    for (int tl = 0; tl < nt; ++tl) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
            if (j >= nsl) break;
            const int sj = s + j < n ? s + j : s + j - n;
            const int grp = warp + j * kStepWarps;
            if (ok && grp < G) {
                const uint8_t* blk = R.base + size_t(sj) * R.bytes + size_t(warp) * kGroupBytes;
                if constexpr (GPW == 1) {
                    group_product<(MB > 1)>(blk, xf1, lane, acc);
                } else {
                    XFrag xf;
                    load_xfrag(xf, xw + size_t(j * MB + (bload ? g : 0)) * 128, bload, lane, xst + j * 16);
                    group_product<(MB > 1)>(blk, xf, lane, acc);
                }
            }
        }
        __syncwarp();
        if (ok && lane == 0)                     // after a failed wait the ring is left alone
            for (int j = 0; j < nsl; ++j) mbar_arrive(&R.empty[s + j < n ? s + j : s + j - n]);
        s = s + nsl < n ? s + nsl : s + nsl - n;
        store_part<MB>(part + (size_t(tl) * kStepWarps + warp) * WS, lane, acc);
    }
    STEP_SUB(ph, 3);
    compute_sync();
    const int per = (gp.epi == EPI_SILU ? 8 : 16) * MB;
    if (ok)
        for (int idx = tid; idx < nt * per; idx += kStepWarps * 32) {
            const int tl = idx / per;
            tile_epilogue<MB>(gp, part + size_t(tl) * kStepWarps * WS, t0 + tl, idx - tl * per, ssw,
                              idx == tid && have_res0, res0);
        }
    STEP_SUB(ph, 4);
    return phase_leave(p, cx, ph, ok);
}

// The CTA's attention items of one layer: (row, KV head, split) with the attention kernel's
// 8-split plan.  Warps 0..7 score; warps 8..15 only pass the ring slots along.
// The RMSNorm weight and rotation of this warp's head for the CTA's first attention item of a
// layer (warps 0..REP: the q heads and k), fetched before the grid wait: they depend only on
// the layer and the row's positions.
template <int MB, int D, int REP>
__device__ __forceinline__ void rope_prefetch(const StepParams& p, const uint16_t* const* norms, int l,
                                              const RowInfo* rows, float* rope) {
    constexpr int EPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int ia, ib;
    share(p.B * p.nkv * kSplits, blockIdx.x, gridDim.x, ia, ib);
    if (ia < ib && warp <= REP && rows[ia / (p.nkv * kSplits)].active) {
        float nw[EPL], cs[EPL], sn[EPL];
        attn_rope_constants<D>(warp < REP ? norms[l * 4 + 2] : norms[l * 4 + 3], p.pos, p.B, ia / (p.nkv * kSplits),
                               p.inv_freq, p.sec0, p.sec1, lane, nw, cs, sn);
        float* r = rope + (warp * 32 + lane) * 3 * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            r[e] = nw[e];
            r[EPL + e] = cs[e];
            r[2 * EPL + e] = sn[e];
        }
    }
}

// Returns the ring position after the phase's slots, with bit 63 set if a wait failed.
template <int MB, int D, int REP, int CH>
__device__ __noinline__ uint64_t attn_phase(const StepParams& p, int l, uint32_t seq) {
    const Ctx<MB, D, REP> cx(p);
    const StepSmem& L = cx.L;
    const Ring& R = cx.R;
    PumpState* ps = cx.ps;
    const RowInfo* rows = cx.rows;
    uint8_t* smem = step_smem;
    const uint8_t* const* bases = reinterpret_cast<const uint8_t* const*>(smem + L.bases);
    const uint16_t* const* norms = reinterpret_cast<const uint16_t* const*>(smem + L.norms);
    uint16_t* const kcache = const_cast<uint16_t*>(reinterpret_cast<const uint16_t*>(bases[l * 6 + SRC_K]));
    uint16_t* const vcache = const_cast<uint16_t*>(reinterpret_cast<const uint16_t*>(bases[l * 6 + SRC_V]));
    const float* rope = reinterpret_cast<const float*>(smem + L.rope);
    const int ph = l * kPhases + 1;
    if (!phase_enter(p, cx, ph)) return uint64_t(seq) | (1ull << 63);
    STEP_SUB(ph, 0);
    constexpr int EPL = D / 32;
    constexpr int kSub = 8 * CH;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    float* qs = reinterpret_cast<float*>(smem + L.qs);
    uint16_t* knew = reinterpret_cast<uint16_t*>(smem + L.knew);
    uint16_t* vnew = reinterpret_cast<uint16_t*>(smem + L.vnew);
    float* wml = reinterpret_cast<float*>(smem + L.wml);
    float* wo = reinterpret_cast<float*>(smem + L.wo);
    volatile int* flag = reinterpret_cast<volatile int*>(smem + L.misc);
    const int qd = p.nq * D, nqkv = (p.nq + 2 * p.nkv) * D;
    const int items = p.B * p.nkv * kSplits;
    int ia, ib;
    share(items, c, G, ia, ib);
    bool ok = true;
    for (int it = ia; it < ib; ++it) {
        const int b = it / (p.nkv * kSplits), h = (it / kSplits) % p.nkv, s = it % kSplits;
        const RowInfo& r = rows[b];
        float* outrow = p.attn + size_t(b) * qd + size_t(h) * REP * D;
        if (!r.active) {
            // finished or invalid row: no K/V traffic, the output is zero (error recorded once)
            if (s == 0 && warp < 8) {
                if (!r.fin && h == 0 && tid == 0) set_error(p.err, r.bad_slot ? KMR_ERR_SLOT_RANGE : KMR_ERR_CACHE_FULL);
                for (int i = tid; i < REP * D; i += 256) outrow[i] = 0.f;
            }
            continue;
        }
        const ItemPlan q = item_plan(r, s, kSub);
        if (s >= q.ns) continue;                              // empty split: nothing to read or merge
        const size_t headoff = (size_t(r.slot) * p.nkv + h) * p.S * D;
        const int cp = r.cp;
        // ---- prologue: q (scaled into base 2), the new k and v (bf16) of this KV head
        const float qscale = __fmul_rn(p.scale, kAttnLog2e);
        if (warp <= REP + 1) {
            const bool isq = warp < REP, isk = warp == REP;
            const float* in = p.qkv + size_t(b) * nqkv;
            const float* src = isq ? in + size_t(h * REP + warp) * D
                                   : (isk ? in + size_t(qd) + size_t(h) * D : in + size_t(qd + p.nkv * D) + size_t(h) * D);
            float x[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[e] = __ldcg(src + lane * EPL + e);
            if (warp <= REP) {
                if (it == ia) {
                    float nw[EPL], cs[EPL], sn[EPL];
                    const float* r = rope + (warp * 32 + lane) * 3 * EPL;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        nw[e] = r[e];
                        cs[e] = r[EPL + e];
                        sn[e] = r[2 * EPL + e];
                    }
                    attn_norm_rope<D>(x, p.qk_norm != 0, p.eps, nw, cs, sn, lane);
                } else {
                    float nw[EPL], cs[EPL], sn[EPL];
                    attn_rope_constants<D>(isq ? norms[l * 4 + 2] : norms[l * 4 + 3], p.pos, p.B, b, p.inv_freq, p.sec0, p.sec1,
                                           lane, nw, cs, sn);
                    attn_norm_rope<D>(x, p.qk_norm != 0, p.eps, nw, cs, sn, lane);
                }
            }
            if (isq) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) qs[warp * D + lane * EPL + e] = __fmul_rn(x[e], qscale);
            } else {
                uint16_t* dst = isk ? knew : vnew;
                uint16_t* cache = isk ? kcache : vcache;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const uint16_t v = f32_to_bf16_rn(x[e]);
                    dst[lane * EPL + e] = v;
                    if (s == q.ns - 1) cache[headoff + size_t(cp) * D + lane * EPL + e] = v;
                }
            }
        }
        compute_sync();
        STEP_SUB(ph, 1);
        // ---- per-warp online softmax over the split's stages
        float qreg[REP][EPL], m[REP], lsum[REP], o[REP][EPL];
#pragma unroll
        for (int hh = 0; hh < REP; ++hh) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qreg[hh][e] = qs[hh * D + lane * EPL + e];
                o[hh][e] = 0.f;
            }
            m[hh] = -INFINITY;
            lsum[hh] = 0.f;
        }
        for (int st = 0; st < q.nsub; ++st) {
            const int pa = q.t0 + st * kSub;
            const int np = min(kSub, q.t1 - pa);              // positions of this stage, the new one included
            const int nch = stage_kv_chunks(q, st, kSub);
            static_assert(kSub <= 2 * kKvChunk, "a stage spans at most two chunks of K and two of V");
            for (int j = 0; j < 2 * nch; ++j)
                if (ok && !ring_acquire(R, ps, seq + j, p.abort_flag, p.err)) ok = false;
            auto slot_ptr = [&](int j) {
                return reinterpret_cast<const uint16_t*>(R.base + size_t((seq + j) % uint32_t(R.n)) * R.bytes);
            };
            const uint16_t* k0 = slot_ptr(0);
            const uint16_t* k1 = slot_ptr(nch > 1 ? 1 : 0);
            const uint16_t* v0 = slot_ptr(nch);
            const uint16_t* v1 = slot_ptr(nch > 1 ? nch + 1 : nch);
            const int c0 = warp * CH;
            if (ok && warp < 8 && c0 < np) {
                const int nv = min(CH, np - c0);
                auto krow = [&](int j) -> const uint16_t* {
                    const int i = c0 + j;
                    return pa + i == cp ? knew : (i < kKvChunk ? k0 + size_t(i) * D : k1 + size_t(i - kKvChunk) * D);
                };
                auto vrow = [&](int j) -> const uint16_t* {
                    const int i = c0 + j;
                    return pa + i == cp ? vnew : (i < kKvChunk ? v0 + size_t(i) * D : v1 + size_t(i - kKvChunk) * D);
                };
                attn_score_chunk<D, REP, CH>(nv, krow, vrow, qreg, m, lsum, o, lane);
            }
            __syncwarp();
            if (ok && lane == 0)
                for (int j = 0; j < 2 * nch; ++j) mbar_arrive(&R.empty[(seq + j) % uint32_t(R.n)]);
            seq += 2 * nch;
        }
        STEP_SUB(ph, 2);
        // ---- the 8 warps' states, merged in warp order, written as this split's state
        if (warp < 8) {
#pragma unroll
            for (int hh = 0; hh < REP; ++hh) {
                if (lane == 0) {
                    wml[(warp * kAttnMaxRep + hh) * 2] = m[hh];
                    wml[(warp * kAttnMaxRep + hh) * 2 + 1] = lsum[hh];
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) wo[(size_t(warp) * REP + hh) * D + lane * EPL + e] = o[hh][e];
            }
        }
        compute_sync();
        float* mypart = p.part + ((size_t(b) * p.nkv + h) * kSplits + s) * REP * (D + 2);
        if (warp < 8) {
            for (int i = tid; i < REP * D; i += 256) {
                const int hh = i / D, dim = i % D;
                float mx, num, den;
                attn_warp_merge<D, REP>(wml, wo, hh, dim, mx, num, den);
                mypart[hh * (D + 2) + 2 + dim] = num;
                if (dim == 0) {
                    mypart[hh * (D + 2)] = mx;
                    mypart[hh * (D + 2) + 1] = den;
                }
            }
            attn_sync();
            if (tid == 0) {
                __threadfence();
                unsigned* ctr = p.merge_cnt + size_t(b) * p.nkv + h;
                const unsigned old = atomicAdd(ctr, 1u);
                flag[0] = old == unsigned(q.ns - 1);
                if (old == unsigned(q.ns - 1)) {
                    *ctr = 0u;                                   // ready for the next layer
                    __threadfence();
                }
            }
            attn_sync();
            STEP_SUB(ph, 3);
            if (flag[0]) {
                // last split of this (row, KV head) to arrive: merge every split in split order
                const float* parts = p.part + (size_t(b) * p.nkv + h) * kSplits * REP * (D + 2);
                for (int i = tid; i < REP * D; i += 256) {
                    const int hh = i / D, dim = i % D;
                    float mr[kSplits], lr[kSplits], nr[kSplits];
#pragma unroll
                    for (int rr = 0; rr < kSplits; ++rr) {
                        mr[rr] = -INFINITY;
                        lr[rr] = nr[rr] = 0.f;
                        if (rr < q.ns) {
                            const float* pr = parts + size_t(rr) * REP * (D + 2) + hh * (D + 2);
                            mr[rr] = __ldcg(pr);
                            lr[rr] = __ldcg(pr + 1);
                            nr[rr] = __ldcg(pr + 2 + dim);
                        }
                    }
                    outrow[i] = attn_split_merge(mr, lr, nr);
                }
            }
        }
        compute_sync();                                   // wml / wo / qs are reused by the next item
        STEP_SUB(ph, 4);
    }
    ok = phase_leave(p, cx, ph, ok);
    return uint64_t(seq) | (ok ? 0ull : (1ull << 63));
}

template <int MB, int D, int REP, int CH>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
    uint8_t* smem = step_smem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    constexpr int kSub = 8 * CH;
    const StepSmem L = step_layout(MB, p.gpw_max, p.max_tiles, D, REP, p.nslots, p.slot_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + L.misc);

    // Row state comes from the previous step (complete before this kernel started).
    RowInfo* rows = reinterpret_cast<RowInfo*>(smem + L.rows);
    if (tid < kStepMaxRows) {
        RowInfo r{0, 0, false, false, false, true};
        if (tid < p.B) {
            r.fin = p.fin[tid] != 0;
            r.slot = p.slot[tid];
            r.cp = p.cpos[tid];
            r.bad_slot = r.slot < 0 || r.slot >= p.slots;
            r.bad_pos = r.cp < 0 || r.cp >= p.S;
            r.active = !r.fin && !r.bad_slot && !r.bad_pos;
        }
        rows[tid] = r;
    }
    // every layer's copy sources (the pump reads them per copy)
    const uint8_t** bases = reinterpret_cast<const uint8_t**>(smem + L.bases);
    for (int i = tid; i < p.L * 4; i += kStepThreads)
        reinterpret_cast<const uint16_t**>(smem + L.norms)[i] = p.layers[i / 4].norm[i % 4];
    for (int i = tid; i < p.L * 6; i += kStepThreads) {
        const StepLayer& ly = p.layers[i / 6];
        const int w = i % 6;
        bases[i] = w == SRC_QKV ? ly.w[0] : w == SRC_K ? reinterpret_cast<const uint8_t*>(ly.kc)
                 : w == SRC_V ? reinterpret_cast<const uint8_t*>(ly.vc) : w == SRC_O ? ly.w[1]
                 : w == SRC_GU ? ly.w[2] : ly.w[3];
    }
    if (tid == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kStepWarps);
        }
        misc[1] = 0;
        misc[3] = 0;
        misc[10] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    STEP_MARK(0);
    pdl_launch_dependents();                       // the LM head may queue behind this kernel

    SchedEntry* sched = reinterpret_cast<SchedEntry*>(smem + L.sched);
    PumpState* ps = reinterpret_cast<PumpState*>(smem + L.misc + 16);
    const Ring R{full, empty, smem + L.ring, p.nslots, p.slot_bytes, sched, bases};
    uint32_t seq = 0;                              // next ring slot this thread's warp consumes
    if (tid == 0) {
        const int n = build_schedule<D>(p, rows, kSub, sched);
        misc[2] = n;
        ps->issued = 0;
        ps->per_layer = n > 0 ? uint32_t(n) : 1u;
        ps->total = n > 0 ? uint32_t(n) * uint32_t(p.L) : 0u;
        ps->pol = policy_evict_first();
        pump(R, ps);                               // the first fill
    }
    compute_sync();
    STEP_MARK(1);
    if (misc[2] < 0) {                             // the host checks the copy count; never taken
        if (tid == 0) set_error(p.err, KMR_ERR_SHAPE);
        return;
    }
    const int qd = p.nq * D, nqkv = (p.nq + 2 * p.nkv) * D;
    unsigned* cnt = p.phase_cnt;
    bool ok = true;
    // a projection phase: publish its descriptor, fetch what does not depend on the previous
    // phase (norm weights, the first residual), wait for the previous phase, run
    GemvParams* gps = reinterpret_cast<GemvParams*>(smem + L.gp);
    auto projection = [&](int idx, const GemvParams& gp) {
        int t0, t1;
        share(gp.tiles, c, G, t0, t1);
        const int gpw = ((gp.K >> 7) + kStepWarps - 1) / kStepWarps;
        if (tid == 0) *gps = gp;                   // read after the barrier in enter()
        const GemvPre pre = gpw == 1 ? gemv_prefetch<MB, 1>(gp, t0, t1) : gemv_prefetch<MB, 3>(gp, t0, t1);
        // the phase waits for the previous one inside (the call's overhead overlaps the wait)
        const bool r = gpw == 1
            ? gemv_phase<MB, 1, D, REP>(p, t0, t1, pre.nwv[0], pre.nwv[1], pre.nwv[2], pre.res0, pre.have_res0, seq, idx)
            : gemv_phase<MB, 3, D, REP>(p, t0, t1, pre.nwv[0], pre.nwv[1], pre.nwv[2], pre.res0, pre.have_res0, seq, idx);
        seq += uint32_t(t1 > t0 ? t1 - t0 : 0) * uint32_t(gpw);
        if (!r) ok = false;
    };
    const uint16_t* const* norms = reinterpret_cast<const uint16_t* const*>(smem + L.norms);
    float* rope = reinterpret_cast<float*>(smem + L.rope);
    for (int l = 0; l < p.L && ok; ++l) {
        const int base = l * kPhases;
        GemvParams gp = {};
        gp.M = p.B;
        gp.eps = p.eps;
        gp.err = p.err;
        // ---- QKV (+ input RMSNorm; layer 0 embeds the tokens)
        gp.N = nqkv;
        gp.K = p.H;
        gp.tiles = nqkv / 16;
        gp.tile_bytes = (p.H >> 7) * kGroupBytes;
        gp.in_kind = l == 0 ? IN_EMBED_NORM : IN_F32_NORM;
        gp.x = p.x;
        gp.embed = p.embed;
        gp.tokens = p.tok;
        gp.vocab = p.vocab;
        gp.x_out = l == 0 ? p.x : nullptr;
        gp.norm_w = norms[l * 4 + 0];
        gp.epi = EPI_STORE;
        gp.y = p.qkv;
        gp.ldy = nqkv;
        projection(base, gp);
        if (!ok) break;
        // ---- attention
        rope_prefetch<MB, D, REP>(p, norms, l, rows, rope);
        {
            const uint64_t r = attn_phase<MB, D, REP, CH>(p, l, seq);
            seq = uint32_t(r);
            if (r >> 63) ok = false;
        }
        if (!ok) break;
        // ---- O + residual
        gp.N = p.H;
        gp.K = qd;
        gp.tiles = p.H / 16;
        gp.tile_bytes = (qd >> 7) * kGroupBytes;
        gp.in_kind = IN_F32;
        gp.x = p.attn;
        gp.x_out = nullptr;
        gp.norm_w = nullptr;
        gp.epi = EPI_RESID;
        gp.y = p.x;
        gp.ldy = p.H;
        projection(base + 2, gp);
        if (!ok) break;
        // ---- gate_up (+ post-attention RMSNorm) -> SiLU(gate) * up
        gp.N = 2 * p.I;
        gp.K = p.H;
        gp.tiles = 2 * p.I / 16;
        gp.tile_bytes = (p.H >> 7) * kGroupBytes;
        gp.in_kind = IN_F32_NORM;
        gp.x = p.x;
        gp.norm_w = norms[l * 4 + 1];
        gp.epi = EPI_SILU;
        gp.y = p.act;
        gp.ldy = p.I;
        projection(base + 3, gp);
        if (!ok) break;
        // ---- down + residual
        gp.N = p.H;
        gp.K = p.I;
        gp.tiles = p.H / 16;
        gp.tile_bytes = (p.I >> 7) * kGroupBytes;
        gp.in_kind = IN_F32;
        gp.x = p.act;
        gp.norm_w = nullptr;
        gp.epi = EPI_RESID;
        gp.y = p.x;
        gp.ldy = p.H;
        projection(base + 4, gp);
    }
    // ---- end of the step: the last CTA out resets the counters for the next step
    compute_sync();
    if (tid == 0) {
        // Every copy issued into this CTA's shared memory must have landed before it exits
        // (after an abort some were never consumed): wait, bounded, for the latest fill of
        // each slot; a slot is refilled only after its previous fill was consumed.
        const uint32_t issued = ps->issued;
        for (uint32_t k = 0; k < uint32_t(p.nslots) && k < issued; ++k) {
            const uint32_t q = issued - 1 - k;
            mbar_wait(&full[q % uint32_t(p.nslots)], (q / uint32_t(p.nslots)) & 1, p.err);
        }
        __threadfence();
        const unsigned old = atomicAdd(p.done_cnt, 1u);
        if (old == unsigned(G - 1)) {
            for (int i = 0; i < p.L * kPhases; ++i) cnt[i] = 0u;
            for (int i = 0; i < p.B * p.nkv; ++i) p.merge_cnt[i] = 0u;
            *p.abort_flag = 0u;
            *p.done_cnt = 0u;
            __threadfence();
        }
    }
}

template <int MB, int D, int REP, int CH>
const void* step_fn() {
    return (const void*)step_kernel<MB, D, REP, CH>;
}

const void* step_fn_for(int MB, int D, int REP, int CH) {
    if (D == 128 && REP == 2 && CH == 16) return MB == 1 ? step_fn<1, 128, 2, 16>() : step_fn<4, 128, 2, 16>();
    if (D == 64 && REP == 2 && CH == 8) return MB == 1 ? step_fn<1, 64, 2, 8>() : step_fn<4, 64, 2, 8>();
    return nullptr;
}

}  // namespace

bool step_supported(int B, int n_layers, int hidden, int nq, int nkv, int d, int inter, int max_len, int sms,
                    StepPlan* plan) {
    if (B < 1 || B > kStepMaxRows || nq % nkv || n_layers < 1 || n_layers > kMaxLayersSmem || sms < 1) return false;
    const int rep = nq / nkv;
    const int ch = attn_chunk(max_len, kAttnClusterSplits, rep);
    if (!step_fn_for(B == 1 ? 1 : 4, d, rep, ch)) return false;
    if (hidden % 128 || inter % 128 || (nq * d) % 128) return false;
    auto gpw = [](int K) { return ((K >> 7) + kStepWarps - 1) / kStepWarps; };
    if (gpw(hidden) != 1 || gpw(nq * d) != 1 || (gpw(inter) != 1 && gpw(inter) != 3)) return false;
    const int G = sms;
    auto maxt = [&](int tiles) { return (tiles + G - 1) / G; };
    const int nqkv = (nq + 2 * nkv) * d;
    int mt = std::max(std::max(maxt(nqkv / 16), maxt(hidden / 16)), std::max(maxt(2 * inter / 16), maxt(hidden / 16)));
    const int MB = B == 1 ? 1 : 4;
    const int slot_bytes = std::max(kStepWarps * kGroupBytes, kKvChunk * d * 2);
    const int gpw_max = std::max(gpw(inter), 1);
    // ring: whatever shared memory is left, at least one stage of attention (4 slots) and a
    // 3-slot tile; at most 16 slots
    const size_t budget = 227 * 1024;
    const size_t fixed = step_layout(MB, gpw_max, mt, d, rep, 0, slot_bytes).total + 16 * 16;
    if (fixed >= budget) return false;
    int nslots = int((budget - fixed) / slot_bytes);
    if (nslots > 16) nslots = 16;
    if (nslots < 4 || nslots < mt) return false;
    // ring copies per CTA per layer must fit the copy list: tiles, plus every attention item's
    // stages of K and V chunks at the longest split the cache allows
    const int tslots = ((inter >> 7) + kStepWarps - 1) / kStepWarps;
    const int ksub = 8 * ch;
    const int chunk_max = (((max_len + kAttnClusterSplits - 1) / kAttnClusterSplits) + 15) & ~15;
    const int per_item = ((chunk_max + ksub - 1) / ksub) * 2 * ((ksub + kKvChunk - 1) / kKvChunk);
    const int items = (B * nkv * kAttnClusterSplits + G - 1) / G;
    const int copies = maxt(nqkv / 16) + items * per_item + maxt(hidden / 16) + maxt(2 * inter / 16) +
                       maxt(hidden / 16) * tslots;
    if (copies > kMaxSched) return false;
    if (plan) {
        plan->MB = MB;
        plan->ch = ch;
        plan->rep = rep;
        plan->gpw_max = gpw_max;
        plan->max_tiles = mt;
        plan->nslots = nslots;
        plan->slot_bytes = slot_bytes;
        plan->smem = step_layout(MB, gpw_max, mt, d, rep, nslots, slot_bytes).total;
        plan->grid = G;
    }
    return true;
}

cudaError_t step_set_attributes() {
    const void* fns[4] = {step_fn<1, 128, 2, 16>(), step_fn<4, 128, 2, 16>(), step_fn<1, 64, 2, 8>(),
                          step_fn<4, 64, 2, 8>()};
    for (const void* k : fns) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_step(const StepParams& p, const StepPlan& plan, int d, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;       // every CTA resident at once (they wait on each other)
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    StepParams q = p;
    void* args[] = {&q};
    return cudaLaunchKernelExC(&cfg, step_fn_for(plan.MB, d, plan.rep, plan.ch), args);
}

int step_max_active_ctas(const StepPlan& plan, int d) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_fn_for(plan.MB, d, plan.rep, plan.ch), kStepThreads,
                                                      plan.smem) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace kmr

#ifdef KMR_STEP_TRACE
extern "C" int kmr_step_trace(unsigned long long* marks, unsigned long long* subs) {
    if (cudaMemcpyFromSymbol(marks, kmr::g_step_trace, sizeof(kmr::g_step_trace)) != cudaSuccess) return -1;
    return cudaMemcpyFromSymbol(subs, kmr::g_step_sub, sizeof(kmr::g_step_sub)) == cudaSuccess ? 0 : -1;
}
#endif
