// kmr_decode_attn_noalloc: the split-KV decode attention for callers that must
// not allocate device memory.
//
// Some callers cannot call cudaMalloc: code running while a CUDA graph is being
// captured in global mode, engines whose memory planner owns every byte of the
// device heap, and latency-critical loops that cannot afford cudaMalloc's
// implicit device synchronisation.  kmr_decode_attn needs a caller-allocated
// workspace for its per-split partial results; this entry point instead uses
// one fixed array that lives in the library's device image, so the caller only
// passes inputs and outputs.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it, so calls that overlap on the GPU (different streams without
// ordering between them) race on it.  The arrival counters that must start at
// zero are cleared with cudaMemsetAsync on the caller's stream before every
// launch; nothing here allocates.
#include <mutex>

#include "kmr_internal.cuh"

namespace kmr {

constexpr size_t kNoallocAttnScratchBytes = KMR_NOALLOC_ATTN_SCRATCH_BYTES;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_attn_scratch[kNoallocAttnScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KMR_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return KMR_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KMR_OK;
}

size_t round16(size_t v) { return (v + 15) & ~size_t(15); }

}  // namespace
}  // namespace kmr

using namespace kmr;

extern "C" int kmr_decode_attn_noalloc(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                       const int32_t* slot_ids, const int32_t* cache_position, int B, int nq,
                                       int nkv, int d, int max_len, int slots, float scale, float* out,
                                       void* stream) {
    if (!q || !k_cache || !v_cache || !slot_ids || !cache_position || !out) return KMR_ERR_INVALID_ARG;
    if (B < 1 || B > 65535) return KMR_ERR_BATCH;
    if (nq < 1 || nkv < 1 || nq % nkv || (nq / nkv) > 4 || (nq / nkv) == 3) return KMR_ERR_SHAPE;
    if ((d != 64 && d != 128) || max_len < 1 || slots < 1) return KMR_ERR_SHAPE;
    if (!(scale == scale)) return KMR_ERR_INVALID_ARG;
    const int tsplit = attn_default_tsplit(nkv);
    const size_t part_bytes = round16(size_t(B) * nq * tsplit * (d + 2) * sizeof(float));
    const size_t cnt_bytes = size_t(B) * nkv * sizeof(int);
    if (part_bytes + cnt_bytes > kNoallocAttnScratchBytes) return KMR_ERR_SHAPE;   // beyond the fixed scratch
    if (ensure_kernel_attributes() != cudaSuccess) return KMR_ERR_CUDA;
    int* err = standalone_error_word();
    if (!err) return KMR_ERR_CUDA;
    void* base = nullptr;
    const int rc = scratch_address(&base);
    if (rc != KMR_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* counters = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + part_bytes);
    if (cudaMemsetAsync(counters, 0, cnt_bytes, st) != cudaSuccess) return KMR_ERR_CUDA;
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
    p.tsplit = tsplit;
    p.out = out;
    p.part = static_cast<float*>(base);
    p.counters = counters;
    p.err = err;
    return launch_attn(p, st, false) == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}
