// KV row migration between static caches ("kaminari — a single-GPU Qwen3-VL inference
// engine, explained", §08 The serving layer: the continuous scheduler's slot pool owns one
// static cache with a physical row per slot, and copy_row_from moves a row's KV state into
// it; §03 State model: the cache buffers are mutated in place).
//
// A row of a cache [L][slots][n_kv][max_len][d] is L * n_kv * 2 (K and V) segments, each
// positions [0, length) of one (layer, head): length * d contiguous bf16 values.  One launch
// copies every segment: blockIdx.y picks the segment, the x-blocks stride over it in
// 16-byte units, four loads in flight per thread before their stores.  HBM-bound: the bytes
// moved are 2 (read + write) * L * n_kv * 2 * length * d * 2.
#include "kmr_internal.cuh"

namespace kmr {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) kv_row_copy_kernel(const KvCopyParams p) {
    const int seg = blockIdx.y;                       // (layer, K/V, head)
    const int l = seg / (2 * p.nkv), kv = (seg / p.nkv) & 1, h = seg % p.nkv;
    const uint16_t* sbase = kv ? p.src_v : p.src_k;
    uint16_t* dbase = kv ? p.dst_v : p.dst_k;
    const uint4* src = reinterpret_cast<const uint4*>(
        sbase + ((size_t(l) * p.src_slots + p.src_row) * p.nkv + h) * size_t(p.src_max_len) * p.d);
    uint4* dst = reinterpret_cast<uint4*>(
        dbase + ((size_t(l) * p.dst_slots + p.dst_row) * p.nkv + h) * size_t(p.dst_max_len) * p.d);
    const long long units = p.units;                  // 16-byte units per segment
    const long long stride = (long long)gridDim.x * kCopyThreads * kCopyUnroll;
    for (long long u0 = (long long)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x; u0 < units; u0 += stride) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int i = 0; i < kCopyUnroll; ++i) {
            const long long u = u0 + (long long)i * kCopyThreads;
            if (u < units) v[i] = __ldcs(src + u);
        }
#pragma unroll
        for (int i = 0; i < kCopyUnroll; ++i) {
            const long long u = u0 + (long long)i * kCopyThreads;
            if (u < units) __stcs(dst + u, v[i]);
        }
    }
}

}  // namespace

cudaError_t launch_kv_row_copy(const KvCopyParams& p, int sms, cudaStream_t st) {
    if (p.units <= 0) return cudaSuccess;
    const long long per_block = (long long)kCopyThreads * kCopyUnroll;
    const int segs = 2 * p.L * p.nkv;
    // enough blocks to fill the GPU a few times over, at most one pass per block
    long long bx = (p.units + per_block - 1) / per_block;
    const long long want = (4LL * sms + segs - 1) / segs;
    if (bx > want) bx = want < 1 ? 1 : want;
    kv_row_copy_kernel<<<dim3(unsigned(bx), unsigned(segs)), kCopyThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kmr
