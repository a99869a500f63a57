// KMR4 packing of canonical int4 weights (q codes, bf16 scale / zero per
// group of 128 along K) into the tile layout the GEMV streams, and back.
// The layout is specified in kmr.h; this file is its only implementation in
// the library (host loop and a device kernel that produce identical bytes).
#include <string.h>

#include "kmr_internal.cuh"

namespace kmr {

bool pack_geom(int N, int K, int group, PackGeom* g) {
    if (group != 128 || N <= 0 || K <= 0 || K % 128 != 0) return false;
    g->N = N;
    g->K = K;
    g->groups = K / 128;
    g->tiles = (N + 15) / 16;
    g->tile_bytes = g->groups * kGroupBytes;
    g->bytes = (long long)g->tiles * g->tile_bytes;
    return true;
}

// Canonical row held by packed row p (-1: padding row).
__host__ __device__ static inline int canon_row(int p, int N, int gate_up) {
    if (!gate_up) return p < N ? p : -1;
    const int t = p >> 4, r = p & 15, half = N >> 1;
    return r < 8 ? 8 * t + r : half + 8 * t + (r - 8);
}

// The 32-bit word of lane l, k-step ks of group gr in tile T: the lane's mma A
// fragment of that 16x16 block.  g = l / 4, t = l % 4, k0 = 128 gr + 16 ks:
//   bits  0-3 (g, k0+2t)      16-19 (g, k0+2t+1)
//   bits  4-7 (g+8, k0+2t)    20-23 (g+8, k0+2t+1)
//   bits  8-11 (g, k0+2t+8)   24-27 (g, k0+2t+9)
//   bits 12-15 (g+8, k0+2t+8) 28-31 (g+8, k0+2t+9)
// stored at T * tile_bytes + gr * 1088 + (ks / 4) * 512 + l * 16 + (ks % 4) * 4.
__host__ __device__ static inline uint32_t code_at(const uint8_t* q, int N, int K, int gate_up, int prow, int k) {
    const int n = canon_row(prow, N, gate_up);
    return n < 0 ? 8u : (uint32_t(q[(size_t)n * K + k]) & 15u);
}
__host__ __device__ static inline uint32_t pack_word(const uint8_t* q, int N, int K, int gate_up, int T, int gr,
                                                     int ks, int l) {
    const int g = l >> 2, t = l & 3, k0 = gr * 128 + ks * 16;
    const int r0 = T * 16 + g, r1 = r0 + 8;
    return code_at(q, N, K, gate_up, r0, k0 + 2 * t) | code_at(q, N, K, gate_up, r0, k0 + 2 * t + 1) << 16 |
           code_at(q, N, K, gate_up, r1, k0 + 2 * t) << 4 | code_at(q, N, K, gate_up, r1, k0 + 2 * t + 1) << 20 |
           code_at(q, N, K, gate_up, r0, k0 + 2 * t + 8) << 8 | code_at(q, N, K, gate_up, r0, k0 + 2 * t + 9) << 24 |
           code_at(q, N, K, gate_up, r1, k0 + 2 * t + 8) << 12 | code_at(q, N, K, gate_up, r1, k0 + 2 * t + 9) << 28;
}
__host__ __device__ static inline size_t word_offset(const PackGeom& g, int T, int gr, int ks, int l) {
    return (size_t)T * g.tile_bytes + (size_t)gr * kGroupBytes + (ks >> 2) * 512 + l * 16 + (ks & 3) * 4;
}
__host__ __device__ static inline void unpack_word(uint32_t w, uint8_t* q, int N, int K, int gate_up, int T, int gr,
                                                   int ks, int l) {
    const int g = l >> 2, t = l & 3, k0 = gr * 128 + ks * 16;
    const int rows[2] = {T * 16 + g, T * 16 + g + 8};
    const int sh[2][4] = {{0, 16, 8, 24}, {4, 20, 12, 28}};
    const int kk[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
    for (int h = 0; h < 2; ++h) {
        const int n = canon_row(rows[h], N, gate_up);
        if (n < 0) continue;
        for (int e = 0; e < 4; ++e) q[(size_t)n * K + k0 + kk[e]] = uint8_t((w >> sh[h][e]) & 15u);
    }
}

// ------------------------------------------------------------------ host
static void pack_host(const uint8_t* q, const uint16_t* s, const uint16_t* z, const PackGeom& g, int gate_up,
                      uint8_t* out) {
    for (int T = 0; T < g.tiles; ++T)
        for (int gr = 0; gr < g.groups; ++gr) {
            for (int ks = 0; ks < 8; ++ks)
                for (int l = 0; l < 32; ++l) {
                    const uint32_t w = pack_word(q, g.N, g.K, gate_up, T, gr, ks, l);
                    memcpy(out + word_offset(g, T, gr, ks, l), &w, 4);   // little-endian host
                }
            uint8_t* szp = out + (size_t)T * g.tile_bytes + (size_t)gr * kGroupBytes + 1024;
            for (int r = 0; r < 16; ++r) {
                const int n = canon_row(T * 16 + r, g.N, gate_up);
                const uint16_t sv = n < 0 ? 0 : s[(size_t)n * g.groups + gr];
                const uint16_t zv = n < 0 ? 0 : z[(size_t)n * g.groups + gr];
                memcpy(szp + 4 * r, &sv, 2);
                memcpy(szp + 4 * r + 2, &zv, 2);
            }
        }
}

static void unpack_host(const uint8_t* in, const PackGeom& g, int gate_up, uint8_t* q, uint16_t* s, uint16_t* z) {
    for (int T = 0; T < g.tiles; ++T)
        for (int gr = 0; gr < g.groups; ++gr) {
            for (int ks = 0; ks < 8; ++ks)
                for (int l = 0; l < 32; ++l) {
                    uint32_t w;
                    memcpy(&w, in + word_offset(g, T, gr, ks, l), 4);
                    unpack_word(w, q, g.N, g.K, gate_up, T, gr, ks, l);
                }
            const uint8_t* szp = in + (size_t)T * g.tile_bytes + (size_t)gr * kGroupBytes + 1024;
            for (int r = 0; r < 16; ++r) {
                const int n = canon_row(T * 16 + r, g.N, gate_up);
                if (n < 0) continue;
                memcpy(&s[(size_t)n * g.groups + gr], szp + 4 * r, 2);
                memcpy(&z[(size_t)n * g.groups + gr], szp + 4 * r + 2, 2);
            }
        }
}

// ------------------------------------------------------------------ device
// One thread per packed word, plus one per (row, group) scale/zero pair.
__global__ void pack_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                            const uint16_t* __restrict__ z, PackGeom g, int gate_up, uint8_t* __restrict__ out) {
    const long long nwords = (long long)g.tiles * g.groups * 256;
    const long long nsz = (long long)g.tiles * g.groups * 16;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < nwords + nsz;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < nwords) {
            const int l = int(idx & 31), ks = int((idx >> 5) & 7);
            const long long tg = idx >> 8;
            const int gr = int(tg % g.groups), T = int(tg / g.groups);
            *reinterpret_cast<uint32_t*>(out + word_offset(g, T, gr, ks, l)) = pack_word(q, g.N, g.K, gate_up, T, gr, ks, l);
        } else {
            const long long k2 = idx - nwords;
            const int r = int(k2 & 15);
            const long long tg = k2 >> 4;
            const int gr = int(tg % g.groups), T = int(tg / g.groups);
            const int n = canon_row(T * 16 + r, g.N, gate_up);
            const uint32_t sv = n < 0 ? 0u : s[(size_t)n * g.groups + gr];
            const uint32_t zv = n < 0 ? 0u : z[(size_t)n * g.groups + gr];
            *reinterpret_cast<uint32_t*>(out + (size_t)T * g.tile_bytes + (size_t)gr * kGroupBytes + 1024 + r * 4) =
                sv | (zv << 16);
        }
    }
}

__global__ void unpack_kernel(const uint8_t* __restrict__ in, PackGeom g, int gate_up, uint8_t* __restrict__ q,
                              uint16_t* __restrict__ s, uint16_t* __restrict__ z) {
    const long long nwords = (long long)g.tiles * g.groups * 256;
    const long long nsz = (long long)g.tiles * g.groups * 16;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < nwords + nsz;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < nwords) {
            const int l = int(idx & 31), ks = int((idx >> 5) & 7);
            const long long tg = idx >> 8;
            const int gr = int(tg % g.groups), T = int(tg / g.groups);
            unpack_word(*reinterpret_cast<const uint32_t*>(in + word_offset(g, T, gr, ks, l)), q, g.N, g.K, gate_up, T,
                        gr, ks, l);
        } else {
            const long long k2 = idx - nwords;
            const int r = int(k2 & 15);
            const long long tg = k2 >> 4;
            const int gr = int(tg % g.groups), T = int(tg / g.groups);
            const int n = canon_row(T * 16 + r, g.N, gate_up);
            if (n < 0) continue;
            const uint32_t v = *reinterpret_cast<const uint32_t*>(in + (size_t)T * g.tile_bytes +
                                                                  (size_t)gr * kGroupBytes + 1024 + r * 4);
            s[(size_t)n * g.groups + gr] = uint16_t(v & 0xFFFFu);
            z[(size_t)n * g.groups + gr] = uint16_t(v >> 16);
        }
    }
}

int pack_run(const uint8_t* q, const uint16_t* s, const uint16_t* z, int N, int K, int group, int flags,
             void* packed, size_t packed_bytes, int on_device, cudaStream_t st) {
    PackGeom g;
    if (!q || !s || !z || !packed) return KMR_ERR_INVALID_ARG;
    if (flags & ~KMR_PACK_GATE_UP) return KMR_ERR_INVALID_ARG;
    if (!pack_geom(N, K, group, &g)) return KMR_ERR_SHAPE;
    const int gate_up = flags & KMR_PACK_GATE_UP;
    if (gate_up && N % 16 != 0) return KMR_ERR_SHAPE;
    if (packed_bytes < (size_t)g.bytes) return KMR_ERR_BUFFER_SIZE;
    if (!on_device) {
        const size_t n = (size_t)N * K;
        for (size_t i = 0; i < n; ++i)
            if (q[i] > 15) return KMR_ERR_INVALID_ARG;
        pack_host(q, s, z, g, gate_up, static_cast<uint8_t*>(packed));
        return KMR_OK;
    }
    pack_kernel<<<4 * num_sms(), 256, 0, st>>>(q, s, z, g, gate_up, static_cast<uint8_t*>(packed));
    return cudaGetLastError() == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

int unpack_run(const void* packed, size_t packed_bytes, int N, int K, int group, int flags, uint8_t* q, uint16_t* s,
               uint16_t* z, int on_device, cudaStream_t st) {
    PackGeom g;
    if (!q || !s || !z || !packed) return KMR_ERR_INVALID_ARG;
    if (flags & ~KMR_PACK_GATE_UP) return KMR_ERR_INVALID_ARG;
    if (!pack_geom(N, K, group, &g)) return KMR_ERR_SHAPE;
    const int gate_up = flags & KMR_PACK_GATE_UP;
    if (gate_up && N % 16 != 0) return KMR_ERR_SHAPE;
    if (packed_bytes < (size_t)g.bytes) return KMR_ERR_BUFFER_SIZE;
    if (!on_device) {
        unpack_host(static_cast<const uint8_t*>(packed), g, gate_up, q, s, z);
        return KMR_OK;
    }
    unpack_kernel<<<4 * num_sms(), 256, 0, st>>>(static_cast<const uint8_t*>(packed), g, gate_up, q, s, z);
    return cudaGetLastError() == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

}  // namespace kmr
