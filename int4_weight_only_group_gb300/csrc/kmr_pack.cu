// KMR4 packing of canonical int4 weights (q codes, bf16 scale / zero per
// group of 128 along K) into the unit layout the GEMV streams, and back.
// The layout is specified in kmr.h; this file is its only implementation in
// the library (host loop and a device kernel that produce identical bytes).
#include <string.h>

#include "kmr_internal.cuh"

namespace kmr {

static const int kBitOff[8] = {0, 16, 4, 20, 8, 24, 12, 28};
__constant__ int c_bitoff[8] = {0, 16, 4, 20, 8, 24, 12, 28};

bool pack_geom(int N, int K, int group, PackGeom* g) {
    if (group != 128 || N <= 0 || K <= 0 || K % 128 != 0) return false;
    int wks = 0;
    for (int w = 1024; w >= 128; w -= 128)
        if (K % w == 0) { wks = w; break; }
    g->N = N;
    g->K = K;
    g->wks = wks;
    g->ksl = K / wks;
    g->tiles = (N + 7) / 8;
    g->unit_bytes = 4 * wks + wks / 4;
    g->bytes = (long long)g->tiles * g->ksl * g->unit_bytes;
    return true;
}

// Canonical row held by packed row p (-1: padding row).
__host__ __device__ static inline int canon_row(int p, int N, int gate_up) {
    if (!gate_up) return p < N ? p : -1;
    const int t = p >> 3, r = p & 7, half = N >> 1;
    return r < 4 ? 4 * t + r : half + 4 * t + (r - 4);
}

// ------------------------------------------------------------------ host
static void pack_host(const uint8_t* q, const uint16_t* s, const uint16_t* z, const PackGeom& g, int gate_up,
                      uint8_t* out) {
    const int W = g.wks, G = W / 128, KG = g.K / 128;
    for (int p = 0; p < g.tiles * 8; ++p) {
        const int n = canon_row(p, g.N, gate_up);
        const int t = p >> 3, r = p & 7;
        for (int j = 0; j < g.ksl; ++j) {
            uint8_t* unit = out + ((size_t)t * g.ksl + j) * g.unit_bytes;
            uint8_t* rowp = unit + (size_t)r * (W / 2);
            for (int i = 0; i < W / 8; ++i) {
                uint32_t word = 0;
                for (int e = 0; e < 8; ++e) {
                    const uint32_t code = n < 0 ? 8u : q[(size_t)n * g.K + (size_t)j * W + 8 * i + e];
                    word |= code << kBitOff[e];
                }
                memcpy(rowp + 4 * i, &word, 4);   // little-endian host
            }
            uint8_t* szp = unit + 4 * W + (size_t)r * G * 4;
            for (int gl = 0; gl < G; ++gl) {
                const uint16_t sv = n < 0 ? 0 : s[(size_t)n * KG + j * G + gl];
                const uint16_t zv = n < 0 ? 0 : z[(size_t)n * KG + j * G + gl];
                memcpy(szp + 4 * gl, &sv, 2);
                memcpy(szp + 4 * gl + 2, &zv, 2);
            }
        }
    }
}

static void unpack_host(const uint8_t* in, const PackGeom& g, int gate_up, uint8_t* q, uint16_t* s, uint16_t* z) {
    const int W = g.wks, G = W / 128, KG = g.K / 128;
    for (int p = 0; p < g.tiles * 8; ++p) {
        const int n = canon_row(p, g.N, gate_up);
        if (n < 0) continue;
        const int t = p >> 3, r = p & 7;
        for (int j = 0; j < g.ksl; ++j) {
            const uint8_t* unit = in + ((size_t)t * g.ksl + j) * g.unit_bytes;
            const uint8_t* rowp = unit + (size_t)r * (W / 2);
            for (int i = 0; i < W / 8; ++i) {
                uint32_t word;
                memcpy(&word, rowp + 4 * i, 4);
                for (int e = 0; e < 8; ++e) q[(size_t)n * g.K + (size_t)j * W + 8 * i + e] = (word >> kBitOff[e]) & 15u;
            }
            const uint8_t* szp = unit + 4 * W + (size_t)r * G * 4;
            for (int gl = 0; gl < G; ++gl) {
                memcpy(&s[(size_t)n * KG + j * G + gl], szp + 4 * gl, 2);
                memcpy(&z[(size_t)n * KG + j * G + gl], szp + 4 * gl + 2, 2);
            }
        }
    }
}

// ------------------------------------------------------------------ device
// One thread per packed 32-bit nibble word, plus one per (row, group) scale/zero pair.
__global__ void pack_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                            const uint16_t* __restrict__ z, PackGeom g, int gate_up, uint8_t* __restrict__ out) {
    const int W = g.wks, G = W / 128, KG = g.K / 128, wpr = g.K / 8;   // words per packed row
    const long long nwords = (long long)g.tiles * 8 * wpr;
    const long long nsz = (long long)g.tiles * 8 * KG;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < nwords + nsz;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < nwords) {
            const int p = int(idx / wpr), wi = int(idx % wpr);
            const int n = canon_row(p, g.N, gate_up);
            const int j = (wi * 8) / W, i = wi - j * (W / 8);
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t code = n < 0 ? 8u : (q[(size_t)n * g.K + (size_t)wi * 8 + e] & 15u);
                word |= code << c_bitoff[e];
            }
            const int t = p >> 3, r = p & 7;
            *reinterpret_cast<uint32_t*>(out + ((size_t)t * g.ksl + j) * g.unit_bytes + (size_t)r * (W / 2) + 4 * i) =
                word;
        } else {
            const long long k2 = idx - nwords;
            const int p = int(k2 / KG), kg = int(k2 % KG);
            const int n = canon_row(p, g.N, gate_up);
            const int j = kg / G, gl = kg % G;
            const int t = p >> 3, r = p & 7;
            const uint32_t sv = n < 0 ? 0u : s[(size_t)n * KG + kg];
            const uint32_t zv = n < 0 ? 0u : z[(size_t)n * KG + kg];
            *reinterpret_cast<uint32_t*>(out + ((size_t)t * g.ksl + j) * g.unit_bytes + 4 * W + ((size_t)r * G + gl) * 4) =
                sv | (zv << 16);
        }
    }
}

__global__ void unpack_kernel(const uint8_t* __restrict__ in, PackGeom g, int gate_up, uint8_t* __restrict__ q,
                              uint16_t* __restrict__ s, uint16_t* __restrict__ z) {
    const int W = g.wks, G = W / 128, KG = g.K / 128, wpr = g.K / 8;
    const long long nwords = (long long)g.tiles * 8 * wpr;
    const long long nsz = (long long)g.tiles * 8 * KG;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < nwords + nsz;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < nwords) {
            const int p = int(idx / wpr), wi = int(idx % wpr);
            const int n = canon_row(p, g.N, gate_up);
            if (n < 0) continue;
            const int j = (wi * 8) / W, i = wi - j * (W / 8);
            const int t = p >> 3, r = p & 7;
            const uint32_t word = *reinterpret_cast<const uint32_t*>(
                in + ((size_t)t * g.ksl + j) * g.unit_bytes + (size_t)r * (W / 2) + 4 * i);
#pragma unroll
            for (int e = 0; e < 8; ++e) q[(size_t)n * g.K + (size_t)wi * 8 + e] = (word >> c_bitoff[e]) & 15u;
        } else {
            const long long k2 = idx - nwords;
            const int p = int(k2 / KG), kg = int(k2 % KG);
            const int n = canon_row(p, g.N, gate_up);
            if (n < 0) continue;
            const int j = kg / G, gl = kg % G;
            const int t = p >> 3, r = p & 7;
            const uint32_t v = *reinterpret_cast<const uint32_t*>(
                in + ((size_t)t * g.ksl + j) * g.unit_bytes + 4 * W + ((size_t)r * G + gl) * 4);
            s[(size_t)n * KG + kg] = uint16_t(v & 0xFFFFu);
            z[(size_t)n * KG + kg] = uint16_t(v >> 16);
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
    if (gate_up && N % 8 != 0) return KMR_ERR_SHAPE;
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
    if (gate_up && N % 8 != 0) return KMR_ERR_SHAPE;
    if (packed_bytes < (size_t)g.bytes) return KMR_ERR_BUFFER_SIZE;
    if (!on_device) {
        unpack_host(static_cast<const uint8_t*>(packed), g, gate_up, q, s, z);
        return KMR_OK;
    }
    unpack_kernel<<<4 * num_sms(), 256, 0, st>>>(static_cast<const uint8_t*>(packed), g, gate_up, q, s, z);
    return cudaGetLastError() == cudaSuccess ? KMR_OK : KMR_ERR_CUDA;
}

}  // namespace kmr
