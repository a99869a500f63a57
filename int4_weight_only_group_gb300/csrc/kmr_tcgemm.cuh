// Prefill projections on the 5th-generation tensor cores (tcgen05): the interface between
// the launcher (kmr_tcgemm.cu) and the host code that queues a prefill (kmr_api.cu).
#pragma once

#include "kmr_internal.cuh"

namespace kmr {

// Staging of one projection's input rows for tc_gemm: row t of x (optionally through the
// RMSNorm weight, or the embedding of tokens[t]) as fp16 scaled by a per-row power of two
// sigma_t, in the tensor cores' K-major core-matrix layout, one contiguous block per
// (token tile of nt rows, 128-input group, quarter of the group):
//     half offset = ((t / nt) * (K / 128) + k / 128) * nt * 128 + ((k % 128) / 32) * nt * 32
//                   + ((t % nt) / 8) * 256 + ((k % 32) / 8) * 64 + (t % 8) * 8 + k % 8
// and rs[t] = r_t / sigma_t (r_t the RMSNorm factor, 1 without norm).  Rows t >= M up to
// the tile boundary are zero with rs = 0.
struct TcStageParams {
    int in_kind;                 // IN_F32, IN_F32_NORM or IN_EMBED_NORM
    const float* x;              // [M][K]
    const uint16_t* embed;       // bf16 [vocab][K] (IN_EMBED_NORM)
    const int32_t* tokens;
    int vocab;
    float* x_out;                // IN_EMBED_NORM: embedded rows [M][K] (or null)
    const uint16_t* norm_w;      // bf16 [K] (IN_*_NORM)
    float eps;
    int M, K, nt;
    uint16_t* xs;                // fp16, ceil(M / nt) * nt * K halves
    float* rs;                   // [ceil(M / nt) * nt]
    int* err;
};

// y[t][n] (+)= rs[t] * sum_k w[n][k] * xs[t][k] for packed weight rows n (N a multiple of 128)
// and token rows t < M: STORE, RESID or SILU (gate / up packing, y[t][j] = silu(g) * u).
struct TcGemmParams {
    const uint8_t* w;            // packed KMR4
    int N, K;
    const uint16_t* xs;
    const float* rs;
    int M, nt, epi;
    int ksplit;                  // CTAs along K (a thread-block cluster): 1, 2 or 4, <= K / 128
    float* y;
    int ldy;
    int* err;
};

struct TcPlan {
    int nt;                      // tokens per CTA: 64, 128 or 256
    int ksplit;
};

bool tc_gemm_supported(int N, int K);
// Staged rows to allocate for M tokens (every tile width's padding).
int tc_rows_pad(int M);
TcPlan tc_gemm_plan(int N, int K, int M, int sms);
cudaError_t tc_gemm_set_attributes();
cudaError_t launch_tc_stage(const TcStageParams& p, cudaStream_t st);
cudaError_t launch_tc_gemm(const TcGemmParams& p, cudaStream_t st);

}  // namespace kmr
