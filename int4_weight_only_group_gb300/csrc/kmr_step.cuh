// Parameter blocks of the persistent decode-step kernel (kmr_step.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kmr {

constexpr int kStepMaxRows = 4;          // rows the persistent step serves (one staging pass)

// One decoder layer's device pointers.
struct StepLayer {
    const uint8_t* w[4];                 // packed QKV, O, gate_up, down (KMR4)
    const uint16_t* norm[4];             // bf16 input, post-attention, q, k RMSNorm weights
    uint16_t* kc;                        // this layer's K cache [slots][nkv][S][d]
    uint16_t* vc;
};

struct StepParams {
    const StepLayer* layers;             // [L] in device memory
    int L, H, nq, nkv, I, vocab, S, slots, B;
    float eps, scale;
    int qk_norm;
    const uint16_t* embed;               // bf16 [vocab][H]
    const float* inv_freq;               // [d/2]
    int sec0, sec1;
    // step state (from the previous step; the LM head advances it)
    const int32_t* tok;
    const int32_t* pos;                  // [3][B]
    const int32_t* cpos;
    const int32_t* slot;
    const uint8_t* fin;
    // model scratch
    float* x;                            // residual [B][H]
    float* qkv;                          // [B][(nq + 2 nkv) d]
    float* attn;                         // [B][nq d]
    float* act;                          // [B][I]
    float* part;                         // split states [B][nkv][8][rep][d + 2]
    unsigned* phase_cnt;                 // [L][5], zero between steps
    unsigned* merge_cnt;                 // [B][nkv], zero between layers
    unsigned* done_cnt;                  // zero between steps
    unsigned* abort_flag;                // zero between steps
    int* err;
    // launch plan
    int nslots, slot_bytes, gpw_max, max_tiles;
};

struct StepPlan {
    int MB, ch, rep, gpw_max, max_tiles, nslots, slot_bytes, grid;
    size_t smem;
};

// Whether the persistent step serves this shape (B rows, model dimensions, SM count), and its
// launch plan.
bool step_supported(int B, int n_layers, int hidden, int nq, int nkv, int d, int inter, int max_len, int sms,
                    StepPlan* plan);
cudaError_t step_set_attributes();
cudaError_t launch_step(const StepParams& p, const StepPlan& plan, int d, cudaStream_t st);
int step_max_active_ctas(const StepPlan& plan, int d);

}  // namespace kmr
