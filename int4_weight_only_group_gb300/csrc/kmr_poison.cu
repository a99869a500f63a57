// Shared-memory poisoning: a diagnostic that fills the shared memory of every
// SM with a caller-chosen 32-bit pattern.  A kernel that reads shared memory
// it did not write in the same launch then sees the pattern (NaN or Inf bits,
// say) instead of whatever an earlier kernel happened to leave there, so a
// test that compares a poisoned run with a clean one bitwise turns such a
// read into a deterministic failure.  Nothing on the decode path depends on
// it; the model enables it with kmr_model_set_smem_poison.
#include "kmr_internal.cuh"

namespace kmr {

namespace {

constexpr int kPoisonThreads = 1024;
constexpr size_t kPoisonBytes = 227 * 1024;   // the whole opt-in shared memory of one CTA

__global__ void __launch_bounds__(kPoisonThreads, 1) poison_kernel(uint32_t pattern) {
    extern __shared__ __align__(16) uint32_t buf[];
    constexpr int words = int(kPoisonBytes / 4);
    // asm stores: nothing reads the buffer in this kernel, so plain stores could be dropped
    const uint32_t base = smem_u32(buf);
    for (int i = threadIdx.x; i < words / 4; i += kPoisonThreads)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + uint32_t(i) * 16u), "r"(pattern)
                     : "memory");
    __syncthreads();
}

}  // namespace

cudaError_t poison_set_attributes() {
    return cudaFuncSetAttribute(poison_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPoisonBytes));
}

// One CTA per SM, each holding the SM's whole shared memory, so every SM is
// covered once the kernel completes.
cudaError_t launch_smem_poison(uint32_t pattern, int sms, cudaStream_t st) {
    poison_kernel<<<sms > 0 ? sms : 1, kPoisonThreads, kPoisonBytes, st>>>(pattern);
    return cudaGetLastError();
}

}  // namespace kmr
