// Shared-memory poisoning: a diagnostic that fills the shared memory of every
// SM with a caller-chosen 32-bit pattern.  A kernel that reads shared memory
// it did not write in the same launch then sees the pattern (NaN or Inf bits,
// say) instead of whatever an earlier kernel happened to leave there, so a
// test that compares a poisoned run with a clean one bitwise turns such a
// read into a deterministic failure.  Nothing on the decode path depends on
// it; the model enables it with kmr_model_set_smem_poison.
//
// Also here: a self-test of the bounded device waits, which waits on an
// mbarrier that nothing completes and must give up with a status, not hang.
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

// One warp waits on a freshly initialised mbarrier that expects one arrival which never
// comes (no copy is in flight, so nothing is left pending when the kernel exits).  Every
// lane's bounded wait gives up after limit_ns and records KMR_ERR_DEVICE_TIMEOUT.
__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    mbar_wait(&bar, 0u, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout(int* err, unsigned long long limit_ns, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

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
