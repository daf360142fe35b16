// selftest_wait.cu -- the bounded-wait failure path, exercised on purpose.
//
// Every wait inside the step kernels is bounded: a wait that runs out sets
// LUCETREE_DEV_TIMEOUT in the caller's status word and the kernel returns, so
// the context stays usable and the host learns of it from the status.  This
// kernel makes such a wait run out: one mbarrier that nothing ever arrives on,
// waited on by four warps with the same helper and the same barrier-OR
// consensus the step kernels use, with a caller-chosen cycle limit.
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace lucetree {

namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) wait_timeout_kernel(uint32_t* status, long long limit_cycles,
                                                                long long* waited_cycles) {
    __shared__ alignas(8) uint64_t never;  // no thread and no copy ever arrives here
    if (threadIdx.x == 0) {
        tc::mbar_init(&never, 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    const long long t0 = clock64();
    const bool landed = tc::mbar_wait(&never, 0, limit_cycles);  // phase 0 never completes
    const bool gave_up = tc::bar_sync_or(1, kThreads, !landed);
    if (threadIdx.x == 0) {
        if (gave_up) atomicOr(status, LUCETREE_DEV_TIMEOUT);
        if (waited_cycles) *waited_cycles = clock64() - t0;
    }
}

}  // namespace

}  // namespace lucetree

extern "C" lucetree_status lucetree_selftest_wait_timeout(uint32_t* status, long long limit_cycles,
                                                          long long* waited_cycles, void* stream) {
    if (!status) return LUCETREE_ERR_INVALID_ARG;
    if (limit_cycles < 1 || limit_cycles > 4000000000ll) return LUCETREE_ERR_INVALID_ARG;
    lucetree::wait_timeout_kernel<<<1, lucetree::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        status, limit_cycles, waited_cycles);
    return cudaGetLastError() == cudaSuccess ? LUCETREE_OK : LUCETREE_ERR_CUDA;
}
