// kla_selftest.cu -- exercises the bounded-wait failure path without a GPU fault.
//
// Every wait of the library's kernels on an mbarrier is bounded: after its poll limit the wait
// gives up, the kernel records kErrTimeout in the device error word, skips its remaining work
// and exits cleanly, so the context stays usable and kla_device_status reports
// KLA_ERR_TIMEOUT. This kernel runs that path on purpose: one thread waits, with the same
// bounded wait, on a barrier phase that nothing completes.
#include "kla_internal.cuh"
#include "sm103_ptx.cuh"

namespace {

__global__ void selftest_wait_kernel(unsigned *err, uint32_t limit) {
    __shared__ uint64_t bar;
    const uint32_t b = kla::ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        kla::ptx::mbar_init(b, 1);
        kla::ptx::fence_mbar_init();
    }
    __syncthreads();
    // a freshly initialised barrier sits in phase 0 and nobody arrives: the wait must give up
    if (threadIdx.x == 0 && !kla::ptx::mbar_wait_bounded(b, 0, limit)) atomicOr(err, kla::kErrTimeout);
}

}  // namespace

namespace kla {

cudaError_t launch_selftest_wait(unsigned *err, unsigned limit, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit);
    return cudaGetLastError();
}

}  // namespace kla
