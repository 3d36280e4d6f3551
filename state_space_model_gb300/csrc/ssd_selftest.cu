// A check of the bounded-wait path every kernel of this library uses: one
// thread waits, with a short limit, on an mbarrier phase nothing completes;
// the wait gives up, the kernel records the timeout in the device error word
// and returns, and the host reads it through ssd_device_status.  Nothing is
// in flight when it gives up (no copy, no tensor-core work), so the context
// stays usable.
#include "ptx_sm100.cuh"
#include "ssd_common.h"

#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr unsigned kErrTimeout = 1u;   // the bit the other kernels set

__global__ void k_wait_selftest(unsigned int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    // phase 0 needs one arrival and gets none
    if (!ptx::mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    k_wait_selftest<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace ssd
