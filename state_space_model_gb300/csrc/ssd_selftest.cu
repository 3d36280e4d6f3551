// A check of the bounded-wait path every kernel of this library uses: one
// thread waits, with a short limit, on an mbarrier phase nothing completes;
// the wait gives up, the kernel records the timeout in the device error word
// and returns, and the host reads it through ssd_device_status.  Nothing is
// in flight when it gives up (no copy, no tensor-core work), so the context
// stays usable.
//
// And a check of the debug build's bounds-check reporting: one thread tests
// an index that is out of range by construction (no memory is touched: the
// check only records the failure and the access it guards is skipped).
#include "ptx_sm100.cuh"
#include "ssd_common.h"
#define SSD_DBG_FILE 5u   // kDbgSelftest
#include "ssd_debug.cuh"

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

__global__ void k_bounds_selftest(unsigned int *err, float *sink) {
    if (threadIdx.x != 0) return;
    const int64_t n = 3, i = 5;   // i is not inside [0, n)
    if (SSD_IDX_OK(err, i, n)) sink[0] = 1.f;   // skipped: never reached
}

}  // namespace

bool bounds_checks_built() {
#ifdef SSD_DEBUG_BOUNDS
    return true;
#else
    return false;
#endif
}

cudaError_t launch_bounds_selftest(cudaStream_t s) {
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    k_bounds_selftest<<<1, 32, 0, s>>>(err, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    k_wait_selftest<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace ssd
