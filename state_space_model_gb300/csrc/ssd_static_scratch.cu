// ssd_chunked_fwd_static_scratch: the SSD forward for callers that cannot
// supply device workspace.  Some callers have no allocator they may use: a
// plug-in living inside a host program that owns every byte of device memory
// and offers no workspace hook, or a fixed-latency loop that cannot afford
// cudaMalloc (which may synchronise the device and takes unbounded time).
// This entry point takes its scratch from one file-scope device array
// instead and allocates nothing.
//
// The array's name, used in host code, is only a host-side stand-in for the
// device symbol, not a device address (a kernel handed it would fault, or on
// systems where the GPU can reach host memory, silently use the wrong bytes).
// The device address is therefore looked up with cudaGetSymbolAddress, once
// per device with that device current, and cached.
#include "ssd.h"
#include "ssd_internal.h"

#include <cuda_runtime.h>

#include <mutex>

#include "ssd_tc.cuh"

// the fused path's split never needs more than the static array holds
static_assert(ssd::kSplitWsMax <= SSD_STATIC_SCRATCH_BYTES, "static scratch below the split cap");

namespace {

// Shared by every call on a device; every GPU that loads this library holds
// it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[SSD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up on the
// first call per device).  Returns the CUDA error on failure.
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status ssd_chunked_fwd_static_scratch(
    const ssd_tensor *x, const ssd_tensor *dt, const ssd_tensor *A, const ssd_tensor *Bm,
    const ssd_tensor *Cm, const ssd_tensor *D, const ssd_tensor *initial_states,
    int64_t chunk_size, int64_t ngroups, ssd_tensor *y, ssd_tensor *final_states,
    void *stream) {
    if (!x || !Bm || x->ndim != 4 || Bm->ndim != 4) {
        // let the full argument checks name the problem
        return ssd_chunked_fwd(x, dt, A, Bm, Cm, D, initial_states, chunk_size, ngroups, y,
                               final_states, nullptr, 0, stream);
    }
    size_t need = 0;
    ssd_status st = ssd_workspace_size(x->shape[0], x->shape[1], x->shape[2], x->shape[3],
                                       Bm->shape[3], ngroups, chunk_size, x->dtype, &need);
    if (st != SSD_OK) return st;
    if (need > SSD_STATIC_SCRATCH_BYTES) {
        ssd::set_error_detail(
            "problem needs %zu bytes of scratch; the static scratch holds %zu bytes "
            "(SSD_STATIC_SCRATCH_BYTES); use ssd_chunked_fwd with a caller workspace",
            need, (size_t)SSD_STATIC_SCRATCH_BYTES);
        return SSD_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        ssd::set_error_detail("static scratch set-up (cudaGetSymbolAddress): %s",
                              cudaGetErrorString(e));
        return SSD_ERR_CUDA;
    }
    return ssd_chunked_fwd(x, dt, A, Bm, Cm, D, initial_states, chunk_size, ngroups, y,
                           final_states, scratch, SSD_STATIC_SCRATCH_BYTES, stream);
}
