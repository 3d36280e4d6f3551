// Device-side bounds checks of the debug build.
//
// Built with -DSSD_DEBUG_BOUNDS (python -m state_space_model_gb300.build
// --debug-bounds, which writes libssd_gb300_debug.so), every global-memory
// index, shared-memory offset and tensor-memory column range that a kernel
// computes itself is checked before use.  A failed check does not trap: it
// sets kErrBounds in the device error word (word 0), records the file and line
// of the first failure in word 1, and the access is skipped, so the kernel
// runs to its end (or a bounded wait gives up) and the host reads the report
// through ssd_device_status.  TMA copies are bounds-checked by the hardware
// (out-of-range boxes are filled or clipped); their shared-memory destinations
// are checked here.  In the normal build the checks compile to `true`.
#pragma once

#include <stdint.h>

namespace ssd {

constexpr unsigned kErrBounds = 4u;   // a debug-build bounds check failed

// File codes of the kernels' translation units (word 1 holds code << 16 | line).
enum : unsigned {
    kDbgFused = 1, kDbgPair = 2, kDbgTc = 3, kDbgSimt = 4, kDbgSelftest = 5, kDbgTcF32 = 6,
};

#ifdef SSD_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(unsigned int *err, bool ok, unsigned file,
                                          unsigned line) {
    if (!ok && err) {
        atomicOr(err, kErrBounds);
        atomicCAS(err + 1, 0u, (file << 16) | (line & 0xffffu));
    }
    return ok;
}
#define SSD_IN_BOUNDS(err, cond) ::ssd::bounds_ok((err), (cond), SSD_DBG_FILE, __LINE__)
#else
#define SSD_IN_BOUNDS(err, cond) true
#endif

// Index i is inside [0, n).
#define SSD_IDX_OK(err, i, n) SSD_IN_BOUNDS((err), (int64_t)(i) >= 0 && (int64_t)(i) < (int64_t)(n))
// The len elements from ptr lie inside the n elements from base.
#define SSD_SPAN_OK(err, ptr, base, n, len) \
    SSD_IN_BOUNDS((err), (ptr) >= (base) && (int64_t)((ptr) - (base)) + (int64_t)(len) <= (int64_t)(n))

}  // namespace ssd
