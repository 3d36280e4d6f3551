// What every kernel file shares: the dtype codes of the argument structs, the
// device error word that bounded waits set, and the bounded-wait test hook.
// Not part of the public ABI.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

namespace ssd {

enum : int { DT_F32 = 0, DT_BF16 = 1 };

// Device address of the per-device error words: word 0 holds the flags that
// bounded waits (and the debug build's bounds checks) set, word 1 the file and
// line of the first failed bounds check.
cudaError_t device_error_word(unsigned int **out);

// One CTA whose wait on an mbarrier nobody arrives at gives up after limit_ns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

// True in the debug build (SSD_DEBUG_BOUNDS); there, one thread records a
// bounds check that fails by construction (the guarded access is skipped).
bool bounds_checks_built();
cudaError_t launch_bounds_selftest(cudaStream_t stream);

}  // namespace ssd
