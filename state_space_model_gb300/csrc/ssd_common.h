// What every kernel file shares: the dtype codes of the argument structs, the
// device error word that bounded waits set, and the bounded-wait test hook.
// Not part of the public ABI.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

namespace ssd {

enum : int { DT_F32 = 0, DT_BF16 = 1 };

// Device address of the per-device error word that bounded waits set.
cudaError_t device_error_word(unsigned int **out);

// One CTA whose wait on an mbarrier nobody arrives at gives up after limit_ns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

}  // namespace ssd
