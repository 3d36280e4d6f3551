// Host helpers: TMA tensor maps (bf16, 128-byte swizzle, zero fill out of
// bounds) and the per-device error word bounded waits report into.
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

namespace ssd {
// dims and box innermost first; strides in bytes for dims 1..rank-1.
cudaError_t make_tmap_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                           const uint64_t *strides, const uint32_t *box);
}  // namespace ssd
