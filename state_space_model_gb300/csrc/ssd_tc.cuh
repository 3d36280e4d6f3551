// Tensor-core (tcgen05 + TMA) variants of the steps (see ssd_tc.cu).
#pragma once
#include "ssd_internal.h"

namespace ssd {
// Device address of the per-device error word that bounded waits set.
cudaError_t device_error_word(unsigned int **out);

bool tc_chunk_state_supported(const Args &a);
cudaError_t tc_chunk_state(const Args &a, cudaStream_t s);
bool tc_chunk_scan_supported(const Args &a);
cudaError_t tc_chunk_scan(const Args &a, cudaStream_t s);
}  // namespace ssd

namespace ssd {
// The fused single-kernel forward (ssd_fused.cu): bf16, P = 64, N = 128,
// Q a multiple of 128.  Needs no workspace.
bool fused_supported(const Dims &d, int xdt);
cudaError_t launch_fused(const Args &a, cudaStream_t s);
}  // namespace ssd
