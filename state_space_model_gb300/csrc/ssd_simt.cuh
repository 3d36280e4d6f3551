// CUDA-core variants of the four steps (see ssd_simt.cu).
#pragma once
#include "ssd_internal.h"

namespace ssd {
cudaError_t simt_chunk_cumsum(const Args &a, cudaStream_t s);
cudaError_t simt_chunk_state(const Args &a, cudaStream_t s);
cudaError_t simt_state_passing(const Args &a, cudaStream_t s);
cudaError_t simt_chunk_scan(const Args &a, cudaStream_t s);
}  // namespace ssd
