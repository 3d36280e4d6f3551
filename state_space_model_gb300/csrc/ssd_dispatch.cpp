// Picks the kernel variant of each step for the problem's dtype and geometry.
#include "ssd_internal.h"
#include "ssd_simt.cuh"

namespace ssd {

cudaError_t launch_chunk_cumsum(const Args &a, cudaStream_t s) { return simt_chunk_cumsum(a, s); }
cudaError_t launch_chunk_state(const Args &a, cudaStream_t s) { return simt_chunk_state(a, s); }
cudaError_t launch_state_passing(const Args &a, cudaStream_t s) {
    return simt_state_passing(a, s);
}
cudaError_t launch_chunk_scan(const Args &a, cudaStream_t s) { return simt_chunk_scan(a, s); }

}  // namespace ssd
