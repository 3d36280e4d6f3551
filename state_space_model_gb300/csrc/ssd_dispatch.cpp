// Picks the kernel variant of each step for the problem's dtype and geometry:
// the tensor-core kernels for bf16 inputs with P = 64, N = 128 (and Q of 128
// or 256 for chunk_scan) and, in the full forward, for fp32 inputs with
// P = 64, N = 128, Q of 128 or 256 (as bf16 hi / lo pairs); the CUDA-core
// kernels for everything else.
#include "ssd_internal.h"
#include "ssd_simt.cuh"
#include "ssd_tc.cuh"

#include <cstdlib>

namespace ssd {
namespace {
// SSD_FORCE_SIMT=1 selects the CUDA-core variants for every shape (for
// comparisons only; read once per process).
bool force_simt() {
    static const bool v = [] {
        const char *e = std::getenv("SSD_FORCE_SIMT");
        return e && e[0] == '1';
    }();
    return v;
}
}  // namespace

// SSD_FORCE_STAGED=1 makes ssd_chunked_fwd run the four separate steps even
// where the fused kernel applies (for comparisons only).
bool use_fused(const Dims &d, int xdt) {
    static const bool staged = [] {
        const char *e = std::getenv("SSD_FORCE_STAGED");
        return e && e[0] == '1';
    }();
    // an empty sequence has nothing to tile (a TMA map cannot have a zero
    // extent); the four-step path then just copies the initial state
    return !staged && !force_simt() && d.L > 0 && fused_supported(d, xdt);
}

bool uses_tc_chunk_state(const Args &a) { return !force_simt() && tc_chunk_state_supported(a); }
bool f32_split_plan(const Dims &d, int xdt) { return !force_simt() && tc_f32_supported(d, xdt); }
bool uses_tc_chunk_scan(const Args &a) { return !force_simt() && tc_chunk_scan_supported(a); }

cudaError_t launch_chunk_cumsum(const Args &a, cudaStream_t s) { return simt_chunk_cumsum(a, s); }

cudaError_t launch_chunk_state(const Args &a, cudaStream_t s) {
    if (!force_simt() && tc_chunk_state_supported(a)) return tc_chunk_state(a, s);
    return simt_chunk_state(a, s);
}

cudaError_t launch_state_passing(const Args &a, cudaStream_t s) {
    return simt_state_passing(a, s);
}

cudaError_t launch_chunk_scan(const Args &a, cudaStream_t s) {
    if (!force_simt() && tc_chunk_scan_supported(a)) return tc_chunk_scan(a, s);
    return simt_chunk_scan(a, s);
}

}  // namespace ssd
