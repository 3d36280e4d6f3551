// Tensor-core (tcgen05 + TMA) variants of the steps (see ssd_tc.cu).
#pragma once
#include "ssd_internal.h"

namespace ssd {

bool tc_chunk_state_supported(const Args &a);
cudaError_t tc_chunk_state(const Args &a, cudaStream_t s);
bool tc_chunk_scan_supported(const Args &a);
cudaError_t tc_chunk_scan(const Args &a, cudaStream_t s);
// fp32 inputs as bf16 hi / lo pairs, three products each (ssd_tc_f32.cu):
// P = 64, N = 128, Q of 128 or 256, with the split copies in a.f32s.
bool tc_f32_supported(const Dims &d, int xdt);
cudaError_t tc_chunk_state_f32(const Args &a, cudaStream_t s);
cudaError_t tc_chunk_scan_f32(const Args &a, cudaStream_t s);
}  // namespace ssd

namespace ssd {
// The fused single-kernel forward (ssd_fused.cu): bf16, P = 64, N = 128,
// Q a multiple of 128.  Needs workspace only when it splits the last wave of
// slabs by sequence (at most kSplitWsMax bytes).
bool fused_supported(const Dims &d, int xdt);
// How the fused path splits the last partial wave of slabs by sequence, and
// the workspace that needs (ws_bytes = 0 when nothing is split).
struct FusedSplit {
    int64_t n_whole = 0, tail = 0, seg_len = 0;
    int nseg = 1;
    size_t ws_bytes = 0, off_state = 0, off_decay = 0, off_hin = 0;
};
constexpr size_t kSplitWsMax = size_t(64) << 20;
FusedSplit fused_split(const Dims &d, int sm_count);
int device_sm_count();   // of the current device; 152 when there is none
cudaError_t launch_fused(const Args &a, cudaStream_t s);

// The pair kernel (ssd_pair.cu): the fused forward over two heads of one group
// per CTA; taken when H and the heads per group are even and there are at
// least as many pair slabs as SMs.  Splits the pair slabs left over after the
// last full wave by sequence, with the same workspace record.
bool pair_supported(const Dims &d, int xdt);
FusedSplit pair_split(const Dims &d, int sm_count);
cudaError_t launch_pair(const Args &a, cudaStream_t s);
}  // namespace ssd
