// Arguments of the decode step's launcher (ssd_state_update,
// ssd_state_update_tokens).  Not part of the public ABI.
#pragma once

#include "ssd_common.h"

namespace ssd {

// T decode steps per sequence (ssd_state_update_tokens; ssd_state_update is
// T = 1): strides in elements; state is packed [B, H, P, N] (f32 or bf16); x, z, out
// [B, T, H, P]; dt [B, T, H]; B, C [B, T, G, N]; intermediate states packed
// [B, T, H, P, N]; parent [B, T] int32.  With slots the state and the
// intermediate states are pools of S slots.
struct SsuArgs {
    int B = 0, T = 1, H = 0, P = 0, N = 0, G = 1;
    int xdt = DT_BF16;                        // dtype of x, B, C, z, out
    int softplus = 0;
    int update = 1;                           // write the final state back
    int sdt = DT_F32;                         // dtype of state and inter
    void *state = nullptr;
    const void *x = nullptr;   int64_t x_sb = 0, x_st = 0, x_sh = 0;
    const float *dt = nullptr; int64_t dt_sb = 0, dt_st = 0;
    const float *A = nullptr;
    const float *D = nullptr;                 // may be null (= 0)
    const float *dt_bias = nullptr;           // may be null (= 0)
    const void *Bm = nullptr;
    const void *Cm = nullptr;  int64_t bc_sb = 0, bc_st = 0, bc_sg = 0;   // B, C share strides
    const void *z = nullptr;   int64_t z_sb = 0, z_st = 0, z_sh = 0;     // may be null
    void *out = nullptr;       int64_t o_sb = 0, o_st = 0, o_sh = 0;
    void *inter = nullptr;                    // may be null (not cached)
    const int32_t *parent = nullptr;          // may be null (a chain)
    int64_t par_sb = 0;
    const int32_t *slots = nullptr;           // may be null (row b uses state b)
    int S = 0;                                // slots in the state pool
};
cudaError_t launch_ssu(const SsuArgs &a, cudaStream_t stream);

}  // namespace ssd
