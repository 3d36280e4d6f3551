// Arguments of the mixer prologue's launcher (ssd_mixer_prologue).  Not part
// of the public ABI.
#pragma once

#include "ssd_common.h"

namespace ssd {

// Mixer prologue (ssd_mixer_prologue): strides in elements.  xBC [B, L, Dc]
// with Dc = H P + 2 G N; conv weight [Dc, W] f32 packed, bias [Dc] f32; conv
// state [B, Dc, W] and windows [B, L, Dc, W] packed, dtype of xBC; outputs x
// [B, L, H, P], B and C [B, L, G, N] in the dtype of xBC; dt and dt_out
// [B, L, H] f32.
struct MixerArgs {
    int B = 0, H = 0, P = 0, G = 1, N = 0, Dc = 0, W = 4;
    int64_t L = 0;
    int xdt = DT_BF16;
    int softplus = 1;
    const void *xBC = nullptr; int64_t in_sb = 0, in_sl = 0;
    const float *conv_w = nullptr;
    const float *conv_b = nullptr;            // may be null (= 0)
    void *state = nullptr;                    // may be null (zero context, not written)
    void *windows = nullptr;                  // may be null
    const int32_t *slots = nullptr;           // may be null (row b uses state b)
    int S = 0;                                // slots in the state / windows pools
    const float *dt = nullptr;  int64_t dt_sb = 0, dt_sl = 0;
    const float *dt_bias = nullptr;           // may be null (= 0)
    float *dt_out = nullptr;    int64_t do_sb = 0, do_sl = 0;
    void *x = nullptr;          int64_t x_sb = 0, x_sl = 0, x_sh = 0;
    void *Bo = nullptr;         int64_t b_sb = 0, b_sl = 0, b_sg = 0;
    void *Co = nullptr;         int64_t c_sb = 0, c_sl = 0, c_sg = 0;
};
cudaError_t launch_mixer_prologue(const MixerArgs &a, cudaStream_t stream);

}  // namespace ssd
