// Internal problem description passed from the host API layer to the kernel
// launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define SSD_HD __host__ __device__
#else
#define SSD_HD
#endif

namespace ssd {

enum : int { DT_F32 = 0, DT_BF16 = 1 };

struct Dims {
    int64_t B, L, H, P, N, G, Q, nc;
    SSD_HD int64_t hpg() const { return H / G; }    // heads per group
    SSD_HD int64_t Lp() const { return nc * Q; }    // zero-padded sequence length
};

// Every pointer is a device pointer.  Strides are in elements; the innermost
// stride of every tensor is 1.  G, S, h_prev, h0 and final are contiguous.
struct Args {
    Dims d{};
    int xdt = DT_BF16;                        // dtype of x, B, C, y
    const void *x = nullptr;   int64_t x_sb = 0, x_sl = 0, x_sh = 0;
    const float *dt = nullptr; int64_t dt_sb = 0, dt_sl = 0;
    const float *A = nullptr;
    const float *D = nullptr;                 // may be null (= 0)
    const void *Bm = nullptr;  int64_t b_sb = 0, b_sl = 0, b_sg = 0;
    const void *Cm = nullptr;  int64_t c_sb = 0, c_sl = 0, c_sg = 0;
    const float *h0 = nullptr;                // may be null (= 0)
    void *y = nullptr;         int64_t y_sb = 0, y_sl = 0, y_sh = 0;
    float *final_states = nullptr;            // may be null (skip)
    float *G = nullptr;                       // [B, H, nc*Q]
    float *S = nullptr;                       // [B, nc, H, P, N]
    void *h_prev = nullptr;                   // [B, nc, H, P, N]
    int hprev_dt = DT_F32;
    char *ws = nullptr;                       // workspace base (fused path's tail split)
    const void *z = nullptr;   int64_t z_sb = 0, z_sl = 0, z_sh = 0;   // output gate, or null
};

// T decode steps per sequence (ssd_state_update_tokens; ssd_state_update is
// T = 1): strides in elements; state is packed [B, H, P, N] f32; x, z, out
// [B, T, H, P]; dt [B, T, H]; B, C [B, T, G, N]; intermediate states packed
// [B, T, H, P, N] f32; parent [B, T] int32.
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
// One CTA whose wait on an mbarrier nobody arrives at gives up after limit_ns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
// y *= silu(z) in place (a.y, a.z with their strides, a.d's B, L, H, P).
cudaError_t launch_gate(const Args &a, cudaStream_t stream);

// Records the text ssd_last_error_detail() returns on this thread.
void set_error_detail(const char *fmt, ...);

// True when ssd_chunked_fwd runs the fused single-kernel path for this problem.
bool use_fused(const Dims &d, int xdt);
// Which variant the four-step path picks for chunk_state / chunk_scan.
bool uses_tc_chunk_state(const Args &a);
bool uses_tc_chunk_scan(const Args &a);

// Kernel launchers (one per step).  Each picks its kernel variant for the
// geometry and dtype, launches on `stream` and returns the launch status.
cudaError_t launch_chunk_cumsum(const Args &a, cudaStream_t stream);
cudaError_t launch_chunk_state(const Args &a, cudaStream_t stream);
cudaError_t launch_state_passing(const Args &a, cudaStream_t stream);
cudaError_t launch_chunk_scan(const Args &a, cudaStream_t stream);

}  // namespace ssd
