// Internal description of a forward (chunked scan) problem passed from the
// host API layer to its kernel launchers.  Not part of the public ABI.
#pragma once

#include "ssd_common.h"

#if defined(__CUDACC__)
#define SSD_HD __host__ __device__
#else
#define SSD_HD
#endif

namespace ssd {

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
    // fp32 inputs on the tensor cores (ssd_tc_f32.cu): contiguous bf16 hi / lo
    // copies of x, B, C and h_prev in the workspace; only the full forward
    // provides them (f32_split), so the per-step entry points keep the
    // CUDA-core kernels for fp32
    bool f32_split = false;
    struct {
        void *x_hi, *x_lo, *b_hi, *b_lo, *c_hi, *c_lo, *hp_hi, *hp_lo;
    } f32s{};
    // filled by the launchers: the device error word, and the element extents
    // (largest index + 1) of the strided tensors, which the debug build's
    // bounds checks use
    unsigned int *err = nullptr;
    int64_t n_x = 0, n_dt = 0, n_b = 0, n_c = 0, n_y = 0;
};

// Largest element index + 1 of each strided tensor of a (innermost stride 1).
inline void fill_extents(Args &a) {
    const Dims &d = a.d;
    auto ext = [](int64_t n0, int64_t s0, int64_t n1, int64_t s1, int64_t n2, int64_t s2,
                  int64_t inner) {
        if (n0 <= 0 || n1 <= 0 || n2 <= 0) return int64_t(0);
        return (n0 - 1) * s0 + (n1 - 1) * s1 + (n2 - 1) * s2 + inner;
    };
    a.n_x = ext(d.B, a.x_sb, d.L, a.x_sl, d.H, a.x_sh, d.P);
    a.n_y = ext(d.B, a.y_sb, d.L, a.y_sl, d.H, a.y_sh, d.P);
    a.n_dt = ext(d.B, a.dt_sb, d.L, a.dt_sl, 1, 0, d.H);
    a.n_b = ext(d.B, a.b_sb, d.L, a.b_sl, d.G, a.b_sg, d.N);
    a.n_c = ext(d.B, a.c_sb, d.L, a.c_sl, d.G, a.c_sg, d.N);
}

// A copy of `in` with the device error word and the extents filled in (what
// the launchers pass to their kernels).
inline cudaError_t debug_args(const Args &in, Args *out) {
    *out = in;
    fill_extents(*out);
    return device_error_word(&out->err);
}


// y *= silu(z) in place (a.y, a.z with their strides, a.d's B, L, H, P).
cudaError_t launch_gate(const Args &a, cudaStream_t stream);

// Records the text ssd_last_error_detail() returns on this thread.
void set_error_detail(const char *fmt, ...);

// True when ssd_chunked_fwd runs the fused single-kernel path for this problem.
bool use_fused(const Dims &d, int xdt);
// Which variant the four-step path picks for chunk_state / chunk_scan.
bool uses_tc_chunk_state(const Args &a);
bool uses_tc_chunk_scan(const Args &a);
// True when the four-step forward runs fp32 inputs on the tensor cores (the
// inputs split into bf16 hi / lo copies in the workspace first).
bool f32_split_plan(const Dims &d, int xdt);
// Writes the bf16 hi / lo copies of x, B, C (a.f32s) for the fp32 tensor-core steps.
cudaError_t split_inputs_f32(const Args &a, cudaStream_t stream);

// Kernel launchers (one per step).  Each picks its kernel variant for the
// geometry and dtype, launches on `stream` and returns the launch status.
cudaError_t launch_chunk_cumsum(const Args &a, cudaStream_t stream);
cudaError_t launch_chunk_state(const Args &a, cudaStream_t stream);
cudaError_t launch_state_passing(const Args &a, cudaStream_t stream);
cudaError_t launch_chunk_scan(const Args &a, cudaStream_t stream);

}  // namespace ssd
