// Mixer prologue: the causal depthwise convolution + SiLU that turns the
// in-projection's xBC channels into the x, B and C the scan reads, and the dt
// preparation (dt + dt_bias, softplus) -- "Optimizing Nemotron v3 Super in
// TensorRT-LLM", sections 6.2, 7.1 (the split into contiguous x / B / C done
// by the same kernel), 8 ("CausalConv1d Optimization") and 10.5 (the conv
// state and its per-token windows for speculative decoding).
//
//   out[b, t, c] = silu(bias[c] + sum_k weight[c, k] u[b, t - (W - 1) + k, c])
//
// with u the inputs preceded by the conv state (the last W inputs of the
// sequence so far, oldest first; zeros when absent).  Channels [0, H P) go to
// x [B, L, H, P], the next G N to B [B, L, G, N], the last G N to C.
//
// One pass over HBM: each thread owns one 8-byte vector of channels and walks
// a run of tokens, kUnroll token vectors in flight at a time, keeping the last
// W inputs of its channels in registers, so every input is read once (plus a
// W - 1 token halo per run) and every output written once, with coalesced
// streaming accesses along the channel axis.  The run length makes the grid
// one wave of resident CTAs.  No tensor cores: the work is a W-tap filter per
// channel.
#include "ssd_mixer.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr int kConvMaxThreads = 256;
constexpr int kUnroll = 10;   // token vectors loaded before any is used

template <typename T>
struct Vec;   // one 8-byte vector of channels (few registers per thread, so
              // many token vectors can be in flight per SM)
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int kN = 4;
    __device__ static uint2 raw(const __nv_bfloat16 *p) {   // read once: streaming
        return __ldcs(reinterpret_cast<const uint2 *>(p));
    }
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[4]) { unpack(raw(p), v); }
    __device__ static void unpack(const uint2 u, float (&v)[4]) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        v[0] = lo.x;
        v[1] = lo.y;
        v[2] = hi.x;
        v[3] = hi.y;
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&v)[4]) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                                                       *reinterpret_cast<const uint32_t *>(&hi)));
    }
};
template <>
struct Vec<float> {
    static constexpr int kN = 2;
    __device__ static uint2 raw(const float *p) { return __ldcs(reinterpret_cast<const uint2 *>(p)); }
    __device__ static void load(const float *p, float (&v)[2]) { unpack(raw(p), v); }
    __device__ static void unpack(const uint2 r, float (&v)[2]) {
        v[0] = __uint_as_float(r.x);
        v[1] = __uint_as_float(r.y);
    }
    __device__ static void store(float *p, const float (&v)[2]) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(v[0], v[1]));
    }
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Where channel vector c0 goes (x, B or C): the address at token 0 of batch
// b, and the token stride.
template <typename T>
__device__ __forceinline__ T *dest(const MixerArgs &a, int b, int c0, int64_t &sl) {
    const int hp = a.H * a.P, gn = a.G * a.N;
    if (c0 < hp) {
        sl = a.x_sl;
        return static_cast<T *>(a.x) + int64_t(b) * a.x_sb + int64_t(c0 / a.P) * a.x_sh + c0 % a.P;
    }
    if (c0 < hp + gn) {
        const int c = c0 - hp;
        sl = a.b_sl;
        return static_cast<T *>(a.Bo) + int64_t(b) * a.b_sb + int64_t(c / a.N) * a.b_sg + c % a.N;
    }
    const int c = c0 - hp - gn;
    sl = a.c_sl;
    return static_cast<T *>(a.Co) + int64_t(b) * a.c_sb + int64_t(c / a.N) * a.c_sg + c % a.N;
}

// grid (ceil(Dc / (V blockDim.x)), ceil(L / run), B).  Thread i of CTA
// (bx, r, b) owns channels [V (bx blockDim.x + i), + V) of tokens
// [r run, + run), kUnroll token vectors in flight at a time.  The CTAs of a
// run also share the dt preparation of its tokens, an equal slice each.  The conv state is written here only when one
// run covers the sequence (gridDim.y = 1), so the thread that read a state
// entry is the one that overwrites it.  With slot indices row b's conv state
// and windows are slot slots[b] of their pools, and a row whose slot is outside
// the pool is padding: nothing is read or written for it.
template <typename T, int W, bool kWindows>
__device__ __forceinline__ void conv_prologue(const MixerArgs &a, int64_t run) {
    constexpr int V = Vec<T>::kN;
    const int b = blockIdx.z;
    int64_t slot = b;
    if (a.slots) {
        slot = a.slots[b];
        if (slot < 0 || slot >= a.S) return;
    }
    const int64_t t0 = int64_t(blockIdx.y) * run;
    const int64_t t1 = t0 + run < a.L ? t0 + run : a.L;
    const bool write_state = gridDim.y == 1;

    {   // dt' = dt + dt_bias, softplus: this CTA's slice of the run's (token, head) pairs
        const int n = int(t1 - t0) * a.H;
        const int per = (n + gridDim.x - 1) / gridDim.x;
        const int lo = blockIdx.x * per, hi = lo + per < n ? lo + per : n;
        for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
            const int64_t t = t0 + i / a.H;
            const int h = i % a.H;
            float d = a.dt[int64_t(b) * a.dt_sb + t * a.dt_sl + h];
            if (a.dt_bias) d += a.dt_bias[h];
            if (a.softplus) d = d <= 20.f ? log1pf(expf(d)) : d;   // = d to fp32 above 20
            a.dt_out[int64_t(b) * a.do_sb + t * a.do_sl + h] = d;
        }
    }
    const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (c0 >= a.Dc) return;

    float w[W][V], bias[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        bias[j] = a.conv_b ? a.conv_b[c0 + j] : 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) w[k][j] = a.conv_w[int64_t(c0 + j) * W + k];
    }
    const T *xin = static_cast<const T *>(a.xBC) + int64_t(b) * a.in_sb + c0;
    T *state = a.state ? static_cast<T *>(a.state) + (slot * a.Dc + c0) * W : nullptr;

    // win[k] = input t - (W - 1) + k for the token t about to be computed;
    // win[W - 1] is filled from token t itself
    float win[W][V];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
        const int64_t tau = t0 - (W - 1) + k;
        if (tau >= 0) {
            Vec<T>::load(xin + tau * a.in_sl, win[k]);
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j)   // state column W + tau of channel c0 + j
                win[k][j] = state ? to_f(state[int64_t(j) * W + (W + tau)]) : 0.f;
        }
    }
    int64_t dsl;
    T *dst = dest<T>(a, b, c0, dsl);
    // one token: filter, silu, store; then slide the window
    auto step = [&](const uint2 r, int64_t t) {
        Vec<T>::unpack(r, win[W - 1]);
        float o[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            float acc = bias[j];
#pragma unroll
            for (int k = 0; k < W; ++k) acc = fmaf(w[k][j], win[k][j], acc);
            // silu with the fast exponential and division: a few instructions
            // instead of the ~20 of expf and an IEEE divide, ~2 ulp (the
            // filter is otherwise issue-bound); for acc far below zero the
            // denominator overflows and the quotient is 0, silu's limit
            o[j] = __fdividef(acc, 1.f + __expf(-acc));
        }
        Vec<T>::store(dst + t * dsl, o);
        if constexpr (kWindows) {   // the state after token t: its last W inputs
            T *wp = static_cast<T *>(a.windows) + ((slot * a.L + t) * a.Dc + c0) * W;
#pragma unroll
            for (int j = 0; j < V; ++j)
#pragma unroll
                for (int k = 0; k < W; ++k) wp[j * W + k] = from_f<T>(win[k][j]);
        }
#pragma unroll
        for (int k = 0; k + 1 < W; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j) win[k][j] = win[k + 1][j];
    };
    int64_t t = t0;
    for (; t + kUnroll <= t1; t += kUnroll) {
        uint2 raw[kUnroll];   // kUnroll token vectors in flight before the first is used
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) raw[u] = Vec<T>::raw(xin + (t + u) * a.in_sl);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) step(raw[u], t + u);
    }
    for (; t < t1; ++t) step(Vec<T>::raw(xin + t * a.in_sl), t);
    if (write_state && state) {
        // after the shift win[0 .. W-2] hold the last W - 1 inputs; the oldest
        // of the W kept is the one before them
        float oldest[V];
        const int64_t tau = a.L - W;   // index of the oldest kept input
        if (tau >= 0) {
            Vec<T>::load(xin + tau * a.in_sl, oldest);
        } else {
            // it came from the state read at the start (column W + tau, tau >= -W)
#pragma unroll
            for (int j = 0; j < V; ++j) oldest[j] = to_f(state[int64_t(j) * W + (W + tau)]);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            state[int64_t(j) * W] = from_f<T>(oldest[j]);
#pragma unroll
            for (int k = 0; k + 1 < W; ++k) state[int64_t(j) * W + k + 1] = from_f<T>(win[k][j]);
        }
    }
}

// Without windows the loads in flight per SM are the limit: 72 registers fit
// four 224-thread CTAs per SM where the unconstrained 74 fit three, with ten
// token vectors in flight per thread (0.172 -> 0.145 ms at the 2.7B shape).
// With windows more values stay live, so no cap.
template <typename T, int W>
__global__ void __maxnreg__(72) k_conv_prologue(const MixerArgs a, int64_t run) {
    conv_prologue<T, W, false>(a, run);
}
template <typename T, int W>
__global__ void __launch_bounds__(kConvMaxThreads) k_conv_prologue_windows(const MixerArgs a,
                                                                           int64_t run) {
    conv_prologue<T, W, true>(a, run);
}

// The conv state after a sequence of L > 8 >= W tokens: its last W inputs
// (read only from xBC, so it runs after the main launch has read the old state).
template <typename T, int W>
__global__ void __launch_bounds__(256) k_conv_state_tail(const MixerArgs a) {
    const int b = blockIdx.y;
    const int i = blockIdx.x * 256 + threadIdx.x;   // (channel, column) of the state
    if (i >= a.Dc * W) return;
    int64_t slot = b;
    if (a.slots) {
        slot = a.slots[b];
        if (slot < 0 || slot >= a.S) return;        // a padding row
    }
    const int c = i / W, k = i % W;
    const T *xin = static_cast<const T *>(a.xBC) + int64_t(b) * a.in_sb;
    static_cast<T *>(a.state)[slot * a.Dc * W + i] = xin[(a.L - W + k) * a.in_sl + c];
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

template <typename T, int W>
cudaError_t launch_w(const MixerArgs &a, cudaStream_t s) {
    constexpr int V = Vec<T>::kN;
    // channel vectors split evenly over the fewest CTAs of at most
    // kConvMaxThreads threads (whole warps), so no CTA is mostly idle
    const int nvec = a.Dc / V;
    const int nbx = (nvec + kConvMaxThreads - 1) / kConvMaxThreads;
    const int threads = ((nvec + nbx - 1) / nbx + 31) / 32 * 32;
    auto kern = a.windows ? k_conv_prologue_windows<T, W> : k_conv_prologue<T, W>;
    // each sequence split into R runs so that the grid is one wave of
    // resident CTAs (no tail wave); runs of at least 8 tokens
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess ||
        per_sm <= 0) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t slots = int64_t(per_sm) * sm_count() / nbx;
    int64_t R = slots / a.B;
    const int64_t rmax = (a.L + 7) / 8;
    R = R < 1 ? 1 : (R > rmax ? rmax : R);
    R = R > 65535 ? 65535 : R;
    const int64_t run = (a.L + R - 1) / R;
    R = (a.L + run - 1) / run;
    kern<<<dim3(unsigned(nbx), unsigned(R), unsigned(a.B)), threads, 0, s>>>(a, run);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || R == 1 || !a.state) return e;
    // R > 1 means L > 8 >= W: the new state is read from xBC alone
    k_conv_state_tail<T, W><<<dim3(unsigned((a.Dc * W + 255) / 256), unsigned(a.B)), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const MixerArgs &a, cudaStream_t s) {
    switch (a.W) {
    case 1: return launch_w<T, 1>(a, s);
    case 2: return launch_w<T, 2>(a, s);
    case 3: return launch_w<T, 3>(a, s);
    case 4: return launch_w<T, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_mixer_prologue(const MixerArgs &a, cudaStream_t s) {
    if (a.B == 0 || a.L == 0) return cudaSuccess;
    return a.xdt == DT_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ssd
