// Decode step of the Mamba-2 layer -- the selective state update of
// "Optimizing Nemotron v3 Super in TensorRT-LLM", section 6.1 "The SSU Math",
// with the dt bias, softplus and z gate of section 6.2's reference:
//     dt' = softplus(dt + dt_bias)          (each step optional)
//     state = exp(A dt') state + dt' x (outer) B        (fp32, in place)
//     out   = (state C + D x) * silu(z)
// for every (batch, head), head h reading group h / (H / G).
//
// The step reads and writes the whole fp32 state once and everything else is
// a few hundred bytes per head, so it is bound by HBM: each thread streams
// four consecutive state columns of one row with 16-byte loads and stores
// (a row is N / 4 contiguous lanes, coalesced), and the row's output is a
// shuffle reduction over those lanes.  No tensor cores: the only contraction
// is a length-N dot product per row.
#include "ssd_internal.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr int kSsuThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// four consecutive elements of a B / C row (16-byte aligned for f32, 8 for bf16)
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// grid (ceil(P / (kRows kR)), H, B); block kSsuThreads = kRows x (N / 4)
// threads; each thread owns four columns of kR rows kRows apart and issues
// all kR state loads before using any, so enough bytes are in flight per SM
// to cover the memory latency.
constexpr int kR = 4;

template <int N, typename T>
__global__ void __launch_bounds__(kSsuThreads)
k_ssu_step(const SsuArgs a) {
    constexpr int kTpr = N / 4;                    // threads per state row
    constexpr int kRows = kSsuThreads / kTpr;      // rows per pass
    const int b = blockIdx.z, h = blockIdx.y;
    const int g = h / (a.H / a.G);
    const int row0 = blockIdx.x * kRows * kR + threadIdx.x / kTpr;
    const int c0 = (threadIdx.x % kTpr) * 4;

    float4 s[kR];
    float4 *sp[kR];
    bool live[kR];
#pragma unroll
    for (int i = 0; i < kR; ++i) {
        const int row = row0 + i * kRows;
        live[i] = row < a.P;
        sp[i] = reinterpret_cast<float4 *>(a.state + ((int64_t(b) * a.H + h) * a.P + row) * N + c0);
        s[i] = live[i] ? *sp[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float d = a.dt[int64_t(b) * a.dt_sb + h];
    if (a.dt_bias) d += a.dt_bias[h];
    if (a.softplus) d = d <= 20.f ? log1pf(expf(d)) : d;   // log(1 + e^d), = d to fp32 above 20
    const float dA = expf(a.A[h] * d);
    const int64_t bc = int64_t(b) * a.bc_sb + int64_t(g) * a.bc_sg + c0;
    const float4 bq = load4(static_cast<const T *>(a.Bm) + bc);
    const float4 cq = load4(static_cast<const T *>(a.Cm) + bc);
    const T *xr = static_cast<const T *>(a.x) + int64_t(b) * a.x_sb + int64_t(h) * a.x_sh;

#pragma unroll
    for (int i = 0; i < kR; ++i) {
        const int row = row0 + i * kRows;
        float partial = 0.f, xv = 0.f;
        if (live[i]) {
            xv = to_f(xr[row]);
            const float u = d * xv;
            s[i].x = fmaf(s[i].x, dA, u * bq.x);
            s[i].y = fmaf(s[i].y, dA, u * bq.y);
            s[i].z = fmaf(s[i].z, dA, u * bq.z);
            s[i].w = fmaf(s[i].w, dA, u * bq.w);
            *sp[i] = s[i];
            partial = fmaf(s[i].x, cq.x, fmaf(s[i].y, cq.y, fmaf(s[i].z, cq.z, s[i].w * cq.w)));
        }
        // sum over the row's kTpr lanes (contiguous within the warp)
#pragma unroll
        for (int off = kTpr / 2; off > 0; off >>= 1)
            partial += __shfl_xor_sync(0xffffffffu, partial, off);
        if (live[i] && threadIdx.x % kTpr == 0) {
            float o = partial;
            if (a.D) o = fmaf(a.D[h], xv, o);
            if (a.z) {
                const float zv = to_f(static_cast<const T *>(a.z)[int64_t(b) * a.z_sb +
                                                                  int64_t(h) * a.z_sh + row]);
                o *= zv / (1.f + expf(-zv));
            }
            static_cast<T *>(a.out)[int64_t(b) * a.o_sb + int64_t(h) * a.o_sh + row] = from_f<T>(o);
        }
    }
}

template <int N, typename T>
cudaError_t launch_n(const SsuArgs &a, cudaStream_t s) {
    constexpr int kRows = kSsuThreads / (N / 4);
    const dim3 grid(unsigned((a.P + kRows * kR - 1) / (kRows * kR)), unsigned(a.H), unsigned(a.B));
    k_ssu_step<N, T><<<grid, kSsuThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const SsuArgs &a, cudaStream_t s) {
    switch (a.N) {
    case 16: return launch_n<16, T>(a, s);
    case 32: return launch_n<32, T>(a, s);
    case 64: return launch_n<64, T>(a, s);
    case 128: return launch_n<128, T>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_ssu(const SsuArgs &a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    return a.xdt == DT_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace ssd
