// The mixer's output gate, y *= silu(z) (the gated forward,
// ssd_chunked_fwd_gated): the z gate of the SSU reference in "Optimizing
// Nemotron v3 Super in TensorRT-LLM", section 6.2, applied to the scan's
// output as one HBM-bound pass after it.
#include "ssd_internal.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

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

// y *= silu(z) in place, [B, L, H, P] with P contiguous (the mixer's output
// gate).  HBM-bound (y read and written, z read once): CTA i takes tokens
// [kGateTok i, + kGateTok) of the B L token rows, one token at a time, each
// thread 16-byte vectors of y and z at a stride of the CTA, four in flight,
// with streaming cache hints.  pv_shift = log2(P / V) (P a power of two).
constexpr int kGateTok = 8;
template <typename T>
__global__ void __launch_bounds__(128) k_gate(const Args a, int pv_shift) {
    constexpr int V = 16 / sizeof(T);
    const int nv = (a.d.H * a.d.P) / V;                 // vectors per token
    const int64_t tok0 = int64_t(blockIdx.x) * kGateTok;
    const int64_t ntok = a.d.B * a.d.L;
    const int ntk = int(ntok - tok0 < kGateTok ? ntok - tok0 : kGateTok);
    for (int tt = 0; tt < ntk; ++tt) {
        const int64_t tok = tok0 + tt;
        const int64_t b = tok / a.d.L, t = tok % a.d.L;
        T *yrow = static_cast<T *>(a.y) + b * a.y_sb + t * a.y_sl;
        const T *zrow = static_cast<const T *>(a.z) + b * a.z_sb + t * a.z_sl;
        for (int v0 = threadIdx.x; v0 < nv; v0 += 4 * 128) {
            uint4 yv[4], zv[4];
            int64_t yo[4], zo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * 128;
                const int hh = v >> pv_shift, pp = (v & ((1 << pv_shift) - 1)) * V;
                yo[u] = int64_t(hh) * a.y_sh + pp;
                zo[u] = int64_t(hh) * a.z_sh + pp;
                if (v < nv) {
                    yv[u] = __ldcs(reinterpret_cast<const uint4 *>(yrow + yo[u]));
                    zv[u] = __ldcs(reinterpret_cast<const uint4 *>(zrow + zo[u]));
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v0 + u * 128 >= nv) break;
                const T *yt = reinterpret_cast<const T *>(&yv[u]);
                const T *zt = reinterpret_cast<const T *>(&zv[u]);
                T o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float zf = to_f(zt[e]);
                    // silu with the fast exponential and division (~2 ulp)
                    o[e] = from_f<T>(to_f(yt[e]) * __fdividef(zf, 1.f + __expf(-zf)));
                }
                __stcs(reinterpret_cast<uint4 *>(yrow + yo[u]), *reinterpret_cast<const uint4 *>(o));
            }
        }
    }
}

}  // namespace

cudaError_t launch_gate(const Args &a, cudaStream_t s) {
    if (a.d.B == 0 || a.d.L == 0) return cudaSuccess;
    const unsigned grid = unsigned((a.d.B * a.d.L + kGateTok - 1) / kGateTok);
    const int V = a.xdt == DT_BF16 ? 8 : 4;
    int pv_shift = 0;
    while ((1 << pv_shift) < a.d.P / V) ++pv_shift;   // P / V is a power of two
    if (a.xdt == DT_BF16)
        k_gate<__nv_bfloat16><<<grid, 128, 0, s>>>(a, pv_shift);
    else
        k_gate<float><<<grid, 128, 0, s>>>(a, pv_shift);
    return cudaGetLastError();
}

}  // namespace ssd
