// CUDA-core kernels of the four steps, for every supported geometry and
// both input dtypes.  They are the path for fp32 inputs (fp32 FMA keeps the
// 1e-4 contract without tensor-core splitting) and for geometries the
// tensor-core kernels do not cover.
//
// Method: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile", sections "Kernel 1: Computing cumulative sums",
// "Kernel 2: fwd_pass_state" and "Kernel 3: compute_out".  G is kept scaled
// by log2(e) so every decay is one exp2.
#include "ssd_internal.h"
#include "ssd_simt.cuh"
#define SSD_DBG_FILE 4u   // kDbgSimt
#include "ssd_debug.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------
// Step 1: in-chunk inclusive cumulative sum of A[h] * dt, scaled by log2(e).
// One warp per (b, chunk, head); lane k owns Q/32 consecutive tokens.  The
// zero padding past L keeps the running sum at the chunk's last real value.
__global__ void __launch_bounds__(256)
k_chunk_cumsum(const float *__restrict__ dt, int64_t dt_sb, int64_t dt_sl,
               const float *__restrict__ A, float *__restrict__ G, int64_t L, int H, int Q,
               int64_t nc, unsigned int *err, int64_t n_dt, int64_t n_G) {
    const int64_t c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 8 + warp;
    const int64_t b = blockIdx.z;
    if (h >= H) return;
    const int R = Q / 32;  // 2, 4 or 8
    const float a = A[h];
    const int64_t t0 = c * Q + int64_t(lane) * R;
    float v[8];
    float run = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (k < R) {
            const int64_t t = t0 + k;
            const float d = (t < L && SSD_IDX_OK(err, b * dt_sb + t * dt_sl + h, n_dt))
                                ? __ldg(dt + b * dt_sb + t * dt_sl + h)
                                : 0.f;
            run += a * d;
            v[k] = run;
        }
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const float excl = incl - run;
    float *g = G + (b * H + h) * (nc * Q) + t0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < R && SSD_IDX_OK(err, (b * H + h) * (nc * Q) + t0 + k, n_G))
            g[k] = (excl + v[k]) * kLog2e;
}

// ---------------------------------------------------------------------------
// Step 2: per-chunk state S[p][n] = sum_j 2^(G_last - G_j) dt_j x_j[p] B_j[n].
// One CTA per (chunk, head, batch); 16 x 16 threads, each owning a
// (P/16) x (N/16) register tile.  Tokens are staged 32 at a time.
template <typename T>
__global__ void __launch_bounds__(256) k_chunk_state_simt(Args a) {
    extern __shared__ float sm[];
    const Dims d = a.d;
    const int P = int(d.P), N = int(d.N), Q = int(d.Q);
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int h = blockIdx.y;
    const int64_t g = h / d.hpg();
    float *xs = sm;               // [32][P], rows scaled by w_j
    float *bs = sm + 32 * P;      // [32][N]
    float *ws = bs + 32 * N;      // [32]
    // the block's G row and S tile (uniform over the block, before any barrier)
    if (!SSD_IN_BOUNDS(a.err, (b * d.H + h) * d.Lp() + c * Q + Q <= d.B * d.H * d.Lp() &&
                                  ((b * d.nc + c) * d.H + h + 1) * int64_t(P) * N <=
                                      d.B * d.nc * d.H * int64_t(P) * N))
        return;
    const float *Grow = a.G + (b * d.H + h) * d.Lp() + c * Q;
    const float g_last = Grow[Q - 1];
    const T *x = static_cast<const T *>(a.x);
    const T *Bm = static_cast<const T *>(a.Bm);
    const int tp = threadIdx.x >> 4, tn = threadIdx.x & 15;
    const int TP = P >> 4, TN = N >> 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = 0.f;

    for (int j0 = 0; j0 < Q; j0 += 32) {
        if (threadIdx.x < 32) {
            const int64_t t = c * Q + j0 + threadIdx.x;
            ws[threadIdx.x] = (t < d.L && SSD_IDX_OK(a.err, b * a.dt_sb + t * a.dt_sl + h, a.n_dt))
                                  ? exp2f(g_last - Grow[j0 + threadIdx.x]) *
                                        __ldg(a.dt + b * a.dt_sb + t * a.dt_sl + h)
                                  : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < 32 * P; e += 256) {
            const int jj = e / P, p = e - jj * P;
            const int64_t t = c * Q + j0 + jj;
            const int64_t xo = b * a.x_sb + t * a.x_sl + h * a.x_sh + p;
            xs[e] = (t < d.L && SSD_IDX_OK(a.err, xo, a.n_x)) ? ws[jj] * to_f(x[xo]) : 0.f;
        }
        for (int e = threadIdx.x; e < 32 * N; e += 256) {
            const int jj = e / N, n = e - jj * N;
            const int64_t t = c * Q + j0 + jj;
            const int64_t bo = b * a.b_sb + t * a.b_sl + g * a.b_sg + n;
            bs[e] = (t < d.L && SSD_IDX_OK(a.err, bo, a.n_b)) ? to_f(Bm[bo]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < 32; ++jj) {
            float xv[8], bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = (i < TP) ? xs[jj * P + tp + 16 * i] : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) bv[k] = (k < TN) ? bs[jj * N + tn + 16 * k] : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[i][k] = fmaf(xv[i], bv[k], acc[i][k]);
        }
        __syncthreads();
    }
    float *S = a.S + ((b * d.nc + c) * d.H + h) * int64_t(P) * N;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i < TP && k < TN) S[(tp + 16 * i) * N + tn + 16 * k] = acc[i][k];
}

// ---------------------------------------------------------------------------
// Step 3: sequential pass over chunks, one CTA per (batch, head) slab.  Each
// thread carries its share of the P x N fp32 state in registers (float4s)
// and streams S[c] while writing the entering state h_prev[c].
template <typename TS>
__device__ __forceinline__ void store4(TS *p, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename TS>
__global__ void __launch_bounds__(256) k_state_passing(Args a) {
    const Dims d = a.d;
    const int64_t slab = blockIdx.x, b = slab / d.H, h = slab % d.H;
    const int64_t PN = d.P * d.N;
    const int nq = int(PN >> 2);  // float4 per state, 64..4096
    if (!SSD_IN_BOUNDS(a.err, (slab + 1) * PN <= d.B * d.H * PN &&
                                  (slab + 1) * d.Lp() <= d.B * d.H * d.Lp() &&
                                  ((b * d.nc + d.nc - 1) * d.H + h + 1) * PN <= d.B * d.nc * d.H * PN))
        return;
    float4 hv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int q = threadIdx.x + 256 * k;
        hv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.h0 && q < nq) hv[k] = reinterpret_cast<const float4 *>(a.h0 + slab * PN)[q];
    }
    const float *Grow = a.G + slab * d.Lp();
    TS *hp = static_cast<TS *>(a.h_prev);
    for (int64_t c = 0; c < d.nc; ++c) {
        const float dec = exp2f(Grow[c * d.Q + d.Q - 1]);
        const int64_t off = ((b * d.nc + c) * d.H + h) * PN;
        const float4 *Sc = reinterpret_cast<const float4 *>(a.S + off);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = threadIdx.x + 256 * k;
            if (q < nq) {
                const float4 s = __ldcs(Sc + q);
                store4<TS>(hp + off + 4 * q, hv[k]);
                hv[k].x = fmaf(dec, hv[k].x, s.x);
                hv[k].y = fmaf(dec, hv[k].y, s.y);
                hv[k].z = fmaf(dec, hv[k].z, s.z);
                hv[k].w = fmaf(dec, hv[k].w, s.w);
            }
        }
    }
    if (a.final_states) {
        float4 *f = reinterpret_cast<float4 *>(a.final_states + slab * PN);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = threadIdx.x + 256 * k;
            if (q < nq) f[q] = hv[k];
        }
    }
}

// ---------------------------------------------------------------------------
// Step 4: outputs of a 64-row block of one chunk for one head:
//   y_i = 2^G_i sum_n C_i[n] h[p][n] + sum_{j<=i} 2^(G_i - G_j) (C_i.B_j) dt_j x_j[p] + D x_i[p]
// The causal selection is taken before the exponent, so no positive exponent
// is ever evaluated.  16 x 16 threads; a thread owns rows ti + 16r (r < 4)
// and columns tj + 16k.
template <typename T, typename TS>
__global__ void __launch_bounds__(256) k_chunk_scan_simt(Args a) {
    extern __shared__ float sm[];
    const Dims d = a.d;
    const int P = int(d.P), N = int(d.N), Q = int(d.Q);
    const int NS = N + 1;  // padded row stride
    const int rbs = Q / 64;
    const int64_t c = blockIdx.x / rbs;
    const int rb = blockIdx.x % rbs;
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z, g = h / d.hpg();
    float *Cs = sm;                 // [64][NS]
    float *Bs = Cs + 64 * NS;       // [64][NS], reused for h_prev rows
    float *Ls = Bs + 64 * NS;       // [64][65]
    float *Xs = Ls + 64 * 65;       // [64][P]  (dt_j x_j)
    float *gi = Xs + 64 * P;        // [64]
    float *gj = gi + 64;            // [64]
    const T *x = static_cast<const T *>(a.x);
    const T *Bm = static_cast<const T *>(a.Bm);
    const T *Cm = static_cast<const T *>(a.Cm);
    if (!SSD_IN_BOUNDS(a.err, (b * d.H + h) * d.Lp() + c * Q + Q <= d.B * d.H * d.Lp() &&
                                  ((b * d.nc + c) * d.H + h + 1) * int64_t(P) * N <=
                                      d.B * d.nc * d.H * int64_t(P) * N))
        return;
    const float *Grow = a.G + (b * d.H + h) * d.Lp() + c * Q;
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    const int TP = P >> 4;
    const int64_t i0 = c * Q + rb * 64;

    for (int e = threadIdx.x; e < 64 * N; e += 256) {
        const int r = e / N, n = e - r * N;
        const int64_t t = i0 + r;
        const int64_t co = b * a.c_sb + t * a.c_sl + g * a.c_sg + n;
        Cs[r * NS + n] = (t < d.L && SSD_IDX_OK(a.err, co, a.n_c)) ? to_f(Cm[co]) : 0.f;
    }
    if (threadIdx.x < 64) gi[threadIdx.x] = Grow[rb * 64 + threadIdx.x];

    float yacc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int k = 0; k < 8; ++k) yacc[r][k] = 0.f;

    for (int jb = 0; jb <= rb; ++jb) {
        const int64_t j0 = c * Q + jb * 64;
        __syncthreads();
        for (int e = threadIdx.x; e < 64 * N; e += 256) {
            const int r = e / N, n = e - r * N;
            const int64_t t = j0 + r;
            const int64_t bo = b * a.b_sb + t * a.b_sl + g * a.b_sg + n;
            Bs[r * NS + n] = (t < d.L && SSD_IDX_OK(a.err, bo, a.n_b)) ? to_f(Bm[bo]) : 0.f;
        }
        for (int e = threadIdx.x; e < 64 * P; e += 256) {
            const int r = e / P, p = e - r * P;
            const int64_t t = j0 + r;
            const int64_t xo = b * a.x_sb + t * a.x_sl + h * a.x_sh + p;
            const int64_t dto = b * a.dt_sb + t * a.dt_sl + h;
            Xs[e] = (t < d.L && SSD_IDX_OK(a.err, xo, a.n_x) && SSD_IDX_OK(a.err, dto, a.n_dt))
                        ? __ldg(a.dt + dto) * to_f(x[xo])
                        : 0.f;
        }
        if (threadIdx.x < 64) gj[threadIdx.x] = Grow[jb * 64 + threadIdx.x];
        __syncthreads();
        float cb[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) cb[r][q] = 0.f;
        for (int n = 0; n < N; ++n) {
            float cv[4], bv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) cv[r] = Cs[(ti + 16 * r) * NS + n];
#pragma unroll
            for (int q = 0; q < 4; ++q) bv[q] = Bs[(tj + 16 * q) * NS + n];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) cb[r][q] = fmaf(cv[r], bv[q], cb[r][q]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ri = ti + 16 * r, cj = tj + 16 * q;
                const bool keep = (jb * 64 + cj) <= (rb * 64 + ri);
                Ls[ri * 65 + cj] = keep ? exp2f(gi[ri] - gj[cj]) * cb[r][q] : 0.f;
            }
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < 64; ++jj) {
            float lv[4], xv[8];
#pragma unroll
            for (int r = 0; r < 4; ++r) lv[r] = Ls[(ti + 16 * r) * 65 + jj];
#pragma unroll
            for (int k = 0; k < 8; ++k) xv[k] = (k < TP) ? Xs[jj * P + tj + 16 * k] : 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int k = 0; k < 8; ++k) yacc[r][k] = fmaf(lv[r], xv[k], yacc[r][k]);
        }
    }

    // carried-state term, 64 state rows (p) at a time through the B buffer
    float inter[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int k = 0; k < 8; ++k) inter[r][k] = 0.f;
    const TS *hp = static_cast<const TS *>(a.h_prev) + ((b * d.nc + c) * d.H + h) * int64_t(P) * N;
    for (int pb = 0; pb < P; pb += 64) {
        const int np = min(64, P - pb);
        __syncthreads();
        for (int e = threadIdx.x; e < np * N; e += 256) {
            const int r = e / N, n = e - r * N;
            Bs[r * NS + n] = to_f(hp[int64_t(pb + r) * N + n]);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int p = tj + 16 * k;
            if (k < TP && p >= pb && p < pb + np) {
                for (int n = 0; n < N; ++n) {
                    const float hv = Bs[(p - pb) * NS + n];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        inter[r][k] = fmaf(Cs[(ti + 16 * r) * NS + n], hv, inter[r][k]);
                }
            }
        }
    }
    const float Dh = a.D && SSD_IDX_OK(a.err, h, d.H) ? a.D[h] : 0.f;
    T *y = static_cast<T *>(a.y);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int ri = ti + 16 * r;
        const int64_t t = i0 + ri;
        if (t >= d.L) continue;
        const float e = exp2f(gi[ri]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < TP) {
                const int p = tj + 16 * k;
                const int64_t xo = b * a.x_sb + t * a.x_sl + h * a.x_sh + p;
                const int64_t yo = b * a.y_sb + t * a.y_sl + h * a.y_sh + p;
                if (!SSD_IDX_OK(a.err, xo, a.n_x) || !SSD_IDX_OK(a.err, yo, a.n_y)) continue;
                const float v = fmaf(e, inter[r][k], yacc[r][k]) + Dh * to_f(x[xo]);
                y[yo] = from_f<T>(v);
            }
        }
    }
}

}  // namespace

cudaError_t simt_chunk_cumsum(const Args &a0, cudaStream_t s) {
    Args a;
    cudaError_t e0 = debug_args(a0, &a);
    if (e0 != cudaSuccess) return e0;
    const Dims &d = a.d;
    dim3 grid(unsigned(d.nc), unsigned((d.H + 7) / 8), unsigned(d.B));
    k_chunk_cumsum<<<grid, 256, 0, s>>>(a.dt, a.dt_sb, a.dt_sl, a.A, a.G, d.L, int(d.H),
                                        int(d.Q), d.nc, a.err, a.n_dt, d.B * d.H * d.Lp());
    return cudaGetLastError();
}

cudaError_t simt_chunk_state(const Args &a0, cudaStream_t s) {
    Args a;
    cudaError_t e0 = debug_args(a0, &a);
    if (e0 != cudaSuccess) return e0;
    const Dims &d = a.d;
    dim3 grid(unsigned(d.nc), unsigned(d.H), unsigned(d.B));
    const size_t smem = sizeof(float) * (32 * d.P + 32 * d.N + 32);
    if (a.xdt == DT_F32) {
        k_chunk_state_simt<float><<<grid, 256, smem, s>>>(a);
    } else {
        k_chunk_state_simt<__nv_bfloat16><<<grid, 256, smem, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t simt_state_passing(const Args &a0, cudaStream_t s) {
    Args a;
    cudaError_t e0 = debug_args(a0, &a);
    if (e0 != cudaSuccess) return e0;
    const Dims &d = a.d;
    dim3 grid(unsigned(d.B * d.H));
    if (a.hprev_dt == DT_F32)
        k_state_passing<float><<<grid, 256, 0, s>>>(a);
    else
        k_state_passing<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t simt_chunk_scan(const Args &a0, cudaStream_t s) {
    Args a;
    cudaError_t e0 = debug_args(a0, &a);
    if (e0 != cudaSuccess) return e0;
    const Dims &d = a.d;
    dim3 grid(unsigned(d.nc * (d.Q / 64)), unsigned(d.H), unsigned(d.B));
    const size_t smem = sizeof(float) * (2 * 64 * (d.N + 1) + 64 * 65 + 64 * d.P + 128);
    cudaError_t e;
    if (a.xdt == DT_F32) {
        auto k = k_chunk_scan_simt<float, float>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        k<<<grid, 256, smem, s>>>(a);
    } else {
        auto k = k_chunk_scan_simt<__nv_bfloat16, __nv_bfloat16>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        k<<<grid, 256, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ssd
