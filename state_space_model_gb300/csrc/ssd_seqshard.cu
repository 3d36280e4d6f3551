// Sequence sharding of the forward over ranks: the steps around the exchange.
//
// "mamba-metal", "The essence of selective scan": the recurrence
// h_t = a_t h_{t-1} + b_t composes over a segment into one pair (a, b) =
// (total decay, state reached from zero), and pairs compose associatively,
// (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2).  A rank that holds a contiguous
// segment of the sequence runs the forward on it from a zero state (the
// ordinary ssd_chunked_fwd) and gets b (its final state) and, from
// k_segment_logdecay, log a = sum_t A dt_t.  After the pairs of all ranks are
// gathered, k_sequence_combine folds the pairs of the earlier ranks in
// sequence order into the state entering this rank's segment, and
// k_shard_correct adds what that state contributes:
//   y_t += e^(cum_t) C_t h_in^T,  cum_t = sum_{k <= t} A dt_k (within the segment),
//   final = e^(log a) h_in + b.
// The output of a token decays with its distance from the segment start, so
// the correction stops at the first 128-token chunk whose decay has
// underflowed to exactly zero (cum decreases: A <= 0, dt >= 0), where every
// later term is exactly zero too.
#include "ssd_internal.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

__device__ __forceinline__ float ld_elem(const void *p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
                : static_cast<const float *>(p)[i];
}

// log a[b, h] = A[h] * sum_t dt[b, t, h] (natural log units), the sum taken in
// fp64 in a fixed order (deterministic).  grid (ceil(H / 32), B), 256 threads:
// lane = head within the block's 32, warp w sums tokens t = w mod 8.
__global__ void __launch_bounds__(256)
k_segment_logdecay(const float *dt, int64_t dt_sb, int64_t dt_sl, const float *A, int64_t L,
                   int H, float *out) {
    __shared__ double part[8][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * 32 + lane;
    const int64_t b = blockIdx.y;
    double acc = 0.0;
    if (h < H)
        for (int64_t t = warp; t < L; t += 8) acc += double(dt[b * dt_sb + t * dt_sl + h]);
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && h < H) {
        double s = 0.0;
        for (int w = 0; w < 8; ++w) s += part[w][lane];
        out[b * H + h] = float(double(A[h]) * s);
    }
}

// h_in[b, h] = fold over ranks q < rank of h <- e^(logdecay[q, b, h]) h + state[q, b, h],
// from h0[b, h] (or zero).  One thread per state element.
__global__ void __launch_bounds__(256)
k_sequence_combine(const float *logdecay, const float *states, const float *h0, int rank,
                   int64_t BH, int64_t PN, float *h_in) {
    const int64_t i = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (i >= BH * PN) return;
    const int64_t bh = i / PN;
    float h = h0 ? h0[i] : 0.f;
    for (int q = 0; q < rank; ++q)
        h = fmaf(expf(logdecay[q * BH + bh]), h, states[q * BH * PN + i]);
    h_in[i] = h;
}

// One CTA per (batch, head): y[b, t, h, :] += e^(cum_t) C_t h_in^T over the
// segment, 128 tokens at a time, and final = e^(logdecay) h_in + final.
// Shared memory: hT [N][P] fp32 (h_in transposed), CT [N][128] fp32 (the
// chunk's C transposed), e [128], a scan buffer.  256 threads; thread j owns
// token j / 2 of the chunk and headdim values (j % 2) * P / 2 ..
struct CorrectArgs {
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *A;
    const void *C;
    int64_t c_sb, c_sl, c_sg;
    const float *h_in;
    const float *logdecay;
    void *y;
    int64_t y_sb, y_sl, y_sh;
    float *final_states;
    int64_t L;
    int H, P, N, hpg, bf16;
};

__global__ void __launch_bounds__(256) k_shard_correct(const CorrectArgs a) {
    extern __shared__ float sm[];
    const int P = a.P, N = a.N;
    float *hT = sm;                  // [N][P]
    float *CT = hT + N * P;          // [N][128]
    float *ev = CT + N * 128;        // [128]
    float *scan = ev + 128;          // [8] warp totals
    const int h = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int g = h / a.hpg;
    const int64_t slab = b * a.H + h;
    const float *hin = a.h_in + slab * int64_t(P) * N;
    for (int e = threadIdx.x; e < P * N; e += 256) {
        const int p = e / N, n = e - p * N;
        hT[n * P + p] = hin[e];
    }
    const float Ah = a.A[h];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok = threadIdx.x >> 1, phalf = threadIdx.x & 1;
    const int np = P / 2;   // headdim values per thread (8 .. 64)
    float carry = 0.f;
    for (int64_t t0 = 0; t0 < a.L; t0 += 128) {
        // cum over the chunk: block inclusive scan of A dt for tokens t0 ..
        __syncthreads();   // the previous chunk's readers of CT / ev are done
        float v = 0.f;
        if (threadIdx.x < 128 && t0 + threadIdx.x < a.L)
            v = Ah * a.dt[b * a.dt_sb + (t0 + threadIdx.x) * a.dt_sl + h];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
        }
        if (lane == 31) scan[warp] = v;
        __syncthreads();
        if (threadIdx.x < 128) {
            float pre = carry;
            for (int w = 0; w < warp; ++w) pre += scan[w];
            ev[threadIdx.x] = t0 + threadIdx.x < a.L ? expf(pre + v) : 0.f;
        }
        carry += scan[0] + scan[1] + scan[2] + scan[3];
        for (int e = threadIdx.x; e < 128 * N; e += 256) {
            const int r = e / N, n = e - r * N;
            const int64_t t = t0 + r;
            CT[n * 128 + r] =
                t < a.L ? ld_elem(a.C, b * a.c_sb + t * a.c_sl + int64_t(g) * a.c_sg + n, a.bf16)
                        : 0.f;
        }
        __syncthreads();
        // the decay at the chunk's first token is the largest of the chunk and
        // of every later chunk: once it is zero, nothing more is added
        if (ev[0] == 0.f) break;
        const int64_t t = t0 + tok;
        if (t < a.L && ev[tok] != 0.f) {
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.f;
            for (int n = 0; n < N; ++n) {
                const float c = CT[n * 128 + tok];
                const float *hr = hT + n * P + phalf * np;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < np) acc[i] = fmaf(c, hr[i], acc[i]);
            }
            const float e = ev[tok];
            const int64_t yo = b * a.y_sb + t * a.y_sl + int64_t(h) * a.y_sh + phalf * np;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                if (i < np) {
                    if (a.bf16) {
                        __nv_bfloat16 *yp = static_cast<__nv_bfloat16 *>(a.y) + yo + i;
                        *yp = __float2bfloat16_rn(fmaf(e, acc[i], __bfloat162float(*yp)));
                    } else {
                        float *yp = static_cast<float *>(a.y) + yo + i;
                        *yp = fmaf(e, acc[i], *yp);
                    }
                }
            }
        }
    }
    if (a.final_states) {
        const float d = expf(a.logdecay[slab]);
        float *f = a.final_states + slab * int64_t(P) * N;
        for (int e = threadIdx.x; e < P * N; e += 256) f[e] = fmaf(d, hin[e], f[e]);
    }
}

}  // namespace

cudaError_t launch_segment_logdecay(const float *dt, int64_t dt_sb, int64_t dt_sl, const float *A,
                                    int64_t B, int64_t L, int64_t H, float *out, cudaStream_t s) {
    k_segment_logdecay<<<dim3(unsigned((H + 31) / 32), unsigned(B)), 256, 0, s>>>(
        dt, dt_sb, dt_sl, A, L, int(H), out);
    return cudaGetLastError();
}

cudaError_t launch_sequence_combine(const float *logdecay, const float *states, const float *h0,
                                    int rank, int64_t BH, int64_t PN, float *h_in,
                                    cudaStream_t s) {
    const int64_t n = BH * PN;
    k_sequence_combine<<<unsigned((n + 255) / 256), 256, 0, s>>>(logdecay, states, h0, rank, BH,
                                                                 PN, h_in);
    return cudaGetLastError();
}

cudaError_t launch_shard_correct(const Args &a, const float *h_in, const float *logdecay,
                                 cudaStream_t s) {
    const Dims &d = a.d;
    CorrectArgs c{a.dt, a.dt_sb, a.dt_sl, a.A, a.Cm, a.c_sb, a.c_sl, a.c_sg, h_in, logdecay,
                  a.y, a.y_sb, a.y_sl, a.y_sh, a.final_states, d.L, int(d.H), int(d.P),
                  int(d.N), int(d.hpg()), a.xdt == DT_BF16 ? 1 : 0};
    const int smem = int((d.N * d.P + d.N * 128 + 128 + 8) * sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(k_shard_correct,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_shard_correct<<<dim3(unsigned(d.H), unsigned(d.B)), 256, smem, s>>>(c);
    return cudaGetLastError();
}

}  // namespace ssd
