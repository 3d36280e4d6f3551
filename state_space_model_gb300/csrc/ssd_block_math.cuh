// Per-block arithmetic shared by the fused tensor-core kernels: the
// cumulative-sum record of a 128-token block, the decay operand L of one
// 32-column block, bf16 packing and the exp2 approximation, and the device
// error flags.  Device code only; each including file gets its own copy.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// device error flags
constexpr unsigned kErrTimeout = 1u;      // a bounded wait gave up
constexpr unsigned kErrSmemAlign = 2u;    // the shared-memory window is not 1024-byte aligned

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 2^x with the hardware approximation (relative error ~2^-22; -inf gives +0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Writes this thread's state row n = r (64 headdim values, bf16) into the
// [128 n][64 p] MN-major, 128-byte-swizzled operand tile.
__device__ __forceinline__ void write_state_row(uint8_t *tile, int r, const float2 (&h)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = make_uint4(pack_bf16(h[4 * c].x, h[4 * c].y),
                                   pack_bf16(h[4 * c + 1].x, h[4 * c + 1].y),
                                   pack_bf16(h[4 * c + 2].x, h[4 * c + 2].y),
                                   pack_bf16(h[4 * c + 3].x, h[4 * c + 3].y));
        *reinterpret_cast<uint4 *>(tile + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

// One 32-column block (columns col0..col0 + 31) of the decay operand for
// row r, from the matching block of C B^T in v.  On the diagonal block the
// entries are cb[j] * 2^(gr + ngd[j]) with ngd[j] = log2(dt_j) - g_j, -inf
// exponents for j > r and dd added at j = r.  Strictly below it, with p the
// block's last row, 2^(g_r - g_j) dt_j = 2^(g_r - g_p) * (2^(g_p - g_j) dt_j),
// both factors <= 1 (times dt), so the entries are cb[j] * u * vcol[j] with
// u = 2^(g_r - g_p) and vcol[j] = 2^(g_p - g_j) dt_j: no exponent per entry.
__device__ __forceinline__ void l_block(const uint32_t (&v)[32], int col0, bool diag, int r,
                                        float gr, float u, const float *ngd, const float *vcol,
                                        float dd, uint32_t (&out)[16]) {
    if (diag) {
        const float2 g2 = make_float2(gr, gr);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4) {
            const int j = col0 + jj;
            const float4 n4 = *reinterpret_cast<const float4 *>(ngd + j);
            float2 a0 = __fadd2_rn(g2, make_float2(n4.x, n4.y));
            float2 a1 = __fadd2_rn(g2, make_float2(n4.z, n4.w));
            if (j > r) a0.x = -INFINITY;
            if (j + 1 > r) a0.y = -INFINITY;
            if (j + 2 > r) a1.x = -INFINITY;
            if (j + 3 > r) a1.y = -INFINITY;
            float2 e0 = __fmul2_rn(make_float2(ex2(a0.x), ex2(a0.y)),
                                   make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])));
            float2 e1 = __fmul2_rn(make_float2(ex2(a1.x), ex2(a1.y)),
                                   make_float2(__uint_as_float(v[jj + 2]),
                                               __uint_as_float(v[jj + 3])));
            if (j == r) e0.x += dd;
            if (j + 1 == r) e0.y += dd;
            if (j + 2 == r) e1.x += dd;
            if (j + 3 == r) e1.y += dd;
            out[jj >> 1] = pack_bf16(e0.x, e0.y);
            out[(jj >> 1) + 1] = pack_bf16(e1.x, e1.y);
        }
    } else {
        const float2 u2 = make_float2(u, u);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4) {
            const float4 c4 = *reinterpret_cast<const float4 *>(vcol + col0 + jj);
            const float2 e0 = __fmul2_rn(
                __fmul2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])),
                           make_float2(c4.x, c4.y)),
                u2);
            const float2 e1 = __fmul2_rn(
                __fmul2_rn(make_float2(__uint_as_float(v[jj + 2]), __uint_as_float(v[jj + 3])),
                           make_float2(c4.z, c4.w)),
                u2);
            out[jj >> 1] = pack_bf16(e0.x, e0.y);
            out[(jj >> 1) + 1] = pack_bf16(e1.x, e1.y);
        }
    }
}

// The cumulative-sum record of one 128-token block, computed by one warp
// whose lane holds dt of rows 32 qq + lane: rec[0..127] = g (block-local
// cumulative sum of A dt, log2 units), rec[128..255] = ngd = log2(dt) - g
// (-inf for dt = 0), rec[256..383] = vcol = 2^(g_p - g) dt with p the last row
// of the row's 32-row quarter, rec[384..387] = g of each quarter's last row,
// rec[388] = g_end.
__device__ __forceinline__ void build_record(const float (&dt)[4], float Ah, int lane,
                                             float *rec) {
    float tot[4], own[4];
    // inclusive scans of the four 32-row quarters, interleaved; a quarter's
    // total is its last lane's scan value
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) own[qq] = Ah * dt[qq];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const float o = __shfl_up_sync(0xffffffffu, own[qq], off);
            if (lane >= off) own[qq] += o;
        }
    }
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) tot[qq] = __shfl_sync(0xffffffffu, own[qq], 31);
    float pre = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int row = 32 * qq + lane;
        const float g = (pre + own[qq]) * kLog2e;
        const float ngd = log2f(dt[qq]) - g;
        const float gp = __shfl_sync(0xffffffffu, g, 31);
        rec[row] = g;
        rec[128 + row] = ngd;
        rec[256 + row] = ex2(gp + ngd);
        if (lane == 0) rec[384 + qq] = gp;
        pre += tot[qq];
    }
    if (lane == 0) rec[388] = (((tot[0] + tot[1]) + tot[2]) + tot[3]) * kLog2e;
}

}  // namespace
}  // namespace ssd
