// Fused SSD forward on tcgen05: all four steps of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile" (the in-chunk
// cumulative sum, the per-chunk state and its sequential pass, and
// compute_out) in one kernel, so x is read once, y written once and no
// intermediate reaches HBM.
//
// One CTA walks one (batch, head) slab -- or one segment of it -- in blocks
// of 128 tokens.  A chunk of Q = 128 k tokens is evaluated as k such blocks:
// its off-diagonal decay blocks are applied through the state at the block
// boundary, by associativity,
//     (C_1 B_0^T o decay) (dt x_0) = 2^(g_1) C_1 (B_0^T (w o x_0)),
// the same product in a different order.  Per block, with g the block-local
// cumulative sum of A dt (log2 units):
//     CB    = C B^T                                  tensor cores -> TMEM
//     inter = C h^T                                  tensor cores -> TMEM
//     L_ij  = [j <= i] CB_ij 2^(g_i - g_j) dt_j      math warps, in place in TMEM (bf16)
//     intra = L x                                    tensor cores, A read from TMEM
//     S^T   = B^T (w o x),  w_j = 2^(g_end - g_j) dt_j   tensor cores -> TMEM
//     y     = 2^(g_i) inter + intra + D x            math warps (drain)
//     h     = 2^(g_end) h + S                        math warps, fp32 in registers
// dt_j is folded into the exponent, 2^(g_i - g_j + log2 dt_j) (dt_j = 0 gives
// 2^-inf = 0), and the causal selection replaces the exponent of masked
// entries by -inf before it is evaluated, so no positive exponent of the
// decay is ever computed.
//
// Roles: warp 0 = TMA producer (128-byte swizzle, no multicast), warp 1 =
// tensor-memory owner and MMA issuer, warps 2..5 = math (thread r owns tile
// row / state row r = TMEM lane r).  Tensor memory (256 columns): [0,64) C B^T
// then L, [64,128) C B^T then S^T, [128,192) inter, [192,256) intra.  Shared
// memory (~99 KB, two CTAs per SM): the C, B and x tiles, and one buffer that
// holds the bf16 carried state [n][p] (inter's operand) and then w o x [j][p]
// (the state product's operand).
#include "ptx_sm100.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#include "ssd_tmap.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct FusedParams {
    int64_t L;            // sequence length
    int64_t seg_len;      // tokens per segment (multiple of 128)
    int B, H, hpg, nseg;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *A;
    const float *D;       // may be null
    const float *h_in;    // [nseg][B][H][P][N] entering state per segment, or null (= 0)
    float *h_out;         // [B][H][P][N] state after the last segment, or null
    __nv_bfloat16 *y;
    int64_t y_sb, y_sl, y_sh;
    unsigned int *err;
};

struct FusedSmem {
    static constexpr int kC = 0;         // 2 x [128 tokens][128 B]  C, K-major (state)
    static constexpr int kB = 32768;     // 2 x [128 tokens][128 B]  B, K-major (state)
    static constexpr int kX = 65536;     // [128 tokens][128 B]      x, MN-major (headdim)
    static constexpr int kXH = 81920;    // [128][128 B]: bf16 state [n][p] / w o x [j][p]
    static constexpr int kF = 98304;     // ngd[128] (float), w2[128] (bf16x2), wsum[4]
    static constexpr int kBar = kF + (2 * 128 + 4) * 4;
    static constexpr int kBytes = kBar + 128 + 1024;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
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

// One 32-column block of the decay operand for row r: entries
// cb[j] * 2^(gr + ngd[j]) with ngd[j] = log2(dt_j) - g_j, and, on the
// diagonal block, -inf exponents for j > r.
__device__ __forceinline__ void l_block(const uint32_t (&v)[32], int col0, bool diag, int r,
                                        float gr, const float *ngd, uint32_t (&out)[16]) {
    const float2 g2 = make_float2(gr, gr);
#pragma unroll
    for (int jj = 0; jj < 32; jj += 4) {
        const float4 n4 = *reinterpret_cast<const float4 *>(ngd + col0 + jj);
        float2 a0 = __fadd2_rn(g2, make_float2(n4.x, n4.y));
        float2 a1 = __fadd2_rn(g2, make_float2(n4.z, n4.w));
        if (diag) {
            const int j = col0 + jj;
            if (j > r) a0.x = -INFINITY;
            if (j + 1 > r) a0.y = -INFINITY;
            if (j + 2 > r) a1.x = -INFINITY;
            if (j + 3 > r) a1.y = -INFINITY;
        }
        const float2 e0 = __fmul2_rn(make_float2(ex2(a0.x), ex2(a0.y)),
                                     make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])));
        const float2 e1 = __fmul2_rn(make_float2(ex2(a1.x), ex2(a1.y)),
                                     make_float2(__uint_as_float(v[jj + 2]),
                                                 __uint_as_float(v[jj + 3])));
        out[jj >> 1] = pack_bf16(e0.x, e0.y);
        out[(jj >> 1) + 1] = pack_bf16(e1.x, e1.y);
    }
}

__global__ void __launch_bounds__(192, 2)
k_ssd_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
            const __grid_constant__ CUtensorMap tm_c, const FusedParams p) {
    using SM = FusedSmem;
    constexpr uint32_t kCols = 256;
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdKmn = ptx::idesc_bf16_f32(128, 64, false, true);   // A K-major, B MN-major
    constexpr uint32_t kIdState = ptx::idesc_bf16_f32(128, 64, true, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *ngd = reinterpret_cast<float *>(smem + SM::kF);
    uint32_t *w2 = reinterpret_cast<uint32_t *>(ngd + 128);
    float *wsum = reinterpret_cast<float *>(w2 + 128);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint64_t *bar_C = bars, *bar_B = bars + 1, *bar_X = bars + 2, *bar_cbi = bars + 3,
             *bar_L = bars + 4, *bar_is = bars + 5, *bar_dr = bars + 6;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 7);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // unit = (segment, batch, head), heads fastest so neighbouring CTAs share B, C in L2
    const int unit = blockIdx.x;
    const int h = unit % p.H;
    const int b = (unit / p.H) % p.B;
    const int seg = unit / (p.H * p.B);
    const int g = h / p.hpg;
    const int64_t t_begin = int64_t(seg) * p.seg_len;
    const int64_t t_end = t_begin + p.seg_len < p.L ? t_begin + p.seg_len : p.L;
    const int nblk = int((t_end - t_begin + 127) / 128);

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_C, 1);
        ptx::mbar_init(bar_B, 1);
        ptx::mbar_init(bar_X, 1);
        ptx::mbar_init(bar_cbi, 1);
        ptx::mbar_init(bar_L, 128);
        ptx::mbar_init(bar_is, 1);
        ptx::mbar_init(bar_dr, 128);
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_b);
        ptx::prefetch_tmap(&tm_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tL = tmem, tS = tmem + 64, tInter = tmem + 128, tIntra = tmem + 192;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            for (int k = 0; k < nblk && ok; ++k) {
                const int t0 = int(t_begin + int64_t(k) * 128);
                if (k > 0 && !ptx::mbar_wait(bar_cbi, (k - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(bar_C, 32768);
                ptx::tma_load_4d(smem + SM::kC, &tm_c, bar_C, 0, g, t0, b);
                ptx::tma_load_4d(smem + SM::kC + 16384, &tm_c, bar_C, 64, g, t0, b);
                if (k > 0 && !ptx::mbar_wait(bar_is, (k - 1) & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(bar_B, 32768);
                ptx::tma_load_4d(smem + SM::kB, &tm_b, bar_B, 0, g, t0, b);
                ptx::tma_load_4d(smem + SM::kB + 16384, &tm_b, bar_B, 64, g, t0, b);
                if (k > 0 && !ptx::mbar_wait(bar_dr, k & 1)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(bar_X, 16384);
                ptx::tma_load_4d(smem + SM::kX, &tm_x, bar_X, 0, h, t0, b);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sC = ptx::smem_u32(smem + SM::kC);
            const uint32_t sB = ptx::smem_u32(smem + SM::kB);
            const uint32_t sX = ptx::smem_u32(smem + SM::kX);
            const uint32_t sXH = ptx::smem_u32(smem + SM::kXH);
            for (int k = 0; k < nblk && ok; ++k) {
                const uint32_t par = k & 1;
                if (!ptx::mbar_wait(bar_C, par) || !ptx::mbar_wait(bar_B, par) ||
                    !ptx::mbar_wait(bar_dr, par)) { ok = false; break; }
                ptx::tc_fence_after();
                // C B^T: K = state, both operands K-major
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::mma_bf16_ss(tmem,
                                     ptx::sdesc(sC + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                     ptx::sdesc(sB + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                     kIdCB, ks != 0);
                // C h^T: K = state; h stored [n][p] (MN-major, 16 state rows per step)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::mma_bf16_ss(tInter,
                                     ptx::sdesc(sC + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                     ptx::sdesc(sXH + ks * 2048, 16384, 1024), kIdKmn, ks != 0);
                ptx::mma_commit(bar_cbi);
                if (!ptx::mbar_wait(bar_L, par)) { ok = false; break; }
                ptx::tc_fence_after();
                // L x: A = L from tensor memory (8 columns per 16 tokens), x [j][p] MN-major
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::mma_bf16_ts(tIntra, tL + ks * 8, ptx::sdesc(sX + ks * 2048, 16384, 1024),
                                     kIdKmn, ks != 0);
                // S^T = B^T (w o x): A = B^T (MN-major, the two state halves 16 KB apart)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    ptx::mma_bf16_ss(tS, ptx::sdesc(sB + ks * 2048, 16384, 1024),
                                     ptx::sdesc(sXH + ks * 2048, 16384, 1024), kIdState, ks != 0);
                ptx::mma_commit(bar_is);
            }
            // the last commit must land before tensor memory is released
            if (ok && nblk > 0 && !ptx::mbar_wait(bar_is, (nblk - 1) & 1)) ok = false;
        }
    } else {
        const int q = warp & 3;
        const int r = 32 * q + lane;               // tile row i, state row n, TMEM lane
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float Ah = p.A[h];
        const float Dh = p.D ? p.D[h] : 0.f;
        const float2 D2 = make_float2(Dh, Dh);
        uint8_t *xh = smem + SM::kXH;
        const uint8_t *xs = smem + SM::kX;
        const size_t slab = size_t(b) * p.H + h;
        // carried state row n = r, pairs of headdim values (2m, 2m + 1), fp32
        float2 hreg[32];
        const float *hin = p.h_in ? p.h_in + (size_t(seg) * p.B * p.H + slab) * 8192 : nullptr;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            hreg[m] = hin ? make_float2(hin[(2 * m) * 128 + r], hin[(2 * m + 1) * 128 + r])
                          : make_float2(0.f, 0.f);
        write_state_row(xh, r, hreg);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar_dr);

        const float *dtp = p.dt + int64_t(b) * p.dt_sb + h;
        float dt_next = (t_begin + r < t_end) ? __ldg(dtp + (t_begin + r) * p.dt_sl) : 0.f;
        for (int k = 0; k < nblk; ++k) {
            const uint32_t par = k & 1;
            const int64_t t = t_begin + int64_t(k) * 128 + r;
            const bool real = t < t_end;
            const float dtr = dt_next;
            if (k + 1 < nblk) {            // the next block's dt, one block ahead
                const int64_t tn = t + 128;
                dt_next = tn < t_end ? __ldg(dtp + tn * p.dt_sl) : 0.f;
            }
            // ---- block-local cumulative sum of A dt (log2 units) ----
            float s = Ah * dtr;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += o;
            }
            if (lane == 31) wsum[q] = s;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            float pre = 0.f;
            for (int qq = 0; qq < q; ++qq) pre += wsum[qq];
            const float tot = ((wsum[0] + wsum[1]) + wsum[2]) + wsum[3];
            const float gr = (pre + s) * kLog2e;
            const float gend = tot * kLog2e;
            ngd[r] = log2f(dtr) - gr;                  // -inf for dt = 0
            const float w = ex2(gend - gr) * dtr;
            w2[r] = pack_bf16(w, w);
            asm volatile("bar.sync 1, 128;" ::: "memory");

            // ---- L: causal-selected decay of C B^T, in place, bf16 pairs ----
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_cbi, par))) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {   // column blocks of 32
                uint32_t out[16];
                if (cb <= q) {                 // rows of warp q see columns j <= 32 q + 31
                    uint32_t v[32];
                    ptx::tmem_ld32(tmem + lane_off + 32 * cb, v);
                    ptx::tmem_ld_wait();
                    l_block(v, 32 * cb, cb == q, r, gr, ngd, out);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) out[jj] = 0u;
                }
                ptx::tmem_st16(tL + lane_off + 16 * cb, out);
            }
            ptx::tmem_st_wait();

            // ---- w o x for the state product (inter has consumed the state operand) ----
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_X, par))) { ok = false; break; }
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int chunk = r + 128 * rr;      // 16-byte chunk; row j = chunk / 8
                const uint32_t wv = w2[chunk >> 3];
                const __nv_bfloat162 wb = *reinterpret_cast<const __nv_bfloat162 *>(&wv);
                uint4 v = reinterpret_cast<const uint4 *>(xs)[chunk];
                __nv_bfloat162 *v2 = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) v2[kk] = __hmul2(v2[kk], wb);
                reinterpret_cast<uint4 *>(xh)[chunk] = v;
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_L);

            // ---- drain: y rows, then the carried state ----
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_is, par))) { ok = false; break; }
            ptx::tc_fence_after();
            {
                const float e_i = ex2(gr);
                const float2 e2 = make_float2(e_i, e_i);
                const uint8_t *xrow = xs + r * 128;
                __nv_bfloat16 *yrow = p.y + int64_t(b) * p.y_sb + t * p.y_sl + int64_t(h) * p.y_sh;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t a[16], d[16];
                    ptx::tmem_ld16(tInter + lane_off + 16 * cb, a);
                    ptx::tmem_ld16(tIntra + lane_off + 16 * cb, d);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c4 = 0; c4 < 2; ++c4) {
                        const int ch = 2 * cb + c4;
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xrow + ((ch ^ (r & 7)) << 4));
                        const uint32_t *xu = reinterpret_cast<const uint32_t *>(&xv);
                        uint32_t o[4];
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int jj = 8 * c4 + 2 * kk;
                            float2 acc = __ffma2_rn(
                                make_float2(__uint_as_float(a[jj]), __uint_as_float(a[jj + 1])), e2,
                                make_float2(__uint_as_float(d[jj]), __uint_as_float(d[jj + 1])));
                            acc = __ffma2_rn(unpack_bf16(xu[kk]), D2, acc);
                            o[kk] = pack_bf16(acc.x, acc.y);
                        }
                        if (real)
                            *reinterpret_cast<uint4 *>(yrow + 8 * ch) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            {
                const float dend = ex2(gend);
                const float2 d2 = make_float2(dend, dend);
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t sv[32];
                    ptx::tmem_ld32(tS + lane_off + 32 * cb, sv);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        hreg[16 * cb + m] =
                            __ffma2_rn(d2, hreg[16 * cb + m],
                                       make_float2(__uint_as_float(sv[2 * m]),
                                                   __uint_as_float(sv[2 * m + 1])));
                }
                write_state_row(xh, r, hreg);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_dr);
        }
        if (ok && p.h_out) {
            float *ho = p.h_out + slab * 8192;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                ho[(2 * m) * 128 + r] = hreg[m].x;
                ho[(2 * m + 1) * 128 + r] = hreg[m].y;
            }
        }
    }
    if (!ok) atomicOr(s_err, 1);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
    if (threadIdx.x == 0 && *s_err) atomicOr(p.err, 1u);
}

}  // namespace

bool fused_supported(const Dims &d, int xdt) {
    return xdt == DT_BF16 && d.P == 64 && d.N == 128 && d.Q % 128 == 0;
}

cudaError_t launch_fused(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    CUtensorMap tm_x, tm_b, tm_c;
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t xd[4] = {64, uint64_t(d.H), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t xs[3] = {uint64_t(a.x_sh) * 2, uint64_t(a.x_sl) * 2, uint64_t(a.x_sb) * 2};
    const uint64_t bd[4] = {128, uint64_t(d.G), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t bs[3] = {uint64_t(a.b_sg) * 2, uint64_t(a.b_sl) * 2, uint64_t(a.b_sb) * 2};
    const uint64_t cs[3] = {uint64_t(a.c_sg) * 2, uint64_t(a.c_sl) * 2, uint64_t(a.c_sb) * 2};
    cudaError_t e = make_tmap_bf16(&tm_x, a.x, 4, xd, xs, box);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_b, a.Bm, 4, bd, bs, box)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_c, a.Cm, 4, bd, cs, box)) != cudaSuccess) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    FusedParams p{};
    p.L = d.L;
    p.seg_len = ((d.L + 127) / 128) * 128;
    p.B = int(d.B);
    p.H = int(d.H);
    p.hpg = int(d.hpg());
    p.nseg = 1;
    p.dt = a.dt;
    p.dt_sb = a.dt_sb;
    p.dt_sl = a.dt_sl;
    p.A = a.A;
    p.D = a.D;
    p.h_in = a.h0;
    p.h_out = a.final_states;
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.y_sb = a.y_sb;
    p.y_sl = a.y_sl;
    p.y_sh = a.y_sh;
    p.err = err;
    const int smem = FusedSmem::kBytes;
    e = cudaFuncSetAttribute(k_ssd_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned units = unsigned(d.B * d.H) * unsigned(p.nseg);
    k_ssd_fused<<<units, 192, smem, s>>>(tm_x, tm_b, tm_c, p);
    return cudaGetLastError();
}

}  // namespace ssd
