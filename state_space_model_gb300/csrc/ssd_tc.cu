// Tensor-core (tcgen05 + TMA) kernels for bf16 inputs, P = 64, N = 128.
//
// chunk_state ("Kernel 2: fwd_pass_state" of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", its jump
// formula without the carried state):
//     S_c^T [n][p] = sum_j B_j[n] * (w_j x_j[p]),   w_j = 2^(G_last - G_j) dt_j
// One CTA per (chunk, pair of heads of one group, batch).  Tokens stream
// through shared memory 64 at a time (TMA, 128-byte swizzle, no multicast);
// four math warps scale the x rows by w_j in place; one thread issues
// tcgen05.mma with B^T as the M = 128 operand (so the group's B tile is
// shared by both heads) and each head's scaled x as an N = 64 operand; the
// fp32 accumulators live in tensor memory and are drained with tcgen05.ld.
#include "ptx_sm100.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#define SSD_DBG_FILE 3u   // kDbgTc
#include "ssd_debug.cuh"
#include "ssd_tmap.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

namespace ssd {
namespace {

// Set by a kernel whose bounded wait gave up (see ssd_device_status).
__device__ unsigned int g_device_error[2];

constexpr int kTile = 8192;  // one 64-row x 128-byte swizzled tile (bf16 64 x 64)

struct StateTcParams {
    int64_t L, Lp;
    int H, hpg, Q;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *G;
    float *S;
    int64_t nc;
    unsigned int *err;
    int64_t n_dt, n_G, n_S;   // element extents (debug build)
};

template <int KH, int NSTG>
struct StateTcSmem {
    static constexpr int kStageBytes = (2 + KH) * kTile;
    static constexpr int kStages = NSTG * kStageBytes;
    static constexpr int kBytes = kStages + KH * 256 * 4 + 256 + 1024;  // + weights, barriers, align
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Multiplies the 8 bf16 values of one 16-byte chunk by w (fp32), in place.
__device__ __forceinline__ void scale_chunk(uint4 *p, float w) {
    uint4 v = *p;
    uint32_t *u = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 h2 = *reinterpret_cast<__nv_bfloat162 *>(&u[k]);
        float2 f = __bfloat1622float2(h2);
        h2 = __floats2bfloat162_rn(f.x * w, f.y * w);
        u[k] = *reinterpret_cast<uint32_t *>(&h2);
    }
    *p = v;
}

template <int KH, int NSTG>
__global__ void __launch_bounds__(192, 1)
k_chunk_state_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                 const StateTcParams p) {
    using SM = StateTcSmem<KH, NSTG>;
    constexpr uint32_t kCols = KH * 64;  // fp32 accumulator columns: KH heads x P
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 64, true, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *wts = reinterpret_cast<float *>(smem + SM::kStages);            // [KH][Q]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kStages + KH * 256 * 4);
    uint64_t *full = bars, *scaled = bars + NSTG, *empty = bars + 2 * NSTG,
             *accfull = bars + 3 * NSTG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * NSTG + 1);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int h0 = blockIdx.y * KH;
    const int g = h0 / p.hpg;
    const int Q = p.Q, nkb = Q / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTG; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&scaled[s], 128);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accfull, 1);
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    if (warp >= 2) {
        // per-token weights w_j = 2^(G_last - G_j) dt_j (0 past the sequence end)
        for (int e = threadIdx.x - 64; e < KH * Q; e += 128) {
            const int i = e / Q, j = e - i * Q;
            const float *Grow = p.G + (b * p.H + h0 + i) * p.Lp + c * Q;
            const int64_t t = c * Q + j;
            const int64_t gb = (b * p.H + h0 + i) * p.Lp + c * Q;
            const int64_t dto = b * p.dt_sb + t * p.dt_sl + h0 + i;
            wts[e] = (t < p.L && SSD_IDX_OK(p.err, gb + Q - 1, p.n_G) &&
                      SSD_IDX_OK(p.err, dto, p.n_dt))
                         ? exp2f(Grow[Q - 1] - Grow[j]) * __ldg(p.dt + dto)
                         : 0.f;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % NSTG, u = kb / NSTG;
                if (u > 0 && !ptx::mbar_wait(&empty[s], (u - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * SM::kStageBytes;
                ptx::mbar_arrive_expect_tx(&full[s], SM::kStageBytes);
                const int t0 = int(c * Q + kb * 64);
                ptx::tma_load_4d(st, &tm_b, &full[s], 0, g, t0, int(b));
                ptx::tma_load_4d(st + kTile, &tm_b, &full[s], 64, g, t0, int(b));
                for (int i = 0; i < KH; ++i)
                    ptx::tma_load_4d(st + (2 + i) * kTile, &tm_x, &full[s], 0, h0 + i, t0, int(b));
            }
            // never leave the CTA with copies in flight
            for (int kb = (nkb > NSTG ? nkb - NSTG : 0); kb < nkb; ++kb)
                if (!ptx::mbar_wait(&full[kb % NSTG], (kb / NSTG) & 1, 200000000ull)) ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % NSTG, u = kb / NSTG;
                if (!ptx::mbar_wait(&scaled[s], u & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sb = ptx::smem_u32(smem + s * SM::kStageBytes);
#pragma unroll
                for (int i = 0; i < KH; ++i) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // A = B^T: M = state (two 64-wide atoms 8 KB apart), K = tokens
                        const uint64_t ad = ptx::sdesc(sb + k * 2048, kTile, 1024);
                        // B = w * x of head i: N = headdim (one atom), K = tokens
                        const uint64_t bd = ptx::sdesc(sb + (2 + i) * kTile + k * 2048, kTile, 1024);
                        ptx::mma_bf16_ss(tmem + i * 64, ad, bd, kIdesc, (kb | k) != 0);
                    }
                }
                ptx::mma_commit(&empty[s]);
            }
            ptx::mma_commit(accfull);
            if (!ptx::mbar_wait(accfull, 0)) ok = false;
        }
    } else {
        const int mt = threadIdx.x - 64;  // 0..127
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % NSTG, u = kb / NSTG;
            if (!ptx::mbar_wait(&full[s], u & 1)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * SM::kStageBytes;
#pragma unroll
            for (int i = 0; i < KH; ++i) {
                uint4 *x = reinterpret_cast<uint4 *>(st + (2 + i) * kTile);
                const float *w = wts + i * Q + kb * 64;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int chunk = mt + 128 * r;    // 16-byte chunk; 8 per 128-byte row
                    scale_chunk(x + chunk, w[chunk >> 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&scaled[s]);
        }
        const bool go = __all_sync(0xffffffffu, ok && ptx::mbar_wait(accfull, 0));
        if (go) {
            ptx::tc_fence_after();
            const int q = warp & 3;
            const int n = 32 * q + lane;
            const uint32_t row = tmem + (uint32_t(32 * q) << 16);
#pragma unroll
            for (int i = 0; i < KH; ++i) {
                const int64_t so = ((b * p.nc + c) * p.H + h0 + i) * (64 * 128);
                if (!SSD_IDX_OK(p.err, so + 64 * 128 - 1, p.n_S)) continue;
                float *S = p.S + so + n;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[16];
                    ptx::tmem_ld16(row + i * 64 + cc * 16, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) S[(cc * 16 + jj) * 128] = __uint_as_float(r[jj]);
                }
            }
        } else {
            ok = false;
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

// ---------------------------------------------------------------------------
// chunk_scan ("Kernel 3: compute_out"): one CTA per (128-row block r of chunk
// c, head h, batch b):
//     y_i = 2^G_i (C_i h_prev^T) + sum_{s<=r} sum_j L_ij x_j + D x_i,
//     L_ij = [j <= i] (C_i . B_j) 2^(G_i - G_j) dt_j
// Tensor memory holds the C B^T blocks (one 128-column fp32 block per column
// block s <= r), the carried-state product and the intra-chunk product.  The
// four math warps turn each C B^T block into the bf16 operand L (causal
// selection before the exponent) in the 128-byte-swizzled K-major layout the
// tensor cores read, then drain both products, add D x and store y.

struct ScanTcParams {
    int64_t L, Lp, nc;
    int H, hpg, Q;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *G;
    const float *D;
    __nv_bfloat16 *y;
    int64_t y_sb, y_sl, y_sh;
    unsigned int *err;
    int64_t n_dt, n_G, n_y;   // element extents (debug build)
};

template <int QB>
struct ScanTcSmem {
    static constexpr int kC = 0;                          // 2 x [128][128 B]
    static constexpr int kHP = 32768;                     // 2 x [64][128 B]
    static constexpr int kB = 49152;                      // QB x 2 x [128][128 B]
    static constexpr int kX = kB + QB * 32768;            // QB x [128][128 B]
    static constexpr int kLt = kX + QB * 16384;           // QB x 2 x [128][128 B]
    static constexpr int kF = kLt + QB * 32768;           // floats: gi[128], gj, dtj [QB*128]
    static constexpr int kBar = kF + (128 + 2 * QB * 128) * 4;
    static constexpr int kBytes = kBar + 256 + 1024;
};

template <int QB>
__global__ void __launch_bounds__(192, 1)
k_chunk_scan_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_hp,
                const ScanTcParams p) {
    using SM = ScanTcSmem<QB>;
    constexpr uint32_t kCols = QB == 1 ? 256 : 512;
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdInter = ptx::idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t kIdIntra = ptx::idesc_bf16_f32(128, 64, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *gi = reinterpret_cast<float *>(smem + SM::kF);
    float *gj = gi + 128;
    float *dtj = gj + QB * 128;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint64_t *bar_in0 = bars, *bar_in = bars + 1, *bar_cb = bars + 1 + QB,
             *bar_L = bars + 1 + 2 * QB, *bar_acc = bars + 1 + 3 * QB;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 + 3 * QB);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x / QB;
    const int r = int(blockIdx.x % QB);
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int g = h / p.hpg;
    const int Q = p.Q;
    const int nblk = r + 1;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_in0, 1);
        for (int s = 0; s < QB; ++s) {
            ptx::mbar_init(&bar_in[s], 1);
            ptx::mbar_init(&bar_cb[s], 1);
            ptx::mbar_init(&bar_L[s], 128);
        }
        ptx::mbar_init(bar_acc, 1);
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_b);
        ptx::prefetch_tmap(&tm_c);
        ptx::prefetch_tmap(&tm_hp);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    if (warp >= 2) {
        const int i = threadIdx.x - 64;
        const int64_t gb = (b * p.H + h) * p.Lp + c * Q;
        const float *Grow = p.G + gb;
        gi[i] = SSD_IDX_OK(p.err, gb + r * 128 + i, p.n_G) ? Grow[r * 128 + i] : 0.f;
        for (int s = 0; s < nblk; ++s) {
            const int64_t t = c * Q + s * 128 + i;
            const int64_t dto = b * p.dt_sb + t * p.dt_sl + h;
            gj[s * 128 + i] = SSD_IDX_OK(p.err, gb + s * 128 + i, p.n_G) ? Grow[s * 128 + i] : 0.f;
            dtj[s * 128 + i] = (t < p.L && SSD_IDX_OK(p.err, dto, p.n_dt)) ? __ldg(p.dt + dto) : 0.f;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_inter = tmem + 128 * QB, t_intra = tmem + 128 * QB + 64;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            const int t_r = int(c * Q + r * 128);
            const int hp_row = int(((b * p.nc + c) * p.H + h) * 64);
            ptx::mbar_arrive_expect_tx(bar_in0, 32768 + 16384);
            ptx::tma_load_4d(smem + SM::kC, &tm_c, bar_in0, 0, g, t_r, int(b));
            ptx::tma_load_4d(smem + SM::kC + 16384, &tm_c, bar_in0, 64, g, t_r, int(b));
            ptx::tma_load_3d(smem + SM::kHP, &tm_hp, bar_in0, 0, hp_row, 0);
            ptx::tma_load_3d(smem + SM::kHP + 8192, &tm_hp, bar_in0, 64, hp_row, 0);
            for (int s = 0; s < nblk; ++s) {
                const int t_s = int(c * Q + s * 128);
                ptx::mbar_arrive_expect_tx(&bar_in[s], 32768 + 16384);
                ptx::tma_load_4d(smem + SM::kB + s * 32768, &tm_b, &bar_in[s], 0, g, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kB + s * 32768 + 16384, &tm_b, &bar_in[s], 64, g, t_s,
                                 int(b));
                ptx::tma_load_4d(smem + SM::kX + s * 16384, &tm_x, &bar_in[s], 0, h, t_s, int(b));
            }
            if (!ptx::mbar_wait(bar_in0, 0)) ok = false;
            for (int s = 0; s < nblk; ++s)
                if (!ptx::mbar_wait(&bar_in[s], 0)) ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sC = ptx::smem_u32(smem + SM::kC);
            ok = ptx::mbar_wait(bar_in0, 0);
            for (int s = 0; s < nblk && ok; ++s) {
                if (!ptx::mbar_wait(&bar_in[s], 0)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sB = ptx::smem_u32(smem + SM::kB + s * 32768);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_bf16_ss(tmem + 128 * s,
                                         ptx::sdesc(sC + kb * 16384 + k * 32, 16, 1024),
                                         ptx::sdesc(sB + kb * 16384 + k * 32, 16, 1024), kIdCB,
                                         (kb | k) != 0);
                ptx::mma_commit(&bar_cb[s]);
            }
            if (ok) {
                const uint32_t sH = ptx::smem_u32(smem + SM::kHP);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_bf16_ss(t_inter, ptx::sdesc(sC + kb * 16384 + k * 32, 16, 1024),
                                         ptx::sdesc(sH + kb * 8192 + k * 32, 16, 1024), kIdInter,
                                         (kb | k) != 0);
            }
            for (int s = 0; s < nblk && ok; ++s) {
                if (!ptx::mbar_wait(&bar_L[s], 0)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sL = ptx::smem_u32(smem + SM::kLt + s * 32768);
                const uint32_t sX = ptx::smem_u32(smem + SM::kX + s * 16384);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_bf16_ss(t_intra, ptx::sdesc(sL + kb * 16384 + k * 32, 16, 1024),
                                         ptx::sdesc(sX + (kb * 4 + k) * 2048, 16384, 1024),
                                         kIdIntra, (s | kb | k) != 0);
            }
            ptx::mma_commit(bar_acc);
            if (!ptx::mbar_wait(bar_acc, 0)) ok = false;
        }
    } else {
        // tile row owned by this thread = the TMEM lane it may access: warp w
        // reaches lanes 32 (w % 4) .. 32 (w % 4) + 31
        const int i = 32 * (warp & 3) + lane;
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const float g_i = gi[i];
        // the 128 math threads share gj / dtj: make them visible to each other
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int s = 0; s < nblk; ++s) {
            const bool go = __all_sync(0xffffffffu, ptx::mbar_wait(&bar_cb[s], 0));
            if (!go) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint8_t *Lrow = smem + SM::kLt + s * 32768 + i * 128;
            const bool diag = (s == r);
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + 128 * s + 32 * cb, v);
                ptx::tmem_ld_wait();
                uint32_t packed[16];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const int j = 32 * cb + jj;
                    float e0 = 0.f, e1 = 0.f;
                    if (!diag || j <= i)
                        e0 = __uint_as_float(v[jj]) * exp2f(g_i - gj[s * 128 + j]) *
                             dtj[s * 128 + j];
                    if (!diag || j + 1 <= i)
                        e1 = __uint_as_float(v[jj + 1]) * exp2f(g_i - gj[s * 128 + j + 1]) *
                             dtj[s * 128 + j + 1];
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
                    packed[jj >> 1] = *reinterpret_cast<uint32_t *>(&h2);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = 4 * cb + q;           // 16-byte chunk 0..15 of the row
                    const int kb = ch >> 3, c8 = ch & 7;
                    uint4 w4 = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                          packed[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(Lrow + kb * 16384 + ((c8 ^ (i & 7)) << 4)) = w4;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bar_L[s]);
        }
        const bool go = __all_sync(0xffffffffu, ok && ptx::mbar_wait(bar_acc, 0));
        if (go) {
            ptx::tc_fence_after();
            const int64_t t = c * Q + r * 128 + i;
            const float e_i = exp2f(g_i);
            const float Dh = p.D && SSD_IDX_OK(p.err, h, p.H) ? p.D[h] : 0.f;
            const uint8_t *Xrow = smem + SM::kX + r * 16384 + i * 128;
            __nv_bfloat16 *yrow = p.y + b * p.y_sb + t * p.y_sl + int64_t(h) * p.y_sh;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t a[32], d[32];
                ptx::tmem_ld32(t_inter + lane_off + 32 * cb, a);
                ptx::tmem_ld32(t_intra + lane_off + 32 * cb, d);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = 4 * cb + q;   // 8 headdim values per 16-byte chunk
                    const uint4 xv = *reinterpret_cast<const uint4 *>(Xrow + ((ch ^ (i & 7)) << 4));
                    const uint32_t *xu = reinterpret_cast<const uint32_t *>(&xv);
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 xf =
                            __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xu[k]));
                        const int jj = 8 * q + 2 * k;
                        const float y0 = fmaf(e_i, __uint_as_float(a[jj]), __uint_as_float(d[jj])) +
                                         Dh * xf.x;
                        const float y1 =
                            fmaf(e_i, __uint_as_float(a[jj + 1]), __uint_as_float(d[jj + 1])) +
                            Dh * xf.y;
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(y0, y1);
                        o[k] = *reinterpret_cast<uint32_t *>(&h2);
                    }
                    if (t < p.L &&
                        SSD_IDX_OK(p.err, b * p.y_sb + t * p.y_sl + int64_t(h) * p.y_sh + 8 * ch + 7,
                                   p.n_y))
                        *reinterpret_cast<uint4 *>(yrow + 8 * ch) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        } else {
            ok = false;
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

// ---------------------------------------------------------------------------
// host side

std::mutex g_mu;
unsigned int *g_err_addr[256] = {};

cudaError_t make_tmap_bf16_4d(CUtensorMap *m, const void *base, const uint64_t dims[4],
                              const uint64_t strides[3], const uint32_t box[4]) {
    return make_tmap_bf16(m, base, 4, dims, strides, box);
}

cudaError_t make_tmap_bf16_3d(CUtensorMap *m, const void *base, const uint64_t dims[3],
                              const uint64_t strides[2], const uint32_t box[3]) {
    return make_tmap_bf16(m, base, 3, dims, strides, box);
}

template <int QB>
cudaError_t launch_scan_tc(const Args &a, cudaStream_t s, const CUtensorMap &tx,
                           const CUtensorMap &tb, const CUtensorMap &tc, const CUtensorMap &thp,
                           const ScanTcParams &p) {
    auto k = k_chunk_scan_tc<QB>;
    const int smem = ScanTcSmem<QB>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const Dims &d = a.d;
    k<<<dim3(unsigned(d.nc * QB), unsigned(d.H), unsigned(d.B)), 192, smem, s>>>(tx, tb, tc, thp,
                                                                                 p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t device_error_word(unsigned int **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_device_error);
        if (e != cudaSuccess) return e;
        g_err_addr[dev] = static_cast<unsigned int *>(ptr);
    }
    *out = g_err_addr[dev];
    return cudaSuccess;
}

bool tc_chunk_state_supported(const Args &a) {
    if (a.xdt == DT_F32) return a.f32_split && tc_f32_supported(a.d, a.xdt);
    return a.xdt == DT_BF16 && a.d.P == 64 && a.d.N == 128 && a.d.Q % 64 == 0 && a.d.Q <= 256;
}

cudaError_t tc_chunk_state(const Args &a, cudaStream_t s) {
    if (a.xdt == DT_F32) return tc_chunk_state_f32(a, s);
    const Dims &d = a.d;
    CUtensorMap tm_x, tm_b;
    const uint64_t xd[4] = {64, uint64_t(d.H), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t xs[3] = {uint64_t(a.x_sh) * 2, uint64_t(a.x_sl) * 2, uint64_t(a.x_sb) * 2};
    const uint64_t bd[4] = {128, uint64_t(d.G), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t bs[3] = {uint64_t(a.b_sg) * 2, uint64_t(a.b_sl) * 2, uint64_t(a.b_sb) * 2};
    const uint32_t box[4] = {64, 1, 64, 1};
    cudaError_t e = make_tmap_bf16_4d(&tm_x, a.x, xd, xs, box);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_bf16_4d(&tm_b, a.Bm, bd, bs, box)) != cudaSuccess) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    Args ax = a;
    fill_extents(ax);
    StateTcParams p{d.L, d.Lp(), int(d.H), int(d.hpg()), int(d.Q), a.dt, a.dt_sb, a.dt_sl,
                    a.G, a.S, d.nc, err, ax.n_dt, d.B * d.H * d.Lp(),
                    d.B * d.nc * d.H * 64 * 128};
    if (d.hpg() % 2 == 0) {
        auto k = k_chunk_state_tc<2, 2>;
        const int smem = StateTcSmem<2, 2>::kBytes;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)))
            return e;
        k<<<dim3(unsigned(d.nc), unsigned(d.H / 2), unsigned(d.B)), 192, smem, s>>>(tm_x, tm_b, p);
    } else {
        auto k = k_chunk_state_tc<1, 2>;
        const int smem = StateTcSmem<1, 2>::kBytes;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)))
            return e;
        k<<<dim3(unsigned(d.nc), unsigned(d.H), unsigned(d.B)), 192, smem, s>>>(tm_x, tm_b, p);
    }
    return cudaGetLastError();
}

bool tc_chunk_scan_supported(const Args &a) {
    if (a.xdt == DT_F32)
        return a.f32_split && a.hprev_dt == DT_F32 && tc_f32_supported(a.d, a.xdt);
    return a.xdt == DT_BF16 && a.hprev_dt == DT_BF16 && a.d.P == 64 && a.d.N == 128 &&
           (a.d.Q == 128 || a.d.Q == 256);
}

cudaError_t tc_chunk_scan(const Args &a, cudaStream_t s) {
    if (a.xdt == DT_F32) return tc_chunk_scan_f32(a, s);
    const Dims &d = a.d;
    CUtensorMap tm_x, tm_b, tm_c, tm_hp;
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t xd[4] = {64, uint64_t(d.H), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t xs[3] = {uint64_t(a.x_sh) * 2, uint64_t(a.x_sl) * 2, uint64_t(a.x_sb) * 2};
    const uint64_t bd[4] = {128, uint64_t(d.G), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t bs[3] = {uint64_t(a.b_sg) * 2, uint64_t(a.b_sl) * 2, uint64_t(a.b_sb) * 2};
    const uint64_t cs[3] = {uint64_t(a.c_sg) * 2, uint64_t(a.c_sl) * 2, uint64_t(a.c_sb) * 2};
    cudaError_t e = make_tmap_bf16_4d(&tm_x, a.x, xd, xs, box);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_bf16_4d(&tm_b, a.Bm, bd, bs, box)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_4d(&tm_c, a.Cm, bd, cs, box)) != cudaSuccess) return e;
    // h_prev [B, nc, H, P, N] viewed as rows of N: {N, B*nc*H*P, 1}
    const uint64_t hd[3] = {128, uint64_t(d.B * d.nc * d.H * 64), 1};
    const uint64_t hs[2] = {128 * 2, uint64_t(d.B * d.nc * d.H * 64) * 256};
    const uint32_t hbox[3] = {64, 64, 1};
    if ((e = make_tmap_bf16_3d(&tm_hp, a.h_prev, hd, hs, hbox)) != cudaSuccess) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    ScanTcParams p{d.L,
                   d.Lp(),
                   d.nc,
                   int(d.H),
                   int(d.hpg()),
                   int(d.Q),
                   a.dt,
                   a.dt_sb,
                   a.dt_sl,
                   a.G,
                   a.D,
                   static_cast<__nv_bfloat16 *>(a.y),
                   a.y_sb,
                   a.y_sl,
                   a.y_sh,
                   err,
                   0,
                   d.B * d.H * d.Lp(),
                   0};
    {
        Args ax = a;
        fill_extents(ax);
        p.n_dt = ax.n_dt;
        p.n_y = ax.n_y;
    }
    return d.Q == 256 ? launch_scan_tc<2>(a, s, tm_x, tm_b, tm_c, tm_hp, p)
                      : launch_scan_tc<1>(a, s, tm_x, tm_b, tm_c, tm_hp, p);
}

}  // namespace ssd
